"""Python binding of libggufdq (the GB300 GGUF block-dequant GEMV / MoE library).

Argument marshalling only: every function here passes device pointers, sizes and the CUDA
stream of PyTorch tensors to the C ABI declared in ``include/ggufdq.h`` and raises
``QGError`` on a non-zero status.  All arithmetic runs in the library's CUDA kernels; there
is no other code path.  If the shared library has not been built, importing works but the
first call raises, naming the build step (``gguf_block_dequant_gb300.build.build()``).
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

Q4_0, Q8_0, Q4_K, Q6_K = 2, 8, 12, 14
BLOCK = {Q8_0: (32, 34), Q4_0: (32, 18), Q4_K: (256, 144), Q6_K: (256, 210)}

QG_OK, QG_EINVAL_SHAPE, QG_EINVAL_PTR, QG_EALIGN, QG_EUNSUPPORTED, QG_ECUDA, QG_EDEVICE_ID, QG_ETIMEOUT, \
    QG_EWORKSPACE = range(9)

_lock = threading.Lock()
_lib = None


class QGError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {strerror(status)} (status {status})")


def lib_path() -> str:
    return _build.LIB


def load():
    """Load libggufdq.so (no fallback: raises if it is missing)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_build.LIB):
            raise RuntimeError(f"{_build.LIB} is not built; run gguf_block_dequant_gb300.build.build()")
        L = ctypes.CDLL(_build.LIB)
        P, I, I64, SZ, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p
        sig = {
            "qg_version": ([], I),
            "qg_strerror": ([I], ctypes.c_char_p),
            "qg_block_shape": ([I, P, P], I),
            "qg_device_status": ([P, I], I),
            "qg_set_static_weights": ([S, I], I),
            "qgemv_q8_0": ([P, P, P, I64, I64, S], I),
            "qgemv_q4_0": ([P, P, P, I64, I64, S], I),
            "qgemv_q4_k": ([P, P, P, I64, I64, S], I),
            "qgemv_q6_k": ([P, P, P, I64, I64, S], I),
            "qgemv_t": ([I, P, P, P, I64, I64, I, S], I),
            "qgemv_multi": ([I, I, P, P, P, I64, P, I, S], I),
            "qgemm_workspace_size": ([I, I64, I64, I64], SZ),
            "qgemm": ([I, P, P, P, I64, I64, I64, P, SZ, S], I),
            "moe_workspace_size": ([I, I, I, I, I], SZ),
            "moe_route_topk": ([P, P, I, I, I, I, P, P, P, P, SZ, S], I),
            "moe_route_topk_noalloc": ([P, P, I, I, I, I, P, P, P, S], I),
            "moe_expert_swiglu": ([I, P, P, I64, P, I, I, P, P, I, I, I, I, P, P, SZ, S], I),
            "moe_combine": ([I, P, I64, P, I, I, P, P, P, I, I, I, I, P, I, P, SZ, S], I),
            "moe_layer": ([I, P, P, P, P, P, I64, P, I, I, I, I, I, I, P, P, P, P, P, SZ, S], I),
            "qg_embed_rows": ([I, P, I64, I64, P, I, ctypes.c_float, P, S], I),
            "qg_rmsnorm": ([P, P, I, I64, ctypes.c_float, ctypes.c_float, P, S], I),
            "moe_expert_act": ([I, P, P, I64, P, I, I, P, P, I, I, I, I, P, P, P, SZ, S], I),
            "moe_combine_ex": ([I, P, I64, P, I, I, P, P, P, I, I, I, I, P, P, I, P, SZ, S], I),
            "moe_layer_ex": ([I, P, P, P, P, P, I64, P, I, I, I, I, I, I, P, P, P, P, P, P, SZ, S], I),
            "qg_argmax_rows": ([P, I, I64, P, S], I),
            "qg_head_argmax": ([I, P, I64, I64, P, I, P, P, S], I),
        }
        for name, (args, res) in sig.items():
            if hasattr(L, name):
                f = getattr(L, name)
                f.argtypes = args
                f.restype = res
        _lib = L
        return L


def strerror(status: int) -> str:
    try:
        return load().qg_strerror(int(status)).decode()
    except Exception:  # noqa: BLE001 - message only
        return f"status {status}"


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch

        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _call(name, *args):
    rc = getattr(load(), name)(*args)
    if rc != QG_OK:
        raise QGError(rc, name)


def version() -> int:
    return load().qg_version()


def device_status(clear: bool = True) -> int:
    v = ctypes.c_uint32(0)
    _call("qg_device_status", ctypes.byref(v), int(clear))
    return v.value


def set_static_weights(enable: bool, stream=None) -> bool:
    """Declare the weight buffers read on `stream` (default: the current stream) immutable:
    GEMVs enqueued there may start streaming them before the preceding kernel finishes.
    Returns the stream's previous setting."""
    prev = load().qg_set_static_weights(_stream(stream), int(bool(enable)))
    if prev < 0:
        raise QGError(QG_ECUDA, "qg_set_static_weights")
    return bool(prev)


def row_bytes(qtype: int, n: int) -> int:
    qk, bb = BLOCK[qtype]
    return (n // qk) * bb


# ---- GEMV / GEMM ---------------------------------------------------------------------------

_GEMV1 = {Q8_0: "qgemv_q8_0", Q4_0: "qgemv_q4_0", Q4_K: "qgemv_q4_k", Q6_K: "qgemv_q6_k"}


def qgemv(qtype, w, x, M, N, y, stream=None):
    """y[m] = W[m] . x for one token (qgemv_q8_0 / _q4_0 / _q4_k / _q6_k)."""
    _call(_GEMV1[qtype], _ptr(w), _ptr(x), _ptr(y), M, N, _stream(stream))
    return y


def qgemv_q8_0(w, x, y, M, N, stream=None):
    return qgemv(Q8_0, w, x, M, N, y, stream)


def qgemv_q4_0(w, x, y, M, N, stream=None):
    return qgemv(Q4_0, w, x, M, N, y, stream)


def qgemv_q4_k(w, x, y, M, N, stream=None):
    return qgemv(Q4_K, w, x, M, N, y, stream)


def qgemv_q6_k(w, x, y, M, N, stream=None):
    return qgemv(Q6_K, w, x, M, N, y, stream)


def qgemv_t(qtype, w, x, y, M, N, T, stream=None):
    """Y[t][m] = W[m] . X[t] for T <= 16 token rows, one weight pass."""
    _call("qgemv_t", qtype, _ptr(w), _ptr(x), _ptr(y), M, N, T, _stream(stream))
    return y


def qgemv_multi(qtype, ws, ys, x, N, T, stream=None):
    """Y_j = W_j . X for up to 4 matrices sharing the activations X [T][N], one launch.
    ws: weight tensors (raw blocks), ys: f32 [T][M_j] outputs; M_j from ys."""
    n = len(ws)
    if n != len(ys):
        raise ValueError("one output per weight tensor")
    W = (ctypes.c_void_p * n)(*[w.data_ptr() for w in ws])
    Y = (ctypes.c_void_p * n)(*[y.data_ptr() for y in ys])
    M = (ctypes.c_int64 * n)(*[int(y.shape[-1]) for y in ys])
    _call("qgemv_multi", qtype, n, W, Y, M, N, _ptr(x), T, _stream(stream))
    return ys


def embed_rows(qtype, table, V, N, ids, out, scale=1.0, stream=None):
    """out[i] = scale * dequantized row ids[i] of the [V][N] table (raw blocks)."""
    _call("qg_embed_rows", qtype, _ptr(table), V, N, _ptr(ids), int(ids.numel()), float(scale), _ptr(out),
          _stream(stream))
    return out


def rmsnorm(x, w, eps, y, k=1.0, stream=None):
    """y[t] = ((x[t] / sqrt(mean(x[t]^2) + eps)) * k) * w for x [T][N] (k = 1: plain RMSNorm)."""
    T, N = (1, x.shape[-1]) if x.dim() == 1 else (x.shape[0], x.shape[1])
    _call("qg_rmsnorm", _ptr(x), _ptr(w), T, N, float(eps), float(k), _ptr(y), _stream(stream))
    return y


def argmax_rows(logits, ids, stream=None):
    """ids[t] = lowest index of the largest value of logits[t] (NaN never picked)."""
    T, n = (1, logits.shape[-1]) if logits.dim() == 1 else (logits.shape[0], logits.shape[1])
    _call("qg_argmax_rows", _ptr(logits), T, n, _ptr(ids), _stream(stream))
    return ids


def head_argmax(qtype, w, x, M, N, T, logits, ids, stream=None):
    """Tied-head GEMV over T <= 16 tokens into logits [T][M], then ids[t] = argmax logits[t]."""
    _call("qg_head_argmax", qtype, _ptr(w), M, N, _ptr(x), T, _ptr(logits), _ptr(ids), _stream(stream))
    return ids


def qgemm_workspace_size(qtype, M, N, T) -> int:
    return int(load().qgemm_workspace_size(qtype, M, N, T))


def qgemm(qtype, w, x, y, M, N, T, workspace=None, stream=None):
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _call("qgemm", qtype, _ptr(w), _ptr(x), _ptr(y), M, N, T, _ptr(workspace), ws_bytes, _stream(stream))
    return y


# ---- MoE -------------------------------------------------------------------------------------

def moe_workspace_size(T, k, E, H, F) -> int:
    return int(load().moe_workspace_size(T, k, E, H, F))


def _nbytes(t):
    return 0 if t is None else t.numel() * t.element_size()


def moe_route_topk(xn, wr, T, H, E, k, ids, weights, logits=None, workspace=None, stream=None):
    _call("moe_route_topk", _ptr(xn), _ptr(wr), T, H, E, k, _ptr(ids), _ptr(weights), _ptr(logits),
          _ptr(workspace), _nbytes(workspace), _stream(stream))
    return ids, weights


def moe_route_topk_noalloc(xn, wr, T, H, E, k, ids, weights, logits=None, stream=None):
    """moe_route_topk without a workspace argument (library-held scratch, T * E <= 16384)."""
    _call("moe_route_topk_noalloc", _ptr(xn), _ptr(wr), T, H, E, k, _ptr(ids), _ptr(weights), _ptr(logits),
          _stream(stream))
    return ids, weights


def moe_expert_swiglu(qtype, w_gate, w_up, expert_stride, slots, n_slots, E, ids, xn, T, k, H, F, act,
                      workspace=None, stream=None):
    _call("moe_expert_swiglu", qtype, _ptr(w_gate), _ptr(w_up), expert_stride, _ptr(slots), n_slots, E, _ptr(ids),
          _ptr(xn), T, k, H, F, _ptr(act), _ptr(workspace), _nbytes(workspace), _stream(stream))
    return act


def moe_combine(qtype, w_down, expert_stride, slots, n_slots, E, ids, weights, act, T, k, H, F, x_inout,
                add_residual=1, workspace=None, stream=None):
    _call("moe_combine", qtype, _ptr(w_down), expert_stride, _ptr(slots), n_slots, E, _ptr(ids), _ptr(weights),
          _ptr(act), T, k, H, F, _ptr(x_inout), int(add_residual), _ptr(workspace), _nbytes(workspace),
          _stream(stream))
    return x_inout


ACT_SILU, ACT_GELU_TANH = 0, 1


class MoeVariant(ctypes.Structure):
    """qg_moe_variant: expert activation, per-expert down scale, sigmoid-gated shared expert."""
    _fields_ = [("act", ctypes.c_int), ("down_scale", ctypes.c_void_p), ("shared_out", ctypes.c_void_p),
                ("shared_gate", ctypes.c_void_p)]


def moe_variant(act=ACT_SILU, down_scale=None, shared_out=None, shared_gate=None):
    """A qg_moe_variant from tensors (None for the fields not used).  The struct keeps the
    tensors alive: it holds their addresses, and the kernels read them when they run."""
    dp = lambda t: None if t is None else t.data_ptr()  # noqa: E731
    v = MoeVariant(int(act), dp(down_scale), dp(shared_out), dp(shared_gate))
    v.tensors = (down_scale, shared_out, shared_gate)
    return v


def _var(v):
    return None if v is None else ctypes.byref(v)


def moe_expert_act(qtype, w_gate, w_up, expert_stride, slots, n_slots, E, ids, xn, T, k, H, F, variant, act,
                   workspace=None, stream=None):
    _call("moe_expert_act", qtype, _ptr(w_gate), _ptr(w_up), expert_stride, _ptr(slots), n_slots, E, _ptr(ids),
          _ptr(xn), T, k, H, F, _var(variant), _ptr(act), _ptr(workspace), _nbytes(workspace), _stream(stream))
    return act


def moe_combine_ex(qtype, w_down, expert_stride, slots, n_slots, E, ids, weights, act, T, k, H, F, variant, x_inout,
                   add_residual=1, workspace=None, stream=None):
    _call("moe_combine_ex", qtype, _ptr(w_down), expert_stride, _ptr(slots), n_slots, E, _ptr(ids), _ptr(weights),
          _ptr(act), T, k, H, F, _var(variant), _ptr(x_inout), int(add_residual), _ptr(workspace),
          _nbytes(workspace), _stream(stream))
    return x_inout


def moe_layer_ex(qtype, xn, wr, w_gate, w_up, w_down, expert_stride, slots, n_slots, T, H, F, E, k, variant, ids,
                 weights, act, x_inout, workspace=None, stream=None):
    _call("moe_layer_ex", qtype, _ptr(xn), _ptr(wr), _ptr(w_gate), _ptr(w_up), _ptr(w_down), expert_stride,
          _ptr(slots), n_slots, T, H, F, E, k, _var(variant), _ptr(ids), _ptr(weights), _ptr(act), _ptr(x_inout),
          _ptr(workspace), _nbytes(workspace), _stream(stream))
    return x_inout


def moe_layer(qtype, xn, wr, w_gate, w_up, w_down, expert_stride, slots, n_slots, T, H, F, E, k, ids, weights, act,
              x_inout, workspace=None, stream=None):
    _call("moe_layer", qtype, _ptr(xn), _ptr(wr), _ptr(w_gate), _ptr(w_up), _ptr(w_down), expert_stride,
          _ptr(slots), n_slots, T, H, F, E, k, _ptr(ids), _ptr(weights), _ptr(act), _ptr(x_inout),
          _ptr(workspace), _nbytes(workspace), _stream(stream))
    return x_inout
