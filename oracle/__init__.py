"""CPU oracle for the GGUF block-dequant GEMV / MoE path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg (and its
``--impl reference`` arm) may import this package.  The product library never does, and it
has no fallback to it.  The arithmetic lives in ``oracle.c`` (plain C11, float64
accumulation); this module compiles it with gcc and wraps it with ctypes and numpy.

Every function cites the engine page it follows in ``oracle.c``.  Pins that tie the oracle
to the pages and to the mathematics, rather than to itself, are in ``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None

Q4_0, Q8_0, Q4_K, Q6_K = 2, 8, 12, 14
BLOCK = {Q8_0: (32, 34), Q4_0: (32, 18), Q4_K: (256, 144), Q6_K: (256, 210)}


def build(force: bool = False) -> str:
    """Compile oracle.c into _build/liboracle.so (OpenMP when gcc has it)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    base = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", _SRC,
            "-o", _LIB_PATH + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I64 = ctypes.c_int64
            I = ctypes.c_int
            L.og_f16_value.argtypes = [ctypes.c_uint16]
            L.og_f16_value.restype = ctypes.c_double
            L.og_block_value.argtypes = [I, P, I]
            L.og_block_value.restype = ctypes.c_float
            L.og_dequant.argtypes = [I, P, I64, I64, P]
            L.og_gemv.argtypes = [I, P, I64, I64, P, I64, P, P, I]
            L.og_router_logits.argtypes = [P, P, I64, I64, I64, P, P]
            L.og_topk.argtypes = [P, I64, I64, I, P, P]
            L.og_swiglu1.argtypes = [ctypes.c_double, ctypes.c_double]
            L.og_swiglu1.restype = ctypes.c_double
            L.og_moe_gate_up.argtypes = [I, P, P, I64, P, P, P, I64, I, I64, I64, P, P, P, P, P, I]
            L.og_moe_down_combine.argtypes = [I, P, I64, P, P, P, P, P, I64, I, I64, I64, I, P, P, P, P, I]
            L.og_max_threads.restype = I
            L.og_embed_rows.argtypes = [I, P, I64, I64, P, I64, ctypes.c_float, P]
            L.og_rmsnorm.argtypes = [P, P, I64, I64, ctypes.c_double, P]
            L.og_argmax_rows.argtypes = [P, I64, I64, P]
            L.og_gelu_tanh.argtypes = [ctypes.c_double]
            L.og_gelu_tanh.restype = ctypes.c_double
            L.og_sigmoid.argtypes = [ctypes.c_double]
            L.og_sigmoid.restype = ctypes.c_double
            L.og_moe_act.argtypes = [I, P, P, I64, P]
            L.og_moe_combine_ex.argtypes = [P, P, P, P, P, I64, P, P, P, I64, I, I64, I, P, P]
            L.og_rmsnorm_k.argtypes = [P, P, I64, I64, ctypes.c_double, ctypes.c_double, P]
            _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _u8(w):
    w = np.ascontiguousarray(w)
    return w.view(np.uint8).reshape(-1)


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} failed with code {rc}")


def max_threads() -> int:
    return lib().og_max_threads()


def f16_value(h: int) -> float:
    return lib().og_f16_value(int(h) & 0xFFFF)


def block_value(qtype: int, block: np.ndarray, i: int) -> np.float32:
    b = _u8(block)
    return np.float32(lib().og_block_value(qtype, _p(b), int(i)))


def dequant(qtype: int, w: np.ndarray, rows: int, n: int) -> np.ndarray:
    b = _u8(w)
    out = np.empty((rows, n), dtype=np.float32)
    _check(lib().og_dequant(qtype, _p(b), rows, n, _p(out)), "dequant")
    return out


def gemv(qtype: int, w: np.ndarray, M: int, N: int, x: np.ndarray, threads: int = 1):
    """y[t][m] = sum_k w[m][k] x[t][k] in float64; returns (y, bound), both [T][M]."""
    b = _u8(w)
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1, N)
    T = x.shape[0]
    y = np.empty((T, M), dtype=np.float64)
    bnd = np.empty((T, M), dtype=np.float64)
    _check(lib().og_gemv(qtype, _p(b), M, N, _p(x), T, _p(y), _p(bnd), threads), "gemv")
    return y, bnd


def router_logits(xn: np.ndarray, wr: np.ndarray):
    xn = np.ascontiguousarray(xn, dtype=np.float32)
    wr = np.ascontiguousarray(wr, dtype=np.float32)
    T, H = xn.shape
    E = wr.shape[0]
    lg = np.empty((T, E), dtype=np.float64)
    bnd = np.empty((T, E), dtype=np.float64)
    _check(lib().og_router_logits(_p(xn), _p(wr), T, H, E, _p(lg), _p(bnd)), "router_logits")
    return lg, bnd


def topk(logits: np.ndarray, k: int):
    lg = np.ascontiguousarray(logits, dtype=np.float64)
    T, E = lg.shape
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    _check(lib().og_topk(_p(lg), T, E, k, _p(ids), _p(w)), "topk")
    return ids, w


def swiglu1(g: float, u: float) -> float:
    return lib().og_swiglu1(float(g), float(u))


def moe_gate_up(qtype, w_gate, w_up, expert_stride, slots, ids, xn, k, H, F, threads=1):
    """Returns (gate, up, act, bound_gate, bound_up), each float64 [T*k][F]."""
    wg = _u8(w_gate)
    wu = _u8(w_up)
    xn = np.ascontiguousarray(xn, dtype=np.float32).reshape(-1, H)
    T = xn.shape[0]
    ids = np.ascontiguousarray(ids, dtype=np.int32).reshape(-1)
    sl = None if slots is None else np.ascontiguousarray(slots, dtype=np.int32)
    outs = [np.empty((T * k, F), dtype=np.float64) for _ in range(5)]
    rc = lib().og_moe_gate_up(qtype, _p(wg), _p(wu), expert_stride, _p(sl), _p(ids), _p(xn), T, k, H, F,
                              *[_p(o) for o in outs], threads)
    _check(rc, "moe_gate_up")
    return tuple(outs)


def moe_down_combine(qtype, w_down, expert_stride, slots, ids, wts, act, x_in, k, H, F, add_residual=1,
                     threads=1):
    """Returns (dn, bound_dn, out, bound_out): dn [T*k][H], out [T][H], all float64."""
    wd = _u8(w_down)
    ids = np.ascontiguousarray(ids, dtype=np.int32).reshape(-1)
    T = ids.size // k
    wts = np.ascontiguousarray(wts, dtype=np.float64).reshape(-1)
    act = np.ascontiguousarray(act, dtype=np.float64).reshape(-1)
    x_in = np.ascontiguousarray(x_in, dtype=np.float32).reshape(-1)
    sl = None if slots is None else np.ascontiguousarray(slots, dtype=np.int32)
    dn = np.empty((T * k, H), dtype=np.float64)
    bdn = np.empty((T * k, H), dtype=np.float64)
    out = np.empty((T, H), dtype=np.float64)
    bout = np.empty((T, H), dtype=np.float64)
    rc = lib().og_moe_down_combine(qtype, _p(wd), expert_stride, _p(sl), _p(ids), _p(wts), _p(act), _p(x_in),
                                   T, k, H, F, int(add_residual), _p(dn), _p(bdn), _p(out), _p(bout), threads)
    _check(rc, "moe_down_combine")
    return dn, bdn, out, bout


def moe_layer(qtype, experts, gate_off, up_off, down_off, expert_stride, wr, xn, x_in, k, H, F, slots=None,
              threads=1):
    """The whole MoE step in float64: router logits, top-k, gate/up + SwiGLU, down, combine.

    ``experts`` is the flat byte array of all expert records; the gate / up / down bases are
    ``experts + *_off``.  Returns a dict of every intermediate."""
    ex = _u8(experts)
    lg, blg = router_logits(xn, wr)
    ids, wts = topk(lg, k)
    g, u, act, bg, bu = moe_gate_up(qtype, ex[gate_off:], ex[up_off:], expert_stride, slots, ids, xn, k, H, F,
                                    threads)
    dn, bdn, out, bout = moe_down_combine(qtype, ex[down_off:], expert_stride, slots, ids, wts, act, x_in, k, H, F,
                                          1, threads)
    return dict(logits=lg, bound_logits=blg, ids=ids, weights=wts, gate=g, up=u, act=act, bound_gate=bg,
                bound_up=bu, dn=dn, bound_dn=bdn, out=out, bound_out=bout)


def embed_rows(qtype: int, table: np.ndarray, V: int, N: int, ids, scale: float = 1.0) -> np.ndarray:
    """out[i][k] = dequantized table[ids[i]][k] * scale (f64 product rounded once to f32)."""
    b = _u8(table)
    ids = np.ascontiguousarray(ids, dtype=np.int32).reshape(-1)
    out = np.empty((ids.size, N), dtype=np.float32)
    _check(lib().og_embed_rows(qtype, _p(b), V, N, _p(ids), ids.size, float(np.float32(scale)), _p(out)), "embed_rows")
    return out


def rmsnorm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """y[t][k] = x[t][k] * w[k] / sqrt(mean_k x[t][k]^2 + eps), float64 [T][N]."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    x2 = x.reshape(-1, x.shape[-1])
    w = np.ascontiguousarray(w, dtype=np.float32).reshape(-1)
    T, N = x2.shape
    y = np.empty((T, N), dtype=np.float64)
    _check(lib().og_rmsnorm(_p(x2), _p(w), T, N, float(eps), _p(y)), "rmsnorm")
    return y


def argmax_rows(v: np.ndarray) -> np.ndarray:
    """Lowest index of each row's largest value (NaN never picked; an all-NaN row gives 0)."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    v2 = v.reshape(-1, v.shape[-1])
    ids = np.empty(v2.shape[0], dtype=np.int32)
    _check(lib().og_argmax_rows(_p(v2), v2.shape[0], v2.shape[1], _p(ids)), "argmax_rows")
    return ids


ACT_SILU, ACT_GELU_TANH = 0, 1


def gelu_tanh(x: float) -> float:
    return lib().og_gelu_tanh(float(x))


def sigmoid(x: float) -> float:
    return lib().og_sigmoid(float(x))


def moe_act(kind: int, gate: np.ndarray, up: np.ndarray) -> np.ndarray:
    """act = SiLU(gate) * up (kind 0) or GELU-tanh(gate) * up (kind 1), float64."""
    g = np.ascontiguousarray(gate, dtype=np.float64)
    u = np.ascontiguousarray(up, dtype=np.float64)
    out = np.empty_like(g)
    _check(lib().og_moe_act(int(kind), _p(g), _p(u), g.size, _p(out)), "moe_act")
    return out


def moe_combine_ex(ids, wts, dn, bound_dn, x_in, k, H, add_residual=1, down_scale=None, E=0, shared_out=None,
                   shared_gate=None):
    """out, bound_out [T][H] (float64) of the combine with a per-expert down scale and a
    sigmoid-gated shared expert, from down rows dn [T*k][H]."""
    ids = np.ascontiguousarray(ids, dtype=np.int32).reshape(-1)
    T = ids.size // k
    wts = np.ascontiguousarray(wts, dtype=np.float64).reshape(-1)
    dn = np.ascontiguousarray(dn, dtype=np.float64).reshape(-1)
    bdn = None if bound_dn is None else np.ascontiguousarray(bound_dn, dtype=np.float64).reshape(-1)
    ds = None if down_scale is None else np.ascontiguousarray(down_scale, dtype=np.float32).reshape(-1)
    sh = None if shared_out is None else np.ascontiguousarray(shared_out, dtype=np.float32).reshape(-1)
    sg = None if shared_gate is None else np.ascontiguousarray(shared_gate, dtype=np.float32).reshape(-1)
    x_in = np.ascontiguousarray(x_in, dtype=np.float32).reshape(-1)
    out = np.empty((T, H), dtype=np.float64)
    bout = np.empty((T, H), dtype=np.float64)
    _check(lib().og_moe_combine_ex(_p(ids), _p(wts), _p(dn), _p(bdn), _p(ds), E, _p(sh), _p(sg), _p(x_in), T, k, H,
                                   int(add_residual), _p(out), _p(bout)), "moe_combine_ex")
    return out, bout


def rmsnorm_k(x: np.ndarray, w: np.ndarray, eps: float, k: float) -> np.ndarray:
    """y[t][i] = ((x[t][i] * s_t) * k) * w[i], float64 [T][N]."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    x2 = x.reshape(-1, x.shape[-1])
    w = np.ascontiguousarray(w, dtype=np.float32).reshape(-1)
    T, N = x2.shape
    y = np.empty((T, N), dtype=np.float64)
    _check(lib().og_rmsnorm_k(_p(x2), _p(w), T, N, float(eps), float(k), _p(y)), "rmsnorm_k")
    return y
