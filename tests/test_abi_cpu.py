"""The C ABI on the CPU: the library builds, loads without a GPU, exports every symbol the
header declares, and rejects bad arguments on the host before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ggufdq.h")


@pytest.fixture(scope="module")
def lib():
    from gguf_block_dequant_gb300 import build

    path = build.build()
    return ctypes.CDLL(path)


def _declared():
    src = open(HEADER).read()
    return re.findall(r"^QG_API [^;(]*?\b([a-z_0-9]+)\(", src, flags=re.M)


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 15, names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in ggufdq.h but not exported"


def test_version_strings_and_block_shapes(lib):
    assert lib.qg_version() == 3
    lib.qg_strerror.restype = ctypes.c_char_p
    assert lib.qg_strerror(0) == b"ok"
    assert lib.qg_strerror(999) == b"unknown status"
    qk, bb = ctypes.c_int(), ctypes.c_int()
    for t, (q, b) in {8: (32, 34), 2: (32, 18), 12: (256, 144), 14: (256, 210)}.items():
        assert lib.qg_block_shape(t, ctypes.byref(qk), ctypes.byref(bb)) == 0
        assert (qk.value, bb.value) == (q, b)
    assert lib.qg_block_shape(1, ctypes.byref(qk), ctypes.byref(bb)) == 4  # QG_EUNSUPPORTED


def test_host_argument_checks_need_no_gpu(lib):
    P, I64 = ctypes.c_void_p, ctypes.c_int64
    lib.qgemv_q8_0.argtypes = [P, P, P, I64, I64, P]
    lib.qgemv_t.argtypes = [ctypes.c_int, P, P, P, I64, I64, ctypes.c_int, P]
    # NULL pointers -> QG_EINVAL_PTR, before any CUDA call
    assert lib.qgemv_q8_0(None, None, None, 4, 64, None) == 2
    fake = P(4096)  # never dereferenced: the shape check fails first
    assert lib.qgemv_q8_0(fake, fake, fake, 4, 48, None) == 1      # N % 32 != 0
    assert lib.qgemv_q8_0(fake, fake, fake, -1, 64, None) == 1     # M < 0
    assert lib.qgemv_t(8, fake, fake, fake, 4, 64, 0, None) == 1   # T < 1
    assert lib.qgemv_t(8, fake, fake, fake, 4, 64, 17, None) == 1  # T > 16
    assert lib.qgemv_t(13, fake, fake, fake, 4, 64, 1, None) == 4  # unsupported type
    odd = P(4096 + 2)
    assert lib.qgemv_q8_0(odd, fake, fake, 4, 64, None) == 3       # misaligned weights
    lib.qgemv_multi.argtypes = [ctypes.c_int, ctypes.c_int, P, P, P, I64, P, ctypes.c_int, P]
    W = (P * 2)(fake, fake)
    Y = (P * 2)(fake, fake)
    M = (I64 * 2)(4, 4)
    assert lib.qgemv_multi(8, 5, W, Y, M, 64, fake, 1, None) == 1  # n > 4
    assert lib.qgemv_multi(8, 2, W, Y, M, 48, fake, 1, None) == 1  # N % 32 != 0
    assert lib.qgemv_multi(8, 2, None, Y, M, 64, fake, 1, None) == 2


def test_head_steps_host_checks_need_no_gpu(lib):
    P, I, I64, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
    lib.qg_embed_rows.argtypes = [I, P, I64, I64, P, I, F, P, P]
    lib.qg_rmsnorm.argtypes = [P, P, I, I64, F, F, P, P]
    lib.qg_argmax_rows.argtypes = [P, I, I64, P, P]
    lib.qg_head_argmax.argtypes = [I, P, I64, I64, P, I, P, P, P]
    fake, odd = P(4096), P(4096 + 2)
    # embedding gather
    assert lib.qg_embed_rows(8, None, 4, 64, fake, 1, 1.0, fake, None) == 2
    assert lib.qg_embed_rows(8, fake, 4, 48, fake, 1, 1.0, fake, None) == 1   # N % 32
    assert lib.qg_embed_rows(14, fake, 4, 64, fake, 1, 1.0, fake, None) == 1  # N % 256 (Q6_K)
    assert lib.qg_embed_rows(8, fake, 0, 64, fake, 1, 1.0, fake, None) == 1   # V < 1
    assert lib.qg_embed_rows(8, fake, 4, 64, fake, -1, 1.0, fake, None) == 1  # n < 0
    assert lib.qg_embed_rows(8, odd, 4, 64, fake, 1, 1.0, fake, None) == 3    # table alignment
    assert lib.qg_embed_rows(1, fake, 4, 64, fake, 1, 1.0, fake, None) == 4   # type
    assert lib.qg_embed_rows(8, fake, 4, 64, fake, 0, 1.0, fake, None) == 0   # n == 0: nothing to do
    # RMSNorm
    assert lib.qg_rmsnorm(None, fake, 1, 64, 1e-6, 1.0, fake, None) == 2
    assert lib.qg_rmsnorm(fake, fake, 1, 62, 1e-6, 1.0, fake, None) == 1           # N % 4
    assert lib.qg_rmsnorm(fake, fake, 1, 64, -1.0, 1.0, fake, None) == 1           # eps < 0
    assert lib.qg_rmsnorm(fake, fake, 1, 64, float("nan"), 1.0, fake, None) == 1
    assert lib.qg_rmsnorm(fake, odd, 1, 64, 1e-6, 1.0, fake, None) == 3
    assert lib.qg_rmsnorm(fake, fake, 0, 64, 1e-6, 1.0, fake, None) == 0           # T == 0
    assert lib.qg_rmsnorm(fake, fake, 1, 64, 1e-6, float("inf"), fake, None) == 1  # k not finite
    # argmax
    assert lib.qg_argmax_rows(None, 1, 64, fake, None) == 2
    assert lib.qg_argmax_rows(fake, 1, 0, fake, None) == 1
    assert lib.qg_argmax_rows(P(4097), 1, 64, fake, None) == 3
    # head + argmax: checked in full before the GEMV is enqueued
    assert lib.qg_head_argmax(8, fake, 64, 64, fake, 1, fake, None, None) == 2
    assert lib.qg_head_argmax(8, fake, 0, 64, fake, 1, fake, fake, None) == 1
    assert lib.qg_head_argmax(8, fake, 64, 64, fake, 17, fake, fake, None) == 1
    assert lib.qg_head_argmax(8, fake, 64, 64, fake, 1, fake, P(4098), None) == 3
    assert lib.qg_head_argmax(3, fake, 64, 64, fake, 1, fake, fake, None) == 4


def test_moe_host_checks_need_no_gpu(lib):
    P, I, I64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    lib.moe_workspace_size.argtypes = [I, I, I, I, I]
    lib.moe_workspace_size.restype = SZ
    lib.moe_route_topk.argtypes = [P, P, I, I, I, I, P, P, P, P, SZ, P]
    lib.moe_expert_swiglu.argtypes = [I, P, P, I64, P, I, I, P, P, I, I, I, I, P, P, SZ, P]
    lib.moe_combine.argtypes = [I, P, I64, P, I, I, P, P, P, I, I, I, I, P, I, P, SZ, P]
    # workspace: the fixed header (one-token grid-barrier and call counters, tagged logits,
    # then one ticket word for each of up to 65535 router tiles), then router logits and dn
    # rows, each rounded up to 256 bytes
    header = (4096 + 65535 * 4 + 255) // 256 * 256
    n = lib.moe_workspace_size(8, 8, 128, 2048, 768)
    assert n == header + 8 * 128 * 4 + 8 * 8 * 2048 * 4
    # a workspace sized for a larger shape covers every smaller one
    assert lib.moe_workspace_size(1, 8, 128, 2048, 768) < n
    assert lib.moe_workspace_size(8, 33, 128, 2048, 768) == 0   # k > 32
    assert lib.moe_workspace_size(8, 8, 300, 2048, 768) == 0    # E > 256
    fake = P(4096)
    assert lib.moe_route_topk(None, fake, 1, 64, 8, 2, fake, fake, None, fake, 1 << 20, None) == 2
    assert lib.moe_route_topk(fake, fake, 1, 64, 8, 9, fake, fake, None, fake, 1 << 20, None) == 1  # k > E
    assert lib.moe_route_topk(fake, fake, 1, 66, 8, 2, fake, fake, None, fake, 1 << 20, None) == 1  # H % 4
    assert lib.moe_route_topk(fake, fake, 2, 64, 8, 2, fake, fake, None, fake, 16, None) == 8       # workspace
    assert lib.moe_expert_swiglu(8, fake, fake, 0, None, 1, 8, fake, fake, 17, 2, 64, 32, fake, None, 0,
                                 None) == 4  # more than 16 tokens: not on this path
    assert lib.moe_expert_swiglu(8, fake, fake, 0, None, 1, 8, fake, fake, 2, 2, 48, 32, fake, None, 0,
                                 None) == 1  # H not a multiple of the block
    assert lib.moe_expert_swiglu(3, fake, fake, 0, None, 1, 8, fake, fake, 2, 2, 64, 32, fake, None, 0,
                                 None) == 4  # unsupported type
    assert lib.moe_combine(8, fake, 0, None, 1, 8, fake, fake, fake, 2, 2, 64, 32, fake, 1, fake, 16,
                           None) == 8  # workspace too small


def test_moe_variant_host_checks_need_no_gpu(lib):
    P, I, I64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t

    class Var(ctypes.Structure):
        _fields_ = [("act", I), ("down_scale", P), ("shared_out", P), ("shared_gate", P)]

    lib.moe_expert_act.argtypes = [I, P, P, I64, P, I, I, P, P, I, I, I, I, P, P, P, SZ, P]
    lib.moe_combine_ex.argtypes = [I, P, I64, P, I, I, P, P, P, I, I, I, I, P, P, I, P, SZ, P]
    lib.moe_layer_ex.argtypes = [I, P, P, P, P, P, I64, P, I, I, I, I, I, I, P, P, P, P, P, P, SZ, P]
    fake = P(4096)
    bad_act = Var(5, None, None, None)
    half_shared = Var(0, None, 4096, None)
    odd_shared = Var(1, None, 4096 + 4, 4096)
    odd_scale = Var(1, 4096 + 2, None, None)
    for v, want in ((bad_act, 1), (half_shared, 2), (odd_shared, 3), (odd_scale, 3)):
        assert lib.moe_expert_act(8, fake, fake, 0, None, 1, 8, fake, fake, 2, 2, 64, 32, ctypes.byref(v), fake,
                                  fake, 1 << 20, None) == want
        assert lib.moe_combine_ex(8, fake, 0, None, 1, 8, fake, fake, fake, 2, 2, 64, 32, ctypes.byref(v), fake, 1,
                                  fake, 1 << 20, None) == want
        assert lib.moe_layer_ex(4, fake, fake, fake, fake, fake, 0, None, 1, 2, 64, 32, 8, 2, ctypes.byref(v), fake,
                                fake, fake, fake, fake, 1 << 20, None) == want
    # a GELU variant goes through the usual shape checks (N % 32 here)
    gelu = Var(1, None, None, None)
    assert lib.moe_expert_act(8, fake, fake, 0, None, 1, 8, fake, fake, 2, 2, 48, 32, ctypes.byref(gelu), fake,
                              fake, 1 << 20, None) == 1


def test_moe_rejects_before_enqueueing_anything(lib):
    """Every check runs before the first launch: on a machine without a GPU a launch attempt
    would return QG_ECUDA, so the argument error itself coming back shows that nothing was
    enqueued ahead of it."""
    P, I, I64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    lib.moe_combine.argtypes = [I, P, I64, P, I, I, P, P, P, I, I, I, I, P, I, P, SZ, P]
    lib.moe_route_topk_noalloc.argtypes = [P, P, I, I, I, I, P, P, P, P]
    lib.moe_layer.argtypes = [I, P, P, P, P, P, I64, P, I, I, I, I, I, I, P, P, P, P, P, SZ, P]
    lib.moe_workspace_size.argtypes = [I, I, I, I, I]
    lib.moe_workspace_size.restype = SZ
    fake, odd = P(1 << 20), P((1 << 20) + 4)
    T, k, E, H, F = 4, 2, 8, 64, 32
    big = 1 << 30
    # misaligned x_inout: the down kernel must not be enqueued first
    assert lib.moe_combine(8, fake, 0, None, 1, E, fake, fake, fake, T, k, H, F, odd, 1, fake, big, None) == 3
    # the whole layer, misaligned act or x_inout, for each token-count path
    for t in (1, 4, 17):
        h, f = (256, 256) if t > 16 else (H, F)
        assert lib.moe_layer(8, fake, fake, fake, fake, fake, 0, None, 1, t, h, f, E, k, fake, fake, odd, fake,
                             fake, big, None) == 3, t
        assert lib.moe_layer(8, fake, fake, fake, fake, fake, 0, None, 1, t, h, f, E, k, fake, fake, fake, odd,
                             fake, big, None) == 3, t
        assert lib.moe_layer(8, fake, fake, fake, fake, fake, 0, None, 1, t, h, f, E, k, fake, fake, fake, fake,
                             fake, 16, None) == 8, t  # workspace too small
    # the router without a workspace: argument errors before its ticket memset
    assert lib.moe_route_topk_noalloc(odd, fake, 1, 64, 8, 2, fake, fake, None, None) == 3
    assert lib.moe_route_topk_noalloc(fake, fake, 1, 64, 8, 9, fake, fake, None, None) == 1  # k > E
    assert lib.moe_route_topk_noalloc(None, fake, 1, 64, 8, 2, fake, fake, None, None) == 2
    # its limits: T * E <= 16384 and at most 1024 tiles of 16 tokens
    assert lib.moe_route_topk_noalloc(fake, fake, 16385, 64, 1, 1, fake, fake, None, None) == 8
    assert lib.moe_route_topk_noalloc(fake, fake, 200, 64, 128, 8, fake, fake, None, None) == 8


def test_static_weights_is_a_setting_of_one_stream(lib):
    """Each stream handle keeps its own setting; enabling it on one stream leaves the others
    (and the legacy default stream) off.  No CUDA work is enqueued, so fake handles serve."""
    lib.qg_set_static_weights.argtypes = [ctypes.c_void_p, ctypes.c_int]
    lib.qg_set_static_weights.restype = ctypes.c_int
    a, b = ctypes.c_void_p(0x1000), ctypes.c_void_p(0x2000)
    try:
        assert lib.qg_set_static_weights(a, 7) == 0  # any non-zero value enables it
        assert lib.qg_set_static_weights(a, 1) == 1
        assert lib.qg_set_static_weights(b, 0) == 0  # the other stream is untouched
        assert lib.qg_set_static_weights(None, 0) == 0
        assert lib.qg_set_static_weights(a, 0) == 1
        assert lib.qg_set_static_weights(a, 0) == 0
    finally:
        lib.qg_set_static_weights(a, 0)
        lib.qg_set_static_weights(b, 0)
