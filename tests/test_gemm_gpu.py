"""Parity of the prefill dequant-GEMM (qgemm, tcgen05 tensor cores) with the CPU oracle.

The weights are decoded to bf16 and the activations rounded to bf16 for the tensor cores,
with f32 accumulation: the bar is |gpu - oracle| <= 2e-3 * sum|w x| + 1e-6 per element.
Inputs that are exact in bf16 (d = 1, small codes, small integer activations) leave only
f32 accumulation, which is exact for these integer sums, so there the GPU must equal the
oracle exactly: a wrong operand layout, descriptor, swizzle or partial-tile reduction cannot
hide inside the tolerance.
"""
import numpy as np
import pytest

import gguf_synth as gs
from helpers import assert_within_bound, to_dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

GEMM_REL = 2e-3


@pytest.fixture(scope="module")
def qg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gguf_block_dequant_gb300 as qg
    from gguf_block_dequant_gb300 import build

    build.build()
    qg.load()
    return qg


def _gemm(qg, w, x, M, N, qtype=gs.Q8_0):
    T = x.shape[0]
    wd, xd = to_dev(w, torch), to_dev(x, torch)
    yd = torch.full((T, M), float("nan"), dtype=torch.float32, device="cuda")
    n = qg.qgemm_workspace_size(qtype, M, N, T)
    ws = torch.empty(max(n, 16), dtype=torch.uint8, device="cuda")
    qg.qgemm(qtype, wd, xd, yd, M, N, T, ws)
    torch.cuda.synchronize()
    assert qg.device_status() == 0
    return yd.cpu().numpy()


def _exact_q8_0(M, N, seed):
    """Q8_0 blocks with d = 1.0 and codes in [-8, 8]: every weight is exact in bf16."""
    rng = np.random.default_rng(seed)
    nb = M * N // 32
    blk = np.empty((nb, 34), np.uint8)
    blk[:, 0] = 0x00
    blk[:, 1] = 0x3C  # f16 1.0, little-endian
    blk[:, 2:] = rng.integers(-8, 9, size=(nb, 32)).astype(np.int8).view(np.uint8)
    return blk.reshape(-1)


@pytest.mark.parametrize("M,N,T", [(128, 256, 256), (300, 512, 300), (256, 2560, 40), (256, 9728, 256),
                                   (1000, 1024, 513)])
def test_gemm_exact_on_bf16_exact_inputs(qg, oracle_lib, M, N, T):
    w = _exact_q8_0(M, N, seed=M + T)
    x = np.random.default_rng(N).integers(-4, 5, size=(T, N)).astype(np.float32)
    y = _gemm(qg, w, x, M, N)
    ref, _ = oracle_lib.gemv(gs.Q8_0, w, M, N, x, threads=8)
    assert np.array_equal(y, ref.astype(np.float32)), f"max diff {np.abs(y - ref).max()}"


@pytest.mark.parametrize("M,N,T", [(128, 256, 17), (257, 768, 100), (640, 1536, 333)])
def test_gemm_parity_random(qg, oracle_lib, M, N, T):
    w = gs.quant_blocks(gs.Q8_0, M, N, seed=M, stream=301)
    x = gs.activations(T, N, seed=T, stream=302)
    y = _gemm(qg, w, x, M, N)
    ref, bnd = oracle_lib.gemv(gs.Q8_0, w, M, N, x, threads=8)
    assert_within_bound(y, ref, bnd, rel=GEMM_REL, what=f"gemm {M}x{N} T={T}")


@pytest.mark.parametrize("M,N", [(9728, 2560), (2560, 9728)])
def test_gemm_prefill_full_size(qg, oracle_lib, M, N):
    """The prefill shapes at T = 512, every token, a sample of rows against the oracle."""
    T = 512
    w = gs.quant_blocks(gs.Q8_0, M, N, seed=0, stream=104 if M == 9728 else 106)
    x = gs.activations(T, N, seed=0, stream=303)
    y = _gemm(qg, w, x, M, N)
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, M // 2, M - 1], rng.integers(0, M, 40)]))
    rb = gs.row_bytes(gs.Q8_0, N)
    ref, bnd = oracle_lib.gemv(gs.Q8_0, w.reshape(M, rb)[rows], len(rows), N, x, threads=8)
    assert_within_bound(y[:, rows], ref, bnd, rel=GEMM_REL, what=f"prefill {M}x{N}")


def test_gemm_small_t_routes_to_exact_gemv(qg, oracle_lib):
    M, N, T = 200, 512, 9
    w = gs.quant_blocks(gs.Q8_0, M, N, seed=1)
    x = gs.activations(T, N, seed=1)
    y = _gemm(qg, w, x, M, N)
    ref, bnd = oracle_lib.gemv(gs.Q8_0, w, M, N, x, threads=8)
    assert_within_bound(y, ref, bnd, what="qgemm T<=16")  # the GEMV bar, not the bf16 one


def test_gemm_repeat_is_deterministic(qg):
    """Stream-K partial tiles are summed in a fixed order: two calls agree bit for bit."""
    M, N, T = 384, 9728, 300
    w = gs.quant_blocks(gs.Q8_0, M, N, seed=2)
    x = gs.activations(T, N, seed=2)
    assert np.array_equal(_gemm(qg, w, x, M, N), _gemm(qg, w, x, M, N))


def test_gemm_rejects(qg):
    f = torch.zeros(1 << 16, dtype=torch.float32, device="cuda")
    u = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(qg.QGError) as e:
        qg.qgemm(gs.Q4_K, u, f, f, 16, 256, 64, u)     # tensor-core path is Q8_0 only
    assert e.value.status == qg.QG_EUNSUPPORTED
    with pytest.raises(qg.QGError) as e:
        qg.qgemm(gs.Q8_0, u, f, f, 16, 288, 64, u)     # rows must be whole 256-element boxes
    assert e.value.status == qg.QG_EUNSUPPORTED
    with pytest.raises(qg.QGError) as e:
        qg.qgemm(gs.Q8_0, u, f, f, 16, 256, 64, u[:64])  # workspace too small
    assert e.value.status == qg.QG_EWORKSPACE
