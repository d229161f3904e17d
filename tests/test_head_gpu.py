"""GPU parity of the steps on either side of the GEMV chain, through the C ABI, against the
oracle: embedding row gathers (bit-exact), RMSNorm (within its bound), per-row argmax
(exact on the same logits) and the tied head with its argmax (vocab scale, Q8_0 and Q6_K)."""
import numpy as np
import pytest
import torch

import gguf_synth as gs
from helpers import assert_within_bound, to_dev

pytestmark = pytest.mark.gpu

TYPES = [gs.Q8_0, gs.Q4_0, gs.Q4_K, gs.Q6_K]


@pytest.fixture(scope="module")
def qg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gguf_block_dequant_gb300 as qg
    from gguf_block_dequant_gb300 import build

    build.build()
    qg.load()
    return qg


def _status(qg, clear=True):
    torch.cuda.synchronize()
    return qg.device_status(clear=clear)


def _embed(qg, qtype, table, V, N, ids, scale=1.0):
    td = to_dev(table, torch)
    idd = torch.from_numpy(np.asarray(ids, dtype=np.int32)).cuda()
    out = torch.full((len(ids), N), float("nan"), dtype=torch.float32, device="cuda")
    qg.embed_rows(qtype, td, V, N, idd, out, scale=scale)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("qtype", TYPES)
@pytest.mark.parametrize("aligned", [True, False])
def test_embed_rows_bit_exact(qg, oracle_lib, qtype, aligned):
    """Rows of 16-byte-multiple length and rows that are not (the last row then ends past the
    table's last 16-byte boundary); first, last and repeated ids; the scale as one rounding."""
    qk, bb = gs.BLOCK[qtype]
    N = (2560 if aligned else 2592) if qk == 32 else (2816 if not aligned else 2048)
    V = 301
    table = gs.quant_blocks(qtype, V, N, seed=31, stream=qtype)
    ids = [0, V - 1, 7, 7, 150, V - 2, 3]
    for scale in (1.0, float(np.sqrt(np.float32(N)))):
        got = _embed(qg, qtype, table, V, N, ids, scale)
        want = oracle_lib.embed_rows(qtype, table, V, N, np.array(ids, dtype=np.int32), scale)
        assert np.array_equal(got, want), (qtype, aligned, scale, np.argwhere(got != want)[:4])
    assert _status(qg) == 0


def test_embed_rows_bad_id_gives_zero_row_and_status(qg, oracle_lib):
    V, N = 10, 256
    table = gs.quant_blocks(gs.Q8_0, V, N, seed=2)
    assert _status(qg) == 0
    got = _embed(qg, gs.Q8_0, table, V, N, [3, V, -1, 9])
    want = oracle_lib.embed_rows(gs.Q8_0, table, V, N, np.array([3, 9], dtype=np.int32))
    assert np.array_equal(got[0], want[0]) and np.array_equal(got[3], want[1])
    assert not got[1].any() and not got[2].any()
    st = _status(qg)
    assert st == (1 << 6), st  # QG_EDEVICE_ID


@pytest.mark.parametrize("qtype,V,N,scale", [(gs.Q8_0, 151936, 2560, 1.0), (gs.Q6_K, 262144, 2816, float(np.sqrt(np.float32(2816))))])
def test_embed_rows_vocab_scale(qg, oracle_lib, qtype, V, N, scale):
    """Qwen3-shaped Q8_0 and Gemma-shaped Q6_K embedding tables (413 / 606 MB): 16 tokens
    including the first and the last row."""
    table = gs.quant_blocks(qtype, V, N, seed=3, stream=qtype)
    rng = np.random.default_rng(5)
    ids = np.concatenate([[0, V - 1], rng.integers(0, V, 14)]).astype(np.int32)
    got = _embed(qg, qtype, table, V, N, ids, scale)
    rb = gs.row_bytes(qtype, N)
    rows = table.reshape(V, rb)[ids]
    want = oracle_lib.embed_rows(qtype, rows, len(ids), N, np.arange(len(ids), dtype=np.int32), scale)
    assert np.array_equal(got, want)
    assert _status(qg) == 0


@pytest.mark.parametrize("T,N", [(1, 2560), (3, 2048), (16, 2560), (5, 4)])
@pytest.mark.parametrize("inplace", [False, True])
def test_rmsnorm(qg, oracle_lib, T, N, inplace):
    """|gpu - oracle| <= 1e-5 |x s w| + 1e-6 per element (s the oracle's row scale): the f32 sum
    of squares and one rounding in each of sqrt, the reciprocal and two products."""
    x = gs.activations(T, N, seed=T + N, stream=9)
    x[0, :3] *= 40.0  # rows with a wide range
    rng = np.random.default_rng(T)
    w = rng.uniform(-1.5, 1.5, N).astype(np.float32)
    eps = 1e-6
    xd = to_dev(x, torch)
    wd = to_dev(w, torch)
    yd = xd if inplace else torch.empty_like(xd)
    qg.rmsnorm(xd, wd, eps, yd)
    torch.cuda.synchronize()
    ref = oracle_lib.rmsnorm(x, w, eps)
    ms = np.mean(x.astype(np.float64) ** 2, axis=1, keepdims=True)
    bound = np.abs(x.astype(np.float64) * w.astype(np.float64)) / np.sqrt(ms + eps)
    assert_within_bound(yd.cpu().numpy(), ref, bound, what=f"rmsnorm T={T} N={N}")


@pytest.mark.parametrize("T,n", [(1, 151936), (16, 151936), (4, 33), (2, 1)])
def test_argmax_rows_exact(qg, oracle_lib, T, n):
    """Random logits with the maximum planted twice (the lower index must win), NaN in places,
    an all -inf row and an all-NaN row: the same f32 values through the oracle."""
    rng = np.random.default_rng(n + T)
    v = rng.standard_normal((T, n)).astype(np.float32)
    for t in range(T):
        if n > 8:
            a, b = sorted(rng.choice(n, 2, replace=False))
            v[t, a] = v[t, b] = np.float32(9.0)
            v[t, rng.choice(n, min(n // 7, 1000), replace=False)] = np.nan
    if T >= 4:
        v[1] = -np.inf
        v[2] = np.nan
    ids = torch.empty(T, dtype=torch.int32, device="cuda")
    qg.argmax_rows(to_dev(v, torch), ids)
    torch.cuda.synchronize()
    want = oracle_lib.argmax_rows(v.astype(np.float64))
    assert np.array_equal(ids.cpu().numpy(), want)


@pytest.mark.parametrize("qtype,M,N,T", [(gs.Q8_0, 151936, 2560, 1), (gs.Q8_0, 151936, 2560, 4),
                                          (gs.Q6_K, 262144, 2816, 1)])
def test_head_argmax_vocab_scale(qg, oracle_lib, qtype, M, N, T):
    """The tied head and its argmax in one call: logits within the GEMV bound of the oracle's
    (every row), ids equal to the argmax of the returned logits, and to the oracle's argmax
    wherever its top two logits are further apart than twice the bound (otherwise the pick's
    oracle logit is within that of the maximum: several answers are correct)."""
    w = gs.quant_blocks(qtype, M, N, seed=8, stream=qtype)
    x = gs.activations(T, N, seed=8)
    wd, xd = to_dev(w, torch), to_dev(x, torch)
    logits = torch.full((T, M), float("nan"), dtype=torch.float32, device="cuda")
    ids = torch.empty(T, dtype=torch.int32, device="cuda")
    qg.head_argmax(qtype, wd, xd, M, N, T, logits, ids)
    torch.cuda.synchronize()
    assert qg.device_status() == 0
    lg = logits.cpu().numpy()
    got = ids.cpu().numpy()
    ref, bnd = oracle_lib.gemv(qtype, w, M, N, x, threads=16)
    assert_within_bound(lg, ref, bnd, what=f"head {qtype} {M}x{N} T={T}")
    assert np.array_equal(got, oracle_lib.argmax_rows(lg.astype(np.float64)))
    tol = 2 * (1e-5 * bnd + 1e-6)
    for t in range(T):
        order = np.argsort(-ref[t], kind="stable")
        top, second = order[0], order[1]
        if ref[t, top] - ref[t, second] > tol[t, top] + tol[t, second]:
            assert got[t] == top, (t, got[t], top)
        else:
            assert ref[t, top] - ref[t, got[t]] <= tol[t, top] + tol[t, got[t]]
