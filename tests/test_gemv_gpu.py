"""Parity of the dense quantized GEMV kernels (qgemv_*, qgemv_t) with the CPU oracle.

Every call goes through the C ABI (libggufdq.so) via the thin Python binding.  Sizes span
several tiles, partial activation groups and ragged row tails; the one-hot cases check that
every dequantized weight comes out of the kernels bit-exact.
"""
import numpy as np
import pytest

import edge_blocks as eb
import gguf_synth as gs
from helpers import assert_within_bound, to_dev

torch = pytest.importorskip("torch")
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


def _run(qg, qtype, w, x, M, N):
    T = x.shape[0]
    wd = to_dev(w, torch)
    xd = to_dev(x, torch)
    yd = torch.full((T, M), float("nan"), dtype=torch.float32, device="cuda")
    if T == 1:
        qg.qgemv(qtype, wd, xd, M, N, yd)
    else:
        qg.qgemv_t(qtype, wd, xd, yd, M, N, T)
    torch.cuda.synchronize()
    assert qg.device_status() == 0
    return yd.cpu().numpy()


def _shapes(qtype):
    qk = gs.BLOCK[qtype][0]
    if qk == 32:   # groups of 256 elements: full groups, a partial group, a single block
        return [(1, 32), (37, 352), (130, 1024), (261, 2816), (9, 4096 + 96)]
    return [(1, 256), (37, 1280), (130, 2048), (67, 5120), (5, 17408)]


@pytest.mark.parametrize("qtype", TYPES)
@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 8, 11, 16])
def test_gemv_parity(qg, oracle_lib, qtype, T):
    for si, (M, N) in enumerate(_shapes(qtype)):
        w = gs.quant_blocks(qtype, M, N, seed=si, stream=qtype)
        x = gs.activations(T, N, seed=si, stream=7)
        y = _run(qg, qtype, w, x, M, N)
        ref, bnd = oracle_lib.gemv(qtype, w, M, N, x, threads=4)
        assert_within_bound(y, ref, bnd, what=f"type {qtype} M={M} N={N} T={T}")


@pytest.mark.parametrize("qtype", TYPES)
def test_gemv_one_hot_is_exact_dequant(qg, oracle_lib, qtype):
    """x = e_k makes every product but one an exact zero, so y must equal column k of the
    dequantized matrix bit for bit: this checks the in-register decode of every type."""
    M, N = 45, 2048 if gs.BLOCK[qtype][0] == 256 else 640
    w = gs.quant_blocks(qtype, M, N, seed=3, stream=qtype)
    W = oracle_lib.dequant(qtype, w, M, N)
    cols = list(range(0, N, 7)) + [N - 1]
    for T in (1, 8):
        for start in range(0, len(cols), T):
            ks = cols[start:start + T]
            x = np.zeros((len(ks), N), np.float32)
            for t, k in enumerate(ks):
                x[t, k] = 1.0
            y = _run(qg, qtype, w, x, M, N)
            for t, k in enumerate(ks):
                # equal as values: exact for every nonzero weight; a zero weight may come out
                # as +0 where the decoded value is -0 (negative Q6_K scales)
                assert np.array_equal(y[t], W[:, k]), (qtype, T, k)


@pytest.mark.parametrize("qtype", TYPES)
@pytest.mark.parametrize("T", [1, 8, 16])
@pytest.mark.parametrize("aligned", [False, True])
def test_gemv_one_hot_edge_blocks(qg, oracle_lib, qtype, T, aligned):
    """The formats' edge values through every CUDA decoder: Q8_0 code 0x80 (-128), negative,
    subnormal and extreme f16 d; Q4_0 negative (ggml's d = max / -8), subnormal and largest d;
    Q4_K d = 0, dmin = 0, all-63 scales and mins, subnormal and negative d; Q6_K scales -32 and
    31 with subnormal and extreme d.  The blocks (tests/golden/hand_blocks.txt and
    tests/edge_blocks.py, pinned on the CPU) are dealt over the rows between random blocks;
    with one-hot activations every output equals one dequantized weight, bit for bit."""
    qk, bb = gs.BLOCK[qtype]
    # rows whose byte length is a multiple of 16 take the lean one-token kernel; the others
    # the general one
    if qk == 32:
        N = 1024 if aligned else 640
    else:
        N = 2048 if aligned or qtype == gs.Q4_K else 1280
    assert ((N // qk) * bb % 16 == 0) == (aligned or qtype == gs.Q4_K)
    M = 26
    w = eb.matrix_with_edge_blocks(qtype, M, N, seed=9)
    W = oracle_lib.dequant(qtype, w, M, N)
    cols = list(range(0, N, 5)) + [N - 1]
    for start in range(0, len(cols), T):
        ks = cols[start:start + T]
        x = np.zeros((len(ks), N), np.float32)
        for t, k in enumerate(ks):
            x[t, k] = 1.0
        y = _run(qg, qtype, w, x, M, N)
        for t, k in enumerate(ks):
            assert np.array_equal(y[t], W[:, k]), (qtype, T, k, np.nonzero(y[t] != W[:, k])[0][:4])


@pytest.mark.parametrize("qtype", [gs.Q8_0, gs.Q4_0, gs.Q4_K, gs.Q6_K])
@pytest.mark.parametrize("M,N,T", [(4874, 1024, 4), (4874, 1024, 16), (26, 4096, 16)])
def test_multi_token_edge_blocks_rows_across_lanes(qg, oracle_lib, qtype, M, N, T):
    """The edge blocks through the rows-across-lanes decoders: 4874 rows are 305 16-row groups
    (at least two per SM, so that kernel goes first, and the last group is partial); 26 rows of
    4096 at T = 16 do not fit one CTA's shared memory with their activations, so K is split
    over a cluster.  One-hot activations: every output is one dequantized weight, bit for bit."""
    w = eb.matrix_with_edge_blocks(qtype, M, N, seed=13)
    W = oracle_lib.dequant(qtype, w, M, N)
    cols = list(range(3, N, 37)) + [0, N - 1]
    for start in range(0, len(cols), T):
        ks = cols[start:start + T]
        x = np.zeros((len(ks), N), np.float32)
        for t, k in enumerate(ks):
            x[t, k] = 1.0
        y = _run(qg, qtype, w, x, M, N)
        for t, k in enumerate(ks):
            assert np.array_equal(y[t], W[:, k]), (qtype, M, N, T, k, np.nonzero(y[t] != W[:, k])[0][:4])


@pytest.mark.parametrize("qtype", TYPES)
def test_gemv_zero_input_and_zero_rows(qg, qtype):
    M, N = 70, 1024
    w = gs.quant_blocks(qtype, M, N, seed=4, stream=qtype)
    y = _run(qg, qtype, w, np.zeros((3, N), np.float32), M, N)
    assert (y == 0).all()


def test_gemv_chunked_activations(qg, oracle_lib):
    """T = 16 over a long row streams the activations in K chunks (y accumulated per chunk)."""
    for qtype, (M, N) in [(gs.Q8_0, (40, 9728)), (gs.Q4_K, (24, 17408)), (gs.Q6_K, (24, 17408)),
                          (gs.Q4_0, (40, 9728))]:
        w = gs.quant_blocks(qtype, M, N, seed=5, stream=qtype)
        x = gs.activations(16, N, seed=5)
        y = _run(qg, qtype, w, x, M, N)
        ref, bnd = oracle_lib.gemv(qtype, w, M, N, x, threads=4)
        assert_within_bound(y, ref, bnd, what=f"chunked type {qtype}")


def test_gemv_rejects_bad_arguments(qg):
    w = torch.zeros(34 * 4, dtype=torch.uint8, device="cuda")
    x = torch.zeros(128, dtype=torch.float32, device="cuda")
    y = torch.zeros(1, dtype=torch.float32, device="cuda")
    with pytest.raises(qg.QGError) as e:
        qg.qgemv(gs.Q8_0, w, x, 1, 100, y)      # N not a multiple of 32
    assert e.value.status == qg.QG_EINVAL_SHAPE
    with pytest.raises(qg.QGError) as e:
        qg.qgemv(gs.Q8_0, w[1:], x, 1, 128, y)  # misaligned weights
    assert e.value.status == qg.QG_EALIGN
    with pytest.raises(qg.QGError) as e:
        qg.qgemv_t(gs.Q8_0, w, x, y, 1, 128, 17)
    assert e.value.status == qg.QG_EINVAL_SHAPE
    with pytest.raises(qg.QGError) as e:
        qg.qgemv_t(5, w, x, y, 1, 128, 1)
    assert e.value.status == qg.QG_EUNSUPPORTED


# ---- full-size workloads (sampled rows) ------------------------------------------------------

def _sample_rows(M, n=96, seed=0):
    rng = np.random.default_rng(seed)
    rows = np.unique(np.concatenate([[0, 1, M // 2, M - 2, M - 1], rng.integers(0, M, n)]))
    return rows


@pytest.mark.parametrize("name", list(gs.QWEN3_4B_PROJ))
@pytest.mark.parametrize("T", [1, 4, 16])
def test_qwen3_4b_projection_full_size(qg, oracle_lib, name, T):
    M, N = gs.QWEN3_4B_PROJ[name]
    w = gs.quant_blocks(gs.Q8_0, M, N, seed=0, stream=100 + list(gs.QWEN3_4B_PROJ).index(name))
    x = gs.activations(T, N, seed=0)
    y = _run(qg, gs.Q8_0, w, x, M, N)
    rows = _sample_rows(M)
    rb = gs.row_bytes(gs.Q8_0, N)
    wsub = w.reshape(M, rb)[rows]
    ref, bnd = oracle_lib.gemv(gs.Q8_0, wsub, len(rows), N, x, threads=4)
    assert_within_bound(y[:, rows], ref, bnd, what=f"{name} T={T}")


@pytest.mark.parametrize("qtype,M,N", [(gs.Q4_K, 17408, 5120), (gs.Q4_K, 5120, 17408), (gs.Q6_K, 17408, 5120),
                                        (gs.Q6_K, 5120, 17408), (gs.Q4_0, 2112, 2816)])
@pytest.mark.parametrize("T", [1, 8])
def test_kquant_full_size(qg, oracle_lib, qtype, M, N, T):
    w = gs.quant_blocks(qtype, M, N, seed=0, stream=200 + qtype)
    x = gs.activations(T, N, seed=0)
    y = _run(qg, qtype, w, x, M, N)
    rows = _sample_rows(M)
    rb = gs.row_bytes(qtype, N)
    ref, bnd = oracle_lib.gemv(qtype, w.reshape(M, rb)[rows], len(rows), N, x, threads=4)
    assert_within_bound(y[:, rows], ref, bnd, what=f"type {qtype} {M}x{N} T={T}")


@pytest.mark.parametrize("qtype,M,N,T", [(gs.Q8_0, 2560, 9728, 1), (gs.Q8_0, 2560, 4096, 1), (gs.Q8_0, 2561, 9728, 4),
                                          (gs.Q8_0, 2560, 9728, 16), (gs.Q4_0, 999, 9728, 8), (gs.Q4_K, 640, 17408, 1),
                                          (gs.Q6_K, 333, 17408, 1), (gs.Q8_0, 31, 9728, 1)])
def test_row_blocks_split_between_warps(qg, oracle_lib, qtype, M, N, T):
    """Few row blocks per CTA and rows cut into K chunks: the CTA's (row block, chunk) items are
    dealt to its warps in contiguous ranges, so many row blocks are summed from the parts of
    two or more warps (and with 31 rows some CTAs have fewer items than warps).  Every row
    against the oracle."""
    w = gs.quant_blocks(qtype, M, N, seed=5, stream=300 + qtype)
    x = gs.activations(T, N, seed=5)
    y = _run(qg, qtype, w, x, M, N)
    ref, bnd = oracle_lib.gemv(qtype, w, M, N, x, threads=8)
    assert_within_bound(y, ref, bnd, what=f"split type {qtype} {M}x{N} T={T}")


def test_config1_full(qg, oracle_lib):
    """Q8_0 1024 x 1024, T = 1, seed 0: every row against the oracle."""
    M = N = 1024
    w = gs.quant_blocks(gs.Q8_0, M, N, seed=0)
    x = gs.activations(1, N, seed=0)
    y = _run(qg, gs.Q8_0, w, x, M, N)
    ref, bnd = oracle_lib.gemv(gs.Q8_0, w, M, N, x, threads=4)
    assert_within_bound(y, ref, bnd, what="config 1")


@pytest.mark.parametrize("qtype", TYPES)
@pytest.mark.parametrize("T", [1, 3, 16])
def test_gemv_multi_matches_separate_calls(qg, oracle_lib, qtype, T):
    """qgemv_multi over matrices of different heights (one empty) equals the oracle per matrix."""
    N = 1024 if gs.BLOCK[qtype][0] == 32 else 2048
    Ms = [130, 37, 0, 261]
    x = gs.activations(T, N, seed=T, stream=71)
    ws = [gs.quant_blocks(qtype, max(M, 1), N, seed=j, stream=80 + j) for j, M in enumerate(Ms)]
    wd = [to_dev(w, torch) for w in ws]
    yd = [torch.full((T, max(M, 1)), float("nan"), dtype=torch.float32, device="cuda")[:, :M] for M in Ms]
    yd = [y.contiguous() for y in yd]
    qg.qgemv_multi(qtype, wd, yd, to_dev(x, torch), N, T)
    torch.cuda.synchronize()
    assert qg.device_status() == 0
    for j, M in enumerate(Ms):
        if M == 0:
            continue
        ref, bnd = oracle_lib.gemv(qtype, ws[j], M, N, x, threads=4)
        assert_within_bound(yd[j].cpu().numpy(), ref, bnd, what=f"multi type {qtype} j={j} T={T}")


@pytest.mark.parametrize("Ms", [[37, 130, 5], [333]])
def test_q6k_one_token_rows_at_any_offset(qg, oracle_lib, Ms):
    """One token over Q6_K rows of 65 super-blocks (13,650 bytes: each row starts 2 bytes further
    past a 16-byte boundary than the one before, through all eight offsets).  The rows are cut
    into chunks copied from the boundary below each row and read at the row's own offset; the
    last row of every matrix ends short of a 16-byte boundary.  Every row against the oracle."""
    N = 16640
    x = gs.activations(1, N, seed=11, stream=72)
    ws = [gs.quant_blocks(gs.Q6_K, M, N, seed=j, stream=90 + j) for j, M in enumerate(Ms)]
    wd = [to_dev(w, torch) for w in ws]
    yd = [torch.full((1, M), float("nan"), dtype=torch.float32, device="cuda") for M in Ms]
    qg.qgemv_multi(gs.Q6_K, wd, yd, to_dev(x, torch), N, 1)
    torch.cuda.synchronize()
    assert qg.device_status() == 0
    for j, M in enumerate(Ms):
        ref, bnd = oracle_lib.gemv(gs.Q6_K, ws[j], M, N, x, threads=8)
        assert_within_bound(yd[j].cpu().numpy(), ref, bnd, what=f"Q6_K offsets j={j} M={M}")


@pytest.mark.parametrize("qtype", [gs.Q8_0, gs.Q4_0, gs.Q4_K, gs.Q6_K])
@pytest.mark.parametrize("T", [5, 16])
def test_gemv_multi_rows_across_lanes(qg, oracle_lib, qtype, T):
    """qgemv_multi over 377 16-row groups (the rows-across-lanes kernel goes first), matrices
    with partial last groups and one empty: every row of every matrix against the oracle."""
    N = 2560
    Ms = [4100, 0, 1000, 903]
    x = gs.activations(T, N, seed=T, stream=72)
    ws = [gs.quant_blocks(qtype, max(M, 1), N, seed=j, stream=90 + j) for j, M in enumerate(Ms)]
    wd = [to_dev(w, torch) for w in ws]
    yd = [torch.full((T, max(M, 1)), float("nan"), dtype=torch.float32, device="cuda")[:, :M].contiguous() for M in Ms]
    qg.qgemv_multi(qtype, wd, yd, to_dev(x, torch), N, T)
    torch.cuda.synchronize()
    assert qg.device_status() == 0
    for j, M in enumerate(Ms):
        if M == 0:
            continue
        ref, bnd = oracle_lib.gemv(qtype, ws[j], M, N, x, threads=8)
        assert_within_bound(yd[j].cpu().numpy(), ref, bnd, what=f"multi rows-across-lanes type {qtype} j={j} T={T}")


def test_gemv_multi_rejects(qg):
    w = torch.zeros(34 * 64, dtype=torch.uint8, device="cuda")
    x = torch.zeros(256, dtype=torch.float32, device="cuda")
    y = torch.zeros((1, 8), dtype=torch.float32, device="cuda")
    with pytest.raises(qg.QGError) as e:
        qg.qgemv_multi(gs.Q8_0, [w] * 5, [y] * 5, x, 256, 1)  # more than 4 matrices
    assert e.value.status == qg.QG_EINVAL_SHAPE


@pytest.mark.parametrize("T", [1, 4])
def test_static_weights_chain_matches_default(qg, oracle_lib, T):
    """With static weights on, each GEMV streams its weights before the preceding GEMV ends,
    but its activations still come from that GEMV's output: a chain y_i -> x_(i+1) equals the
    fully stream-ordered run bit for bit, and every link is within the oracle's bound."""
    dims = [1024, 2048, 512, 1024, 1024]  # N_0, M_0 = N_1, ...
    ws = [gs.quant_blocks(gs.Q8_0, dims[i + 1], dims[i], seed=i, stream=90) for i in range(len(dims) - 1)]
    wd = [to_dev(w, torch) for w in ws]
    x0 = to_dev(gs.activations(T, dims[0], seed=T, stream=91), torch)

    def chain():
        ys, x = [], x0
        for i, w in enumerate(wd):
            y = torch.empty((T, dims[i + 1]), dtype=torch.float32, device="cuda")
            qg.qgemv_t(gs.Q8_0, w, x, y, dims[i + 1], dims[i], T)
            ys.append(y)
            x = y
        torch.cuda.synchronize()
        assert qg.device_status() == 0
        return [y.cpu().numpy() for y in ys]

    prev = qg.set_static_weights(False)
    try:
        base = chain()
        qg.set_static_weights(True)
        fast = chain()
    finally:
        qg.set_static_weights(prev)
    xin = x0.cpu().numpy()
    for i, (a, b) in enumerate(zip(base, fast)):
        assert np.array_equal(a, b), f"link {i} differs"
        ref, bnd = oracle_lib.gemv(gs.Q8_0, ws[i], dims[i + 1], dims[i], xin, threads=4)
        assert_within_bound(b, ref, bnd, what=f"chain link {i} T={T}")
        xin = b


@pytest.mark.parametrize("qtype,N", [(gs.Q8_0, 1024), (gs.Q8_0, 2560), (gs.Q8_0, 2304), (gs.Q4_0, 2048), (gs.Q4_0, 1792)])
def test_tall_matrix_one_token(qg, oracle_lib, qtype, N):
    """One token over more than 65536 rows takes the tall-matrix shape (4-row blocks, the
    activations held in registers); a row count that leaves a partial last block, sampled rows
    against the oracle, plus every row of the last blocks.  2304 and 1792 end in a partial
    512-element group (4.5 and 3.5 groups per row)."""
    M = 65536 + 7
    w = gs.quant_blocks(qtype, M, N, seed=11, stream=qtype)
    x = gs.activations(1, N, seed=11)
    y = _run(qg, qtype, w, x, M, N)
    rows = np.unique(np.concatenate([_sample_rows(M, n=200, seed=3), np.arange(M - 12, M)]))
    rb = gs.row_bytes(qtype, N)
    ref, bnd = oracle_lib.gemv(qtype, w.reshape(M, rb)[rows], len(rows), N, x, threads=4)
    assert_within_bound(y[:, rows], ref, bnd, what=f"tall type {qtype} N={N}")
