"""Pins of the oracle's row dot, router, SwiGLU and combine to things other than itself.

- row dot: closed forms (x = 0, all-ones x on hand blocks, one-hot x gives a column),
  the T-token form equals T single-token calls, and the special case that reduces to a
  library matmul (numpy float64 on the dequantized matrix).
- router: brute force over all k-subsets on tiny inputs (with seeded ties), the full
  softmax when k = E (scipy), forced routing.
- SwiGLU: scipy's logistic function; closed forms.
- MoE: one-hot combine weights, linearity, and a tiny MoE recomputed with numpy matmuls
  on dequantized experts (gate rows before up rows, slot indirection, residual last).
"""
import itertools

import numpy as np
import pytest
from scipy.special import expit, softmax

import gguf_synth as gs

TYPES = [gs.Q8_0, gs.Q4_0, gs.Q4_K, gs.Q6_K]


@pytest.mark.parametrize("qtype", TYPES)
def test_gemv_matches_library_matmul(oracle_lib, qtype):
    M, N, T = 37, 512, 5
    w = gs.quant_blocks(qtype, M, N, seed=11)
    x = gs.activations(T, N, seed=11)
    y, b = oracle_lib.gemv(qtype, w, M, N, x)
    W = oracle_lib.dequant(qtype, w, M, N).astype(np.float64)
    ref = x.astype(np.float64) @ W.T
    assert y.shape == (T, M)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(b, np.abs(x.astype(np.float64)) @ np.abs(W).T, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("qtype", TYPES)
def test_gemv_closed_forms(oracle_lib, qtype):
    M, N = 9, 512
    w = gs.quant_blocks(qtype, M, N, seed=12)
    y0, b0 = oracle_lib.gemv(qtype, w, M, N, np.zeros((1, N), np.float32))
    assert not y0.any() and not b0.any()
    W = oracle_lib.dequant(qtype, w, M, N)
    # one-hot x returns column k exactly
    for k in (0, 1, 31, 32, 255, 256, N - 1):
        e = np.zeros((1, N), np.float32)
        e[0, k] = 1.0
        yk, _ = oracle_lib.gemv(qtype, w, M, N, e)
        assert np.array_equal(yk[0], W[:, k].astype(np.float64))
    # T tokens at once == T single-token calls
    x = gs.activations(16, N, seed=13)
    yT, bT = oracle_lib.gemv(qtype, w, M, N, x)
    for t in range(16):
        y1, b1 = oracle_lib.gemv(qtype, w, M, N, x[t:t + 1])
        assert np.array_equal(yT[t], y1[0]) and np.array_equal(bT[t], b1[0])


def test_gemv_hand_block_row_sums(oracle_lib):
    """Q8_0 block with d = 1, q_i = i - 16 sums to -16; a row of 8 such blocks against
    all-ones x gives -128; against x_i = i gives sum_i i*((i mod 32) - 16)."""
    blk = bytes.fromhex("003c" + bytes(np.arange(-16, 16, dtype=np.int8).view(np.uint8)).hex())
    row = np.frombuffer(blk * 8, dtype=np.uint8)
    y, _ = oracle_lib.gemv(gs.Q8_0, row, 1, 256, np.ones((1, 256), np.float32))
    assert y[0, 0] == -128.0
    xi = np.arange(256, dtype=np.float32)[None]
    y, _ = oracle_lib.gemv(gs.Q8_0, row, 1, 256, xi)
    assert y[0, 0] == sum(i * ((i % 32) - 16) for i in range(256))


def test_gemv_shapes_and_errors(oracle_lib):
    w = gs.quant_blocks(gs.Q8_0, 2, 64)
    with pytest.raises(ValueError):
        oracle_lib.gemv(gs.Q8_0, w, 2, 48, np.zeros((1, 48), np.float32))  # 48 % 32 != 0
    y, b = oracle_lib.gemv(gs.Q8_0, w, 0, 64, np.zeros((1, 64), np.float32))
    assert y.shape == (1, 0)


# ---- router ----------------------------------------------------------------------------

def _brute_topk(l, k):
    """Highest-sum k-subset; among equal sums, the subset whose sorted-descending logits
    list picks lower indices first (the greedy order with ties to the lowest index)."""
    best = None
    for sub in itertools.combinations(range(len(l)), k):
        key = (sum(l[i] for i in sub),)
        order = sorted(sub, key=lambda i: (-l[i], i))
        cand = (key, [-i for i in order])
        if best is None or cand > best[0]:
            best = (cand, order)
    return best[1]


def test_topk_brute_force_small(oracle_lib):
    rng = np.random.default_rng(0)
    for trial in range(300):
        E = int(rng.integers(2, 13))
        k = int(rng.integers(1, min(E, 4) + 1))
        if trial % 3 == 0:   # seeded ties: few distinct values
            l = rng.integers(0, 3, E).astype(np.float64)
        else:
            l = rng.normal(size=E)
        ids, w = oracle_lib.topk(l[None], k)
        assert ids[0].tolist() == _brute_topk(l.tolist(), k)
        p = softmax(l)
        np.testing.assert_allclose(w[0], p[ids[0]] / p[ids[0]].sum(), rtol=1e-13)


def test_topk_full_softmax_and_forced(oracle_lib):
    l = np.random.default_rng(1).normal(size=(3, 128)) * 3
    ids, w = oracle_lib.topk(l, 128)
    for t in range(3):
        assert sorted(ids[t].tolist()) == list(range(128))
        np.testing.assert_allclose(w[t], softmax(l[t])[ids[t]], rtol=1e-12)
        assert abs(w[t].sum() - 1.0) < 1e-14
    # forced routing: one logit 10 above the rest is picked first
    l2 = np.zeros((1, 128))
    l2[0, 77] = 10.0
    ids, w = oracle_lib.topk(l2, 8)
    assert ids[0].tolist() == [77, 0, 1, 2, 3, 4, 5, 6]
    np.testing.assert_allclose(w[0, 0], np.exp(10) / (np.exp(10) + 7), rtol=1e-14)


def test_router_logits_library(oracle_lib):
    xn = gs.activations(4, 2048, seed=2)
    wr = gs.router_weights(128, 2048, seed=2)
    lg, b = oracle_lib.router_logits(xn, wr)
    np.testing.assert_allclose(lg, xn.astype(np.float64) @ wr.astype(np.float64).T, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(b, np.abs(xn.astype(np.float64)) @ np.abs(wr.astype(np.float64)).T, rtol=1e-12)


def test_swiglu(oracle_lib):
    for g, u in [(0.0, 5.0), (1.5, -2.0), (-3.0, 0.25), (30.0, 1.0), (-30.0, 1.0), (7.0, 0.0)]:
        assert oracle_lib.swiglu1(g, u) == pytest.approx(g * expit(g) * u, rel=1e-15, abs=1e-300)
    assert oracle_lib.swiglu1(0.0, 123.0) == 0.0


# ---- MoE -------------------------------------------------------------------------------

def _tiny_moe(qtype=gs.Q8_0, E=6, H=64, F=32, T=3, k=2, seed=4):
    go, uo, do, stride = gs.moe_expert_record_layout(H, F, qtype)
    ex = gs.moe_experts(E, H, F, qtype, seed=seed)
    wr = gs.router_weights(E, H, seed=seed) * 20
    xn = gs.activations(T, H, seed=seed, stream=5)
    x = gs.activations(T, H, seed=seed, stream=6)
    return ex, (go, uo, do, stride), wr, xn, x


@pytest.mark.parametrize("qtype", [gs.Q8_0, gs.Q4_0])
def test_moe_layer_against_library_matmuls(oracle_lib, qtype):
    E, H, F, T, k = 6, 64, 32, 3, 2
    ex, (go, uo, do, stride), wr, xn, x = _tiny_moe(qtype, E, H, F, T, k)
    slots = np.array([3, 0, 5, 1, 4, 2], np.int32)   # expert e lives in record slots[e]
    r = oracle_lib.moe_layer(qtype, ex, go, uo, do, stride, wr, xn, x, k, H, F, slots=slots)
    # numpy restatement with dequantized experts
    lg = xn.astype(np.float64) @ wr.astype(np.float64).T
    out = x.astype(np.float64).copy()
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-lg[t, e], e))[:k]
        assert r["ids"][t].tolist() == order
        p = softmax(lg[t])[order]
        p = p / p.sum()
        acc = np.zeros(H)
        for j, e in enumerate(order):
            rec = ex.reshape(E, stride)[slots[e]]
            Wg = oracle_lib.dequant(qtype, rec[go:uo], F, H).astype(np.float64)
            Wu = oracle_lib.dequant(qtype, rec[uo:do], F, H).astype(np.float64)
            Wd = oracle_lib.dequant(qtype, rec[do:stride], H, F).astype(np.float64)
            g, u = Wg @ xn[t].astype(np.float64), Wu @ xn[t].astype(np.float64)
            act = g * expit(g) * u
            np.testing.assert_allclose(r["act"][t * k + j], act, rtol=1e-12, atol=1e-15)
            acc += p[j] * (Wd @ act)
        out[t] += acc
    np.testing.assert_allclose(r["out"], out, rtol=1e-11, atol=1e-13)


def test_moe_combine_one_hot_and_linearity(oracle_lib):
    E, H, F, T, k = 5, 64, 32, 2, 3
    ex, (go, uo, do, stride), wr, xn, x = _tiny_moe(gs.Q8_0, E, H, F, T, k)
    ids = np.array([[4, 0, 2], [1, 3, 0]], np.int32)
    act = gs.activations(T * k, F, seed=9).astype(np.float64)
    exd = ex.reshape(-1)[do:]
    for j in range(k):
        wts = np.zeros((T, k))
        wts[:, j] = 1.0
        dn, _, out, _ = oracle_lib.moe_down_combine(gs.Q8_0, exd, stride, None, ids, wts, act, x, k, H, F)
        np.testing.assert_array_equal(out, x.astype(np.float64) + dn[j::k])
    w1 = np.random.default_rng(0).random((T, k))
    w2 = np.random.default_rng(1).random((T, k))
    o1 = oracle_lib.moe_down_combine(gs.Q8_0, exd, stride, None, ids, w1, act, x, k, H, F, add_residual=0)[2]
    o2 = oracle_lib.moe_down_combine(gs.Q8_0, exd, stride, None, ids, w2, act, x, k, H, F, add_residual=0)[2]
    o12 = oracle_lib.moe_down_combine(gs.Q8_0, exd, stride, None, ids, w1 + w2, act, x, k, H, F,
                                      add_residual=0)[2]
    np.testing.assert_allclose(o12, o1 + o2, rtol=1e-12, atol=1e-12)


def test_moe_gate_before_up(oracle_lib):
    """The SiLU takes the gate rows: zeroing the gate's codes zeroes the activation, zeroing
    the up rows' codes too; swapping the two bases changes the result."""
    E, H, F, T, k = 2, 64, 32, 1, 1
    ex, (go, uo, do, stride), wr, xn, x = _tiny_moe(gs.Q8_0, E, H, F, T, k)
    ids = np.array([[1]], np.int32)
    exz = ex.copy().reshape(E, stride)
    blocks = exz[:, go:uo].reshape(E, -1, 34)
    blocks[:, :, 2:] = 0                      # gate codes all zero -> gate = 0 -> act = 0
    exz[:, go:uo] = blocks.reshape(E, -1)
    flat = exz.reshape(-1)
    g, u, act, _, _ = oracle_lib.moe_gate_up(gs.Q8_0, flat[go:], flat[uo:], stride, None, ids, xn, k, H, F)
    assert not g.any() and not act.any() and u.any()
    g2, u2, act2, _, _ = oracle_lib.moe_gate_up(gs.Q8_0, flat[uo:], flat[go:], stride, None, ids, xn, k, H, F)
    assert np.array_equal(g2, u) and not u2.any()
