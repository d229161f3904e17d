"""Pins of the oracle's MoE variants (GELU-tanh experts, per-expert down scale, sigmoid-gated
shared expert, the router's scaled RMSNorm) to things other than themselves.

- GELU-tanh: the identity gelu(x) - gelu(-x) = x of the tanh form (the clamp is odd, so it
  holds beyond it too), within 1e-3 of the exact GELU x * Phi(x) (scipy's normal CDF) where the
  tanh form approximates it, gelu(0) = 0, and the page's clamp at |a| = 10.
- sigmoid: scipy's logistic function.
- combine variants: with no scale and no shared expert the combine equals the pinned MoE
  combine exactly; one-hot pick weights give one scaled down row; the shared gate at 0 and at
  +-60 gives half, all or none of the shared row.
- scaled RMSNorm: k = 1 is RMSNorm exactly, k a power of two scales it exactly.
"""
import numpy as np
import pytest
from scipy.special import expit, ndtr

import gguf_synth as gs


def test_gelu_tanh_identities_and_exact_gelu(oracle_lib):
    xs = np.concatenate([np.linspace(-12, 12, 241), [0.0, 1e-8, -1e-8, 35.0, -35.0]])
    for x in xs:
        g, gm = oracle_lib.gelu_tanh(x), oracle_lib.gelu_tanh(-x)
        assert g - gm == pytest.approx(x, abs=1e-12 * max(1.0, abs(x)))
        if abs(x) <= 6:
            assert abs(g - x * ndtr(x)) <= 1e-3
    assert oracle_lib.gelu_tanh(0.0) == 0.0
    # the page clamps the tanh argument at 10: for x = 20 the result is 10 (1 + tanh 10), not 20
    assert oracle_lib.gelu_tanh(20.0) == pytest.approx(10.0 * (1.0 + np.tanh(10.0)), rel=1e-15)
    assert oracle_lib.gelu_tanh(20.0) < 20.0


def test_sigmoid_matches_scipy(oracle_lib):
    for x in np.linspace(-30, 30, 121):
        assert oracle_lib.sigmoid(x) == pytest.approx(float(expit(x)), rel=1e-14, abs=1e-300)


def test_moe_act_kinds(oracle_lib):
    rng = np.random.default_rng(2)
    g = rng.standard_normal(500) * 3
    u = rng.standard_normal(500)
    silu = oracle_lib.moe_act(oracle_lib.ACT_SILU, g, u)
    assert np.allclose(silu, g * expit(g) * u, rtol=1e-13, atol=1e-300)
    gelu = oracle_lib.moe_act(oracle_lib.ACT_GELU_TANH, g, u)
    assert np.all(np.abs(gelu - g * ndtr(g) * u) <= 1e-3 * np.abs(u) + 1e-300)
    with pytest.raises(ValueError):
        oracle_lib.moe_act(2, g, u)


def _tiny(seed=1, T=3, k=2, E=5, H=64, F=32):
    rng = np.random.default_rng(seed)
    w_down = gs.quant_blocks(gs.Q8_0, E * H, F, seed=seed, stream=41)
    stride = gs.tensor_bytes(gs.Q8_0, H, F)
    ids = np.array([[(t + j) % E for j in range(k)] for t in range(T)], dtype=np.int32)
    wts = rng.uniform(0.1, 1.0, (T, k))
    act = rng.standard_normal((T * k, F))
    x = rng.standard_normal((T, H)).astype(np.float32)
    return w_down, stride, ids, wts, act, x, T, k, E, H, F


def test_combine_ex_reduces_to_the_pinned_combine(oracle_lib):
    w_down, stride, ids, wts, act, x, T, k, E, H, F = _tiny()
    dn, bdn, out, bout = oracle_lib.moe_down_combine(gs.Q8_0, w_down, stride, None, ids, wts, act, x, k, H, F)
    out2, bout2 = oracle_lib.moe_combine_ex(ids, wts, dn, bdn, x, k, H)
    assert np.array_equal(out, out2) and np.array_equal(bout, bout2)


def test_combine_ex_down_scale_and_shared_expert_closed_forms(oracle_lib):
    w_down, stride, ids, wts, act, x, T, k, E, H, F = _tiny(seed=3)
    dn, bdn, _, _ = oracle_lib.moe_down_combine(gs.Q8_0, w_down, stride, None, ids, wts, act, x, k, H, F)
    ds = np.array([0.5, 2.0, -1.0, 4.0, 0.25], dtype=np.float32)
    onehot = np.zeros((T, k))
    onehot[:, 1] = 1.0
    out, _ = oracle_lib.moe_combine_ex(ids, onehot, dn, bdn, x, k, H, add_residual=0, down_scale=ds, E=E)
    for t in range(T):
        z = t * k + 1
        assert np.array_equal(out[t], dn[z] * float(ds[ids[t, 1]]))
    sh = np.random.default_rng(4).standard_normal((T, H)).astype(np.float32)
    base, _ = oracle_lib.moe_combine_ex(ids, wts, dn, bdn, x, k, H, down_scale=ds, E=E)
    for gate, frac in ((0.0, 0.5), (60.0, 1.0), (-60.0, 0.0)):
        sg = np.full(T, gate, dtype=np.float32)
        got, _ = oracle_lib.moe_combine_ex(ids, wts, dn, bdn, x, k, H, down_scale=ds, E=E, shared_out=sh,
                                           shared_gate=sg)
        want_no_res = (base - x.astype(np.float64)) + frac * sh.astype(np.float64)
        assert np.allclose(got - x.astype(np.float64), want_no_res, rtol=1e-12, atol=1e-20)


def test_rmsnorm_k_closed_forms(oracle_lib):
    rng = np.random.default_rng(9)
    x = rng.standard_normal((2, 2048)).astype(np.float32)
    w = rng.uniform(0.5, 1.5, 2048).astype(np.float32)
    assert np.array_equal(oracle_lib.rmsnorm_k(x, w, 1e-6, 1.0), oracle_lib.rmsnorm(x, w, 1e-6))
    assert np.array_equal(oracle_lib.rmsnorm_k(x, w, 1e-6, 0.125), oracle_lib.rmsnorm(x, w, 1e-6) * 0.125)
