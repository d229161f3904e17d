"""GPU parity of the MoE variants through the C ABI: GELU-tanh experts (geglu), the per-expert
down scale (moeSum), the sigmoid-gated shared expert (moeAccumShared), the whole layer with a
variant, and the router's scaled RMSNorm (rmsnormK).

- act against the oracle's GELU of its own gate/up rows, the GEMV bound carried through
  GELU-tanh's derivative (plus a few f32 roundings of tanh and the products);
- the combine against the oracle's combine fed the GPU's act and weights;
- more than 16 tokens (Q8_0, tensor cores): the same at the prefill bar."""
import numpy as np
import pytest

import gguf_synth as gs
from helpers import ABS, REL, assert_within_bound, to_dev
from test_moe_gpu import Experts, _rand_ids, _route, _ws, check_route

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

PREFILL_REL = 2e-3


@pytest.fixture(scope="module")
def qg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gguf_block_dequant_gb300 as qg
    from gguf_block_dequant_gb300 import build

    build.build()
    qg.load()
    return qg


def _gelu_act_bound(g, u, bg, bu, rel=REL):
    eg = rel * bg + ABS
    eu = rel * bu + ABS
    a = 0.7978845608 * g * (1.0 + 0.044715 * g * g)
    inside = np.abs(a) < 10.0
    th = np.tanh(np.clip(a, -10, 10))
    da = 0.7978845608 * (1.0 + 3 * 0.044715 * g * g) * inside
    gelu = 0.5 * g * (1.0 + th)
    dgelu = 0.5 * (1.0 + th) + 0.5 * g * (1.0 - th * th) * da
    act = gelu * u
    # first order in the gate and up errors, then the second-order terms (|gelu''| <= 0.8,
    # |gelu'| <= 1.13), then f32 rounding of tanh and the products and the bar's absolute term
    return (np.abs(dgelu * u) * eg + np.abs(gelu) * eu + 1.13 * eg * eu + 0.4 * eg * eg * np.abs(u) +
            1e-6 * (np.abs(act) + 0.5 * np.abs(g * u)) + ABS)


def _check_gelu_act(oracle_lib, ex, ids, xn, k, act, rel=REL, what=""):
    g, u, _, bg, bu = oracle_lib.moe_gate_up(ex.qtype, ex.host[ex.offs[0]:], ex.host[ex.offs[1]:], ex.stride, None,
                                             ids, xn, k, ex.H, ex.F, threads=8)
    ref = oracle_lib.moe_act(oracle_lib.ACT_GELU_TANH, g, u)
    lim = _gelu_act_bound(g, u, bg, bu, rel)
    err = np.abs(act.astype(np.float64) - ref)
    assert np.isfinite(act).all(), what
    bad = err > lim
    assert not bad.any(), f"{what}: {bad.sum()} act elements out of bound, worst {(err / lim).max():.2f}x"


def _variant_inputs(ex, T, seed):
    rng = np.random.default_rng(seed)
    ds = rng.uniform(-2.0, 2.0, ex.E).astype(np.float32)
    sh = rng.standard_normal((T, ex.H)).astype(np.float32)
    sg = rng.uniform(-4.0, 4.0, T).astype(np.float32)
    return ds, sh, sg


def _check_combine_ex(oracle_lib, ex, ids, wts, act, x, k, out, ds, sh, sg, rel=REL, what=""):
    dn, bdn, _, _ = oracle_lib.moe_down_combine(ex.qtype, ex.host[ex.offs[2]:], ex.stride, None, ids, wts, act, x, k,
                                                ex.H, ex.F, 1, threads=8)
    ref, bnd = oracle_lib.moe_combine_ex(ids, wts, dn, bdn, x, k, ex.H, add_residual=1, down_scale=ds, E=ex.E,
                                         shared_out=sh, shared_gate=sg)
    assert_within_bound(out, ref, bnd, rel=rel, what=f"{what} combine")


# the Gemma-4-shaped experts (hidden 2816) at T <= 8: the T <= 16 expert kernel keeps every
# token's activation row in shared memory, and 16 rows of 2816 do not fit beside its ring
@pytest.mark.parametrize("qtype,H,F,E,k,T", [(q, 512, 96 if q != gs.Q6_K else 256, 16, 4, T)
                                             for q in (gs.Q4_0, gs.Q8_0, gs.Q6_K) for T in (1, 3, 16)] +
                         [(gs.Q4_0, 2816, 704, 128, 8, T) for T in (1, 3, 8)])
def test_gelu_experts_down_scale_and_shared_expert(qg, oracle_lib, qtype, H, F, E, k, T):
    ex = Experts(qtype, E, H, F, seed=qtype + T)
    ids = _rand_ids(T, k, E, seed=T + 1)
    xn = gs.activations(T, H, seed=T, stream=31)
    gate, up, down = ex.bases()
    act = torch.full((T * k, F), float("nan"), dtype=torch.float32, device="cuda")
    ws = _ws(qg, T, k, E, H, F)
    v = qg.moe_variant(act=qg.ACT_GELU_TANH)
    qg.moe_expert_act(qtype, gate, up, ex.stride, None, E, E, to_dev(ids, torch), to_dev(xn, torch), T, k, H, F, v, act,
                      ws)
    torch.cuda.synchronize()
    assert qg.device_status() == 0
    act_h = act.cpu().numpy()
    _check_gelu_act(oracle_lib, ex, ids, xn, k, act_h, what=f"gelu type {qtype} T={T}")
    wts = np.random.default_rng(T).random((T, k)).astype(np.float32)
    x = gs.activations(T, H, seed=T, stream=32)
    ds, sh, sg = _variant_inputs(ex, T, seed=T)
    dsd, shd, sgd = to_dev(ds, torch), to_dev(sh, torch), to_dev(sg, torch)
    for with_shared in (False, True):
        var = qg.moe_variant(act=qg.ACT_GELU_TANH, down_scale=dsd, shared_out=shd if with_shared else None,
                             shared_gate=sgd if with_shared else None)
        xd = to_dev(x, torch)
        qg.moe_combine_ex(qtype, down, ex.stride, None, E, E, to_dev(ids, torch), to_dev(wts, torch), act, T, k, H, F,
                          var, xd, 1, ws)
        torch.cuda.synchronize()
        assert qg.device_status() == 0
        _check_combine_ex(oracle_lib, ex, ids, wts, act_h, x, k, xd.cpu().numpy(), ds, sh if with_shared else None,
                          sg if with_shared else None, what=f"type {qtype} T={T} shared={with_shared}")


def test_variants_more_than_16_tokens(qg, oracle_lib):
    """T = 40 Q8_0: the grouped tensor-core expert steps with the GELU epilogue and the
    variant combine, at the prefill bar."""
    qtype, H, F, E, k, T = gs.Q8_0, 512, 256, 16, 4, 40
    ex = Experts(qtype, E, H, F, seed=3)
    ids = _rand_ids(T, k, E, seed=9)
    xn = gs.activations(T, H, seed=4, stream=33)
    gate, up, down = ex.bases()
    act = torch.full((T * k, F), float("nan"), dtype=torch.float32, device="cuda")
    ws = _ws(qg, T, k, E, H, F)
    qg.moe_expert_act(qtype, gate, up, ex.stride, None, E, E, to_dev(ids, torch), to_dev(xn, torch), T, k, H, F,
                      qg.moe_variant(act=qg.ACT_GELU_TANH), act, ws)
    torch.cuda.synchronize()
    assert qg.device_status() == 0
    act_h = act.cpu().numpy()
    _check_gelu_act(oracle_lib, ex, ids, xn, k, act_h, rel=PREFILL_REL, what="gelu T=40")
    wts = np.random.default_rng(5).random((T, k)).astype(np.float32)
    x = gs.activations(T, H, seed=5, stream=34)
    ds, sh, sg = _variant_inputs(ex, T, seed=6)
    var = qg.moe_variant(act=qg.ACT_GELU_TANH, down_scale=to_dev(ds, torch), shared_out=to_dev(sh, torch),
                         shared_gate=to_dev(sg, torch))
    xd = to_dev(x, torch)
    qg.moe_combine_ex(qtype, down, ex.stride, None, E, E, to_dev(ids, torch), to_dev(wts, torch), act, T, k, H, F, var,
                      xd, 1, ws)
    torch.cuda.synchronize()
    assert qg.device_status() == 0
    _check_combine_ex(oracle_lib, ex, ids, wts, act_h, x, k, xd.cpu().numpy(), ds, sh, sg, rel=PREFILL_REL,
                      what="T=40")


@pytest.mark.parametrize("T", [1, 4])
def test_moe_layer_ex_gemma_like(qg, oracle_lib, T):
    """A Gemma-4-like layer: Q4_0 experts, GELU, per-expert down scale, router on the scaled
    RMSNorm of the residual stream (qg_rmsnorm with k = 1/sqrt(H)); and the same call with a
    shared expert.  Stage by stage against the oracle, as the Qwen3 layer test does."""
    qtype, H, F, E, k = gs.Q4_0, 1024, 352, 32, 8
    ex = Experts(qtype, E, H, F, seed=11)
    gate, up, down = ex.bases()
    x = gs.activations(T, H, seed=T, stream=35)
    gw = np.random.default_rng(2).uniform(0.5, 1.5, H).astype(np.float32)
    xn_d = torch.empty((T, H), dtype=torch.float32, device="cuda")
    kf = float(np.float32(1.0 / np.sqrt(H)))
    qg.rmsnorm(to_dev(x, torch), to_dev(gw, torch), 1e-6, xn_d, k=kf)
    torch.cuda.synchronize()
    xn = xn_d.cpu().numpy()
    ref = oracle_lib.rmsnorm_k(x, gw, 1e-6, kf)
    ms = np.mean(x.astype(np.float64) ** 2, axis=1, keepdims=True)
    assert_within_bound(xn, ref, np.abs(x.astype(np.float64) * gw * kf) / np.sqrt(ms + 1e-6), what="router rmsnormK")
    wr = gs.router_weights(E, H, seed=3)
    ds, sh, sg = _variant_inputs(ex, T, seed=12)
    for with_shared in (False, True):
        var = qg.moe_variant(act=qg.ACT_GELU_TANH, down_scale=to_dev(ds, torch),
                             shared_out=to_dev(sh, torch) if with_shared else None,
                             shared_gate=to_dev(sg, torch) if with_shared else None)
        ids = torch.zeros((T, k), dtype=torch.int32, device="cuda")
        wts = torch.zeros((T, k), dtype=torch.float32, device="cuda")
        act = torch.zeros((T * k, F), dtype=torch.float32, device="cuda")
        xd = to_dev(x, torch)
        ws = _ws(qg, T, k, E, H, F)
        qg.moe_layer_ex(qtype, xn_d, to_dev(wr, torch), gate, up, down, ex.stride, None, E, T, H, F, E, k, var, ids, wts,
                        act, xd, ws)
        torch.cuda.synchronize()
        assert qg.device_status() == 0
        ids_h, wts_h, act_h = ids.cpu().numpy(), wts.cpu().numpy(), act.cpu().numpy()
        i2, w2, lg = _route(qg, xn, wr, k)
        assert np.array_equal(i2, ids_h) and np.array_equal(w2, wts_h)
        check_route(oracle_lib, xn, wr, k, ids_h, wts_h, lg, what=f"gemma layer T={T}")
        _check_gelu_act(oracle_lib, ex, ids_h, xn, k, act_h, what=f"gemma layer T={T}")
        _check_combine_ex(oracle_lib, ex, ids_h, wts_h, act_h, x, k, xd.cpu().numpy(), ds,
                          sh if with_shared else None, sg if with_shared else None, what=f"gemma layer T={T}")


def test_moe_layer_ex_default_variant_is_moe_layer(qg):
    """A NULL variant and a default one give moe_layer's result, bit for bit (the one-token
    launch at T = 1)."""
    qtype, H, F, E, k, T = gs.Q8_0, 512, 96, 16, 4, 1
    ex = Experts(qtype, E, H, F, seed=21)
    gate, up, down = ex.bases()
    xn = to_dev(gs.activations(T, H, seed=1, stream=36), torch)
    wr = to_dev(gs.router_weights(E, H, seed=4), torch)
    x = gs.activations(T, H, seed=2, stream=37)
    outs = []
    for mode in ("layer", "ex_null", "ex_default"):
        ids = torch.zeros((T, k), dtype=torch.int32, device="cuda")
        wts = torch.zeros((T, k), dtype=torch.float32, device="cuda")
        act = torch.zeros((T * k, F), dtype=torch.float32, device="cuda")
        xd = to_dev(x, torch)
        ws = _ws(qg, T, k, E, H, F)
        if mode == "layer":
            qg.moe_layer(qtype, xn, wr, gate, up, down, ex.stride, None, E, T, H, F, E, k, ids, wts, act, xd, ws)
        else:
            var = None if mode == "ex_null" else qg.moe_variant()
            qg.moe_layer_ex(qtype, xn, wr, gate, up, down, ex.stride, None, E, T, H, F, E, k, var, ids, wts, act, xd,
                            ws)
        torch.cuda.synchronize()
        outs.append(xd.cpu().numpy())
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])
    assert qg.device_status() == 0
