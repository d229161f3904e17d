"""Parity of the MoE step (moe_route_topk, moe_expert_swiglu, moe_combine, moe_layer) with the
CPU oracle, through the C ABI.

Stage-wise checks, as the oracle's readings fix them:
  - router logits within 1e-5 * sum|w x| + 1e-6; top-k ids bit-exact wherever the oracle's
    logit gaps around the picks exceed the two logits' error bounds, and otherwise the GPU ids
    must be exactly the top-k of the GPU's own logits (several answers are then correct);
    weights against the oracle's softmax-over-picks of the GPU logits;
  - act against the oracle's SwiGLU of its own gate/up rows, the GEMV bound propagated
    through silu(g) * u;
  - the combine against the oracle run on the GPU's act and weights.
"""
import numpy as np
import pytest

import gguf_synth as gs
from helpers import ABS, REL, assert_within_bound, to_dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gguf_block_dequant_gb300 as qg
    from gguf_block_dequant_gb300 import build

    build.build()
    qg.load()
    return qg


def _ws(qg, T, k, E, H, F):
    n = qg.moe_workspace_size(T, k, E, H, F)
    assert n > 0
    return torch.zeros(n, dtype=torch.uint8, device="cuda")


# ---- router ----------------------------------------------------------------------------------

def _route(qg, xn, wr, k):
    T, H = xn.shape
    E = wr.shape[0]
    ids = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    wts = torch.full((T, k), float("nan"), dtype=torch.float32, device="cuda")
    lg = torch.full((T, E), float("nan"), dtype=torch.float32, device="cuda")
    ws = _ws(qg, T, k, E, H, 32)
    qg.moe_route_topk(to_dev(xn, torch), to_dev(wr, torch), T, H, E, k, ids, wts, lg, ws)
    torch.cuda.synchronize()
    assert qg.device_status() == 0
    return ids.cpu().numpy(), wts.cpu().numpy(), lg.cpu().numpy()


def check_route(oracle_lib, xn, wr, k, ids, wts, lg, what=""):
    ref_lg, bnd = oracle_lib.router_logits(xn, wr)
    assert_within_bound(lg, ref_lg, bnd, what=f"{what} logits")
    tol = REL * bnd + ABS
    # the GPU's picks are the exact top-k of its own logits, with their weights
    own_ids, own_w = oracle_lib.topk(lg.astype(np.float64), k)
    assert np.array_equal(ids, own_ids), f"{what}: ids are not the top-k of the GPU logits"
    assert np.allclose(wts, own_w, rtol=2e-6, atol=1e-7), f"{what}: weights"
    # where the oracle's order is clear of the error bounds, the ids are the oracle's
    ref_ids, _ = oracle_lib.topk(ref_lg, k)
    stable = 0
    for t in range(ref_lg.shape[0]):
        order = np.lexsort((np.arange(ref_lg.shape[1]), -ref_lg[t]))
        top = order[:min(k + 1, len(order))]
        gaps = ref_lg[t, top[:-1]] - ref_lg[t, top[1:]]
        if np.all(gaps > tol[t, top[:-1]] + tol[t, top[1:]]):
            stable += 1
            assert np.array_equal(ids[t], ref_ids[t]), f"{what}: token {t} ids differ from the oracle"
    return stable


@pytest.mark.parametrize("T", [1, 3, 8, 16, 33, 512])
def test_router_qwen3_moe_shape(qg, oracle_lib, T):
    H, E, k = gs.MOE_H, gs.MOE_E, gs.MOE_K
    xn = gs.activations(T, H, seed=T, stream=11)
    wr = gs.router_weights(E, H, seed=0)
    ids, wts, lg = _route(qg, xn, wr, k)
    stable = check_route(oracle_lib, xn, wr, k, ids, wts, lg, what=f"T={T}")
    assert stable >= 0.9 * T


@pytest.mark.parametrize("E,k", [(12, 4), (33, 1), (64, 32), (200, 8), (256, 16), (8, 8)])
def test_router_other_shapes(qg, oracle_lib, E, k):
    T, H = 5, 96
    xn = gs.activations(T, H, seed=E, stream=12)
    wr = gs.router_weights(E, H, seed=E)
    ids, wts, lg = _route(qg, xn, wr, k)
    check_route(oracle_lib, xn, wr, k, ids, wts, lg, what=f"E={E} k={k}")
    if k == E:  # every expert picked: the weights are the full softmax
        assert np.allclose(wts.sum(axis=1), 1.0, rtol=1e-6)


@pytest.mark.parametrize("T,E,H", [(512, 128, 2048), (64, 200, 96), (77, 33, 3072)])
def test_router_many_tiles_same_logits_as_one_tile_calls(qg, T, E, H):
    """From four 16-token tiles on, the router stages each tile in shared memory and runs a share
    of the experts over it; it sums every logit in the same order as the one-tile router, so the
    logits (and picks and weights) equal those of calls of at most 16 tokens, bit for bit."""
    k = min(8, E)
    xn = gs.activations(T, H, seed=T + E, stream=14)
    wr = gs.router_weights(E, H, seed=E)
    ids, wts, lg = _route(qg, xn, wr, k)
    for t0 in range(0, T, 16):
        sub = xn[t0:t0 + 16]
        ids1, wts1, lg1 = _route(qg, sub, wr, k)
        assert np.array_equal(lg[t0:t0 + 16].view(np.uint32), lg1.view(np.uint32)), t0
        assert np.array_equal(ids[t0:t0 + 16], ids1) and np.array_equal(wts[t0:t0 + 16], wts1), t0


def test_router_ties_go_to_the_lowest_id(qg, oracle_lib):
    """Identical router rows give bit-identical logits: the lower expert id is picked first."""
    T, H, E, k = 4, 128, 12, 4
    wr = gs.router_weights(E, H, seed=3)
    wr[7] = wr[2]
    wr[9] = wr[2]
    xn = gs.activations(T, H, seed=3)
    xn[:, :] = np.sign(wr[2])[None, :] * np.abs(xn)  # makes expert 2 (and 7, 9) score highest
    ids, wts, lg = _route(qg, xn, wr, k)
    for t in range(T):
        assert lg[t, 2] == lg[t, 7] == lg[t, 9]
        assert list(ids[t, :3]) == [2, 7, 9]
        assert wts[t, 0] == wts[t, 1] == wts[t, 2]
    check_route(oracle_lib, xn, wr, k, ids, wts, lg, what="ties")


# ---- experts ---------------------------------------------------------------------------------

class Experts:
    """E expert records (gate || up || down) as one device buffer, plus optional slot map."""

    def __init__(self, qtype, E, H, F, n_slots=None, seed=0):
        self.qtype, self.E, self.H, self.F = qtype, E, H, F
        n_slots = n_slots or E
        self.n_slots = n_slots
        go, uo, do, stride = gs.moe_expert_record_layout(H, F, qtype)
        self.offs, self.stride = (go, uo, do), stride
        self.host = gs.moe_experts(n_slots, H, F, qtype, seed=seed).reshape(-1)
        self.dev = to_dev(self.host, torch)

    def bases(self):
        return [self.dev[o:] for o in self.offs]


def _act_bound(g, u, bg, bu):
    """|act_gpu - act_oracle| bound: the gate/up GEMV bound carried through silu(g) * u, plus
    a few f32 roundings of the SwiGLU itself."""
    eg = REL * bg + ABS
    eu = REL * bu + ABS
    sig = 1.0 / (1.0 + np.exp(-g))
    ds = sig * (1.0 + g * (1.0 - sig))
    act = g * sig * u
    return np.abs(ds * u) * eg + np.abs(g * sig) * eu + 6e-7 * np.abs(act) + 1e-30


def _rand_ids(T, k, E, seed):
    rng = np.random.default_rng(seed)
    return np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)


def run_swiglu(qg, ex, ids, xn, k, slots=None):
    T = xn.shape[0]
    gate, up, _ = ex.bases()
    act = torch.full((T * k, ex.F), float("nan"), dtype=torch.float32, device="cuda")
    sl = None if slots is None else to_dev(slots.astype(np.int32), torch)
    qg.moe_expert_swiglu(ex.qtype, gate, up, ex.stride, sl, ex.n_slots, ex.E, to_dev(ids, torch), to_dev(xn, torch),
                         T, k, ex.H, ex.F, act)
    torch.cuda.synchronize()
    return act.cpu().numpy()


def check_swiglu(oracle_lib, ex, ids, xn, k, act, slots=None, what=""):
    g, u, ref, bg, bu = oracle_lib.moe_gate_up(ex.qtype, ex.host[ex.offs[0]:], ex.host[ex.offs[1]:], ex.stride,
                                               slots, ids, xn, k, ex.H, ex.F, threads=8)
    lim = _act_bound(g, u, bg, bu)
    err = np.abs(act.astype(np.float64) - ref)
    assert np.isfinite(act).all(), what
    bad = err > lim
    assert not bad.any(), f"{what}: {bad.sum()} act elements out of bound, worst {(err / lim).max():.2f}x"


def run_combine(qg, ex, ids, wts, act, x, k, add_residual=1, slots=None, ws=None):
    T, H = x.shape
    _, _, down = ex.bases()
    xd = to_dev(x, torch)
    ws = ws if ws is not None else _ws(qg, T, k, ex.E, H, ex.F)
    sl = None if slots is None else to_dev(slots.astype(np.int32), torch)
    qg.moe_combine(ex.qtype, down, ex.stride, sl, ex.n_slots, ex.E, to_dev(ids, torch), to_dev(wts, torch),
                   to_dev(act, torch), T, k, H, ex.F, xd, add_residual, ws)
    torch.cuda.synchronize()
    return xd.cpu().numpy()


def check_combine(oracle_lib, ex, ids, wts, act, x, k, out, add_residual=1, slots=None, what=""):
    _, _, ref, bnd = oracle_lib.moe_down_combine(ex.qtype, ex.host[ex.offs[2]:], ex.stride, slots, ids, wts, act, x,
                                                 k, ex.H, ex.F, add_residual, threads=8)
    assert_within_bound(out, ref, bnd, what=f"{what} combine")


SMALL = {gs.Q8_0: (512, 96), gs.Q4_0: (512, 96), gs.Q4_K: (512, 256), gs.Q6_K: (512, 256)}


@pytest.mark.parametrize("qtype", [gs.Q8_0, gs.Q4_0, gs.Q4_K, gs.Q6_K])
@pytest.mark.parametrize("T", [1, 2, 3, 5, 8, 16])
def test_experts_small(qg, oracle_lib, qtype, T):
    H, F = SMALL[qtype]
    E, k = 16, 4
    ex = Experts(qtype, E, H, F, seed=qtype)
    ids = _rand_ids(T, k, E, seed=T)
    xn = gs.activations(T, H, seed=T, stream=21)
    act = run_swiglu(qg, ex, ids, xn, k)
    assert qg.device_status() == 0
    check_swiglu(oracle_lib, ex, ids, xn, k, act, what=f"type {qtype} T={T}")
    rng = np.random.default_rng(T)
    wts = rng.random((T, k)).astype(np.float32)
    x = gs.activations(T, H, seed=T, stream=22)
    out = run_combine(qg, ex, ids, wts, act, x, k)
    assert qg.device_status() == 0
    check_combine(oracle_lib, ex, ids, wts, act, x, k, out, what=f"type {qtype} T={T}")


def test_experts_slot_map_and_repeated_ids(qg, oracle_lib):
    """Experts in permuted pool slots, and a token that picks the same expert twice."""
    H, F, E, k, T = 256, 64, 10, 3, 4
    ex = Experts(gs.Q8_0, E, H, F, n_slots=13, seed=5)
    slots = np.random.default_rng(1).permutation(13)[:E].astype(np.int32)
    ids = _rand_ids(T, k, E, seed=2)
    ids[1] = [4, 4, 9]
    xn = gs.activations(T, H, seed=6)
    act = run_swiglu(qg, ex, ids, xn, k, slots=slots)
    check_swiglu(oracle_lib, ex, ids, xn, k, act, slots=slots, what="slots")
    wts = np.full((T, k), 0.25, np.float32)
    x = gs.activations(T, H, seed=7)
    for res in (1, 0):
        out = run_combine(qg, ex, ids, wts, act, x, k, add_residual=res, slots=slots)
        check_combine(oracle_lib, ex, ids, wts, act, x, k, out, add_residual=res, slots=slots, what=f"slots res={res}")
    assert qg.device_status() == 0


def test_experts_bad_ids_flagged(qg, oracle_lib):
    """An out-of-range id sets the device status; that pair's act row is zero and the combine
    skips it."""
    H, F, E, k, T = 256, 64, 8, 2, 3
    ex = Experts(gs.Q8_0, E, H, F, seed=8)
    ids = _rand_ids(T, k, E, seed=3)
    ids[2, 1] = E + 5
    xn = gs.activations(T, H, seed=9)
    act = run_swiglu(qg, ex, ids, xn, k)
    assert qg.device_status() & (1 << qg.QG_EDEVICE_ID)
    assert (act[2 * k + 1] == 0).all()
    good = [z for z in range(T * k) if z != 2 * k + 1]
    ids_ok = ids.copy()
    ids_ok[2, 1] = ids[2, 0]  # any valid id: its act row is all we compare
    g, u, ref, bg, bu = oracle_lib.moe_gate_up(ex.qtype, ex.host[ex.offs[0]:], ex.host[ex.offs[1]:], ex.stride, None,
                                               ids_ok, xn, k, H, F)
    lim = _act_bound(g, u, bg, bu)
    assert (np.abs(act[good] - ref[good]) <= lim[good]).all()
    wts = np.full((T, k), 0.5, np.float32)
    x = gs.activations(T, H, seed=10)
    out = run_combine(qg, ex, ids, wts, act, x, k)
    assert qg.device_status() & (1 << qg.QG_EDEVICE_ID)
    wts_ok = wts.copy()
    wts_ok[2, 1] = 0.0  # the skipped pick contributes nothing
    check_combine(oracle_lib, ex, ids_ok, wts_ok, act, x, k, out, what="bad id")


def test_moe_shape_errors(qg):
    d = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    f = torch.zeros(4096, dtype=torch.float32, device="cuda")
    i = torch.zeros(64, dtype=torch.int32, device="cuda")
    with pytest.raises(qg.QGError) as e:
        qg.moe_route_topk(f, f, 1, 64, 8, 33, i, f, None, d)   # k > 32
    assert e.value.status == qg.QG_EINVAL_SHAPE
    with pytest.raises(qg.QGError) as e:
        qg.moe_route_topk(f, f, 1, 64, 300, 8, i, f, None, d)  # E > 256
    assert e.value.status == qg.QG_EINVAL_SHAPE
    with pytest.raises(qg.QGError) as e:
        qg.moe_route_topk(f, f, 4, 64, 8, 2, i, f, None, d[:16])  # workspace too small
    assert e.value.status == qg.QG_EWORKSPACE
    with pytest.raises(qg.QGError) as e:  # more than 16 tokens needs rows in whole 256-element boxes
        qg.moe_expert_swiglu(gs.Q8_0, d, d, 0, None, 1, 8, i, f, 17, 2, 64, 32, f)
    assert e.value.status == qg.QG_EUNSUPPORTED


# ---- the Qwen3-30B-A3B-shaped layer ----------------------------------------------------------

@pytest.fixture(scope="module")
def a3b():
    return Experts(gs.Q8_0, gs.MOE_E, gs.MOE_H, gs.MOE_F, seed=0)


@pytest.mark.parametrize("T", [1, 8, 16])
def test_moe_layer_qwen3_30b_a3b(qg, oracle_lib, a3b, T):
    H, F, E, k = gs.MOE_H, gs.MOE_F, gs.MOE_E, gs.MOE_K
    ex = a3b
    wr = gs.router_weights(E, H, seed=0)
    xn = gs.activations(T, H, seed=T, stream=31)
    x = gs.activations(T, H, seed=T, stream=32)
    gate, up, down = ex.bases()
    ids = torch.zeros((T, k), dtype=torch.int32, device="cuda")
    wts = torch.zeros((T, k), dtype=torch.float32, device="cuda")
    act = torch.zeros((T * k, F), dtype=torch.float32, device="cuda")
    ws = _ws(qg, T, k, E, H, F)
    outs = []
    for _ in range(2):  # twice on one workspace: the counters must be back at zero
        xd = to_dev(x, torch)
        qg.moe_layer(gs.Q8_0, to_dev(xn, torch), to_dev(wr, torch), gate, up, down, ex.stride, None, E, T, H, F, E, k,
                     ids, wts, act, xd, ws)
        torch.cuda.synchronize()
        assert qg.device_status() == 0
        outs.append(xd.cpu().numpy())
    assert np.array_equal(outs[0], outs[1])
    ids_h, wts_h, act_h = ids.cpu().numpy(), wts.cpu().numpy(), act.cpu().numpy()
    # router stage (logits are not returned by moe_layer: recompute them with the standalone call)
    i2, w2, lg = _route(qg, xn, wr, k)
    assert np.array_equal(i2, ids_h) and np.array_equal(w2, wts_h)
    check_route(oracle_lib, xn, wr, k, ids_h, wts_h, lg, what=f"layer T={T}")
    check_swiglu(oracle_lib, ex, ids_h, xn, k, act_h, what=f"layer T={T}")
    check_combine(oracle_lib, ex, ids_h, wts_h, act_h, x, k, outs[0], what=f"layer T={T}")


# ---- more than 16 tokens: grouped tensor-core path (bf16 operands, f32 accumulation) ----------

PREFILL_REL = 2e-3  # the prefill bar: |gpu - oracle| <= 2e-3 * sum|w x| + 1e-6


class ExactExperts(Experts):
    """Q8_0 expert records with d = 1.0 and codes in [-4, 4]: exact in bf16."""

    def __init__(self, E, H, F, seed=0):
        self.qtype, self.E, self.H, self.F, self.n_slots = gs.Q8_0, E, H, F, E
        go, uo, do, stride = gs.moe_expert_record_layout(H, F, gs.Q8_0)
        self.offs, self.stride = (go, uo, do), stride
        rng = np.random.default_rng(seed)
        blk = np.empty((E * stride // 34, 34), np.uint8)
        blk[:, 0], blk[:, 1] = 0x00, 0x3C
        blk[:, 2:] = rng.integers(-4, 5, size=(blk.shape[0], 32)).astype(np.int8).view(np.uint8)
        self.host = blk.reshape(-1)
        self.dev = to_dev(self.host, torch)


def test_grouped_gate_up_exact_products(qg, oracle_lib):
    """Integer weights and activations: every gate/up product and sum is exact, so act can
    differ from the oracle only by the f32 evaluation of silu(g) * u."""
    E, H, F, k, T = 8, 256, 256, 2, 40
    ex = ExactExperts(E, H, F, seed=1)
    ids = _rand_ids(T, k, E, seed=4)
    xn = np.random.default_rng(5).integers(-2, 3, size=(T, H)).astype(np.float32)
    gate, up, _ = ex.bases()
    act = torch.full((T * k, F), float("nan"), dtype=torch.float32, device="cuda")
    ws = _ws(qg, T, k, E, H, F)
    qg.moe_expert_swiglu(gs.Q8_0, gate, up, ex.stride, None, E, E, to_dev(ids, torch), to_dev(xn, torch), T, k, H, F,
                         act, ws)
    torch.cuda.synchronize()
    assert qg.device_status() == 0
    g, u, ref, _, _ = oracle_lib.moe_gate_up(gs.Q8_0, ex.host[ex.offs[0]:], ex.host[ex.offs[1]:], ex.stride, None, ids,
                                             xn, k, H, F)
    assert np.array_equal(np.round(g), g) and np.array_equal(np.round(u), u)
    got = act.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref) <= 1e-6 * np.abs(ref) + 1e-30), np.abs(got - ref).max()


@pytest.mark.parametrize("T", [17, 100])
def test_grouped_experts_slots_and_bad_id(qg, oracle_lib, T):
    H, F, E, k = 512, 256, 12, 3
    ex = Experts(gs.Q8_0, E, H, F, n_slots=15, seed=6)
    slots = np.random.default_rng(2).permutation(15)[:E].astype(np.int32)
    ids = _rand_ids(T, k, E, seed=T)
    ids[T // 2, 1] = -3  # bad id: flagged, act row zero, left out of the combine
    xn = gs.activations(T, H, seed=T, stream=51)
    gate, up, down = ex.bases()
    ws = _ws(qg, T, k, E, H, F)
    act = torch.full((T * k, F), float("nan"), dtype=torch.float32, device="cuda")
    sl = to_dev(slots, torch)
    qg.moe_expert_swiglu(gs.Q8_0, gate, up, ex.stride, sl, ex.n_slots, E, to_dev(ids, torch), to_dev(xn, torch), T, k,
                         H, F, act, ws)
    torch.cuda.synchronize()
    assert qg.device_status() & (1 << qg.QG_EDEVICE_ID)
    act_h = act.cpu().numpy()
    bad = (T // 2) * k + 1
    assert (act_h[bad] == 0).all()
    ids_ok = ids.copy()
    ids_ok[T // 2, 1] = ids[T // 2, 0]
    g, u, ref, bg, bu = oracle_lib.moe_gate_up(gs.Q8_0, ex.host[ex.offs[0]:], ex.host[ex.offs[1]:], ex.stride, slots,
                                               ids_ok, xn, k, H, F, threads=8)
    eg, eu = PREFILL_REL * bg + 1e-6, PREFILL_REL * bu + 1e-6
    sig = 1.0 / (1.0 + np.exp(-g))
    lim = np.abs(sig * (1 + g * (1 - sig)) * u) * eg + np.abs(g * sig) * eu + 1e-6
    good = np.ones(T * k, bool)
    good[bad] = False
    assert (np.abs(act_h[good] - ref[good]) <= lim[good]).all()
    wts = np.random.default_rng(T).random((T, k)).astype(np.float32)
    x = gs.activations(T, H, seed=T, stream=52)
    xd = to_dev(x, torch)
    qg.moe_combine(gs.Q8_0, down, ex.stride, sl, ex.n_slots, E, to_dev(ids, torch), to_dev(wts, torch),
                   to_dev(act_h, torch), T, k, H, F, xd, 1, ws)
    torch.cuda.synchronize()
    assert qg.device_status() & (1 << qg.QG_EDEVICE_ID)
    wts_ok = wts.copy()
    wts_ok[T // 2, 1] = 0.0
    _, _, out_ref, bout = oracle_lib.moe_down_combine(gs.Q8_0, ex.host[ex.offs[2]:], ex.stride, slots, ids_ok, wts_ok,
                                                      act_h, x, k, H, F, 1, threads=8)
    assert_within_bound(xd.cpu().numpy(), out_ref, bout, rel=PREFILL_REL, what=f"grouped combine T={T}")


@pytest.mark.parametrize("T", [64, 512])
def test_moe_layer_prefill_grouped(qg, oracle_lib, a3b, T):
    """The Qwen3-30B-A3B-shaped layer on a prefill batch: router and top-k as in decode, the
    expert steps grouped per expert on the tensor cores."""
    H, F, E, k = gs.MOE_H, gs.MOE_F, gs.MOE_E, gs.MOE_K
    ex = a3b
    wr = gs.router_weights(E, H, seed=0)
    xn = gs.activations(T, H, seed=T, stream=61)
    x = gs.activations(T, H, seed=T, stream=62)
    gate, up, down = ex.bases()
    ids = torch.zeros((T, k), dtype=torch.int32, device="cuda")
    wts = torch.zeros((T, k), dtype=torch.float32, device="cuda")
    act = torch.zeros((T * k, F), dtype=torch.float32, device="cuda")
    ws = _ws(qg, T, k, E, H, F)
    xd = to_dev(x, torch)
    qg.moe_layer(gs.Q8_0, to_dev(xn, torch), to_dev(wr, torch), gate, up, down, ex.stride, None, E, T, H, F, E, k, ids,
                 wts, act, xd, ws)
    torch.cuda.synchronize()
    assert qg.device_status() == 0
    ids_h, wts_h, act_h = ids.cpu().numpy(), wts.cpu().numpy(), act.cpu().numpy()
    i2, w2, lg = _route(qg, xn, wr, k)
    assert np.array_equal(i2, ids_h) and np.array_equal(w2, wts_h)
    check_route(oracle_lib, xn, wr, k, ids_h, wts_h, lg, what=f"prefill T={T}")
    # sampled pairs for the gate/up stage (the oracle's full stage at T = 512 is slow)
    rng = np.random.default_rng(T)
    toks = np.unique(np.concatenate([[0, T - 1], rng.integers(0, T, 12)]))
    g, u, ref, bg, bu = oracle_lib.moe_gate_up(gs.Q8_0, ex.host[ex.offs[0]:], ex.host[ex.offs[1]:], ex.stride, None,
                                               ids_h[toks], xn[toks], k, H, F, threads=16)
    eg, eu = PREFILL_REL * bg + 1e-6, PREFILL_REL * bu + 1e-6
    sig = 1.0 / (1.0 + np.exp(-g))
    lim = np.abs(sig * (1 + g * (1 - sig)) * u) * eg + np.abs(g * sig) * eu + 1e-6
    rows = (toks[:, None] * k + np.arange(k)[None, :]).reshape(-1)
    assert (np.abs(act_h[rows] - ref) <= lim).all(), "prefill act"
    _, _, out_ref, bout = oracle_lib.moe_down_combine(gs.Q8_0, ex.host[ex.offs[2]:], ex.stride, None, ids_h[toks],
                                                      wts_h[toks], act_h[rows], x[toks], k, H, F, 1, threads=16)
    assert_within_bound(xd.cpu().numpy()[toks], out_ref, bout, rel=PREFILL_REL, what=f"prefill combine T={T}")
