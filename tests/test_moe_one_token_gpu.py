"""The one-token MoE layer (moe_layer at T = 1: router, picks, gate/up, down and combine in one
cooperative launch) against the oracle, for every block type, with a slot map, a pick whose
slot is invalid, and many calls on one workspace (its grid-barrier counter only grows)."""
import numpy as np
import pytest

import edge_blocks as eb
import gguf_synth as gs
from helpers import to_dev
from test_moe_gpu import Experts, _act_bound, _route, _ws, check_combine, check_route, check_swiglu

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SHAPES = {gs.Q8_0: (512, 96), gs.Q4_0: (512, 96), gs.Q4_K: (512, 256), gs.Q6_K: (512, 256)}


@pytest.fixture(scope="module")
def qg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gguf_block_dequant_gb300 as qg
    from gguf_block_dequant_gb300 import build

    build.build()
    qg.load()
    return qg


def _layer(qg, ex, xn, wr, x, k, slots=None, ws=None):
    E, H, F = ex.E, ex.H, ex.F
    gate, up, down = ex.bases()
    ids = torch.full((1, k), -7, dtype=torch.int32, device="cuda")
    wts = torch.full((1, k), float("nan"), dtype=torch.float32, device="cuda")
    act = torch.full((k, F), float("nan"), dtype=torch.float32, device="cuda")
    xd = to_dev(x, torch)
    ws = ws if ws is not None else _ws(qg, 1, k, E, H, F)
    sl = None if slots is None else to_dev(slots.astype(np.int32), torch)
    qg.moe_layer(ex.qtype, to_dev(xn, torch), to_dev(wr, torch), gate, up, down, ex.stride, sl, ex.n_slots, 1, H, F,
                 E, k, ids, wts, act, xd, ws)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), wts.cpu().numpy(), act.cpu().numpy(), xd.cpu().numpy()


@pytest.mark.parametrize("qtype", [gs.Q8_0, gs.Q4_0, gs.Q4_K, gs.Q6_K])
def test_one_token_layer_every_type_with_slot_map(qg, oracle_lib, qtype):
    H, F = SHAPES[qtype]
    E, k, n_slots = 16, 4, 19
    ex = Experts(qtype, E, H, F, n_slots=n_slots, seed=40 + qtype)
    slots = np.random.default_rng(qtype).permutation(n_slots)[:E].astype(np.int32)
    wr = gs.router_weights(E, H, seed=qtype)
    xn = gs.activations(1, H, seed=qtype, stream=50)
    x = gs.activations(1, H, seed=qtype, stream=51)
    ids, wts, act, out = _layer(qg, ex, xn, wr, x, k, slots=slots)
    assert qg.device_status() == 0
    i2, w2, lg = _route(qg, xn, wr, k)
    assert np.array_equal(i2, ids) and np.array_equal(w2, wts)  # the standalone router's picks, bit for bit
    check_route(oracle_lib, xn, wr, k, ids, wts, lg, what=f"one token type {qtype}")
    check_swiglu(oracle_lib, ex, ids, xn, k, act, slots=slots, what=f"one token type {qtype}")
    check_combine(oracle_lib, ex, ids, wts, act, x, k, out, slots=slots, what=f"one token type {qtype}")


def test_one_token_pick_with_invalid_slot(qg, oracle_lib):
    """The top pick's expert maps to no slot: the status word reports it, its act row is zero
    and the combine leaves it out; the other picks keep their weights."""
    H, F, E, k = 512, 96, 16, 4
    ex = Experts(gs.Q8_0, E, H, F, seed=61)
    wr = gs.router_weights(E, H, seed=61)
    xn = gs.activations(1, H, seed=61, stream=52)
    x = gs.activations(1, H, seed=61, stream=53)
    picks, _, _ = _route(qg, xn, wr, k)
    slots = np.arange(E, dtype=np.int32)
    slots[picks[0, 0]] = E + 3  # out of range
    qg.device_status()  # clear
    ids, wts, act, out = _layer(qg, ex, xn, wr, x, k, slots=slots)
    assert qg.device_status() & (1 << qg.QG_EDEVICE_ID)
    assert np.array_equal(ids, picks)
    assert (act[0] == 0).all()
    ok_slots = np.arange(E, dtype=np.int32)  # any valid slot for the bad pick: its act row and weight are zeroed
    good = np.ones(k, bool)
    good[0] = False
    g, u, ref, bg, bu = oracle_lib.moe_gate_up(ex.qtype, ex.host[ex.offs[0]:], ex.host[ex.offs[1]:], ex.stride,
                                               ok_slots, ids, xn, k, H, F)
    lim = _act_bound(g, u, bg, bu)
    assert (np.abs(act[good] - ref[good]) <= lim[good]).all()
    wts_ok = wts.copy()
    wts_ok[0, 0] = 0.0
    check_combine(oracle_lib, ex, ids, wts_ok, act, x, k, out, slots=ok_slots, what="invalid slot")


def test_one_token_many_calls_one_workspace(qg):
    """Eager calls and graph replays on one workspace give the first call's result every time
    (the grid barrier's counter is never reset between calls)."""
    H, F, E, k = 512, 96, 16, 4
    ex = Experts(gs.Q8_0, E, H, F, seed=71)
    wr = to_dev(gs.router_weights(E, H, seed=71), torch)
    xn = to_dev(gs.activations(1, H, seed=71, stream=54), torch)
    x0 = to_dev(gs.activations(1, H, seed=71, stream=55), torch)
    gate, up, down = ex.bases()
    ws = _ws(qg, 1, k, E, H, F)
    ids = torch.zeros((1, k), dtype=torch.int32, device="cuda")
    wts = torch.zeros((1, k), dtype=torch.float32, device="cuda")
    act = torch.zeros((k, F), dtype=torch.float32, device="cuda")
    x = torch.empty_like(x0)

    def call():
        x.copy_(x0)
        qg.moe_layer(gs.Q8_0, xn, wr, gate, up, down, ex.stride, None, E, 1, H, F, E, k, ids, wts, act, x, ws)

    call()
    torch.cuda.synchronize()
    first = x.cpu().numpy().copy()
    for _ in range(37):
        call()
    torch.cuda.synchronize()
    assert np.array_equal(x.cpu().numpy(), first)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        call()
        s.synchronize()
        with torch.cuda.graph(g, stream=s):
            for _ in range(5):
                call()
    for _ in range(10):
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(x.cpu().numpy(), first)
    assert qg.device_status() == 0


@pytest.mark.parametrize("E,k", [(5, 4), (13, 8), (40, 8), (97, 1)])
def test_one_token_expert_counts_not_multiple_of_four(qg, oracle_lib, E, k):
    """The fused ranking splits the experts into four quarters (the last one short or empty when
    E is not a multiple of four): picks and weights still equal the standalone router's."""
    H, F = 512, 96
    ex = Experts(gs.Q8_0, E, H, F, seed=80 + E)
    wr = gs.router_weights(E, H, seed=E)
    xn = gs.activations(1, H, seed=E, stream=56)
    x = gs.activations(1, H, seed=E, stream=57)
    ids, wts, act, out = _layer(qg, ex, xn, wr, x, k)
    assert qg.device_status() == 0
    i2, w2, lg = _route(qg, xn, wr, k)
    assert np.array_equal(i2, ids) and np.array_equal(w2, wts)
    check_route(oracle_lib, xn, wr, k, ids, wts, lg, what=f"one token E={E} k={k}")
    check_combine(oracle_lib, ex, ids, wts, act, x, k, out, what=f"one token E={E} k={k}")


@pytest.mark.parametrize("qtype", [gs.Q8_0, gs.Q4_0, gs.Q4_K, gs.Q6_K])
def test_one_token_layer_with_edge_blocks(qg, oracle_lib, qtype):
    """Edge-value blocks (code -128, negative / subnormal / extreme d, zero d or dmin, extreme
    scales) dealt over every expert's gate, up and down rows: the fused one-token layer still
    matches the oracle stage by stage."""
    H, F = SHAPES[qtype]
    E, k = 16, 4
    ex = Experts(qtype, E, H, F, seed=90 + qtype)
    qk, bb = gs.BLOCK[qtype]
    edge = eb.edge_blocks(qtype)
    go, uo, do = ex.offs
    host = ex.host.copy()
    nb = 0
    for e in range(E):
        for base, rows, K in ((go, F, H), (uo, F, H), (do, H, F)):
            off = e * ex.stride + base
            blocks = host[off:off + rows * (K // qk) * bb].reshape(-1, bb)
            for i in range(0, blocks.shape[0], 7):
                blocks[i] = edge[(i // 7 + e) % len(edge)]
                nb += 1
    assert nb > 0
    ex.host = host
    ex.dev = to_dev(host, torch)
    wr = gs.router_weights(E, H, seed=qtype + 3)
    xn = gs.activations(1, H, seed=qtype, stream=58)
    x = gs.activations(1, H, seed=qtype, stream=59)
    ids, wts, act, out = _layer(qg, ex, xn, wr, x, k)
    assert qg.device_status() == 0
    i2, w2, lg = _route(qg, xn, wr, k)
    assert np.array_equal(i2, ids) and np.array_equal(w2, wts)
    check_route(oracle_lib, xn, wr, k, ids, wts, lg, what=f"edge blocks type {qtype}")
    check_swiglu(oracle_lib, ex, ids, xn, k, act, what=f"edge blocks type {qtype}")
    check_combine(oracle_lib, ex, ids, wts, act, x, k, out, what=f"edge blocks type {qtype}")


def test_one_workspace_serves_every_token_count(qg, oracle_lib):
    """One workspace sized for T = 8 serves moe_layer at T = 8, 1, 8, 1, 3 in turn and then the
    standalone router: the one-token grid-barrier counter and the router tickets sit in a fixed
    header, so no call's scratch (logits, dn rows) lands on them, and every result still
    matches the oracle."""
    H, F, E, k = 512, 96, 16, 4
    ex = Experts(gs.Q8_0, E, H, F, seed=73)
    gate, up, down = ex.bases()
    wr = gs.router_weights(E, H, seed=73)
    wrd = to_dev(wr, torch)
    ws = _ws(qg, 8, k, E, H, F)
    for i, T in enumerate((8, 1, 8, 1, 3)):
        xn = gs.activations(T, H, seed=i, stream=60)
        x = gs.activations(T, H, seed=i, stream=61)
        ids = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
        wts = torch.full((T, k), float("nan"), dtype=torch.float32, device="cuda")
        act = torch.full((T * k, F), float("nan"), dtype=torch.float32, device="cuda")
        xd = to_dev(x, torch)
        qg.moe_layer(gs.Q8_0, to_dev(xn, torch), wrd, gate, up, down, ex.stride, None, E, T, H, F, E, k, ids, wts,
                     act, xd, ws)
        torch.cuda.synchronize()
        assert qg.device_status() == 0, T
        ids_h, wts_h, act_h, out = ids.cpu().numpy(), wts.cpu().numpy(), act.cpu().numpy(), xd.cpu().numpy()
        i2, w2, lg = _route(qg, xn, wr, k)
        assert np.array_equal(i2, ids_h), T
        check_route(oracle_lib, xn, wr, k, ids_h, wts_h, lg, what=f"shared workspace T={T}")
        check_swiglu(oracle_lib, ex, ids_h, xn, k, act_h, what=f"shared workspace T={T}")
        check_combine(oracle_lib, ex, ids_h, wts_h, act_h, x, k, out, what=f"shared workspace T={T}")
    # the standalone router on the same workspace: its tickets read zero again
    xn = gs.activations(8, H, seed=9, stream=62)
    ids = torch.full((8, k), -7, dtype=torch.int32, device="cuda")
    wts = torch.full((8, k), float("nan"), dtype=torch.float32, device="cuda")
    qg.moe_route_topk(to_dev(xn, torch), wrd, 8, H, E, k, ids, wts, None, ws)
    torch.cuda.synchronize()
    i2, w2, _ = _route(qg, xn, wr, k)
    assert np.array_equal(ids.cpu().numpy(), i2) and np.array_equal(wts.cpu().numpy(), w2)


@pytest.mark.parametrize("T", [1, 4])
def test_nan_router_input_leaves_no_pick_unset(qg, T):
    """A NaN token row makes every router logit NaN, so every expert ranks first and ranks 1..k-1
    have no expert: those picks come back -1 and the status word reports invalid ids, while the
    call still completes (T = 1 ranks inside the one-token kernel, T = 4 inside the gate/up
    kernel).  The other rows of the T = 4 call are finite and keep valid picks."""
    H, F, E, k = 512, 96, 16, 4
    ex = Experts(gs.Q8_0, E, H, F, seed=75)
    gate, up, down = ex.bases()
    wr = to_dev(gs.router_weights(E, H, seed=75), torch)
    xn = gs.activations(T, H, seed=75, stream=63)
    xn[0] = np.nan
    ids = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    wts = torch.zeros((T, k), dtype=torch.float32, device="cuda")
    act = torch.zeros((T * k, F), dtype=torch.float32, device="cuda")
    x = to_dev(gs.activations(T, H, seed=75, stream=64), torch)
    ws = _ws(qg, T, k, E, H, F)
    qg.device_status()  # clear
    qg.moe_layer(gs.Q8_0, to_dev(xn, torch), wr, gate, up, down, ex.stride, None, E, T, H, F, E, k, ids, wts, act, x,
                 ws)
    torch.cuda.synchronize()
    assert qg.device_status() & (1 << qg.QG_EDEVICE_ID)
    got = ids.cpu().numpy()
    assert 0 <= got[0, 0] < E and (got[0, 1:] == -1).all(), got[0]
    for t in range(1, T):
        assert ((got[t] >= 0) & (got[t] < E)).all() and len(set(got[t])) == k, got[t]
