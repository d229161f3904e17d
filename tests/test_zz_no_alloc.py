"""moe_route_topk_noalloc: the router with the library's own fixed scratch (no workspace, no
allocation) gives the same ids, weights and logits as moe_route_topk, call after call.

Kept in its own file, collected last, so that it also runs after every other GPU test."""
import numpy as np
import pytest

import gguf_synth as gs
from helpers import to_dev

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


def _outs(T, k, E):
    return (torch.full((T, k), -1, dtype=torch.int32, device="cuda"),
            torch.full((T, k), float("nan"), dtype=torch.float32, device="cuda"),
            torch.full((T, E), float("nan"), dtype=torch.float32, device="cuda"))


def _workspace_route(qg, xn, wr, T, H, E, k):
    ids, wts, lg = _outs(T, k, E)
    ws = torch.zeros(qg.moe_workspace_size(T, k, E, H, 64), dtype=torch.uint8, device="cuda")
    qg.moe_route_topk(xn, wr, T, H, E, k, ids, wts, lg, ws)
    torch.cuda.synchronize()
    return [t.cpu().numpy() for t in (ids, wts, lg)]


@pytest.mark.parametrize("with_logits", [True, False])
@pytest.mark.parametrize("T,E,k", [(1, 128, 8), (8, 128, 8), (33, 64, 4), (100, 128, 8), (16384, 1, 1)])
def test_noalloc_router_matches_workspace_router(qg, T, E, k, with_logits):
    """Same ids, weights (and logits, when asked for) as the workspace router, on two calls in
    a row; without logits_out the router keeps its logits in the fixed scratch.  T = 16384,
    E = 1 is the edge of the documented limit (T * E = 16384, 1024 tiles)."""
    H = 2048 if E == 128 else 512 if E > 1 else 64
    xn = to_dev(gs.activations(T, H, seed=T, stream=91), torch)
    wr = to_dev(gs.router_weights(E, H, seed=E), torch)
    ref = _workspace_route(qg, xn, wr, T, H, E, k)
    for _ in range(2):  # twice in a row: the scratch's tickets must be clear again
        ids2, wts2, lg2 = _outs(T, k, E)
        qg.moe_route_topk_noalloc(xn, wr, T, H, E, k, ids2, wts2, lg2 if with_logits else None)
        torch.cuda.synchronize()
        assert qg.device_status() == 0
        assert np.array_equal(ref[0], ids2.cpu().numpy())
        assert np.array_equal(ref[1], wts2.cpu().numpy())
        if with_logits:
            assert np.array_equal(ref[2], lg2.cpu().numpy())


def test_noalloc_router_large_then_small_shape(qg):
    """A call with many tiles, then one-token calls, then the large shape again: every call sees
    its own tickets at zero whatever the previous call's shape was."""
    shapes = [(100, 128, 8, 2048), (1, 128, 8, 2048), (1, 64, 4, 512), (100, 128, 8, 2048), (17, 96, 6, 512)]
    for i, (T, E, k, H) in enumerate(shapes):
        xn = to_dev(gs.activations(T, H, seed=i, stream=92), torch)
        wr = to_dev(gs.router_weights(E, H, seed=i), torch)
        ref = _workspace_route(qg, xn, wr, T, H, E, k)
        ids2, wts2, _ = _outs(T, k, E)
        qg.moe_route_topk_noalloc(xn, wr, T, H, E, k, ids2, wts2, None)
        torch.cuda.synchronize()
        assert qg.device_status() == 0
        assert np.array_equal(ref[0], ids2.cpu().numpy()), (T, E, k)
        assert np.array_equal(ref[1], wts2.cpu().numpy()), (T, E, k)


def test_noalloc_router_rejects_too_large(qg):
    T, E, k, H = 200, 128, 8, 64
    xn = torch.zeros((T, H), dtype=torch.float32, device="cuda")
    wr = torch.zeros((E, H), dtype=torch.float32, device="cuda")
    ids, wts, lg = _outs(T, k, E)
    with pytest.raises(qg.QGError) as e:
        qg.moe_route_topk_noalloc(xn, wr, T, H, E, k, ids, wts, lg)  # T * E > 16384
    assert e.value.status == qg.QG_EWORKSPACE
