"""The seeded generators: determinism, layouts and the stated distributions."""
import numpy as np

import gguf_synth as gs


def test_deterministic_and_streams_differ():
    a = gs.quant_blocks(gs.Q8_0, 8, 256, seed=0, stream=1)
    b = gs.quant_blocks(gs.Q8_0, 8, 256, seed=0, stream=1)
    c = gs.quant_blocks(gs.Q8_0, 8, 256, seed=0, stream=2)
    assert np.array_equal(a, b) and not np.array_equal(a, c)
    assert a.size == gs.tensor_bytes(gs.Q8_0, 8, 256)


def test_q8_0_fields():
    w = gs.quant_blocks(gs.Q8_0, 64, 1024, seed=0).reshape(-1, 34)
    d = w[:, 0:2].copy().view(np.float16).astype(np.float64).reshape(-1)
    q = w[:, 2:].view(np.int8)
    assert (d >= 0).all() and 0.01 < d.mean() < 0.02      # |N(0,1)|*0.02 has mean 0.016
    assert q.min() == -127 and q.max() == 127            # -128 is never produced
    assert abs(q.astype(np.float64).mean()) < 1.0


def test_q6_k_scales_range():
    w = gs.quant_blocks(gs.Q6_K, 16, 1024, seed=0).reshape(-1, 210)
    sc = w[:, 192:208].view(np.int8)
    assert sc.min() == -32 and sc.max() == 31


def test_activation_stats():
    x = gs.activations(4, 4096, seed=0)
    assert x.dtype == np.float32 and x.shape == (4, 4096)
    assert abs(x.mean()) < 0.05 and 0.95 < x.std() < 1.05
    wr = gs.router_weights(128, 2048)
    assert 0.019 < wr.std() < 0.021
