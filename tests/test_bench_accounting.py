"""The byte accounting behind bench.py's headline numbers, checked against the block formula
(Q8_0: 34 bytes per 32 weights) for the Qwen3-4B-shaped decode step, independently of the
generator module's own byte counter."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

# (rows, row length) of the step's projections: q, k, v, o, gate, up, down; then the tied head
LAYER = [(4096, 2560), (1024, 2560), (1024, 2560), (2560, 4096), (9728, 2560), (9728, 2560), (2560, 9728)]
HEAD = (151936, 2560)


def q8_bytes(m, n):
    return m * (n // 32) * 34


def test_weight_bytes_per_step():
    assert q8_bytes(*HEAD) == 413_265_920
    assert sum(q8_bytes(m, n) for m, n in LAYER) == 107_233_280
    assert bench.step_weight_bytes(36) == 36 * 107_233_280 + 413_265_920 == 4_273_664_000
    assert bench.step_weight_bytes(1) == 107_233_280 + 413_265_920


@pytest.mark.parametrize("T", [1, 4, 16])
def test_activation_bytes_per_step(T):
    per_layer = sum(T * (m + n) * 4 for m, n in LAYER)
    assert bench.step_act_bytes(36, T) == 36 * per_layer + T * (HEAD[0] + HEAD[1]) * 4


def test_algorithmic_bytes_per_launch():
    """The roofline's per-launch bytes: weights + activations of the whole step over its 145
    launches (every launch of the step is the one-token GEMV kernel)."""
    per = (bench.step_weight_bytes(36) + bench.step_act_bytes(36, 1)) / (4 * 36 + 1)
    assert per == pytest.approx(29_534_755.3, abs=0.1)
