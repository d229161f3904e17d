"""Pins of the oracle's embedding gather, RMSNorm and argmax to things other than itself.

- embedding gather (embedQ8 / embedQ6K): Q8_0 and Q4_0 rows against a numpy decode of the
  block bytes written here from the format (f16 d, int8 codes / nibbles - 8); Q4_K and Q6_K
  rows against the pages' dequant loops restated in test_oracle_blocks.py; the scale as one
  f32 rounding of the exact product; ids outside the table rejected.
- RMSNorm (rmsnorm): closed forms (constant rows, the row (3, 4)), the RMS of y / w equal to 1
  when eps = 0, invariance of the result under scaling x when eps = 0.
- argmax (argmax / argmaxRows): brute force over small integer rows full of ties, NaN never
  picked, all-NaN rows give 0, -inf rows give their first index.
"""
from fractions import Fraction

import numpy as np
import pytest

import gguf_synth as gs
from test_oracle_blocks import _dequant_q4k_page_loop, _dequant_q6k_page_loop


def _f16_col(blocks, off):
    return blocks[:, off:off + 2].copy().view(np.float16).astype(np.float64)[:, 0]


def _decode_q8_0(raw, rows, n):
    blk = raw.reshape(-1, 34)
    d = _f16_col(blk, 0)
    q = blk[:, 2:].view(np.int8).astype(np.float64)
    return (d[:, None] * q).astype(np.float32).reshape(rows, n)


def _decode_q4_0(raw, rows, n):
    blk = raw.reshape(-1, 18)
    d = _f16_col(blk, 0)
    qs = blk[:, 2:].astype(np.int64)
    vals = np.concatenate([(qs & 15) - 8, (qs >> 4) - 8], axis=1).astype(np.float64)
    return (d[:, None] * vals).astype(np.float32).reshape(rows, n)


@pytest.mark.parametrize("qtype", [gs.Q8_0, gs.Q4_0, gs.Q4_K, gs.Q6_K])
def test_embed_rows_match_independent_decode(oracle_lib, qtype):
    qk, bb = gs.BLOCK[qtype]
    V, N = 37, 2 * 256
    table = gs.quant_blocks(qtype, V, N, seed=21, stream=qtype)
    ids = np.array([0, 36, 5, 5, 17], dtype=np.int32)
    got = oracle_lib.embed_rows(qtype, table, V, N, ids)
    rows = table.reshape(V, -1)
    for i, r in enumerate(ids):
        raw = rows[r]
        if qtype == gs.Q8_0:
            want = _decode_q8_0(raw, 1, N)[0]
        elif qtype == gs.Q4_0:
            want = _decode_q4_0(raw, 1, N)[0]
        elif qtype == gs.Q4_K:
            want = np.concatenate([_dequant_q4k_page_loop(b) for b in raw.reshape(-1, 144)])
        else:
            want = np.array([float(v) for b in raw.reshape(-1, 210) for v in _dequant_q6k_page_loop(b.astype(np.int64))],
                            dtype=np.float32)
        if qtype == gs.Q6_K:
            # the page loop runs in exact rationals, which carry no sign of zero: compare values
            assert np.array_equal(got[i], want), (qtype, i)
        else:
            assert np.array_equal(got[i].view(np.uint32), want.view(np.uint32)), (qtype, i)


def test_embed_rows_scale_is_one_rounding(oracle_lib):
    V, N = 9, 256
    table = gs.quant_blocks(gs.Q6_K, V, N, seed=22, stream=5)
    s = np.float32(np.sqrt(np.float32(2816.0)))
    ids = np.arange(V, dtype=np.int32)
    base = oracle_lib.embed_rows(gs.Q6_K, table, V, N, ids)
    got = oracle_lib.embed_rows(gs.Q6_K, table, V, N, ids, scale=float(s))
    # the dequantized value times the f32 scale, exactly (two 24-bit significands fit a double),
    # rounded once to f32 (nearest even)
    for i in range(0, V):
        for k in range(0, N, 17):
            exact = Fraction(float(base[i, k])) * Fraction(float(s))
            assert float(exact) == float(base[i, k]) * float(s)
            assert got[i, k] == np.float32(float(exact))


def test_embed_rows_rejects_bad_ids(oracle_lib):
    table = gs.quant_blocks(gs.Q8_0, 4, 32, seed=1)
    with pytest.raises(ValueError):
        oracle_lib.embed_rows(gs.Q8_0, table, 4, 32, np.array([4], dtype=np.int32))
    with pytest.raises(ValueError):
        oracle_lib.embed_rows(gs.Q8_0, table, 4, 32, np.array([-1], dtype=np.int32))


def test_rmsnorm_closed_forms(oracle_lib):
    w = np.array([1.0, 2.0], dtype=np.float32)
    y = oracle_lib.rmsnorm(np.array([[3.0, 4.0]], dtype=np.float32), w, 0.0)
    # mean of squares 12.5: 3 / sqrt(12.5) and 2 * 4 / sqrt(12.5)
    assert y[0, 0] == pytest.approx(3.0 / np.sqrt(12.5), rel=1e-15)
    assert y[0, 1] == pytest.approx(8.0 / np.sqrt(12.5), rel=1e-15)
    c, eps = 0.75, 1e-6
    x = np.full((2, 64), c, dtype=np.float32)
    x[1] = -c
    wv = np.linspace(-2, 2, 64).astype(np.float32)
    y = oracle_lib.rmsnorm(x, wv, eps)
    scale = 1.0 / np.sqrt(c * c + eps)
    assert np.allclose(y[0], c * scale * wv.astype(np.float64), rtol=1e-14, atol=0)
    assert np.allclose(y[1], -c * scale * wv.astype(np.float64), rtol=1e-14, atol=0)


def test_rmsnorm_unit_rms_and_scale_invariance(oracle_lib):
    rng = np.random.default_rng(3)
    x = rng.standard_normal((3, 2560)).astype(np.float32)
    w = rng.uniform(0.5, 1.5, 2560).astype(np.float32)
    y = oracle_lib.rmsnorm(x, w, 0.0)
    z = y / w.astype(np.float64)
    assert np.allclose(np.sqrt(np.mean(z * z, axis=1)), 1.0, rtol=1e-12)
    y2 = oracle_lib.rmsnorm((x * np.float32(4.0)).astype(np.float32), w, 0.0)
    assert np.allclose(y, y2, rtol=1e-12, atol=0)
    # eps moves every row's scale by the same closed form
    eps = 0.5
    ye = oracle_lib.rmsnorm(x, w, eps)
    ms = np.mean(x.astype(np.float64) ** 2, axis=1)
    assert np.allclose(ye / y, np.sqrt(ms / (ms + eps))[:, None], rtol=1e-12)


def _brute_argmax(row):
    best = None
    for i, v in enumerate(row):
        if np.isnan(v):
            continue
        if best is None or v > row[best]:
            best = i
    return 0 if best is None else best


def test_argmax_brute_force_with_ties(oracle_lib):
    rng = np.random.default_rng(7)
    v = rng.integers(-3, 4, size=(200, 23)).astype(np.float64)
    v[rng.random(v.shape) < 0.1] = np.nan
    v[5] = np.nan
    v[6] = -np.inf
    v[7, :] = np.nan
    v[7, 9] = -np.inf
    ids = oracle_lib.argmax_rows(v)
    assert [int(i) for i in ids] == [_brute_argmax(r) for r in v]
    assert ids[5] == 0 and ids[6] == 0 and ids[7] == 9
