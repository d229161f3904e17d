"""Pins of the oracle's f16 conversion and block decoders to things other than itself.

- f16: exhaustive against numpy's IEEE binary16 conversion (a library routine).
- Q8_0 / Q4_0: hand-built blocks (tests/golden/hand_blocks.txt) with closed-form values.
- Q4_K: blocks packed by an encoder written here from the 6-bit scale/min layout (the
  inverse of the decoder), values in closed form; random blocks checked against exact
  rational arithmetic rounded once to f32; and the page's own chunk-loop formulation
  (dequantQ4K in ternary_bonsai_2_dflash.js), restated here as a loop, against the oracle's
  per-element formula.
- Q6_K: the chunk-loop formulation of dequantQ6K (ternary_bonsai_2_dflash.js) restated here
  against the oracle's per-index q6v form (gemma4_moe_ssd.js); one-bit-set blocks.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

import edge_blocks as eb
import gguf_synth as gs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_blocks.txt")


def _hand_blocks():
    out = {}
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        name, typ, hx = line.split()
        out[name] = (typ, np.frombuffer(bytes.fromhex(hx), dtype=np.uint8).copy())
    return out


def _vals(oracle, qtype, blk, n):
    return oracle.dequant(qtype, blk, 1, n)[0]


def _f16(bits):
    return float(np.array([bits], dtype=np.uint16).view(np.float16)[0])


def test_f16_exhaustive(oracle_lib):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle_lib.f16_value(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signed zero and the f32 view
    assert np.signbit(got[0x8000]) and not np.signbit(got[0])


def test_q8_0_hand_blocks(oracle_lib):
    hb = _hand_blocks()
    a = _vals(oracle_lib, gs.Q8_0, hb["q8_hand_a"][1], 32)
    assert a.tolist() == [float(i - 16) for i in range(32)]
    b = _vals(oracle_lib, gs.Q8_0, hb["q8_hand_b"][1], 32)
    assert b.tolist() == [float((127 - 8 * i) * 2.0 ** -14) for i in range(32)]
    c = _vals(oracle_lib, gs.Q8_0, hb["q8_hand_c"][1], 32)
    assert c.tolist() == [float((-1) ** i * i * 2.0 ** -24) for i in range(32)]
    d = _vals(oracle_lib, gs.Q8_0, hb["q8_hand_d"][1], 32)
    assert d.tolist() == [-65504.0 if i == 5 else 0.0 for i in range(32)]


def test_q4_0_hand_blocks(oracle_lib):
    hb = _hand_blocks()
    a = _vals(oracle_lib, gs.Q4_0, hb["q4_hand_a"][1], 32)
    assert a[:16].tolist() == [float(7 - j) for j in range(16)]
    assert a[16:].tolist() == [float(j - 8) for j in range(16)]
    b = _vals(oracle_lib, gs.Q4_0, hb["q4_hand_b"][1], 32)
    exp = [0.0] * 32
    exp[3], exp[19] = -4.0, 3.5
    assert b.tolist() == exp


def test_q8_0_edge_hand_blocks(oracle_lib):
    """Code 0x80 (-128), a negative d, the smallest subnormal d and the most negative d."""
    hb = _hand_blocks()
    e = _vals(oracle_lib, gs.Q8_0, hb["q8_hand_e"][1], 32)
    assert e.tolist() == [-128.0 if i % 2 == 0 else 127.0 for i in range(32)]
    f = _vals(oracle_lib, gs.Q8_0, hb["q8_hand_f"][1], 32)
    assert f.tolist() == [(16 - i) / 2 for i in range(32)]
    g = _vals(oracle_lib, gs.Q8_0, hb["q8_hand_g"][1], 32)
    assert g.tolist() == [-(2.0 ** -17)] * 32
    h = _vals(oracle_lib, gs.Q8_0, hb["q8_hand_h"][1], 32)
    q = [-128] + [i - 16 for i in range(1, 31)] + [127]
    assert h.tolist() == [-65504.0 * v for v in q]


def test_q4_0_edge_hand_blocks(oracle_lib):
    """A negative d (ggml's d = max / -8), a subnormal d and the largest finite d."""
    hb = _hand_blocks()
    c = _vals(oracle_lib, gs.Q4_0, hb["q4_hand_c"][1], 32)
    assert c[:16].tolist() == [(j - 7) / 4 for j in range(16)]
    assert c[16:].tolist() == [(8 - j) / 4 for j in range(16)]
    d = _vals(oracle_lib, gs.Q4_0, hb["q4_hand_d"][1], 32)
    assert d[:16].tolist() == [3 * (j - 8) * 2.0 ** -24 for j in range(16)]
    assert d[16:].tolist() == [3 * (7 - j) * 2.0 ** -24 for j in range(16)]
    e = _vals(oracle_lib, gs.Q4_0, hb["q4_hand_e"][1], 32)
    assert e.tolist() == [7 * 65504.0] * 16 + [-8 * 65504.0] * 16


def test_q8_q4_products_exact(oracle_lib):
    """d * q needs at most 11 + 7 significant bits, so it is exact in f32: the oracle's f32
    value equals the exact rational product for every element of random blocks."""
    for qtype in (gs.Q8_0, gs.Q4_0):
        w = gs.quant_blocks(qtype, 4, 256, seed=7)
        qk, bb = gs.BLOCK[qtype]
        vals = oracle_lib.dequant(qtype, w, 4, 256).reshape(-1)
        blocks = w.reshape(-1, bb)
        for bi, blk in enumerate(blocks):
            d = Fraction(_f16(int(blk[0]) | (int(blk[1]) << 8)))
            for i in range(qk):
                if qtype == gs.Q8_0:
                    q = int(np.int8(blk[2 + i]))
                else:
                    byte = int(blk[2 + (i % 16)])
                    q = (byte & 15 if i < 16 else byte >> 4) - 8
                assert Fraction(float(vals[bi * qk + i])) == d * q


# ---- Q4_K ------------------------------------------------------------------------------

def _pack_q4k_scales(sc, mn):
    """Pack 8 six-bit scales and mins into 12 bytes (the layout of block_q4_K.scales):
    j < 4: byte j low 6 bits = sc[j], byte j+4 low 6 bits = mn[j]; the top 2 bits of byte j /
    byte j+4 carry bits 4..5 of sc[j+4] / mn[j+4]; byte j+8 = (sc[j+4] & 15) | (mn[j+4] & 15) << 4."""
    b = [0] * 12
    for j in range(4):
        b[j] = (sc[j] & 63) | ((sc[j + 4] >> 4) << 6)
        b[j + 4] = (mn[j] & 63) | ((mn[j + 4] >> 4) << 6)
        b[j + 8] = (sc[j + 4] & 15) | ((mn[j + 4] & 15) << 4)
    return b


def _q4k_block(dbits, dminbits, sc, mn, qs):
    blk = np.zeros(144, dtype=np.uint8)
    blk[0:2] = [dbits & 255, dbits >> 8]
    blk[2:4] = [dminbits & 255, dminbits >> 8]
    blk[4:16] = _pack_q4k_scales(sc, mn)
    blk[16:144] = qs
    return blk


def _q4k_closed_form(dbits, dminbits, sc, mn, qs):
    """w[64c + l] = d*sc[2c]*lo(qs[32c+l]) - dmin*mn[2c]; w[64c+32+l] = d*sc[2c+1]*hi(..) - dmin*mn[2c+1]."""
    d, dm = Fraction(_f16(dbits)), Fraction(_f16(dminbits))
    out = []
    for c in range(4):
        for half in range(2):
            s = 2 * c + half
            for l in range(32):
                byte = int(qs[32 * c + l])
                q = (byte & 15) if half == 0 else (byte >> 4)
                out.append(d * sc[s] * q - dm * mn[s])
    return out


def _round_f32(fr):
    """Exact rational -> nearest f32 (ties to even), checked by bracketing."""
    f = np.float32(float(fr))
    # float(fr) is the nearest double; verify the f32 is the nearest f32 to the exact value
    lo = np.nextafter(f, np.float32(-np.inf))
    hi = np.nextafter(f, np.float32(np.inf))
    e = abs(Fraction(float(f)) - fr)
    assert e <= abs(Fraction(float(lo)) - fr) and e <= abs(Fraction(float(hi)) - fr)
    return f


@pytest.mark.parametrize("case", range(4))
def test_q4_k_hand_blocks(oracle_lib, case):
    rng = np.random.default_rng(100 + case)
    if case == 0:    # both scale paths, extreme values
        sc, mn = [0, 1, 63, 17, 63, 1, 0, 42], [63, 0, 1, 5, 0, 63, 33, 1]
        qs = np.array([(15 if (i % 3) else 0) | ((0 if (i % 5) else 15) << 4) for i in range(128)], np.uint8)
        dbits, dminbits = 0x3C00, 0x3800          # d = 1, dmin = 0.5
    elif case == 1:  # dmin = 0 -> w = d * sc * q
        sc, mn = [1, 2, 3, 4, 5, 6, 7, 8], [9] * 8
        qs = np.full(128, 0x21, np.uint8)
        dbits, dminbits = 0x4000, 0x0000          # d = 2, dmin = 0
    elif case == 2:  # d = 0 -> w = -dmin * mn
        sc, mn = [63] * 8, [0, 1, 2, 3, 60, 61, 62, 63]
        qs = rng.integers(0, 256, 128).astype(np.uint8)
        dbits, dminbits = 0x0000, 0x2E66          # dmin ~ 0.1
    else:            # random fields
        sc, mn = rng.integers(0, 64, 8).tolist(), rng.integers(0, 64, 8).tolist()
        qs = rng.integers(0, 256, 128).astype(np.uint8)
        dbits, dminbits = 0x1F5C, 0x2123          # small normal scales
    blk = _q4k_block(dbits, dminbits, sc, mn, qs)
    got = _vals(oracle_lib, gs.Q4_K, blk, 256)
    exp = [_round_f32(v) for v in _q4k_closed_form(dbits, dminbits, sc, mn, qs)]
    assert got.tolist() == [float(e) for e in exp]


@pytest.mark.parametrize("idx", range(len(eb.Q4K_EDGE)))
def test_q4_k_edge_blocks(oracle_lib, idx):
    """d = 0, dmin = 0, all-63 scales and mins, subnormal and negative d, the largest d: the
    oracle equals the exact d*sc*q - dmin*m rounded once, from the fields."""
    name, blk, (dbits, dminbits, sc, mn, qs) = eb.q4k_edge_blocks()[idx]
    got = _vals(oracle_lib, gs.Q4_K, blk, 256)
    exp = [_round_f32(v) for v in _q4k_closed_form(dbits, dminbits, sc, mn, qs)]
    assert got.tolist() == [float(v) for v in exp], name


@pytest.mark.parametrize("idx", range(len(eb.Q6K_EDGE)))
def test_q6_k_edge_blocks(oracle_lib, idx):
    """Scales -32 and 31 with a subnormal, an extreme and a normal d; uniform ql / qh bytes give
    one 6-bit code per quarter, so w_i = d * sc[i // 16] * (Q[(i % 128) // 32] - 32)."""
    name, blk, (dbits, sc, ql, qh) = eb.q6k_edge_blocks()[idx]
    Q = [((ql >> (4 * (qd >> 1))) & 15) | (((qh >> (2 * qd)) & 3) << 4) for qd in range(4)]
    d = Fraction(_f16(dbits))
    exp = [d * sc[i // 16] * (Q[(i % 128) // 32] - 32) for i in range(256)]
    got = _vals(oracle_lib, gs.Q6_K, blk, 256)
    assert [Fraction(float(v)) for v in got] == exp, name


def _scale_min_page(j, sc):
    # the page's get_scale_min_k4 (scaleMinK4), restated
    if j < 4:
        return sc[j] & 63, sc[j + 4] & 63
    return (sc[j + 4] & 0xF) | ((sc[j - 4] >> 6) << 4), (sc[j + 4] >> 4) | ((sc[j] >> 6) << 4)


def _dequant_q4k_page_loop(blk):
    """dequantQ4K of ternary_bonsai_2_dflash.js restated as its chunk loop, computing the
    f32 sequence d1 = d*s, m1 = dmin*m, w = d1*q - m1 (each product exact)."""
    d = np.float32(_f16(int(blk[0]) | (int(blk[1]) << 8)))
    dmin = np.float32(_f16(int(blk[2]) | (int(blk[3]) << 8)))
    sc = [int(v) for v in blk[4:16]]
    q = 16
    out = []
    for j in range(0, 256, 64):
        is_ = j // 32
        s1, m1 = _scale_min_page(is_, sc)
        s2, m2 = _scale_min_page(is_ + 1, sc)
        d1, mm1, d2, mm2 = d * np.float32(s1), dmin * np.float32(m1), d * np.float32(s2), dmin * np.float32(m2)
        lo = [np.float32(d1 * np.float32(int(blk[q + l]) & 15)) - mm1 for l in range(32)]
        hi = [np.float32(d2 * np.float32(int(blk[q + l]) >> 4)) - mm2 for l in range(32)]
        out += lo + hi
        q += 32
    return np.array(out, dtype=np.float32)


def test_q4_k_random_blocks_match_page_loop_and_exact(oracle_lib):
    w = gs.quant_blocks(gs.Q4_K, 3, 1024, seed=3)
    vals = oracle_lib.dequant(gs.Q4_K, w, 3, 1024).reshape(-1, 256)
    for bi, blk in enumerate(w.reshape(-1, 144)):
        page = _dequant_q4k_page_loop(blk)
        assert np.array_equal(vals[bi].view(np.uint32), page.view(np.uint32))
        sc = [int(v) for v in blk[4:16]]
        smn = [_scale_min_page(j, sc) for j in range(8)]
        exact = _q4k_closed_form(int(blk[0]) | (int(blk[1]) << 8), int(blk[2]) | (int(blk[3]) << 8),
                                 [s for s, _ in smn], [m for _, m in smn], blk[16:144])
        for i in range(0, 256, 7):
            assert float(vals[bi, i]) == float(_round_f32(exact[i]))


# ---- Q6_K ------------------------------------------------------------------------------

def _dequant_q6k_page_loop(blk):
    """dequantQ6K of ternary_bonsai_2_dflash.js restated as its loop over two halves."""
    d = Fraction(_f16(int(blk[208]) | (int(blk[209]) << 8)))
    out = [None] * 256
    ql, qh, sc, y = 0, 128, 192, 0
    s8 = lambda v: int(np.int8(np.uint8(v)))  # noqa: E731
    for _half in range(2):
        for l in range(32):
            is_ = l // 16
            q1 = ((blk[ql + l] & 0xF) | (((blk[qh + l] >> 0) & 3) << 4)) - 32
            q2 = ((blk[ql + l + 32] & 0xF) | (((blk[qh + l] >> 2) & 3) << 4)) - 32
            q3 = ((blk[ql + l] >> 4) | (((blk[qh + l] >> 4) & 3) << 4)) - 32
            q4 = ((blk[ql + l + 32] >> 4) | (((blk[qh + l] >> 6) & 3) << 4)) - 32
            out[y + l] = d * s8(blk[sc + is_]) * int(q1)
            out[y + l + 32] = d * s8(blk[sc + is_ + 2]) * int(q2)
            out[y + l + 64] = d * s8(blk[sc + is_ + 4]) * int(q3)
            out[y + l + 96] = d * s8(blk[sc + is_ + 6]) * int(q4)
        y += 128
        ql += 64
        qh += 32
        sc += 8
    return out


def test_q6_k_random_blocks_match_page_loop(oracle_lib):
    w = gs.quant_blocks(gs.Q6_K, 3, 1024, seed=5)
    vals = oracle_lib.dequant(gs.Q6_K, w, 3, 1024).reshape(-1, 256)
    for bi, blk in enumerate(w.reshape(-1, 210)):
        exact = _dequant_q6k_page_loop(blk.astype(np.int64))
        # d*scale*(q-32) has at most 23 significant bits: exact in f32
        assert [Fraction(float(v)) for v in vals[bi]] == exact


def test_q6_k_one_bit_blocks(oracle_lib):
    """Every element reads its own low-4 and high-2 bits: set exactly one code bit and check
    that exactly one element moves, by the amount its bit weight says."""
    base = np.zeros(210, dtype=np.uint8)
    base[192:208] = np.arange(1, 17, dtype=np.uint8)     # scales 1..16 -> scale index visible
    base[208:210] = [0x00, 0x3C]                         # d = 1
    v0 = _vals(oracle_lib, gs.Q6_K, base, 256)
    # all codes 0 -> q - 32 = -32: element i has value -32 * scale(i)
    for i in range(256):
        n, r = divmod(i, 128)
        qd, l = divmod(r, 32)
        assert v0[i] == -32.0 * (8 * n + l // 16 + 2 * qd + 1)
    for byte in list(range(0, 192, 5)) + [191]:
        for bit in (0, 3, 4, 7):
            blk = base.copy()
            blk[byte] |= np.uint8(1 << bit)
            diff = np.nonzero(_vals(oracle_lib, gs.Q6_K, blk, 256) != v0)[0]
            assert diff.size == 1, (byte, bit)
            i = int(diff[0])
            n, r = divmod(i, 128)
            qd, l = divmod(r, 32)
            if byte < 128:   # ql: element uses low nibble (qd < 2) or high nibble
                assert byte == 64 * n + l + 32 * (qd & 1)
                assert (bit >= 4) == (qd >= 2)
                weight = 1 << (bit % 4)
            else:            # qh: bits 2qd, 2qd + 1 are the element's bits 4, 5
                assert byte - 128 == 32 * n + l and bit // 2 == qd
                weight = 16 << (bit % 2)
            scale = 8 * n + l // 16 + 2 * qd + 1
            assert _vals(oracle_lib, gs.Q6_K, blk, 256)[i] - v0[i] == weight * scale


def test_block_value_sizes(oracle_lib):
    assert gs.row_bytes(gs.Q8_0, 2560) == 2720
    assert gs.row_bytes(gs.Q4_0, 2816) == 1584
    assert gs.row_bytes(gs.Q4_K, 5120) == 2880
    assert gs.row_bytes(gs.Q6_K, 5120) == 4200
    # one expert record of the Qwen3-30B-A3B-shaped MoE: 5,013,504 bytes
    assert gs.moe_expert_record_layout()[3] == 5013504
