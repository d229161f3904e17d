"""Hand-built GGUF blocks whose fields sit at the formats' edge values.

The blocks are packed from named fields (byte layout only, no decoding and no products): the
CPU pins (test_oracle_blocks.py) check the oracle's dequantized values against closed forms of
these fields, and the GPU one-hot tests feed the same blocks through every CUDA decoder.

Q8_0 / Q4_0 blocks come from tests/golden/hand_blocks.txt.  Q4_K and Q6_K blocks are packed
here from their fields, following the layouts of ternary_bonsai_2_dflash.js ("Layouts follow
ggml-quants.c": dequantQ4K with scaleMinK4, dequantQ6K).
"""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_blocks.txt")


def hand_blocks():
    """name -> (type name, block bytes) for every line of the golden file."""
    out = {}
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        name, typ, hx = line.split()
        out[name] = (typ, np.frombuffer(bytes.fromhex(hx), dtype=np.uint8).copy())
    return out


def pack_q4k_scales(sc, mn):
    """8 six-bit scales and mins into the 12 bytes of block_q4_K.scales: for j < 4 the low
    6 bits of byte j / j + 4 are sc[j] / mn[j] and their top 2 bits carry bits 4..5 of
    sc[j + 4] / mn[j + 4]; byte j + 8 holds the low 4 bits of sc[j + 4] and mn[j + 4]."""
    b = [0] * 12
    for j in range(4):
        b[j] = (sc[j] & 63) | ((sc[j + 4] >> 4) << 6)
        b[j + 4] = (mn[j] & 63) | ((mn[j + 4] >> 4) << 6)
        b[j + 8] = (sc[j + 4] & 15) | ((mn[j + 4] & 15) << 4)
    return b


def q4k_block(dbits, dminbits, sc, mn, qs):
    blk = np.zeros(144, dtype=np.uint8)
    blk[0:2] = [dbits & 255, dbits >> 8]
    blk[2:4] = [dminbits & 255, dminbits >> 8]
    blk[4:16] = pack_q4k_scales(sc, mn)
    blk[16:144] = np.asarray(qs, dtype=np.uint8)
    return blk


def q6k_block(dbits, sc, ql_byte, qh_byte):
    """Q6_K block with every ql byte = ql_byte, every qh byte = qh_byte, int8 scales sc[16]."""
    blk = np.zeros(210, dtype=np.uint8)
    blk[0:128] = ql_byte
    blk[128:192] = qh_byte
    blk[192:208] = np.asarray(sc, dtype=np.int8).view(np.uint8)
    blk[208:210] = [dbits & 255, dbits >> 8]
    return blk


# (name, d bits, dmin bits, scales, mins, qs byte pattern as a function of the byte index)
Q4K_EDGE = [
    ("q4k_d_zero", 0x0000, 0x3C00, [1, 2, 3, 4, 5, 6, 7, 8], [0, 1, 2, 63, 5, 6, 7, 63],
     lambda i: (i % 16) | ((15 - i % 16) << 4)),                      # w = -dmin * m
    ("q4k_dmin_zero_all63", 0x3800, 0x0000, [63] * 8, [63] * 8,
     lambda i: 0xF0 if i % 2 else 0x0F),                              # w = d * 63 * q
    ("q4k_subnormal", 0x0001, 0x0003, [63] * 8, [63] * 8, lambda i: 0xFF),
    ("q4k_negative_d", 0xBC00, 0x0001, [63, 0, 31, 32, 1, 62, 15, 48], [48, 15, 62, 1, 32, 31, 0, 63],
     lambda i: (i * 37) & 0xFF),                                      # one rounding of -sc q - 2^-24 m
    ("q4k_extreme", 0x7BFF, 0x7BFF, [63, 63, 0, 0, 63, 1, 1, 63], [0, 63, 63, 0, 1, 63, 63, 1],
     lambda i: 0xF0 | (i & 15)),
]

# (name, d bits, int8 scales, ql byte, qh byte): every element has the same 6-bit code per
# quarter qd = (i % 128) // 32, so w_i = d * sc[i // 16] * (Q[qd] - 32)
Q6K_EDGE = [
    ("q6k_subnormal_d", 0x0001, [-32, 31] * 8, 0xFF, 0xFF),          # Q = 63 everywhere
    ("q6k_extreme_d", 0xFBFF, [31, -32, 1, -1] * 4, 0x00, 0x00),      # Q = 0 everywhere
    ("q6k_mixed_quarters", 0x3C00, list(range(-32, 32, 4)), 0xF0, 0xCC),  # Q = [0, 48, 15, 63]
    ("q6k_small_normal", 0x0400, [31, -32] * 8, 0x5A, 0x96),
]


def q4k_edge_blocks():
    out = []
    for name, d, dm, sc, mn, pat in Q4K_EDGE:
        qs = [pat(i) & 0xFF for i in range(128)]
        out.append((name, q4k_block(d, dm, sc, mn, qs), (d, dm, sc, mn, qs)))
    return out


def q6k_edge_blocks():
    return [(name, q6k_block(d, sc, ql, qh), (d, sc, ql, qh)) for name, d, sc, ql, qh in Q6K_EDGE]


def edge_blocks(qtype):
    """All edge blocks of one type, as a list of uint8 arrays (one block each)."""
    import gguf_synth as gs

    if qtype in (gs.Q8_0, gs.Q4_0):
        tname = "Q8_0" if qtype == gs.Q8_0 else "Q4_0"
        return [b for _, (t, b) in sorted(hand_blocks().items()) if t == tname]
    if qtype == gs.Q4_K:
        return [b for _, b, _ in q4k_edge_blocks()]
    return [b for _, b, _ in q6k_edge_blocks()]


def matrix_with_edge_blocks(qtype, M, N, seed):
    """Raw [M][N] weights: seeded random blocks with the edge blocks dealt over the rows and
    block columns (row m, block column b holds edge block (m + 3 b) mod n_edge wherever
    (m + b) is even)."""
    import gguf_synth as gs

    qk, bb = gs.BLOCK[qtype]
    w = gs.quant_blocks(qtype, M, N, seed=seed, stream=qtype).reshape(M, N // qk, bb).copy()
    edge = edge_blocks(qtype)
    for m in range(M):
        for b in range(N // qk):
            if (m + b) % 2 == 0:
                w[m, b] = edge[(m + 3 * b) % len(edge)]
    return w.reshape(-1)
