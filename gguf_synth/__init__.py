"""Seeded synthetic inputs: raw GGUF block bytes, activations and router weights.

This module is shared by the CPU oracle's tests, the CUDA parity tests and the
benchmark.  It holds no arithmetic of the method itself: it only draws random
bits and packs them into the byte layouts that the block formats define
(ggml-quants block structs, as the engine pages describe them:
`qwen3_moe_ssd.js` header comment for Q8_0, `gemma4_moe_ssd.js` Q4_0 comment,
`ternary_bonsai_2_dflash.js` "Layouts follow ggml-quants.c" for Q4_K / Q6_K).
It never decodes a block and never forms a product.

Random bits come from numpy's Philox4x64-10 bit generator (a published
counter-based generator, Salmon et al., SC'11) keyed by (seed, stream), read
through ``random_raw`` so that the stream does not depend on numpy's
distribution code.  Normals are Box-Muller in float64; f16 scales are produced
by numpy's round-to-nearest-even float16 cast.
"""
from __future__ import annotations

import numpy as np

# ggml type ids (the pages' GGML table uses the same numbering)
Q4_0 = 2
Q8_0 = 8
Q4_K = 12
Q6_K = 14

# type -> (elements per block, bytes per block)
BLOCK = {Q8_0: (32, 34), Q4_0: (32, 18), Q4_K: (256, 144), Q6_K: (256, 210)}
TYPE_NAME = {Q8_0: "q8_0", Q4_0: "q4_0", Q4_K: "q4_k", Q6_K: "q6_k"}
TYPE_BY_NAME = {v: k for k, v in TYPE_NAME.items()}

_CHUNK = 1 << 22  # u64 words drawn per Philox call (32 MiB)


def row_bytes(qtype: int, n: int) -> int:
    qk, bb = BLOCK[qtype]
    if n % qk:
        raise ValueError(f"row length {n} is not a multiple of {qk}")
    return (n // qk) * bb


def tensor_bytes(qtype: int, rows: int, n: int) -> int:
    return rows * row_bytes(qtype, n)


class Stream:
    """Counter-based stream of 64-bit words for one (seed, stream id)."""

    def __init__(self, seed: int, stream: int):
        key = np.array([seed & 0xFFFFFFFFFFFFFFFF, stream & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
        # full-range uint64 draws return the generator's raw words unchanged (the same
        # sequence as Philox.random_raw), through numpy's faster bulk fill
        self._gen = np.random.Generator(np.random.Philox(key=key))

    def words(self, n: int) -> np.ndarray:
        out = np.empty(n, dtype=np.uint64)
        for s in range(0, n, _CHUNK):
            e = min(n, s + _CHUNK)
            out[s:e] = self._gen.integers(0, 1 << 64, size=e - s, dtype=np.uint64, endpoint=False)
        return out

    def bytes(self, n: int) -> np.ndarray:
        w = self.words((n + 7) // 8)
        return w.view(np.uint8)[:n].copy()

    def uniform01(self, n: int) -> np.ndarray:
        """Doubles in (0, 1]: 53 high bits of each word, shifted off zero."""
        w = self.words(n)
        return ((w >> np.uint64(11)).astype(np.float64) + 1.0) * (1.0 / 9007199254740992.0)

    def normal(self, n: int) -> np.ndarray:
        """N(0, 1) doubles by Box-Muller (cosine branch only)."""
        u1 = self.uniform01(n)
        u2 = self.uniform01(n)
        return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)

    def ints(self, n: int, lo: int, hi: int, dtype=np.int32) -> np.ndarray:
        """Integers uniform in [lo, hi] (hi - lo < 65536) by 16-bit multiply-shift: value i
        comes from the i-th 16-bit piece of the word stream (4 pieces per word, low first)."""
        span = hi - lo + 1
        if not 0 < span <= 65536:
            raise ValueError("span out of range")
        out = np.empty(n, dtype=dtype)
        step = 4 * _CHUNK  # a multiple of 4 values: chunking never splits a word
        for s in range(0, n, step):
            e = min(n, s + step)
            w = self.words((e - s + 3) // 4)
            u = w.view(np.uint16)[:e - s].astype(np.uint32)
            u *= np.uint32(span)
            u >>= np.uint32(16)
            v = u.view(np.int32)
            v += lo
            out[s:e] = v
        return out


def _f16_bytes(v: np.ndarray) -> np.ndarray:
    """float64 values -> little-endian f16 bytes (RNE), shape [n, 2]."""
    h = v.astype(np.float16).view(np.uint16).astype("<u2")
    return h.view(np.uint8).reshape(-1, 2)


# stream ids inside one tensor, so that every field has its own counter space
_S_D, _S_Q, _S_DMIN, _S_SC, _S_QH = 1, 2, 3, 4, 5


def _sub(stream_id: int, field: int) -> int:
    return (stream_id << 8) | field


def quant_blocks(qtype: int, rows: int, n: int, seed: int = 0, stream: int = 0) -> np.ndarray:
    """Raw GGUF blocks for a [rows][n] tensor, row-major, as a flat uint8 array.

    Distributions (one draw per field, every field from its own stream):
      Q8_0: d = f16(|N(0,1)| * 0.02); 32 codes uniform in [-127, 127]
      Q4_0: d = f16(|N(0,1)| * 0.02); 16 bytes uniform (both nibbles uniform 0..15)
      Q4_K: d, dmin = f16(|N(0,1)| * 0.01); 12 scale bytes uniform; 128 nibble bytes uniform
      Q6_K: ql, qh bytes uniform; 16 int8 scales uniform in [-32, 31]; d = f16(|N(0,1)| * 0.01)
    """
    qk, bb = BLOCK[qtype]
    nblk = rows * (n // qk)
    row_bytes(qtype, n)  # validates n
    out = np.empty((nblk, bb), dtype=np.uint8)
    g = lambda f: Stream(seed, _sub(stream, f))  # noqa: E731
    if qtype == Q8_0:
        out[:, 0:2] = _f16_bytes(np.abs(g(_S_D).normal(nblk)) * 0.02)
        out[:, 2:34] = g(_S_Q).ints(nblk * 32, -127, 127, np.int8).view(np.uint8).reshape(nblk, 32)
    elif qtype == Q4_0:
        out[:, 0:2] = _f16_bytes(np.abs(g(_S_D).normal(nblk)) * 0.02)
        out[:, 2:18] = g(_S_Q).bytes(nblk * 16).reshape(nblk, 16)
    elif qtype == Q4_K:
        out[:, 0:2] = _f16_bytes(np.abs(g(_S_D).normal(nblk)) * 0.01)
        out[:, 2:4] = _f16_bytes(np.abs(g(_S_DMIN).normal(nblk)) * 0.01)
        out[:, 4:16] = g(_S_SC).bytes(nblk * 12).reshape(nblk, 12)
        out[:, 16:144] = g(_S_Q).bytes(nblk * 128).reshape(nblk, 128)
    elif qtype == Q6_K:
        out[:, 0:128] = g(_S_Q).bytes(nblk * 128).reshape(nblk, 128)
        out[:, 128:192] = g(_S_QH).bytes(nblk * 64).reshape(nblk, 64)
        out[:, 192:208] = g(_S_SC).ints(nblk * 16, -32, 31, np.int8).view(np.uint8).reshape(nblk, 16)
        out[:, 208:210] = _f16_bytes(np.abs(g(_S_D).normal(nblk)) * 0.01)
    else:
        raise ValueError(f"unsupported type {qtype}")
    return out.reshape(-1)


def activations(T: int, n: int, seed: int = 0, stream: int = 1000, scale: float = 1.0) -> np.ndarray:
    """f32 [T][n] token-major activations, N(0, scale^2)."""
    return (Stream(seed, stream).normal(T * n) * scale).astype(np.float32).reshape(T, n)


def router_weights(E: int, H: int, seed: int = 0, stream: int = 2000) -> np.ndarray:
    """f32 [E][H] router matrix, N(0, 0.02^2)."""
    return (Stream(seed, stream).normal(E * H) * 0.02).astype(np.float32).reshape(E, H)


# ---- shapes of the workloads ----------------------------------------------------------

# Qwen3-4B-shaped dense decode projections: name -> (M rows, N row length)
QWEN3_4B_PROJ = {
    "attn_q": (4096, 2560),
    "attn_k": (1024, 2560),
    "attn_v": (1024, 2560),
    "attn_output": (2560, 4096),
    "ffn_gate": (9728, 2560),
    "ffn_up": (9728, 2560),
    "ffn_down": (2560, 9728),
    "output_tied": (151936, 2560),
}

# Qwen3-30B-A3B-shaped MoE layer
MOE_H, MOE_F, MOE_E, MOE_K = 2048, 768, 128, 8


def moe_expert_record_layout(H: int = MOE_H, F: int = MOE_F, qtype: int = Q8_0):
    """Byte layout of one expert record: gate rows (F x H), then up rows (F x H), then
    down rows (H x F), each as raw blocks.  Returns (gate_off, up_off, down_off, stride)."""
    g = tensor_bytes(qtype, F, H)
    d = tensor_bytes(qtype, H, F)
    return 0, g, 2 * g, 2 * g + d


def moe_experts(E: int = MOE_E, H: int = MOE_H, F: int = MOE_F, qtype: int = Q8_0,
                seed: int = 0, stream: int = 3000) -> np.ndarray:
    """All E expert records, contiguous: [E][stride] bytes."""
    go, uo, do, stride = moe_expert_record_layout(H, F, qtype)
    out = np.empty((E, stride), dtype=np.uint8)
    gate = quant_blocks(qtype, E * F, H, seed, stream + 1).reshape(E, -1)
    out[:, go:uo] = gate
    del gate
    up = quant_blocks(qtype, E * F, H, seed, stream + 2).reshape(E, -1)
    out[:, uo:do] = up
    del up
    out[:, do:stride] = quant_blocks(qtype, E * H, F, seed, stream + 3).reshape(E, -1)
    return out
