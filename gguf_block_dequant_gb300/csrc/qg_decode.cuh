// qg_decode.cuh -- per-block-type lane decoders shared by the GEMV and MoE kernels.
//
// A warp step covers one "group" of SG consecutive elements of a row.  Lane l owns a fixed
// unit of the group (16 elements for Q8_0 / Q4_0, 32 for Q4_K / Q6_K) and reads that unit's
// bytes straight from the raw GGUF block in shared memory.  The unit is delivered in NCH
// chunks of 4 values; chunk ch of lane l multiplies the activations at 32-float row
// xrow(l, ch) of the group and 16-byte unit xunit(l, ch) of that row.  The activations sit
// in shared memory with the TMA 128-byte swizzle (16-byte unit u of row R stored at
// u ^ (R & 7)); the lane -> (row, unit) maps below make every 16-byte activation load of a
// warp touch each bank group exactly four times (no bank conflicts).
//
// Block layouts (ggml-quants, as the engine pages describe them):
//   Q8_0  34 B: f16 d, int8 q[32]                              w = d * q
//   Q4_0  18 B: f16 d, u8 qs[16]; byte j -> elements j (low nibble), j + 16 (high)
//                                                              w = d * (nibble - 8)
//   Q4_K 144 B: f16 d, f16 dmin, u8 scales[12], u8 qs[128]; element 64c + l (l < 32) is the
//               low nibble of qs[32c + l] in sub-block 2c, element 64c + 32 + l the high
//               nibble in sub-block 2c + 1;                     w = d*sc*q - dmin*m
//   Q6_K 210 B: u8 ql[128], u8 qh[64], int8 sc[16], f16 d; element 128n + 32qd + l takes
//               4 bits of ql[64n + 32(qd & 1) + l] (low nibble for qd < 2) and 2 bits of
//               qh[32n + l] at bit 2qd; scale sc[8n + l/16 + 2qd]; w = d * sc * (q - 32)
//
// Codes become exact floats with the magic-number method (the integer placed in the low
// mantissa bits of 2^23, then 2^23 plus the format's bias subtracted); every dequantized
// weight equals the oracle's value.
#pragma once

#include "qg_common.cuh"

// 8 bytes starting at a 2-byte (or 1-byte) aligned shared address, as two words
QG_DEVICE void lds8_any(uint32_t addr, uint32_t &lo, uint32_t &hi) {
  const uint32_t b = addr & ~3u, sh = (addr & 3u) * 8u;
  uint32_t w0, w1, w2;
  QG_LDS32(b, 0, w0);
  QG_LDS32(b, 4, w1);
  QG_LDS32(b, 8, w2);
  lo = __funnelshift_r(w0, w1, sh);
  hi = __funnelshift_r(w1, w2, sh);
}

QG_DEVICE void magic4(uint32_t v, float off, f2 &a, f2 &b) {
  const f2 o = mk2(off, off);
  a = add2(mk2(magic_byte(v, 0), magic_byte(v, 1)), o);
  b = add2(mk2(magic_byte(v, 2), magic_byte(v, 3)), o);
}

template <int QT>
struct Dec;

// ---------------------------------------------------------------------------------------
template <>
struct Dec<QG_TYPE_Q8_0> {
  static constexpr int QK = 32, BB = 34, SG = 512, NCH = 4, GB = 16 * 34;
  // lane = 2 * bl + h: block bl of the group, code bytes 16h .. 16h + 15 (elements 16h ..)
  QG_DEVICE static int block_first(int lane) { return 32 * (lane >> 1); }
  QG_DEVICE static int woff(int lane) { return 34 * (lane >> 1); }
  QG_DEVICE static int xrow(int lane, int) { return lane >> 1; }
  QG_DEVICE static int xunit(int lane, int ch) { return 4 * (lane & 1) + ch; }
  struct U {
    float d;
    uint32_t c[4];
  };
  QG_DEVICE static U load(uint32_t blk, int lane) {
    U u;
    uint32_t d16;
    QG_LDS16(blk, 0, d16);
    u.d = h2f(d16);
    const uint32_t a = blk + 2u + 16u * static_cast<uint32_t>(lane & 1), b = a & ~3u, sh = (a & 3u) * 8u;
    uint32_t w0, w1, w2, w3, w4;
    QG_LDS32(b, 0, w0);
    QG_LDS32(b, 4, w1);
    QG_LDS32(b, 8, w2);
    QG_LDS32(b, 12, w3);
    QG_LDS32(b, 16, w4);
    u.c[0] = __funnelshift_r(w0, w1, sh);
    u.c[1] = __funnelshift_r(w1, w2, sh);
    u.c[2] = __funnelshift_r(w2, w3, sh);
    u.c[3] = __funnelshift_r(w3, w4, sh);
    return u;
  }
  QG_DEVICE static void codes(const U &u, int ch, f2 &q01, f2 &q23) {
    magic4(u.c[ch] ^ 0x80808080u, -8388736.0f, q01, q23);  // int8 q + 128, then -(2^23 + 128)
  }
  QG_DEVICE static void weights(const U &u, int ch, f2 &w01, f2 &w23) {
    f2 q01, q23;
    codes(u, ch, q01, q23);
    const f2 d2 = mk2(u.d, u.d);
    w01 = mul2(q01, d2);
    w23 = mul2(q23, d2);
  }
  QG_DEVICE static float xaux(const float4 *) { return 0.f; }
  QG_DEVICE static float dot1(const U &u, const float4 *xc, float) {
    f2 s = mk2(0.f, 0.f);
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch) {
      f2 q01, q23;
      codes(u, ch, q01, q23);
      s = fma2(q01, mk2(xc[ch].x, xc[ch].y), s);
      s = fma2(q23, mk2(xc[ch].z, xc[ch].w), s);
    }
    return u.d * (s.x + s.y);
  }
};

// ---------------------------------------------------------------------------------------
template <>
struct Dec<QG_TYPE_Q4_0> {
  static constexpr int QK = 32, BB = 18, SG = 512, NCH = 4, GB = 16 * 18;
  // lane = 2 * bl + h: code bytes 8h .. 8h + 7 of block bl; chunks 0, 1 = their low nibbles
  // (elements 8h + 4ch ..), chunks 2, 3 = their high nibbles (elements 16 + 8h + 4(ch - 2) ..)
  QG_DEVICE static int block_first(int lane) { return 32 * (lane >> 1); }
  QG_DEVICE static int woff(int lane) { return 18 * (lane >> 1); }
  QG_DEVICE static int xrow(int lane, int) { return lane >> 1; }
  QG_DEVICE static int xunit(int lane, int ch) { return 4 * (ch >> 1) + 2 * (lane & 1) + (ch & 1); }
  struct U {
    float d;
    uint32_t c[2];
  };
  QG_DEVICE static U load(uint32_t blk, int lane) {
    U u;
    uint32_t d16;
    QG_LDS16(blk, 0, d16);
    u.d = h2f(d16);
    lds8_any(blk + 2u + 8u * static_cast<uint32_t>(lane & 1), u.c[0], u.c[1]);
    return u;
  }
  QG_DEVICE static void codes(const U &u, int ch, f2 &q01, f2 &q23) {
    magic4((u.c[ch & 1] >> (4 * (ch >> 1))) & 0x0F0F0F0Fu, -8388616.0f, q01, q23);  // -(2^23 + 8)
  }
  QG_DEVICE static void weights(const U &u, int ch, f2 &w01, f2 &w23) {
    f2 q01, q23;
    codes(u, ch, q01, q23);
    const f2 d2 = mk2(u.d, u.d);
    w01 = mul2(q01, d2);
    w23 = mul2(q23, d2);
  }
  QG_DEVICE static float xaux(const float4 *) { return 0.f; }
  // one-token dot: the high nibbles are used in place (byte & 0xF0 = 16 q), which gives
  // 16 (q - 8) after subtracting 2^23 + 128; their sum is scaled by 1/16 (exact)
  QG_DEVICE static float dot1(const U &u, const float4 *xc, float) {
    f2 lo = mk2(0.f, 0.f), hi = mk2(0.f, 0.f);
#pragma unroll
    for (int ch = 0; ch < 2; ++ch) {
      f2 q01, q23;
      magic4(u.c[ch] & 0x0F0F0F0Fu, -8388616.0f, q01, q23);  // q - 8
      lo = fma2(q01, mk2(xc[ch].x, xc[ch].y), lo);
      lo = fma2(q23, mk2(xc[ch].z, xc[ch].w), lo);
      magic4(u.c[ch] & 0xF0F0F0F0u, -8388736.0f, q01, q23);  // 16 (q - 8)
      hi = fma2(q01, mk2(xc[ch + 2].x, xc[ch + 2].y), hi);
      hi = fma2(q23, mk2(xc[ch + 2].z, xc[ch + 2].w), hi);
    }
    return u.d * fmaf(hi.x + hi.y, 0.0625f, lo.x + lo.y);
  }
};

// ---------------------------------------------------------------------------------------
template <>
struct Dec<QG_TYPE_Q4_K> {
  static constexpr int QK = 256, BB = 144, SG = 1024, NCH = 8, GB = 4 * 144;
  // lane = 8 * bl + s: sub-block s of block bl (elements 32s .. 32s + 31), the low (s even)
  // or high (s odd) nibbles of qs[32 (s >> 1) .. + 32]; chunk ch = elements 32s + 4ch ..
  QG_DEVICE static int block_first(int lane) { return 256 * (lane >> 3); }
  QG_DEVICE static int woff(int lane) { return 144 * (lane >> 3); }
  QG_DEVICE static int xrow(int lane, int) { return lane; }
  QG_DEVICE static int xunit(int, int ch) { return ch; }
  struct U {
    float dsc, dm;
    uint4 q0, q1;
    uint32_t sh;
  };
  // one-token path: odd sub-blocks use their high nibbles in place (byte & 0xF0 = 16 q)
  QG_DEVICE static uint32_t dot_mask(int lane) { return (lane & 1) ? 0xF0F0F0F0u : 0x0F0F0F0Fu; }
  QG_DEVICE static U load(uint32_t blk, int lane) {
    uint4 h;  // d | dmin, scales[0..3], scales[4..7], scales[8..11]
    QG_LDS128(blk, 0, h.x, h.y, h.z, h.w);
    const int s = lane & 7, j = s & 3;
    const uint32_t a0 = (h.y >> (8 * j)) & 0xFFu, a1 = (h.z >> (8 * j)) & 0xFFu, a2 = (h.w >> (8 * j)) & 0xFFu;
    // 6-bit scale and min of sub-block s (get_scale_min_k4)
    const uint32_t sc = (s < 4) ? (a0 & 63u) : ((a2 & 15u) | ((a0 >> 6) << 4));
    const uint32_t mn = (s < 4) ? (a1 & 63u) : ((a2 >> 4) | ((a1 >> 6) << 4));
    U u;
    u.dsc = h2f(h.x) * static_cast<float>(sc);       // exact (<= 17 significant bits)
    u.dm = h2f(h.x >> 16) * static_cast<float>(mn);  // exact
    const uint32_t qb = blk + 16u + 32u * static_cast<uint32_t>(s >> 1);
    QG_LDS128(qb, 0, u.q0.x, u.q0.y, u.q0.z, u.q0.w);
    QG_LDS128(qb, 16, u.q1.x, u.q1.y, u.q1.z, u.q1.w);
    u.sh = 4u * static_cast<uint32_t>(s & 1);
    return u;
  }
  QG_DEVICE static uint32_t word(const U &u, int ch) {
    switch (ch) {
      case 0: return u.q0.x;
      case 1: return u.q0.y;
      case 2: return u.q0.z;
      case 3: return u.q0.w;
      case 4: return u.q1.x;
      case 5: return u.q1.y;
      case 6: return u.q1.z;
      default: return u.q1.w;
    }
  }
  QG_DEVICE static void codes(const U &u, int ch, f2 &q01, f2 &q23) {
    magic4((word(u, ch) >> u.sh) & 0x0F0F0F0Fu, -8388608.0f, q01, q23);  // -2^23
  }
  // w = d*sc*q - dmin*m with one rounding (both products exact), as the format defines
  QG_DEVICE static void weights(const U &u, int ch, f2 &w01, f2 &w23) {
    f2 q01, q23;
    codes(u, ch, q01, q23);
    const f2 a = mk2(u.dsc, u.dsc), b = mk2(-u.dm, -u.dm);
    w01 = fma2(a, q01, b);
    w23 = fma2(a, q23, b);
  }
  QG_DEVICE static float xaux(const float4 *xc) {  // sum of the unit's 32 activations
    f2 s = mk2(0.f, 0.f);
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch) s = add2(s, add2(mk2(xc[ch].x, xc[ch].y), mk2(xc[ch].z, xc[ch].w)));
    return s.x + s.y;
  }
  // one-token dot in the factored form d*sc*sum(q x) - dmin*m*sum(x); odd sub-blocks read
  // 16 q from the high nibbles in place and scale d*sc by 1/16 (exact)
  QG_DEVICE static float dot1(const U &u, const float4 *xc, float xsum) {
    const uint32_t mask = (u.sh != 0u) ? 0xF0F0F0F0u : 0x0F0F0F0Fu;
    f2 s = mk2(0.f, 0.f);
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch) {
      f2 q01, q23;
      magic4(word(u, ch) & mask, -8388608.0f, q01, q23);
      s = fma2(q01, mk2(xc[ch].x, xc[ch].y), s);
      s = fma2(q23, mk2(xc[ch].z, xc[ch].w), s);
    }
    const float dsc = (u.sh != 0u) ? u.dsc * 0.0625f : u.dsc;
    return fmaf(dsc, s.x + s.y, -u.dm * xsum);
  }
};

// ---------------------------------------------------------------------------------------
template <>
struct Dec<QG_TYPE_Q6_K> {
  static constexpr int QK = 256, BB = 210, SG = 1024, NCH = 8, GB = 4 * 210;
  // lane = 8 * bl + 4 * n + a: half n of block bl, l in [8a, 8a + 8), all four quarters qd.
  // Chunk ch = (qd = ch >> 1, hh = (ch & 1) ^ n) covers l = 8a + 4hh .. + 3, i.e. elements
  // 128n + 32qd + 8a + 4hh ..; the hh swap on odd halves spreads the activation loads over
  // all bank groups.
  QG_DEVICE static int block_first(int lane) { return 256 * (lane >> 3); }
  QG_DEVICE static int woff(int lane) { return 210 * (lane >> 3); }
  QG_DEVICE static int xrow(int lane, int ch) { return (lane & ~7) + 4 * ((lane >> 2) & 1) + (ch >> 1); }
  QG_DEVICE static int xunit(int lane, int ch) { return 2 * (lane & 3) + ((ch & 1) ^ ((lane >> 2) & 1)); }
  struct U {
    uint32_t A[2], B[2], H[2];  // ql[64n + 8a ..], ql[64n + 32 + 8a ..], qh[32n + 8a ..]
    float ds[4];                // d * sc for qd = 0..3
    uint32_t n;
  };
  QG_DEVICE static U load(uint32_t blk, int lane) {
    const uint32_t n = static_cast<uint32_t>((lane >> 2) & 1), a = static_cast<uint32_t>(lane & 3);
    U u;
    u.n = n;
    lds8_any(blk + 64u * n + 8u * a, u.A[0], u.A[1]);
    lds8_any(blk + 64u * n + 32u + 8u * a, u.B[0], u.B[1]);
    lds8_any(blk + 128u + 32u * n + 8u * a, u.H[0], u.H[1]);
    // scales sc[8n + a/2 + 2qd] are bytes 0, 2, 4, 6 of the 8 bytes from sc[8n + a/2]
    uint32_t s0, s1, d16;
    lds8_any(blk + 192u + 8u * n + (a >> 1), s0, s1);
    QG_LDS16(blk, 208, d16);
    const float d = h2f(d16);
    u.ds[0] = d * static_cast<float>(static_cast<int8_t>(s0 & 0xFFu));
    u.ds[1] = d * static_cast<float>(static_cast<int8_t>((s0 >> 16) & 0xFFu));
    u.ds[2] = d * static_cast<float>(static_cast<int8_t>(s1 & 0xFFu));
    u.ds[3] = d * static_cast<float>(static_cast<int8_t>((s1 >> 16) & 0xFFu));
    return u;
  }
  QG_DEVICE static void codes(const U &u, int ch, f2 &q01, f2 &q23) {
    const int qd = ch >> 1;
    const uint32_t hh = static_cast<uint32_t>(ch & 1) ^ u.n;
    const uint32_t lo = (qd & 1) ? (hh ? u.B[1] : u.B[0]) : (hh ? u.A[1] : u.A[0]);
    const uint32_t hi = hh ? u.H[1] : u.H[0];
    const uint32_t q = ((lo >> (4 * (qd >> 1))) & 0x0F0F0F0Fu) | (((hi >> (2 * qd)) & 0x03030303u) << 4);
    magic4(q, -8388640.0f, q01, q23);  // -(2^23 + 32)
  }
  QG_DEVICE static void weights(const U &u, int ch, f2 &w01, f2 &w23) {
    f2 q01, q23;
    codes(u, ch, q01, q23);
    const float s = u.ds[ch >> 1];
    const f2 s2 = mk2(s, s);
    w01 = mul2(q01, s2);
    w23 = mul2(q23, s2);
  }
  QG_DEVICE static float xaux(const float4 *) { return 0.f; }
  QG_DEVICE static float dot1(const U &u, const float4 *xc, float) {
    float acc = 0.f;
#pragma unroll
    for (int qd = 0; qd < 4; ++qd) {
      f2 s = mk2(0.f, 0.f);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int ch = 2 * qd + h;
        f2 q01, q23;
        codes(u, ch, q01, q23);
        s = fma2(q01, mk2(xc[ch].x, xc[ch].y), s);
        s = fma2(q23, mk2(xc[ch].z, xc[ch].w), s);
      }
      acc = fmaf(u.ds[qd], s.x + s.y, acc);
    }
    return acc;
  }
};

// Byte offset, inside a group's activations, of chunk ch of lane `lane` in a buffer written
// by the TMA with the 128-byte swizzle.  Valid whenever the group's first row is a multiple
// of 8 rows from a 1024-byte aligned base (SG / 32 is 16 or 32 rows).
template <int QT>
QG_DEVICE uint32_t x_lane_off(int lane, int ch) {
  using D = Dec<QT>;
  const int R = D::xrow(lane, ch);
  return 128u * static_cast<uint32_t>(R) + 16u * static_cast<uint32_t>(D::xunit(lane, ch) ^ (R & 7));
}

// A lane's unit addresses prepared once per row for the one-token loop.  Consecutive groups
// of a row are GB bytes apart and GB is a multiple of 4 for every type, so the alignment of
// the lane's unit inside its 32-bit words is the same in every group of the row: the
// word-aligned base and the funnel-shift amount are computed once, and a group costs one add
// per address.
template <int QT>
struct RowPrep {
  uint32_t blk;
  QG_DEVICE void init(uint32_t b, int) { blk = b; }
  QG_DEVICE typename Dec<QT>::U load(uint32_t goff, int lane) const { return Dec<QT>::load(blk + goff, lane); }
};

template <>
struct RowPrep<QG_TYPE_Q8_0> {
  static_assert(Dec<QG_TYPE_Q8_0>::GB % 4 == 0, "groups keep the word alignment");
  uint32_t dp, cw, sh;  // the block's scale, the first word holding the lane's codes, shift
  QG_DEVICE void init(uint32_t b, int lane) {
    const uint32_t a = b + 2u + 16u * static_cast<uint32_t>(lane & 1);
    dp = b;
    cw = a & ~3u;
    sh = (a & 3u) * 8u;
  }
  QG_DEVICE Dec<QG_TYPE_Q8_0>::U load(uint32_t goff, int) const {
    Dec<QG_TYPE_Q8_0>::U u;
    uint32_t d16;
    QG_LDS16(dp + goff, 0, d16);
    u.d = h2f(d16);
    const uint32_t b = cw + goff;
    uint32_t w0, w1, w2, w3, w4;
    QG_LDS32(b, 0, w0);
    QG_LDS32(b, 4, w1);
    QG_LDS32(b, 8, w2);
    QG_LDS32(b, 12, w3);
    QG_LDS32(b, 16, w4);
    u.c[0] = __funnelshift_r(w0, w1, sh);
    u.c[1] = __funnelshift_r(w1, w2, sh);
    u.c[2] = __funnelshift_r(w2, w3, sh);
    u.c[3] = __funnelshift_r(w3, w4, sh);
    return u;
  }
};

template <>
struct RowPrep<QG_TYPE_Q4_0> {
  static_assert(Dec<QG_TYPE_Q4_0>::GB % 4 == 0, "groups keep the word alignment");
  uint32_t dp, cw, sh;
  QG_DEVICE void init(uint32_t b, int lane) {
    const uint32_t a = b + 2u + 8u * static_cast<uint32_t>(lane & 1);
    dp = b;
    cw = a & ~3u;
    sh = (a & 3u) * 8u;
  }
  QG_DEVICE Dec<QG_TYPE_Q4_0>::U load(uint32_t goff, int) const {
    Dec<QG_TYPE_Q4_0>::U u;
    uint32_t d16;
    QG_LDS16(dp + goff, 0, d16);
    u.d = h2f(d16);
    const uint32_t b = cw + goff;
    uint32_t w0, w1, w2;
    QG_LDS32(b, 0, w0);
    QG_LDS32(b, 4, w1);
    QG_LDS32(b, 8, w2);
    u.c[0] = __funnelshift_r(w0, w1, sh);
    u.c[1] = __funnelshift_r(w1, w2, sh);
    return u;
  }
};
