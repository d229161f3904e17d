// qg_gemv_mt.cu -- quantized GEMV over several token columns (2 <= T <= 16) for Q8_0 / Q4_0 /
// Q4_K / Q6_K rows of whole 256-element units.
//
// Y[t][m] = sum_k W[m][k] * X[t][k]  (matmulQ8T / matmulQ4T of the engine pages: one pass
// over the weights serves every token column), raw GGUF blocks decoded in registers, f32
// accumulation.
//
// Why a separate kernel from the one-token path: with T columns every decoded weight meets T
// activations, so the activation reads, not the weight decode, set the cost.  Here a lane
// owns ROWS, not a slice of K: lane (i, q) = lane i + 8 q holds rows i and i + 8 of a
// 16-row group and the 16-byte activation units q and q + 4 of every 32-element block.  The
// eight lanes with the same q read the same activation unit, so a warp-wide 16-byte load is
// one shared-memory wavefront (instead of four), and each loaded unit (4 values of one token)
// feeds four packed FMAs (two rows x two pairs).
//
// Work mapping: persistent CTAs, one per SM.  Items are (16-row group, chunk of 8 or 16
// blocks) pairs, dealt to the CTA's warps in contiguous ranges equal to within one item;
// every warp streams its items through a private ring of shared-memory slots with one bulk
// copy per row segment (rows are 16-byte aligned).  A group whose chunks span two warps'
// ranges is summed from their parts in chunk order.  The activations of the CTA's K range
// stay resident in shared memory (2-D tensor copies, 128-byte swizzle).  When all of K does
// not fit, a cluster of KS CTAs splits K: rank r covers the r-th K range of the same row
// groups, and after a cluster barrier every rank sums a share of the groups over the ranks'
// shared memory (distributed shared memory, rank order: deterministic) and writes Y.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "qg_decode.cuh"
#include "qg_host.h"
#include "qg_pipe.cuh"

__device__ unsigned int g_qg_status_mt;  // this translation unit's device status word

namespace {

constexpr int kNS = 4;     // most slots per warp
constexpr int kMats = 4;   // matrices per launch (sharing x)
constexpr int kRG = 16;    // rows per group

struct MtArgs {
  const uint8_t *w[kMats];
  float *y[kMats];
  uint32_t rg0[kMats + 1];  // matrix j owns row groups [rg0[j], rg0[j + 1])
  uint32_t M[kMats];
  int nmat;
  uint32_t row_bytes;       // multiple of 16
  uint32_t groups;          // row groups of the launch
  int N, T;
  int KS;                   // CTAs per cluster (K ranges)
  int units;                // 8-block units per row (N / 256)
  int cbu;                  // units per chunk (1 or 2)
  uint32_t seg;             // slot bytes per row: cbu * 8 blocks
  uint32_t stage_bytes;     // 16 rows x seg
  int NS;
  int xR;                   // activation rows (32 floats) per token in the buffer (>= the CTA's range)
  int box_rows;
  int max_groups;           // most row groups of one cluster (KS > 1: size of `outs`)
  uint32_t off_x, off_ring, off_outs;
  int early_weights;
  uintptr_t mend[kMats];  // Q6_K: last 16-byte boundary of each matrix (its rows are not 16-byte multiples)
};

QG_DEVICE void mt_status(unsigned int bits) { atomicOr(&g_qg_status_mt, bits); }

// bytes of one 256-element unit of a row: eight 32-element blocks (Q8_0, Q4_0) or one
// super-block (Q4_K)
template <int QT>
__host__ __device__ constexpr uint32_t unit_bytes() {
  return QT == QG_TYPE_Q8_0 ? 8u * 34u : QT == QG_TYPE_Q4_0 ? 8u * 18u : QT == QG_TYPE_Q4_K ? 144u : 210u;
}

QG_DEVICE uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
QG_DEVICE void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// address of the same shared-memory location in CTA `rank` of the cluster
QG_DEVICE uint32_t map_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
QG_DEVICE float ld_cluster_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}
QG_DEVICE float4 ld_cluster_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// 4 code bytes at a shared address that is 4-byte aligned (ALIGNED) or 2 bytes past it
template <bool ALIGNED>
QG_DEVICE uint32_t lds_code4(uint32_t addr) {
  if constexpr (ALIGNED) {
    return lds_u32(addr);
  } else {
    return __byte_perm(lds_u32(addr - 2u), lds_u32(addr + 2u), 0x5432);
  }
}

// Weights of rows (i, i + 8) for the activation units q and q + 4 of block `blk` of a chunk:
// w[r][h] holds the four values of unit q + 4h as two pairs.
template <int QT, int BLK>
QG_DEVICE void mt_weights(uint32_t row_i, uint32_t row_j, int q, f2 (&w)[2][2][2]) {
  constexpr uint32_t BB = QT == QG_TYPE_Q8_0 ? 34u : 18u;
  // the block starts at BB * BLK from a 4-byte aligned row; its codes at +2 are 4-byte
  // aligned exactly when BB * BLK + 2 is
  constexpr bool AL = ((BB * BLK + 2u) & 3u) == 0;
  const uint32_t rows[2] = {row_i + BB * BLK, row_j + BB * BLK};
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const float d = h2f(lds_u16(rows[r]));
    const f2 d2 = mk2(d, d);
    if constexpr (QT == QG_TYPE_Q8_0) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t c = lds_code4<AL>(rows[r] + 2u + 16u * h + 4u * q);
        f2 a, b;
        magic4(c ^ 0x80808080u, -8388736.0f, a, b);  // int8 q + 128, then -(2^23 + 128)
        w[r][h][0] = mul2(a, d2);
        w[r][h][1] = mul2(b, d2);
      }
    } else {
      // byte j of the nibbles holds element j (low) and j + 16 (high): unit q is the low
      // nibbles of bytes 4q .. 4q + 3, unit q + 4 their high nibbles
      const uint32_t c = lds_code4<AL>(rows[r] + 2u + 4u * q);
      f2 a, b;
      magic4(c & 0x0F0F0F0Fu, -8388616.0f, a, b);  // nibble - 8
      w[r][0][0] = mul2(a, d2);
      w[r][0][1] = mul2(b, d2);
      magic4((c >> 4) & 0x0F0F0F0Fu, -8388616.0f, a, b);
      w[r][1][0] = mul2(a, d2);
      w[r][1][1] = mul2(b, d2);
    }
  }
}

// Q4_K: the 16-byte head of a super-block (f16 d, f16 dmin, 12 bytes of packed 6-bit scales
// and mins) for rows i and i + 8
struct Q4kHead {
  float d, dmin;
  uint32_t s0, s1, s2;  // scale bytes 0-3, 4-7, 8-11
};
QG_DEVICE Q4kHead q4k_head(uint32_t blk) {
  const uint4 v = lds_v4(blk);
  Q4kHead h;
  h.d = h2f(v.x & 0xFFFFu);
  h.dmin = h2f(v.x >> 16);
  h.s0 = v.y;
  h.s1 = v.z;
  h.s2 = v.w;
  return h;
}
QG_DEVICE uint32_t q4k_byte(const Q4kHead &h, int i) {
  const uint32_t w = i < 4 ? h.s0 : i < 8 ? h.s1 : h.s2;
  return (w >> (8 * (i & 3))) & 0xFFu;
}
// Weights of sub-block SB (elements 32 SB .. 32 SB + 31) of a Q4_K super-block for rows i and
// i + 8, activation units q and q + 4: w = (d sc) q - dmin m as one fused multiply-add (both
// products are exact in f32, so this is the single rounding of the exact value).  Sub-block
// 2c takes the low nibbles of qs[32c ..], 2c + 1 the high ones; its 6-bit scale and min are
// unpacked from the 12 packed bytes as ggml's get_scale_min_k4 lays them out.
template <int SB>
QG_DEVICE void mt_weights_q4k(uint32_t blk_i, uint32_t blk_j, const Q4kHead (&hd)[2], int q, f2 (&w)[2][2][2]) {
  const uint32_t rows[2] = {blk_i, blk_j};
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    uint32_t sc, mn;
    if constexpr (SB < 4) {
      sc = q4k_byte(hd[r], SB) & 63u;
      mn = q4k_byte(hd[r], SB + 4) & 63u;
    } else {
      sc = (q4k_byte(hd[r], SB + 4) & 15u) | ((q4k_byte(hd[r], SB - 4) >> 6) << 4);
      mn = (q4k_byte(hd[r], SB + 4) >> 4) | ((q4k_byte(hd[r], SB) >> 6) << 4);
    }
    const float A = hd[r].d * static_cast<float>(sc), B = hd[r].dmin * static_cast<float>(mn);
    const f2 A2 = mk2(A, A), nB2 = mk2(-B, -B);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t c = lds_u32(rows[r] + 16u + 32u * (SB >> 1) + 16u * h + 4u * q);
      f2 a, b;
      magic4((c >> (4 * (SB & 1))) & 0x0F0F0F0Fu, -8388608.0f, a, b);  // nibble, exactly
      w[r][h][0] = fma2(a, A2, nB2);
      w[r][h][1] = fma2(b, A2, nB2);
    }
  }
}

// 4 bytes at an even shared address (a Q6_K row starts 2-byte aligned in its slot)
QG_DEVICE uint32_t lds_u32_even(uint32_t addr) {
  const uint32_t b = addr & ~3u;
  return __byte_perm(lds_u32(b), lds_u32(b + 4u), (addr & 2u) ? 0x5432u : 0x3210u);
}
// Weights of sub-block SB of a Q6_K super-block (ql[128], qh[64], int8 sc[16], f16 d) for rows
// i and i + 8, activation units q and q + 4.  Element 128 n + 32 qd + l (SB = 4 n + qd) is
// d * sc[8 n + l / 16 + 2 qd] * (q - 32), q = 4 bits of ql[64 n + 32 (qd & 1) + l] (the low
// nibble for qd < 2) and 2 bits of qh[32 n + l] at bit 2 qd; (d sc)(q - 32) has at most 23
// significant bits, so the f32 product is exact.
template <int SB>
QG_DEVICE void mt_weights_q6k(uint32_t blk_i, uint32_t blk_j, int q, f2 (&w)[2][2][2]) {
  constexpr uint32_t n = SB >> 2, qd = SB & 3;
  const uint32_t rows[2] = {blk_i, blk_j};
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const float d = h2f(lds_u16(rows[r] + 208u));
    const uint32_t scw = lds_u16(rows[r] + 192u + 8u * n + 2u * qd);
    const float A[2] = {d * static_cast<float>(static_cast<int8_t>(scw & 0xFFu)),
                        d * static_cast<float>(static_cast<int8_t>(scw >> 8))};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t lo = lds_u32_even(rows[r] + 64u * n + 32u * (qd & 1u) + 16u * h + 4u * q);
      const uint32_t hi = lds_u32_even(rows[r] + 128u + 32u * n + 16u * h + 4u * q);
      const uint32_t qv = ((lo >> (4u * (qd >> 1))) & 0x0F0F0F0Fu) | (((hi >> (2u * qd)) & 0x03030303u) << 4);
      f2 a, b;
      magic4(qv, -8388640.0f, a, b);  // q - 32: -(2^23 + 32)
      const f2 A2 = mk2(A[h], A[h]);
      w[r][h][0] = mul2(a, A2);
      w[r][h][1] = mul2(b, A2);
    }
  }
}

template <int QT, int TT, int NWM>
__global__ void __launch_bounds__(NWM * 32, 1) qgemv_mt_kernel(const __grid_constant__ CUtensorMap xmap, const MtArgs a) {
  constexpr uint32_t UB = unit_bytes<QT>();
  constexpr int TH = TT / 2;  // outputs per lane per group (2 rows x TT tokens over 4 lanes)
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t *wbar = reinterpret_cast<uint64_t *>(smem);  // [NWM][kNS]
  uint64_t *xfull = wbar + NWM * kNS;
  uint8_t *xs = smem + a.off_x;

  const int nw = static_cast<int>(blockDim.x >> 5);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int li = lane & 7, lq = lane >> 3;
  const int KS = a.KS;
  const uint32_t rank = KS > 1 ? cluster_rank() : 0u;
  const uint32_t cl = blockIdx.x / static_cast<uint32_t>(KS), ncl = gridDim.x / static_cast<uint32_t>(KS);
  const uint32_t gA = static_cast<uint32_t>(static_cast<unsigned long long>(cl) * a.groups / ncl);
  const uint32_t gB = static_cast<uint32_t>(static_cast<unsigned long long>(cl + 1) * a.groups / ncl);
  const int nrg = static_cast<int>(gB - gA);
  // this CTA's K range in 8-block units, cut into chunks of cbu units (the last may be short)
  const int uA = static_cast<int>(rank) * a.units / KS, uB = (static_cast<int>(rank) + 1) * a.units / KS;
  const int nc = (uB - uA + a.cbu - 1) / a.cbu;
  const int n_items = nrg * nc;
  const int NWa = max(1, min(nw, n_items));
  auto kb = [&](int w) { return w * n_items / NWa; };
  const int k0 = warp < NWa ? kb(warp) : 0;
  const int items = warp < NWa ? kb(warp + 1) - k0 : 0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NWM * kNS; ++i) mbar_init(&wbar[i], 1);
    mbar_init(xfull, 1);
    fence_mbar_init();
  }
  __syncthreads();

  uint64_t *mybar = wbar + warp * kNS;
  const uint32_t ring_s = smem_u32(smem + a.off_ring) + static_cast<uint32_t>(warp * a.NS) * a.stage_bytes;
  uint8_t *ring = smem + a.off_ring + static_cast<uint32_t>(warp * a.NS) * a.stage_bytes;

  auto locate = [&](uint32_t g, int &j, uint32_t &row0) {
    j = 0;
#pragma unroll
    for (int m = 1; m < kMats; ++m)
      if (m < a.nmat && g >= a.rg0[m]) j = m;
    row0 = (g - a.rg0[j]) * kRG;
  };
  auto chunk_units = [&](int c) { return min(a.cbu, uB - uA - c * a.cbu); };

  // issue chunk c of the cluster's row group gl into slot s: one copy per row (lanes 0..15)
  auto issue = [&](int gl, int c, int s) {
    int j;
    uint32_t row0;
    locate(gA + static_cast<uint32_t>(gl), j, row0);
    const uint32_t nr = min(static_cast<uint32_t>(kRG), a.M[j] - row0);
    const uint32_t cb = static_cast<uint32_t>(chunk_units(c)) * UB;
    if constexpr (QT == QG_TYPE_Q6_K) {
      // rows of 210-byte blocks: each row segment is copied from the 16-byte boundary below
      // it (the slot holds it at its offset from that boundary)
      const uintptr_t src = reinterpret_cast<uintptr_t>(a.w[j]) + static_cast<uintptr_t>(row0 + lane) * a.row_bytes +
                            static_cast<uintptr_t>(uA + c * a.cbu) * UB;
      warp_bulk_copies<true>(ring + s * a.stage_bytes + lane * a.seg, src,
                             static_cast<uint32_t>(lane) < nr ? cb : 0u, a.mend[j], &mybar[s], lane);
    } else {
      if (lane == 0) mbar_arrive_expect_tx(&mybar[s], nr * cb);
      __syncwarp();
      if (static_cast<uint32_t>(lane) < nr)
        bulk_g2s<true>(ring + s * a.stage_bytes + lane * a.seg,
                       a.w[j] + (row0 + lane) * a.row_bytes + static_cast<uint32_t>(uA + c * a.cbu) * UB, cb,
                       &mybar[s]);
    }
  };

  int ii = k0 / nc, ic = k0 - (k0 / nc) * nc, is = 0, issued = 0;
  auto advance_issue = [&]() {
    if (++ic == nc) {
      ic = 0;
      ++ii;
    }
    is = (is + 1 == a.NS) ? 0 : is + 1;
    ++issued;
  };
  auto prologue = [&](int upto) {
    while (issued < upto && issued < items) {
      issue(ii, ic, is);
      advance_issue();
    }
  };
  if (KS > 1) cluster_sync();  // every rank's barriers exist before any rank reads its memory
  if (a.early_weights) prologue(1);
  pdl_wait();
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    // the K range's activation rows, TT token slots each (slots >= T are zero-filled)
    const int rows = (uB - uA) * 8;
    mbar_arrive_expect_tx(xfull, static_cast<uint32_t>(rows * TT) * 128u);
    for (int b = 0; b < rows; b += a.box_rows) tma_load_3d(xs + b * TT * 128, &xmap, 0, 0, uA * 8 + b, xfull);
  }
  prologue(a.NS - 1);

  // activation unit u of token slot t of row R sits at 128 (R TT + t) + 16 (u ^ ((R TT + t) & 7));
  // with u = q + 4h the lane-dependent part is 16 (q ^ (phase & 3)): four base offsets
  const uint32_t xs_s = smem_u32(xs);
  uint32_t xq[4];
#pragma unroll
  for (int m = 0; m < 4; ++m) xq[m] = 16u * static_cast<uint32_t>(lq ^ m);
  bool ok = mbar_wait(xfull, 0);

  f2 acc[2][TT];
  float held[TH];  // the first segment of this warp's range when it is the tail of a split group
  int held_slot = -1, tail_slot = -1;
  float tail[TH];
  int i = k0 / nc, c = k0 - (k0 / nc) * nc, cs = 0, done = 0, c_first = c;
  uint32_t phase = 0;
  for (int it = 0; it < items; ++it) {
    if (ok && issued < items) {
      issue(ii, ic, is);
      advance_issue();
    }
    if (c == 0 || it == 0) {
      c_first = c;
#pragma unroll
      for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int t = 0; t < TT; ++t) acc[r][t] = mk2(0.f, 0.f);
    }
    if (ok && !mbar_wait(&mybar[cs], phase)) ok = false;
    if (ok) {
      ++done;
      const uint32_t st = ring_s + static_cast<uint32_t>(cs) * a.stage_bytes;
      uint32_t row_i = st + static_cast<uint32_t>(li) * a.seg, row_j = row_i + 8u * a.seg;
      if constexpr (QT == QG_TYPE_Q6_K) {
        // each row sits at its source's offset from a 16-byte boundary
        int j;
        uint32_t row0;
        locate(gA + static_cast<uint32_t>(i), j, row0);
        const uintptr_t s0 = reinterpret_cast<uintptr_t>(a.w[j]) + static_cast<uintptr_t>(uA + c * a.cbu) * UB;
        row_i += static_cast<uint32_t>((s0 + static_cast<uintptr_t>(row0 + li) * a.row_bytes) & 15u);
        row_j += static_cast<uint32_t>((s0 + static_cast<uintptr_t>(row0 + li + 8) * a.row_bytes) & 15u);
      }
      const int nu = chunk_units(c);
      for (int u = 0; u < nu; ++u) {
        // activation rows of this unit: 8 blocks x TT token slots, from a 1024-byte boundary
        const uint32_t xu = xs_s + static_cast<uint32_t>((c * a.cbu + u) * 8 * TT) * 128u;
        uint32_t xb[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) xb[m] = xu + xq[m];
        const uint32_t wu = static_cast<uint32_t>(u) * UB;
        Q4kHead hd[2];
        if constexpr (QT == QG_TYPE_Q4_K) {
          hd[0] = q4k_head(row_i + wu);
          hd[1] = q4k_head(row_j + wu);
        }
        auto block = [&](auto blk_c) {
          constexpr int BLK = decltype(blk_c)::value;
          f2 w[2][2][2];
          if constexpr (QT == QG_TYPE_Q4_K) {
            mt_weights_q4k<BLK>(row_i + wu, row_j + wu, hd, lq, w);
          } else if constexpr (QT == QG_TYPE_Q6_K) {
            mt_weights_q6k<BLK>(row_i + wu, row_j + wu, lq, w);
          } else {
            mt_weights<QT, BLK>(row_i + wu, row_j + wu, lq, w);
          }
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float4 xv[TT];
#pragma unroll
            for (int t = 0; t < TT; ++t) {
              const int row = BLK * TT + t, ph = row & 7;
              xv[t] = lds_f4(xb[ph & 3] + static_cast<uint32_t>(128 * row + 16 * ((4 * h) ^ (ph & 4))));
            }
#pragma unroll
            for (int r = 0; r < 2; ++r)
#pragma unroll
              for (int t = 0; t < TT; ++t) acc[r][t] = fma2(w[r][h][0], mk2(xv[t].x, xv[t].y), acc[r][t]);
#pragma unroll
            for (int r = 0; r < 2; ++r)
#pragma unroll
              for (int t = 0; t < TT; ++t) acc[r][t] = fma2(w[r][h][1], mk2(xv[t].z, xv[t].w), acc[r][t]);
          }
        };
        block(std::integral_constant<int, 0>{});
        block(std::integral_constant<int, 1>{});
        block(std::integral_constant<int, 2>{});
        block(std::integral_constant<int, 3>{});
        block(std::integral_constant<int, 4>{});
        block(std::integral_constant<int, 5>{});
        block(std::integral_constant<int, 6>{});
        block(std::integral_constant<int, 7>{});
      }
    }
    __syncwarp();  // every lane is done reading this slot before it is refilled
    if (++cs == a.NS) {
      cs = 0;
      phase ^= 1u;
    }
    if (c == nc - 1 || it == items - 1) {
      // end of a segment: reduce over the four lanes of each row (lanes i, i+8, i+16, i+24)
      // so that lane (i, q) owns row i + 8 (q >> 1), tokens (q & 1) TH .. + TH - 1
      float v[TH];
      {
        const bool hi = (lane & 16) != 0;
        float k[TT];
#pragma unroll
        for (int t = 0; t < TT; ++t) {
          const float v0 = acc[0][t].x + acc[0][t].y, v1 = acc[1][t].x + acc[1][t].y;
          k[t] = (hi ? v1 : v0) + __shfl_xor_sync(0xFFFFFFFFu, hi ? v0 : v1, 16);
        }
        const bool hi2 = (lane & 8) != 0;
#pragma unroll
        for (int t = 0; t < TH; ++t)
          v[t] = (hi2 ? k[t + TH] : k[t]) + __shfl_xor_sync(0xFFFFFFFFu, hi2 ? k[t] : k[t + TH], 8);
      }
      if (c_first == 0 && c == nc - 1) {
        if (KS == 1) {
          int j;
          uint32_t row0;
          locate(gA + static_cast<uint32_t>(i), j, row0);
          const uint32_t row = row0 + static_cast<uint32_t>(li + 8 * (lq >> 1)), M = a.M[j];
          const int t0 = (lq & 1) * TH;
#pragma unroll
          for (int t = 0; t < TH; ++t)
            if (ok && t0 + t < a.T && row < M) a.y[j][static_cast<size_t>(t0 + t) * M + row] = v[t];
        } else {
          float *o = reinterpret_cast<float *>(smem + a.off_outs) + (i * 32 + lane) * TH;
#pragma unroll
          for (int t = 0; t < TH; ++t) o[t] = v[t];
        }
      } else if (c_first != 0 && it + 1 == c - c_first + 1 && held_slot < 0) {
        // the warp's first segment, starting inside a group: its part goes to slot 2 w + 1
        held_slot = 2 * warp + 1;
#pragma unroll
        for (int t = 0; t < TH; ++t) held[t] = v[t];
      } else {
        // a segment that ends the warp's range inside a group (it began at chunk 0): slot 2 (w + 1)
        tail_slot = c_first == 0 ? 2 * (warp + 1) : 2 * warp + 1;
#pragma unroll
        for (int t = 0; t < TH; ++t) tail[t] = v[t];
      }
    }
    if (++c == nc) {
      c = 0;
      ++i;
    }
  }
  if (!ok) {
    if (lane == 0) mt_status(QG_STATUS_BIT_TIMEOUT);
    // never leave this warp's copies in flight (the ring is reused below)
    if (lane == 0)
      for (int k = done; k < issued; ++k) mbar_wait(&mybar[k % a.NS], (k / a.NS) & 1);
    __syncwarp();
  }
  if (nc > 1) {
    // groups split between warps: parts into slots laid over the (now idle) rings, then warp
    // w, the first boundary inside such a group, sums them in chunk order
    __syncthreads();
    float *slots = reinterpret_cast<float *>(smem + a.off_ring);  // [2 NWM][32][TH]
    if (held_slot >= 0)
#pragma unroll
      for (int t = 0; t < TH; ++t) slots[(held_slot * 32 + lane) * TH + t] = held[t];
    if (tail_slot >= 0)
#pragma unroll
      for (int t = 0; t < TH; ++t) slots[(tail_slot * 32 + lane) * TH + t] = tail[t];
    __syncthreads();
    if (warp >= 1 && warp < NWa) {
      const int b = kb(warp);
      const int gl = b / nc, lo = gl * nc;
      if (b != lo && kb(warp - 1) <= lo) {
        float s[TH];
#pragma unroll
        for (int t = 0; t < TH; ++t) s[t] = slots[(2 * warp * 32 + lane) * TH + t];
        for (int w = warp; w < NWa && kb(w) < lo + nc; ++w)
#pragma unroll
          for (int t = 0; t < TH; ++t) s[t] += slots[((2 * w + 1) * 32 + lane) * TH + t];
        if (KS == 1) {
          int j;
          uint32_t row0;
          locate(gA + static_cast<uint32_t>(gl), j, row0);
          const uint32_t row = row0 + static_cast<uint32_t>(li + 8 * (lq >> 1)), M = a.M[j];
          const int t0 = (lq & 1) * TH;
#pragma unroll
          for (int t = 0; t < TH; ++t)
            if (ok && t0 + t < a.T && row < M) a.y[j][static_cast<size_t>(t0 + t) * M + row] = s[t];
        } else {
          float *o = reinterpret_cast<float *>(smem + a.off_outs) + (gl * 32 + lane) * TH;
#pragma unroll
          for (int t = 0; t < TH; ++t) o[t] = s[t];
        }
      }
    }
  }
  if (KS > 1) {
    // every rank holds its K range's sums of all the cluster's groups; rank r adds up groups
    // r, r + KS, ... over the ranks in rank order and writes them
    cluster_sync();
    const uint32_t outs_s = smem_u32(smem + a.off_outs);
    for (int gl = static_cast<int>(rank) + KS * warp; gl < nrg; gl += KS * nw) {
      float s[TH];
#pragma unroll
      for (int t = 0; t < TH; ++t) s[t] = 0.f;
      const uint32_t off = static_cast<uint32_t>((gl * 32 + lane) * TH) * 4u;
      for (int rr = 0; rr < KS; ++rr) {
        const uint32_t src = map_rank(outs_s + off, static_cast<uint32_t>(rr));
        if constexpr (TH % 4 == 0) {
#pragma unroll
          for (int t = 0; t < TH; t += 4) {
            const float4 p = ld_cluster_f4(src + 4u * t);
            s[t] += p.x;
            s[t + 1] += p.y;
            s[t + 2] += p.z;
            s[t + 3] += p.w;
          }
        } else {
#pragma unroll
          for (int t = 0; t < TH; ++t) s[t] += ld_cluster_f32(src + 4u * t);
        }
      }
      int j;
      uint32_t row0;
      locate(gA + static_cast<uint32_t>(gl), j, row0);
      const uint32_t row = row0 + static_cast<uint32_t>(li + 8 * (lq >> 1)), M = a.M[j];
      const int t0 = (lq & 1) * TH;
#pragma unroll
      for (int t = 0; t < TH; ++t)
        if (ok && t0 + t < a.T && row < M) a.y[j][static_cast<size_t>(t0 + t) * M + row] = s[t];
    }
    cluster_sync();  // no rank leaves while another still reads its memory
  }
}

}  // namespace

namespace qg {

struct MtPlan {
  MtArgs a;
  CUtensorMap map;
  unsigned grid;
  uint32_t smem;
  int nw;
};

// Clusters of KS one-CTA-per-SM CTAs that can be resident at once (a cluster's CTAs share one
// GPU processing cluster, so this can be below sms / KS); cached per device and KS.
template <int QT, int TT, int NWM>
long long cluster_fit(int KS) {
  static long long cache[64][4] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  const int idx = KS == 2 ? 0 : KS == 4 ? 1 : KS == 8 ? 2 : 3;
  if (cache[dev][idx] > 0) return cache[dev][idx];
  auto kern = qgemv_mt_kernel<QT, TT, NWM>;
  const uint32_t smem = static_cast<uint32_t>(device_info().smem_optin);
  if (!set_smem_attr(reinterpret_cast<const void *>(kern), smem)) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(KS * (device_info().sms / KS)));
  cfg.blockDim = dim3(NWM * 32);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(KS);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n < 1) {
    cudaGetLastError();
    return 0;
  }
  cache[dev][idx] = n;
  return n;
}

// Plans the kernel for token tile TT; QG_EUNSUPPORTED when the shape is outside its scope.
template <int QT, int TT, int NWM>
qg_status gemv_mt_plan(int nmat, const void *const *w, const float *x, float *const *y, const int64_t *Ms, int64_t N,
                       int T, MtPlan &P) {
  constexpr uint32_t UB = unit_bytes<QT>();
  const DeviceInfo &dev = device_info();
  if (!dev.ok) return QG_ECUDA;
  if (N % 256 != 0) return QG_EUNSUPPORTED;  // rows of whole 256-element units (16-byte aligned)
  const long long row_bytes = N / 256 * UB;
  MtArgs a{};
  unsigned long long groups = 0;
  for (int j = 0; j < nmat; ++j) {
    if (static_cast<unsigned long long>(Ms[j]) * row_bytes >= (1ull << 32)) return QG_EUNSUPPORTED;
    a.w[j] = static_cast<const uint8_t *>(w[j]);
    a.y[j] = y[j];
    a.M[j] = static_cast<uint32_t>(Ms[j]);
    a.rg0[j] = static_cast<uint32_t>(groups);
    a.mend[j] = (reinterpret_cast<uintptr_t>(w[j]) + static_cast<uintptr_t>(Ms[j] * row_bytes)) & ~static_cast<uintptr_t>(15);
    groups += (Ms[j] + kRG - 1) / kRG;
  }
  if (groups == 0 || groups >= (1ull << 31)) return QG_EUNSUPPORTED;
  for (int j = nmat; j <= kMats; ++j) a.rg0[j] = static_cast<uint32_t>(groups);
  a.nmat = nmat;
  a.row_bytes = static_cast<uint32_t>(row_bytes);
  a.groups = static_cast<uint32_t>(groups);
  a.N = static_cast<int>(N);
  a.T = T;
  a.units = static_cast<int>(N / 256);
  const long long budget = dev.smem_optin;
  const uint32_t hdr = 1024;
  // K ranges per cluster: the fewest that let one rank's activations stay resident beside a
  // ring of at least two slots per warp (7 or 8 warps)
  for (int KS : {1, 2, 4, 8}) {
    if (KS > a.units) break;
    const int umax = (a.units + KS - 1) / KS;
    const long long xbytes = static_cast<long long>(TT) * umax * 8 * 128;  // TT token slots per row
    long long ncl = std::min<long long>(dev.sms / KS, static_cast<long long>(groups));
    if (KS > 1) ncl = std::min<long long>(ncl, cluster_fit<QT, TT, NWM>(KS));
    if (ncl < 1) continue;
    const long long gmax = (static_cast<long long>(groups) + ncl - 1) / ncl;
    const long long outs = KS > 1 ? gmax * kRG * TT * 4 : 0;
    for (int cbu : {2, 1}) {
      // Q6_K rows are copied from the 16-byte boundary below them: 16 bytes of slack per row
      long long seg = QT == QG_TYPE_Q6_K ? (static_cast<long long>(cbu) * UB + 15) / 16 * 16 + 16
                                         : static_cast<long long>(cbu) * UB;
      // an odd number of 16-byte units per row: the eight rows that a warp reads at one offset
      // then fall in eight different bank groups (544-byte rows put rows i and i + 4 in one)
      if ((seg / 16) % 2 == 0) seg += 16;
      const long long stage = kRG * seg;
      // all NWM warps per CTA: at T = 16 a 2-CTA cluster split of K with 8 warps beat one CTA of
      // 7 warps that held all of K (decode step 5.02 -> 4.67 ms)
      for (const int nw : {NWM}) {
        const long long fixed = 1024 /*alignment*/ + hdr + ((xbytes + 1023) / 1024) * 1024 + ((outs + 1023) / 1024) * 1024;
        const long long ring_avail = budget - fixed;
        // split-group parts are laid over the rings after the loop
        const long long parts = 2LL * NWM * 32 * (TT / 2) * 4;
        if (ring_avail < 2LL * nw * stage || ring_avail < parts) continue;
        const int NS = static_cast<int>(std::min<long long>(kNS, ring_avail / (nw * stage)));
        if (NS * nw * stage < parts) continue;
        a.KS = KS;
        a.cbu = cbu;
        a.seg = static_cast<uint32_t>(seg);
        a.stage_bytes = static_cast<uint32_t>(stage);
        a.NS = NS;
        a.xR = umax * 8;
        // the box height divides both range lengths (umax and umax - 1 units)
        const int ulo = a.units / KS;
        int g = umax;
        for (int v = ulo; v > 0;) {
          const int t2 = g % v;
          g = v;
          v = t2;
        }
        int box = 8;
        for (int d = 1; d <= 32; ++d)
          if (g % d == 0 && 8 * d * TT * 128 <= 32768) box = 8 * d;
        a.box_rows = box;
        a.max_groups = static_cast<int>(gmax);
        a.off_x = hdr;
        a.off_outs = static_cast<uint32_t>(a.off_x + ((xbytes + 1023) / 1024) * 1024);
        a.off_ring = static_cast<uint32_t>(a.off_outs + ((outs + 1023) / 1024) * 1024);
        P.a = a;
        P.nw = nw;
        P.grid = static_cast<unsigned>(ncl * KS);
        P.smem = static_cast<uint32_t>(a.off_ring + static_cast<long long>(NS) * nw * stage + 1024);
        if (!encode_x_map_tok(&P.map, x, T, N, TT, box)) return QG_ECUDA;
        return QG_OK;
      }
    }
  }
  return QG_EUNSUPPORTED;
}

template <int QT, int TT, int NWM>
qg_status gemv_mt_run(MtPlan &P, cudaStream_t stream) {
  auto kern = qgemv_mt_kernel<QT, TT, NWM>;
  if (!set_smem_attr(reinterpret_cast<const void *>(kern), P.smem)) return QG_ECUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(P.nw * 32);
  cfg.dynamicSmemBytes = P.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(P.a.KS);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cfg.gridDim = dim3(P.grid);
  P.a.early_weights = static_weights(stream) ? 1 : 0;
  if (cudaLaunchKernelEx(&cfg, kern, P.map, P.a) != cudaSuccess) return QG_ECUDA;
  return cudaGetLastError() == cudaSuccess ? QG_OK : QG_ECUDA;
}

template <int QT>
qg_status gemv_mt_launch(int nmat, const void *const *w, const float *x, float *const *y, const int64_t *Ms, int64_t N,
                         int T, cudaStream_t stream) {
  {
    if (T < 2 || T > 16) return QG_EUNSUPPORTED;
    MtPlan P;
    qg_status r;
    if (T <= 4) {
      // up to 4 tokens over fewer than two 16-row groups per SM (the launches this kernel
      // takes when the lean kernel cannot hold their activations): 16 warps per CTA, whose
      // rings leave room for only half of K's activations, so K is split over a 2-CTA cluster
      // (2560 x 9728: 22.9 -> 18.2 us); with more groups 8 warps per CTA are faster
      // (19456 x 2560: 18.5 vs 20.2 us)
      long long groups = 0;
      for (int j = 0; j < nmat; ++j) groups += (Ms[j] + kRG - 1) / kRG;
      if (groups < 2LL * device_info().sms) {
        r = gemv_mt_plan<QT, 4, 16>(nmat, w, x, y, Ms, N, T, P);
        if (r == QG_OK) return gemv_mt_run<QT, 4, 16>(P, stream);
        if (r != QG_EUNSUPPORTED) return r;
      }
      r = gemv_mt_plan<QT, 4, 8>(nmat, w, x, y, Ms, N, T, P);
      return r == QG_OK ? gemv_mt_run<QT, 4, 8>(P, stream) : r;
    }
    if (T <= 8) {
      r = gemv_mt_plan<QT, 8, 8>(nmat, w, x, y, Ms, N, T, P);
      return r == QG_OK ? gemv_mt_run<QT, 8, 8>(P, stream) : r;
    }
    r = gemv_mt_plan<QT, 16, 8>(nmat, w, x, y, Ms, N, T, P);
    return r == QG_OK ? gemv_mt_run<QT, 16, 8>(P, stream) : r;
  }
}

unsigned int read_status_mt(bool clear) {
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_qg_status_mt, sizeof(v)) != cudaSuccess) return 0xFFFFFFFFu;
  if (clear) {
    const unsigned int z = 0;
    cudaMemcpyToSymbol(g_qg_status_mt, &z, sizeof(z));
  }
  return v;
}

template qg_status gemv_mt_launch<QG_TYPE_Q8_0>(int, const void *const *, const float *, float *const *,
                                                const int64_t *, int64_t, int, cudaStream_t);
template qg_status gemv_mt_launch<QG_TYPE_Q4_0>(int, const void *const *, const float *, float *const *,
                                                const int64_t *, int64_t, int, cudaStream_t);
template qg_status gemv_mt_launch<QG_TYPE_Q4_K>(int, const void *const *, const float *, float *const *,
                                                const int64_t *, int64_t, int, cudaStream_t);
template qg_status gemv_mt_launch<QG_TYPE_Q6_K>(int, const void *const *, const float *, float *const *,
                                                const int64_t *, int64_t, int, cudaStream_t);

}  // namespace qg
