// qg_gemm.cu -- prefill dequant-GEMM on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// Y[t][m] = sum_k W[m][k] * X[t][k] for T >= 17 token rows: the tiled matmulQ8T of the
// engine pages (qwen35_moe_ssd.js BATCH_KERNELS) grown into a prefill chunk, with the
// pages' f16 8x8x8 subgroup-matrix path (qwen35_dense.js) as prior art only.  W stays in
// raw Q8_0 blocks in HBM; it is decoded to bf16 inside the kernel, X is rounded to bf16,
// products accumulate in f32 in tensor memory.
//
// One persistent CTA per SM, warp-specialised:
//   warp 0      TMA producer: raw weight tiles (128 rows x 256 k = 8 blocks of 34 bytes per
//               row, a 272-byte box of a 16-bit view of the rows) into a 2-slot raw ring,
//               and bf16 activation tiles (256 tokens x 64 k, 128-byte swizzle) into the
//               3-slot operand ring;
//   warp 1      TMEM allocation and the single MMA-issuing thread: per 64-k stage four
//               tcgen05.mma.kind::f16 (M 128, N 256, K 16, bf16 x bf16 -> f32), then
//               tcgen05.commit to the stage's "empty" barrier;
//   warps 2-17  converters: decode the stage's 128 x 64 weights from the raw ring (d * q in
//               f32, one rounding to bf16) into the A slot in the UMMA K-major 128-byte
//               swizzled layout; after a tile's last stage they are the epilogue (tcgen05.ld
//               of the accumulator, coalesced f32 stores of Y).
//
// Work split: the (tile, 256-k step) space is cut into equal contiguous ranges, one per CTA
// (stream-K), so shapes with few tiles and long K still fill every SM.  A tile whose k
// steps span several CTAs is finished by its last-arriving part, which sums the parts'
// partial tiles in CTA order (deterministic) and writes Y.
//
// Every wait is bounded; a wait that expires raises a CTA-wide abort flag so that the other
// roles stop at their next wait, the status word records QG_ETIMEOUT, in-flight copies and
// MMAs are waited for, and TMEM is released before the CTA exits.
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>

#include "qg_common.cuh"
#include "qg_host.h"
#include "qg_pipe.cuh"

__device__ unsigned int g_qg_status_gemm;

namespace {

constexpr int BM = 128;   // weight rows per tile (MMA M)
constexpr int BT = 256;   // tokens per tile (MMA N)
constexpr int BK = 64;    // k per operand stage: one 128-byte swizzle atom of bf16
constexpr int RK = 256;   // k per raw weight stage: 8 Q8_0 blocks, 272 bytes per row
constexpr int NSTAGE = 3;
constexpr int NRAW = 2;
constexpr int NCONV = 16;  // converter / epilogue warps
constexpr int NTHREADS = (2 + NCONV) * 32;
constexpr uint32_t A_BYTES = BM * BK * 2;       // 16 KB
constexpr uint32_t B_BYTES = BT * BK * 2;       // 32 KB
constexpr uint32_t RAW_ROW = (RK / 32) * 34;    // 272
constexpr uint32_t RAW_BYTES = BM * RAW_ROW;    // 34816
constexpr uint32_t OFF_A = 0;
constexpr uint32_t OFF_B = OFF_A + NSTAGE * A_BYTES;
constexpr uint32_t OFF_RAW = OFF_B + NSTAGE * B_BYTES;
constexpr uint32_t OFF_BAR = OFF_RAW + NRAW * RAW_BYTES;
constexpr uint32_t OFF_PARTS = OFF_BAR + 256;  // slot list of a split tile's parts
constexpr int MAX_PARTS = 128;
constexpr uint32_t SMEM_BYTES = OFF_PARTS + MAX_PARTS * 4 + 1024;  // + alignment slack
constexpr uint32_t TMEM_COLS = 256;

QG_DEVICE void gemm_status(unsigned int bits) { atomicOr(&g_qg_status_gemm, bits); }

// ---- tcgen05 wrappers --------------------------------------------------------------------
QG_DEVICE void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
QG_DEVICE void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
QG_DEVICE void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
QG_DEVICE void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

QG_DEVICE void tc_mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accum)
      : "memory");
}
// arrives once on `bar` when every MMA this thread issued before it has completed
QG_DEVICE void tc_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// 32 consecutive f32 columns of this thread's TMEM lane
QG_DEVICE void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor of a K-major operand tile in the 128-byte swizzled
// layout: rows of 128 bytes, 8-row (1024-byte) swizzle atoms stacked along M/N.
//   bits  0-13  start address >> 4        bits 16-29  leading byte offset >> 4 (unused here)
//   bits 32-45  stride byte offset >> 4 (1024: next 8-row group)
//   bits 46-47  descriptor version 1      bits 61-63  layout: 2 = 128-byte swizzle
QG_DEVICE uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>(1u) << 16;
  d |= static_cast<uint64_t>((1024u >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}

// Instruction descriptor, kind::f16: f32 accumulator, bf16 A and B, both K-major.
__host__ __device__ constexpr uint32_t make_idesc(int m, int n) {
  return (1u << 4)                                 // D format f32
         | (1u << 7)                               // A format bf16
         | (1u << 10)                              // B format bf16
         | (static_cast<uint32_t>(n >> 3) << 17)   // N / 8
         | (static_cast<uint32_t>(m >> 4) << 24);  // M / 16
}

// ---- abort-aware bounded waits -------------------------------------------------------------
QG_DEVICE bool wait_or_abort(uint64_t *bar, uint32_t parity, volatile int *abort_flag) {
  if (mbar_try_wait_sleep(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (true) {
    if (mbar_try_wait_sleep(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_ns() - t0 > QG_WAIT_NS) break;
  }
  *abort_flag = 1;
  gemm_status(QG_STATUS_BIT_TIMEOUT);
  return false;
}

// short bounded wait used only while shutting down
QG_DEVICE void cleanup_wait(uint64_t *bar, uint32_t parity) {
  for (uint32_t i = 0; i < (1u << 16); ++i)
    if (mbar_try_wait(bar, parity)) return;
}

struct GemmArgs {
  float *y;
  float *part;           // partial tiles: [2 * gridDim.x][BT][BM]
  unsigned int *cnt;     // per-tile arrival counters (zeroed by the conversion kernel)
  int M, N, T;
  int n_mt, n_tt, KS;    // m tiles, token tiles, 256-k steps per tile
  long long total;       // tiles * KS
};

// CTA b's contiguous range of the (tile, k step) space starts at s(b)
QG_DEVICE long long range_start(long long b, long long total, int G) { return b * total / G; }
// the CTA whose range holds position p
QG_DEVICE int range_owner(long long p, long long total, int G) {
  return static_cast<int>(((p + 1) * G + total - 1) / total - 1);
}

// Decode 16 Q8_0 weights (half hb & 1 of block hb >> 1 of the 64-k stage `sub`) of one row
// from the raw stage into the A slot.  raw_row: shared address of the row's 272 raw bytes;
// a_row: shared address of the row in the A slot (128 bytes, 16-byte chunks swizzled by
// row & 7).  The 16 code bytes are fetched with two aligned 16-byte loads (eight lanes of
// consecutive rows hit eight different bank groups: the raw row pitch is 17 chunks).
QG_DEVICE void convert_half(uint32_t raw_row, int sub, int hb, uint32_t a_row, int row) {
  const uint32_t blk = raw_row + 68u * static_cast<uint32_t>(sub) + 34u * static_cast<uint32_t>(hb >> 1);
  uint32_t d16;
  QG_LDS16(blk, 0, d16);
  const float d = h2f(d16);
  const uint32_t o = blk + 2u + 16u * static_cast<uint32_t>(hb & 1);
  const uint32_t a16 = o & ~15u, off = o & 15u;
  const uint4 v0 = lds_v4(a16), v1 = lds_v4(a16 + 16u);
  const uint64_t q0 = (static_cast<uint64_t>(v0.y) << 32) | v0.x, q1 = (static_cast<uint64_t>(v0.w) << 32) | v0.z;
  const uint64_t q2 = (static_cast<uint64_t>(v1.y) << 32) | v1.x, q3 = (static_cast<uint64_t>(v1.w) << 32) | v1.z;
  const bool hi8 = off >= 8u;
  const uint32_t sh = (off & 7u) * 8u;
  const uint64_t l0 = hi8 ? q1 : q0, l1 = hi8 ? q2 : q1, l2 = hi8 ? q3 : q2;
  const uint64_t lo = sh ? (l0 >> sh) | (l1 << (64u - sh)) : l0;
  const uint64_t hi = sh ? (l1 >> sh) | (l2 << (64u - sh)) : l1;
  const uint32_t cw[4] = {static_cast<uint32_t>(lo), static_cast<uint32_t>(lo >> 32), static_cast<uint32_t>(hi),
                          static_cast<uint32_t>(hi >> 32)};
  const f2 d2 = mk2(d, d);
  const f2 bias = mk2(-8388736.0f, -8388736.0f);  // -(2^23 + 128)
#pragma unroll
  for (int c = 0; c < 2; ++c) {  // two 16-byte chunks of 8 weights
    uint32_t outw[4];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t word = cw[2 * c + h] ^ 0x80808080u;
      const f2 w01 = mul2(add2(mk2(magic_byte(word, 0), magic_byte(word, 1)), bias), d2);
      const f2 w23 = mul2(add2(mk2(magic_byte(word, 2), magic_byte(word, 3)), bias), d2);
      const __nv_bfloat162 b01 = __floats2bfloat162_rn(w01.x, w01.y);
      const __nv_bfloat162 b23 = __floats2bfloat162_rn(w23.x, w23.y);
      outw[2 * h] = *reinterpret_cast<const uint32_t *>(&b01);
      outw[2 * h + 1] = *reinterpret_cast<const uint32_t *>(&b23);
    }
    const uint32_t chunk = static_cast<uint32_t>((2 * hb + c) ^ (row & 7));
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a_row + chunk * 16u), "r"(outw[0]), "r"(outw[1]),
                 "r"(outw[2]), "r"(outw[3])
                 : "memory");
  }
}

__global__ void __launch_bounds__(NTHREADS, 1)
    qgemm_q8_0_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap xmap,
                      const GemmArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + OFF_BAR);  // [NSTAGE]
  uint64_t *empty = full + NSTAGE;                                 // [NSTAGE]
  uint64_t *rfull = empty + NSTAGE;                                // [NRAW]
  uint64_t *rempty = rfull + NRAW;                                 // [NRAW]
  uint64_t *acc_full = rempty + NRAW;
  uint64_t *acc_empty = acc_full + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(acc_empty + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  volatile unsigned int *s_last = reinterpret_cast<volatile unsigned int *>(tmem_slot + 2);
  volatile int *s_nparts = reinterpret_cast<volatile int *>(tmem_slot + 3);
  int *s_parts = reinterpret_cast<int *>(smem + OFF_PARTS);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = static_cast<int>(gridDim.x);
  const long long beg = range_start(blockIdx.x, a.total, G);
  const long long end = range_start(blockIdx.x + 1, a.total, G);

  if (threadIdx.x == 0) {
    for (int i = 0; i < NSTAGE; ++i) {
      mbar_init(&full[i], 1 + NCONV);  // producer's expect_tx arrival + one per converter warp
      mbar_init(&empty[i], 1);         // MMA commit
    }
    for (int i = 0; i < NRAW; ++i) {
      mbar_init(&rfull[i], 1);
      mbar_init(&rempty[i], NCONV);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, NCONV);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_wait();
  pdl_launch_dependents();
  const uint32_t tmem = *tmem_slot;

  const uint32_t sA = smem_u32(smem + OFF_A), sB = smem_u32(smem + OFF_B), sRaw = smem_u32(smem + OFF_RAW);

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      long long it = 0, rit = 0;
      bool ok = true;
      for (long long pos = beg; pos < end && ok;) {
        const int tile = static_cast<int>(pos / a.KS);
        const int k0 = static_cast<int>(pos - static_cast<long long>(tile) * a.KS);
        const int k1 = static_cast<int>(k0 + (end - pos) < a.KS ? k0 + (end - pos) : a.KS);
        const int mt = tile / a.n_tt, tt = tile - mt * a.n_tt;
        for (int ks = k0; ks < k1 && ok; ++ks, ++rit) {
          const int r = static_cast<int>(rit % NRAW);
          if (!wait_or_abort(&rempty[r], static_cast<uint32_t>(((rit / NRAW) & 1) ^ 1), abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&rfull[r], RAW_BYTES);
          tma_load_2d(smem + OFF_RAW + r * RAW_BYTES, &wmap, ks * (RK / 32) * 17, mt * BM, &rfull[r]);
          for (int sub = 0; sub < RK / BK; ++sub, ++it) {
            const int s = static_cast<int>(it % NSTAGE);
            if (!wait_or_abort(&empty[s], static_cast<uint32_t>(((it / NSTAGE) & 1) ^ 1), abort_flag)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&full[s], B_BYTES);
            tma_load_2d(smem + OFF_B + s * B_BYTES, &xmap, ks * RK + sub * BK, tt * BT, &full[s]);
          }
        }
        pos += k1 - k0;
      }
      // after an abort, the copies already issued must land before the CTA exits (a
      // normal run consumed every one of them)
      if (*abort_flag) {
        for (long long j = (it > NSTAGE ? it - NSTAGE : 0); j < it; ++j)
          cleanup_wait(&full[j % NSTAGE], static_cast<uint32_t>((j / NSTAGE) & 1));
        for (long long j = (rit > NRAW ? rit - NRAW : 0); j < rit; ++j)
          cleanup_wait(&rfull[j % NRAW], static_cast<uint32_t>((j / NRAW) & 1));
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc(BM, BT);
      long long it = 0;
      int si = 0;
      bool ok = true;
      for (long long pos = beg; pos < end && ok; ++si) {
        const int tile = static_cast<int>(pos / a.KS);
        const int k0 = static_cast<int>(pos - static_cast<long long>(tile) * a.KS);
        const int k1 = static_cast<int>(k0 + (end - pos) < a.KS ? k0 + (end - pos) : a.KS);
        if (!wait_or_abort(acc_empty, static_cast<uint32_t>((si & 1) ^ 1), abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int ks = k0; ks < k1 && ok; ++ks) {
          for (int sub = 0; sub < RK / BK; ++sub, ++it) {
            const int s = static_cast<int>(it % NSTAGE);
            if (!wait_or_abort(&full[s], static_cast<uint32_t>((it / NSTAGE) & 1), abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t aa = sA + s * A_BYTES, bb = sB + s * B_BYTES;
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              const uint32_t accum = (ks == k0 && sub == 0 && kk == 0) ? 0u : 1u;
              tc_mma_bf16(tmem, sw128_desc(aa + kk * 32), sw128_desc(bb + kk * 32), idesc, accum);
            }
            tc_commit(&empty[s]);  // the stage's A and B slots are free once these MMAs finish
          }
        }
        if (ok) tc_commit(acc_full);
        pos += k1 - k0;
      }
      // every MMA this thread issued is complete before TMEM is released
      if (it > 0) cleanup_wait(&empty[(it - 1) % NSTAGE], static_cast<uint32_t>(((it - 1) / NSTAGE) & 1));
    }
  } else {
    // ---------------- converters, then epilogue ----------------
    const int ct = threadIdx.x - 64;          // 0 .. NCONV * 32 - 1
    const int crow = 8 * (ct >> 5) + (lane & 7);  // weight row this thread converts
    const int chb = lane >> 3;                   // its 16-weight quarter of the 64-k stage
    const int q = warp & 3;                      // TMEM lane quarter this warp may read
    const int cgrp = (warp - 2) >> 2;            // which 64 accumulator columns
    long long it = 0, rit = 0;
    int si = 0;
    bool ok = true;
    for (long long pos = beg; pos < end && ok; ++si) {
      const int tile = static_cast<int>(pos / a.KS);
      const int k0 = static_cast<int>(pos - static_cast<long long>(tile) * a.KS);
      const int k1 = static_cast<int>(k0 + (end - pos) < a.KS ? k0 + (end - pos) : a.KS);
      const int mt = tile / a.n_tt, tt = tile - mt * a.n_tt;
      for (int ks = k0; ks < k1 && ok; ++ks, ++rit) {
        const int r = static_cast<int>(rit % NRAW);
        if (!wait_or_abort(&rfull[r], static_cast<uint32_t>((rit / NRAW) & 1), abort_flag)) {
          ok = false;
          break;
        }
        for (int sub = 0; sub < RK / BK; ++sub, ++it) {
          const int s = static_cast<int>(it % NSTAGE);
          if (!wait_or_abort(&empty[s], static_cast<uint32_t>(((it / NSTAGE) & 1) ^ 1), abort_flag)) {
            ok = false;
            break;
          }
          convert_half(sRaw + r * RAW_BYTES + static_cast<uint32_t>(crow) * RAW_ROW, sub, chb,
                       sA + s * A_BYTES + static_cast<uint32_t>(crow) * 128u, crow);
          fence_proxy_async_smem();  // generic-proxy stores -> tensor-core reads
          __syncwarp();
          if (lane == 0) mbar_arrive(&full[s]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&rempty[r]);
      }
      if (!ok) break;
      // ---- epilogue of this segment
      if (!wait_or_abort(acc_full, static_cast<uint32_t>(si & 1), abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const bool whole = (k0 == 0 && k1 == a.KS);
      const int m_loc = 32 * q + lane;
      const int m = mt * BM + m_loc;
      int slot = 0;
      if (!whole) slot = 2 * static_cast<int>(blockIdx.x) + (beg < static_cast<long long>(tile) * a.KS ? 1 : 0);
      float *dst = whole ? a.y : a.part + static_cast<size_t>(slot) * BT * BM;
#pragma unroll 1
      for (int cc = 0; cc < 2; ++cc) {
        const int col0 = cgrp * 64 + cc * 32;
        float v[32];
        tmem_ld32(tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(col0), v);
        if (whole) {
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const int t = tt * BT + col0 + c;
            if (t < a.T && m < a.M) dst[static_cast<size_t>(t) * a.M + m] = v[c];
          }
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) dst[static_cast<size_t>(col0 + c) * BM + m_loc] = v[c];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty);
      if (!whole) {
        // count this part; the last part of the tile sums all parts in CTA order
        __threadfence();
        named_bar_sync(1, NCONV * 32);
        if (ct == 0) {
          const long long ts = static_cast<long long>(tile) * a.KS, te = ts + a.KS;
          const int bf = range_owner(ts, a.total, G), bl = range_owner(te - 1, a.total, G);
          int parts = 0;
          for (int bp = bf; bp <= bl; ++bp) {
            const long long sbp = range_start(bp, a.total, G);
            if (sbp < range_start(bp + 1, a.total, G)) {
              if (parts < MAX_PARTS) s_parts[parts] = 2 * bp + (sbp < ts ? 1 : 0);
              ++parts;
            }
          }
          const unsigned int old = atomicAdd(&a.cnt[tile], 1u);
          *s_last = (old + 1u == static_cast<unsigned int>(parts)) ? 1u : 0u;
          *s_nparts = parts;
        }
        named_bar_sync(1, NCONV * 32);
        if (*s_last) {
          __threadfence();
          const int parts = *s_nparts;
          // thread: rows 4 m4 .. 4 m4 + 3, columns cs + NCONV j, in two batches of 8 columns
          // (8 independent float4 loads in flight per part)
          const int m4 = ct & 31, cs = ct >> 5;
          constexpr int NJ = BT / NCONV, NB = 8;
          const int mg = mt * BM + 4 * m4;
#pragma unroll 1
          for (int j0 = 0; j0 < NJ; j0 += NB) {
            float4 acc[NB];
#pragma unroll
            for (int j = 0; j < NB; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int pi = 0; pi < parts; ++pi) {
              int sl;
              if (pi < MAX_PARTS) {
                sl = s_parts[pi];
              } else {  // more parts than the list holds: recompute this one
                const long long ts = static_cast<long long>(tile) * a.KS;
                int bp = range_owner(ts, a.total, G), seen = -1;
                for (;; ++bp)
                  if (range_start(bp, a.total, G) < range_start(bp + 1, a.total, G) && ++seen == pi) break;
                sl = 2 * bp + (range_start(bp, a.total, G) < ts ? 1 : 0);
              }
              const float4 *pp = reinterpret_cast<const float4 *>(a.part + static_cast<size_t>(sl) * BT * BM);
#pragma unroll
              for (int j = 0; j < NB; ++j) {
                const float4 v = __ldcg(pp + (cs + NCONV * (j0 + j)) * (BM / 4) + m4);
                acc[j].x += v.x;
                acc[j].y += v.y;
                acc[j].z += v.z;
                acc[j].w += v.w;
              }
            }
#pragma unroll
            for (int j = 0; j < NB; ++j) {
              const int t = tt * BT + cs + NCONV * (j0 + j);
              if (t >= a.T) continue;
              float *yr = a.y + static_cast<size_t>(t) * a.M;
              if (mg + 3 < a.M && (a.M & 3) == 0) {
                *reinterpret_cast<float4 *>(yr + mg) = acc[j];
              } else {
                if (mg < a.M) yr[mg] = acc[j].x;
                if (mg + 1 < a.M) yr[mg + 1] = acc[j].y;
                if (mg + 2 < a.M) yr[mg + 2] = acc[j].z;
                if (mg + 3 < a.M) yr[mg + 3] = acc[j].w;
              }
            }
          }
          named_bar_sync(1, NCONV * 32);
          if (ct == 0) a.cnt[tile] = 0u;
        }
      }
      pos += k1 - k0;
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// f32 -> bf16 (round to nearest even) copy of X, and zeroed tile counters
__global__ void qgemm_prep_kernel(const float4 *__restrict__ x, uint2 *__restrict__ xb, long long n4,
                                  unsigned int *cnt, int ncnt) {
  pdl_wait();
  pdl_launch_dependents();
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += stride) {
    const float4 v = __ldg(x + i);
    const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
    xb[i] = make_uint2(*reinterpret_cast<const uint32_t *>(&lo), *reinterpret_cast<const uint32_t *>(&hi));
  }
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < ncnt; i += stride)
    cnt[i] = 0u;
}

struct GemmPlan {
  int n_mt, n_tt, KS, G;
  long long total;
  size_t off_xb, off_cnt, off_part, bytes;
};

GemmPlan plan_gemm(int64_t M, int64_t N, int64_t T, int sms) {
  GemmPlan p{};
  p.n_mt = static_cast<int>((M + BM - 1) / BM);
  p.n_tt = static_cast<int>((T + BT - 1) / BT);
  p.KS = static_cast<int>((N + RK - 1) / RK);
  p.total = static_cast<long long>(p.n_mt) * p.n_tt * p.KS;
  p.G = static_cast<int>(std::min<long long>(sms, p.total));
  auto up = [](size_t v) { return (v + 255) & ~static_cast<size_t>(255); };
  p.off_xb = 0;
  p.off_cnt = up(static_cast<size_t>(T) * N * 2);
  p.off_part = p.off_cnt + up(static_cast<size_t>(p.n_mt) * p.n_tt * 4);
  p.bytes = p.off_part + static_cast<size_t>(2) * p.G * BT * BM * 4;
  return p;
}

bool gemm_shape_ok(int type, int64_t M, int64_t N, int64_t T) {
  if (type != QG_TYPE_Q8_0) return false;
  if (M < 1 || N < RK || N % RK || T < 17) return false;  // raw rows must be whole 272-byte boxes
  if (M > INT32_MAX || N > INT32_MAX || T > INT32_MAX || T * N > (1LL << 31) || T * M > (1LL << 31)) return false;
  return true;
}

qg_status gemm_tc(const void *w, const float *x, float *y, int64_t M, int64_t N, int64_t T, void *ws,
                  size_t ws_bytes, cudaStream_t s) {
  const qg::DeviceInfo &dev = qg::device_info();
  if (!dev.ok) return QG_ECUDA;
  const GemmPlan p = plan_gemm(M, N, T, dev.sms);
  if (!ws) return QG_EINVAL_PTR;
  if (!qg::aligned16(ws)) return QG_EALIGN;
  if (ws_bytes < p.bytes) return QG_EWORKSPACE;
  uint8_t *wsb = static_cast<uint8_t *>(ws);
  __nv_bfloat16 *xb = reinterpret_cast<__nv_bfloat16 *>(wsb + p.off_xb);
  unsigned int *cnt = reinterpret_cast<unsigned int *>(wsb + p.off_cnt);
  float *part = reinterpret_cast<float *>(wsb + p.off_part);

  auto enc = qg::encode_fn();
  if (!enc) return QG_ECUDA;
  // raw weights as a 16-bit [M][row_bytes / 2] tensor, boxes of 136 x 128 (272 bytes x 128 rows)
  const long long row_bytes = N / 32 * 34;
  CUtensorMap wmap, xmap;
  {
    const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(row_bytes / 2), static_cast<cuuint64_t>(M)};
    const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(row_bytes)};
    const cuuint32_t box[2] = {RAW_ROW / 2, BM};
    const cuuint32_t es[2] = {1, 1};
    if (enc(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void *>(w), gdim, gstride, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return QG_ECUDA;
  }
  {
    const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(T)};
    const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(N * 2)};
    const cuuint32_t box[2] = {BK, BT};
    const cuuint32_t es[2] = {1, 1};
    if (enc(&xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, xb, gdim, gstride, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return QG_ECUDA;
  }
  const long long n4 = T * N / 4;
  const int pb = static_cast<int>(std::min<long long>(4LL * dev.sms, (n4 + 255) / 256));
  if (qg::launch_pdl(qgemm_prep_kernel, dim3(std::max(pb, 1)), dim3(256), 0, s, reinterpret_cast<const float4 *>(x),
                     reinterpret_cast<uint2 *>(xb), n4, cnt, p.n_mt * p.n_tt) != cudaSuccess)
    return QG_ECUDA;

  GemmArgs a{};
  a.y = y;
  a.part = part;
  a.cnt = cnt;
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(N);
  a.T = static_cast<int>(T);
  a.n_mt = p.n_mt;
  a.n_tt = p.n_tt;
  a.KS = p.KS;
  a.total = p.total;
  if (!qg::set_smem_attr(reinterpret_cast<const void *>(qgemm_q8_0_kernel), SMEM_BYTES)) return QG_ECUDA;
  if (qg::launch_pdl(qgemm_q8_0_kernel, dim3(p.G), dim3(NTHREADS), SMEM_BYTES, s, wmap, xmap, a) != cudaSuccess)
    return QG_ECUDA;
  return cudaGetLastError() == cudaSuccess ? QG_OK : QG_ECUDA;
}

}  // namespace

namespace qg {
unsigned int read_status_gemm(bool clear) {
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_qg_status_gemm, sizeof(v)) != cudaSuccess) return 0xFFFFFFFFu;
  if (clear) {
    const unsigned int z = 0;
    cudaMemcpyToSymbol(g_qg_status_gemm, &z, sizeof(z));
  }
  return v;
}
}  // namespace qg

extern "C" {

size_t qgemm_workspace_size(int type, int64_t M, int64_t N, int64_t T) {
  if (T <= 16) return 0;
  if (!gemm_shape_ok(type, M, N, T)) return 0;
  const qg::DeviceInfo &dev = qg::device_info();
  if (!dev.ok) return 0;
  return plan_gemm(M, N, T, dev.sms).bytes;
}

qg_status qgemm(int type, const void *w, const float *x, float *y, int64_t M, int64_t N, int64_t T, void *ws,
                size_t ws_bytes, qg_stream_t stream) {
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int qk = 0, bb = 0;
  if (qg_block_shape(type, &qk, &bb) != QG_OK) return QG_EUNSUPPORTED;
  if (!w || !x || !y) return QG_EINVAL_PTR;
  if (M < 0 || N <= 0 || N % qk || T < 1) return QG_EINVAL_SHAPE;
  if (T <= 16) return qg::gemv_dispatch(type, w, x, y, M, N, static_cast<int>(T), s);
  if (M == 0) return QG_OK;
  if (!gemm_shape_ok(type, M, N, T)) return QG_EUNSUPPORTED;
  if (!qg::aligned16(w) || !qg::aligned16(x) || !qg::aligned16(y)) return QG_EALIGN;
  return gemm_tc(w, x, y, M, N, T, ws, ws_bytes, s);
}

}  // extern "C"
