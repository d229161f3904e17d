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
// steps span several CTAs leaves one partial tile per CTA; a second kernel sums each split
// tile's parts in CTA order (deterministic) over all SMs at once and writes Y.
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
#include "qg_tc.cuh"

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
constexpr uint32_t SMEM_BYTES = OFF_BAR + 256 + 1024;  // + alignment slack
constexpr uint32_t TMEM_COLS = 256;

QG_DEVICE void gemm_status(unsigned int bits) { atomicOr(&g_qg_status_gemm, bits); }
QG_DEVICE bool wait_or_abort_g(uint64_t *bar, uint32_t parity, volatile int *abort_flag) {
  return wait_or_abort(bar, parity, abort_flag, &g_qg_status_gemm);
}

struct GemmArgs {
  float *y;
  float *part;           // partial tiles: [2 * gridDim.x][BT][BM]
  int M, N, T;
  int n_mt, n_tt, KS;    // m tiles, token tiles, 256-k steps per tile
  long long total;       // tiles * KS
};

// CTA b's contiguous range of the (tile, k step) space starts at s(b)
__host__ __device__ inline long long range_start(long long b, long long total, int G) { return b * total / G; }
// the CTA whose range holds position p
__host__ __device__ inline int range_owner(long long p, long long total, int G) {
  return static_cast<int>(((p + 1) * G + total - 1) / total - 1);
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
          if (!wait_or_abort_g(&rempty[r], static_cast<uint32_t>(((rit / NRAW) & 1) ^ 1), abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&rfull[r], RAW_BYTES);
          tma_load_2d(smem + OFF_RAW + r * RAW_BYTES, &wmap, ks * (RK / 32) * 17, mt * BM, &rfull[r]);
          for (int sub = 0; sub < RK / BK; ++sub, ++it) {
            const int s = static_cast<int>(it % NSTAGE);
            if (!wait_or_abort_g(&empty[s], static_cast<uint32_t>(((it / NSTAGE) & 1) ^ 1), abort_flag)) {
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
        if (!wait_or_abort_g(acc_empty, static_cast<uint32_t>((si & 1) ^ 1), abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int ks = k0; ks < k1 && ok; ++ks) {
          for (int sub = 0; sub < RK / BK; ++sub, ++it) {
            const int s = static_cast<int>(it % NSTAGE);
            if (!wait_or_abort_g(&full[s], static_cast<uint32_t>((it / NSTAGE) & 1), abort_flag)) {
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
        if (!wait_or_abort_g(&rfull[r], static_cast<uint32_t>((rit / NRAW) & 1), abort_flag)) {
          ok = false;
          break;
        }
        for (int sub = 0; sub < RK / BK; ++sub, ++it) {
          const int s = static_cast<int>(it % NSTAGE);
          if (!wait_or_abort_g(&empty[s], static_cast<uint32_t>(((it / NSTAGE) & 1) ^ 1), abort_flag)) {
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
      if (!wait_or_abort_g(acc_full, static_cast<uint32_t>(si & 1), abort_flag)) {
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
      pos += k1 - k0;
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// Y of the split tiles: part sum in CTA order.  Block (tile, 8-column slice): thread = 4
// consecutive rows of one column; whole tiles (written by their CTA) are skipped.
__global__ void __launch_bounds__(256) qgemm_reduce_kernel(const GemmArgs a, int G) {
  pdl_wait();
  pdl_launch_dependents();
  const int tile = static_cast<int>(blockIdx.y);
  const long long ts = static_cast<long long>(tile) * a.KS, te = ts + a.KS;
  const int bf = range_owner(ts, a.total, G), bl = range_owner(te - 1, a.total, G);
  if (bf == bl) return;  // one CTA held the whole tile
  const int mt = tile / a.n_tt, tt = tile - mt * a.n_tt;
  const int m4 = threadIdx.x & 31, col = static_cast<int>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int bp = bf; bp <= bl; ++bp) {
    const long long sbp = range_start(bp, a.total, G);
    if (sbp >= range_start(bp + 1, a.total, G)) continue;  // an empty range
    const int sl = 2 * bp + (sbp < ts ? 1 : 0);
    const float4 v = __ldcg(reinterpret_cast<const float4 *>(a.part + static_cast<size_t>(sl) * BT * BM) + col * (BM / 4) + m4);
    acc.x += v.x;
    acc.y += v.y;
    acc.z += v.z;
    acc.w += v.w;
  }
  const int t = tt * BT + col, mg = mt * BM + 4 * m4;
  if (t >= a.T) return;
  float *yr = a.y + static_cast<size_t>(t) * a.M;
  if (mg + 3 < a.M && (a.M & 3) == 0) {
    *reinterpret_cast<float4 *>(yr + mg) = acc;
  } else {
    if (mg < a.M) yr[mg] = acc.x;
    if (mg + 1 < a.M) yr[mg + 1] = acc.y;
    if (mg + 2 < a.M) yr[mg + 2] = acc.z;
    if (mg + 3 < a.M) yr[mg + 3] = acc.w;
  }
}

// f32 -> bf16 (round to nearest even) copy of X
__global__ void qgemm_prep_kernel(const float4 *__restrict__ x, uint2 *__restrict__ xb, long long n4) {
  pdl_wait();
  pdl_launch_dependents();
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  // eight independent loads in flight per thread, then their conversions and stores: one
  // memory round trip per eight elements instead of one each
  constexpr int U = 8;
  for (long long i0 = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i0 < n4; i0 += U * stride) {
    float4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const long long i = i0 + u * stride;
      v[u] = i < n4 ? __ldg(x + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const long long i = i0 + u * stride;
      if (i < n4) {
        const __nv_bfloat162 lo = __floats2bfloat162_rn(v[u].x, v[u].y), hi = __floats2bfloat162_rn(v[u].z, v[u].w);
        xb[i] = make_uint2(*reinterpret_cast<const uint32_t *>(&lo), *reinterpret_cast<const uint32_t *>(&hi));
      }
    }
  }
}

struct GemmPlan {
  int n_mt, n_tt, KS, G;
  long long total;
  size_t off_xb, off_part, bytes;
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
  p.off_part = up(static_cast<size_t>(T) * N * 2);
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
  const int pb = static_cast<int>(std::min<long long>(4LL * dev.sms, (n4 + 8 * 256 - 1) / (8 * 256)));
  if (qg::launch_pdl(qgemm_prep_kernel, dim3(std::max(pb, 1)), dim3(256), 0, s, reinterpret_cast<const float4 *>(x),
                     reinterpret_cast<uint2 *>(xb), n4) != cudaSuccess)
    return QG_ECUDA;

  GemmArgs a{};
  a.y = y;
  a.part = part;
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
  // tiles whose k steps span several CTAs: their parts are summed by all SMs at once
  const int tiles = p.n_mt * p.n_tt;
  bool split = false;
  for (int t = 0; t < tiles && !split; ++t)
    split = range_owner(static_cast<long long>(t) * p.KS, p.total, p.G) !=
            range_owner(static_cast<long long>(t + 1) * p.KS - 1, p.total, p.G);
  if (split && qg::launch_pdl(qgemm_reduce_kernel, dim3(BT / 8, tiles), dim3(256), 0, s, a, p.G) != cudaSuccess)
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
