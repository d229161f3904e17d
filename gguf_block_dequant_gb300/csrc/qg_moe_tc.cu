// qg_moe_tc.cu -- the MoE expert step for prefill-sized batches (T > 16 tokens) on the
// sm_103a tensor cores, with the (token, pick) pairs grouped per expert so that each picked
// expert's rows cross HBM once for all of its tokens (the engine pages load the union of
// the picked experts once per chunk; here the products are grouped the same way).
//
//   plan     one CTA counts the pairs of every expert, lays them out expert by expert
//            (perm: position -> pair) and numbers each expert's 64-token tiles
//   gather   bf16 rows of the tokens (gate/up) or of the pairs' SwiGLU outputs (down) in
//            that order, so that a token tile of an expert is a contiguous block of rows
//   gemm     persistent, warp-specialised like the prefill GEMM: raw Q8_0 expert rows come
//            by TMA through 3-D tensor maps over the expert pool (slot is the third
//            coordinate), converter warps decode them to bf16, one thread issues
//            tcgen05.mma (M 128 weight rows, N 64 tokens, f32 in TMEM), and four epilogue
//            warps read one of two TMEM accumulators while the next tile's MMAs fill the
//            other.  Gate/up tiles hold 64 gate rows and the same 64 up rows, so the epilogue
//            forms act = g / (1 + exp(-g)) * u (or the GELU-tanh form) in place; down tiles
//            write dn rows of their pairs.  Inside moe_layer the down step reuses the gate/up
//            step's plan and the bf16 act rows its epilogue wrote in expert order.
//   combine  x[t] = x[t] + sum_j w_j dn[t, j] in pick order (then the residual, as the pages
//            order it)
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>

#include "qg_common.cuh"
#include "qg_host.h"
#include "qg_pipe.cuh"
#include "qg_tc.cuh"

__device__ unsigned int g_qg_status_moetc;  // this translation unit's device status word

namespace {

constexpr int BM = 128;  // weight rows per tile (MMA M)
constexpr int BT = 64;   // tokens per tile (MMA N)
constexpr int BK = 64;   // k per MMA step (one 128-byte swizzle atom of bf16)
constexpr int RK = 256;  // k per raw stage (8 Q8_0 blocks, 272 bytes per row)
// Separate rings per operand: the A slots are filled by the converters from shared memory
// (short latency: two slots keep them a step ahead of the MMA), the B slots and the raw
// weight stages come by TMA from L2 and HBM (long latency: deeper rings).
constexpr int NA = 2;
constexpr int NB = 8;
constexpr int NRAW = 3;
constexpr int NCONV = 16;
constexpr int NEPI = 4;   // epilogue warps, one per TMEM lane quarter
constexpr int NTHREADS = (2 + NCONV + NEPI) * 32;
constexpr uint32_t A_BYTES = BM * BK * 2;
constexpr uint32_t B_BYTES = BT * BK * 2;
constexpr uint32_t RAW_ROW = (RK / 32) * 34;
constexpr uint32_t RAW_BYTES = BM * RAW_ROW;
constexpr int U_PITCH = BT + 1;  // up-row staging pitch (floats), odd to spread banks
constexpr uint32_t OFF_A = 0;
constexpr uint32_t OFF_B = OFF_A + NA * A_BYTES;
constexpr uint32_t OFF_RAW = OFF_B + NB * B_BYTES;
constexpr uint32_t OFF_U = OFF_RAW + NRAW * RAW_BYTES;
constexpr uint32_t OFF_BAR = OFF_U + ((64 * U_PITCH * 4 + 1023) & ~1023u);
constexpr uint32_t OFF_TOFF = OFF_BAR + 512;
constexpr uint32_t SMEM_BYTES = OFF_TOFF + 260 * 4 + 1024;
constexpr uint32_t TMEM_COLS = 2 * BT;  // two accumulators: a tile's epilogue overlaps the next tile
constexpr int kMaxE = 256;

struct Plan {
  unsigned int *cnt;  // [E] pairs per expert
  int *off;           // [E + 1] first position of each expert
  int *toff;          // [E + 1] first tile of each expert
  int *perm;          // [P] position -> pair
};

QG_DEVICE bool pair_valid(const int32_t *ids, const int32_t *slots, int n_slots, int E, int z, int &e) {
  e = __ldg(ids + z);
  if (e < 0 || e >= E) return false;
  const int s = slots ? __ldg(slots + e) : e;
  return s >= 0 && s < n_slots;
}

// One CTA of 1024 threads.  Pairs with a bad id or slot are left out (status bit set); their
// act rows are zeroed when act_zero is given.
__global__ void __launch_bounds__(1024) moe_tc_plan_kernel(const int32_t *ids, const int32_t *slots, int n_slots,
                                                           int E, int P, float *act_zero, int F, Plan pl) {
  __shared__ unsigned int s_cnt[kMaxE], s_fill[kMaxE];
  __shared__ int s_off[kMaxE + 1];
  pdl_wait();
  pdl_launch_dependents();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    s_cnt[e] = 0u;
    s_fill[e] = 0u;
  }
  __syncthreads();
  for (int z = threadIdx.x; z < P; z += blockDim.x) {
    int e;
    if (pair_valid(ids, slots, n_slots, E, z, e)) {
      atomicAdd(&s_cnt[e], 1u);
    } else {
      atomicOr(&g_qg_status_moetc, QG_STATUS_BIT_ID);
      if (act_zero)
        for (int f = 0; f < F; ++f) act_zero[static_cast<size_t>(z) * F + f] = 0.f;
    }
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    // exclusive scans of the pair counts and of the tile counts: lane l holds experts
    // kMaxE / 32 * l .., the lane totals are scanned with shuffles
    constexpr int PER = kMaxE / 32;
    const int lane = threadIdx.x;
    int c[PER], o_loc = 0, t_loc = 0;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int e = lane * PER + i;
      c[i] = e < E ? static_cast<int>(s_cnt[e]) : 0;
      o_loc += c[i];
      t_loc += (c[i] + BT - 1) / BT;
    }
    int o_inc = o_loc, t_inc = t_loc;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int oa = __shfl_up_sync(0xFFFFFFFFu, o_inc, d), ta = __shfl_up_sync(0xFFFFFFFFu, t_inc, d);
      if (lane >= d) {
        o_inc += oa;
        t_inc += ta;
      }
    }
    int o = o_inc - o_loc, t = t_inc - t_loc;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int e = lane * PER + i;
      if (e < E) {
        s_off[e] = o;
        pl.off[e] = o;
        pl.toff[e] = t;
        pl.cnt[e] = static_cast<unsigned int>(c[i]);
      }
      o += c[i];
      t += (c[i] + BT - 1) / BT;
    }
    if (lane == 31) {
      pl.off[E] = o_inc;
      pl.toff[E] = t_inc;
    }
  }
  __syncthreads();
  for (int z = threadIdx.x; z < P; z += blockDim.x) {
    int e;
    if (pair_valid(ids, slots, n_slots, E, z, e)) pl.perm[s_off[e] + atomicAdd(&s_fill[e], 1u)] = z;
  }
}

// dst[pos][0..K) = bf16(src[row(pos)][0..K)) for every grouped position, row = pair / k
// (token rows) or the pair itself; K % 8 == 0.
template <bool BY_TOKEN>
__global__ void moe_tc_gather_kernel(const float *__restrict__ src, int K, int k, const int *perm, const int *n_valid,
                                     __nv_bfloat16 *dst, int P) {
  pdl_wait();
  pdl_launch_dependents();
  const int np = min(*n_valid, P);
  const long long K8 = K / 8;
  const long long total = static_cast<long long>(np) * K8;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int pos = static_cast<int>(i / K8);
    const int c8 = static_cast<int>(i - static_cast<long long>(pos) * K8);
    const int z = perm[pos];
    const int row = BY_TOKEN ? z / k : z;
    const float4 *sp = reinterpret_cast<const float4 *>(src + static_cast<size_t>(row) * K + 8 * c8);
    const float4 a = __ldg(sp), b = __ldg(sp + 1);
    const __nv_bfloat162 p0 = __floats2bfloat162_rn(a.x, a.y), p1 = __floats2bfloat162_rn(a.z, a.w);
    const __nv_bfloat162 p2 = __floats2bfloat162_rn(b.x, b.y), p3 = __floats2bfloat162_rn(b.z, b.w);
    uint4 o;
    o.x = *reinterpret_cast<const uint32_t *>(&p0);
    o.y = *reinterpret_cast<const uint32_t *>(&p1);
    o.z = *reinterpret_cast<const uint32_t *>(&p2);
    o.w = *reinterpret_cast<const uint32_t *>(&p3);
    *reinterpret_cast<uint4 *>(dst + static_cast<size_t>(pos) * K + 8 * c8) = o;
  }
}

struct TcArgs {
  Plan pl;
  const int32_t *slots;
  int E, n_mt, KS, k, F, H;
  float *act;                 // gate/up: act [P][F] f32
  __nv_bfloat16 *act_sorted;  // gate/up: act in grouped order [P][F] bf16
  float *dn;                  // down: dn [P][H] f32 (row = pair)
  int act_kind;               // gate/up: 0 SiLU(g) u, 1 GELU-tanh(g) u
};

QG_DEVICE bool tc_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag) {
  return wait_or_abort(bar, parity, abort_flag, &g_qg_status_moetc);
}

// Work item -> expert, first grouped row, valid rows, m tile.
struct Item {
  int e, row0, nrows, mt, slot;
};

QG_DEVICE Item item_of(long long it, const TcArgs &a, const int *s_toff) {
  Item r;
  const int tile = static_cast<int>(it / a.n_mt);
  r.mt = static_cast<int>(it - static_cast<long long>(tile) * a.n_mt);
  int lo = 0, hi = a.E;  // largest e with toff[e] <= tile
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s_toff[mid] <= tile) lo = mid;
    else hi = mid;
  }
  while (lo + 1 < a.E && s_toff[lo + 1] <= tile) ++lo;  // skip experts without tiles
  r.e = lo;
  const int tt = tile - s_toff[lo];
  r.row0 = a.pl.off[lo] + tt * BT;
  r.nrows = min(BT, static_cast<int>(a.pl.cnt[lo]) - tt * BT);
  r.slot = a.slots ? __ldg(a.slots + lo) : lo;
  return r;
}

template <bool GATEUP>
__global__ void __launch_bounds__(NTHREADS, 1)
    moe_tc_gemm_kernel(const __grid_constant__ CUtensorMap wmap_a, const __grid_constant__ CUtensorMap wmap_b,
                       const __grid_constant__ CUtensorMap xmap, const TcArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t *afull = reinterpret_cast<uint64_t *>(smem + OFF_BAR);  // [NA] converters done
  uint64_t *aempty = afull + NA;                                     // [NA] MMA done with the slot
  uint64_t *bfull = aempty + NA;                                     // [NB] B tile landed
  uint64_t *bempty = bfull + NB;                                     // [NB] MMA done with the slot
  uint64_t *rfull = bempty + NB;
  uint64_t *rempty = rfull + NRAW;
  uint64_t *acc_full = rempty + NRAW;  // [2]
  uint64_t *acc_empty = acc_full + 2;  // [2]
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(acc_empty + 2);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  int *s_toff = reinterpret_cast<int *>(smem + OFF_TOFF);
  float *s_u = reinterpret_cast<float *>(smem + OFF_U);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = static_cast<int>(gridDim.x);
  if (threadIdx.x == 0) {
    for (int i = 0; i < NA; ++i) {
      mbar_init(&afull[i], NCONV);
      mbar_init(&aempty[i], 1);
    }
    for (int i = 0; i < NB; ++i) {
      mbar_init(&bfull[i], 1);
      mbar_init(&bempty[i], 1);
    }
    for (int i = 0; i < NRAW; ++i) {
      mbar_init(&rfull[i], 1);
      mbar_init(&rempty[i], NCONV);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], NEPI);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, TMEM_COLS);
  pdl_wait();
  pdl_launch_dependents();
  for (int e = threadIdx.x; e <= a.E; e += blockDim.x) s_toff[e] = a.pl.toff[e];
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const long long n_items = static_cast<long long>(s_toff[a.E]) * a.n_mt;
  const long long beg = static_cast<long long>(blockIdx.x) * n_items / G;
  const long long end = static_cast<long long>(blockIdx.x + 1) * n_items / G;
  const uint32_t sA = smem_u32(smem + OFF_A), sB = smem_u32(smem + OFF_B), sRaw = smem_u32(smem + OFF_RAW);

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      long long st = 0, rt = 0;
      bool ok = true;
      for (long long it = beg; it < end && ok; ++it) {
        const Item w = item_of(it, a, s_toff);
        for (int ks = 0; ks < a.KS && ok; ++ks, ++rt) {
          const int r = static_cast<int>(rt % NRAW);
          if (!tc_wait(&rempty[r], static_cast<uint32_t>(((rt / NRAW) & 1) ^ 1), abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&rfull[r], RAW_BYTES);
          uint8_t *raw = smem + OFF_RAW + r * RAW_BYTES;
          if (GATEUP) {
            tma_load_3d(raw, &wmap_a, ks * (RK / 32) * 17, w.mt * (BM / 2), w.slot, &rfull[r]);
            tma_load_3d(raw + (BM / 2) * RAW_ROW, &wmap_b, ks * (RK / 32) * 17, w.mt * (BM / 2), w.slot, &rfull[r]);
          } else {
            tma_load_3d(raw, &wmap_a, ks * (RK / 32) * 17, w.mt * BM, w.slot, &rfull[r]);
          }
          for (int sub = 0; sub < RK / BK; ++sub, ++st) {
            const int s = static_cast<int>(st % NB);
            if (!tc_wait(&bempty[s], static_cast<uint32_t>(((st / NB) & 1) ^ 1), abort_flag)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&bfull[s], B_BYTES);
            tma_load_2d(smem + OFF_B + s * B_BYTES, &xmap, ks * RK + sub * BK, w.row0, &bfull[s]);
          }
        }
      }
      if (*abort_flag) {
        for (long long j = (st > NB ? st - NB : 0); j < st; ++j)
          cleanup_wait(&bfull[j % NB], static_cast<uint32_t>((j / NB) & 1));
        for (long long j = (rt > NRAW ? rt - NRAW : 0); j < rt; ++j)
          cleanup_wait(&rfull[j % NRAW], static_cast<uint32_t>((j / NRAW) & 1));
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc(BM, BT);
      long long st = 0;
      int ii = 0;
      bool ok = true;
      for (long long it = beg; it < end && ok; ++it, ++ii) {
        const int b = ii & 1;  // this tile's accumulator; its previous tile's epilogue must be done
        if (!tc_wait(&acc_empty[b], static_cast<uint32_t>(((ii >> 1) & 1) ^ 1), abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int ks = 0; ks < a.KS && ok; ++ks) {
          for (int sub = 0; sub < RK / BK; ++sub, ++st) {
            const int sa = static_cast<int>(st % NA), sb = static_cast<int>(st % NB);
            if (!tc_wait(&bfull[sb], static_cast<uint32_t>((st / NB) & 1), abort_flag) ||
                !tc_wait(&afull[sa], static_cast<uint32_t>((st / NA) & 1), abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t aa = sA + sa * A_BYTES, bb = sB + sb * B_BYTES;
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)
              tc_mma_bf16(tmem + static_cast<uint32_t>(b * BT), sw128_desc(aa + kk * 32), sw128_desc(bb + kk * 32),
                          idesc, (ks == 0 && sub == 0 && kk == 0) ? 0u : 1u);
            tc_commit(&aempty[sa]);  // both slots are free once these MMAs finish
            tc_commit(&bempty[sb]);
          }
        }
        if (ok) tc_commit(&acc_full[b]);
      }
      if (st > 0) cleanup_wait(&bempty[(st - 1) % NB], static_cast<uint32_t>(((st - 1) / NB) & 1));
    }
  } else if (warp < 2 + NCONV) {
    // ---------------- converters ----------------
    const int ct = threadIdx.x - 64;
    const int crow = 8 * (ct >> 5) + (lane & 7);
    const int chb = lane >> 3;
    long long st = 0, rt = 0;
    bool ok = true;
    for (long long it = beg; it < end && ok; ++it) {
      for (int ks = 0; ks < a.KS && ok; ++ks, ++rt) {
        const int r = static_cast<int>(rt % NRAW);
        if (!tc_wait(&rfull[r], static_cast<uint32_t>((rt / NRAW) & 1), abort_flag)) {
          ok = false;
          break;
        }
        for (int sub = 0; sub < RK / BK; ++sub, ++st) {
          const int s = static_cast<int>(st % NA);
          if (!tc_wait(&aempty[s], static_cast<uint32_t>(((st / NA) & 1) ^ 1), abort_flag)) {
            ok = false;
            break;
          }
          convert_half(sRaw + r * RAW_BYTES + static_cast<uint32_t>(crow) * RAW_ROW, sub, chb,
                       sA + s * A_BYTES + static_cast<uint32_t>(crow) * 128u, crow);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&afull[s]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&rempty[r]);
      }
    }
  } else {
    // ---------------- epilogue: warp w reads TMEM lanes 32 (w % 4) .. + 31 ----------------
    const int q = warp & 3;
    int ii = 0;
    bool ok = true;
    for (long long it = beg; it < end && ok; ++it, ++ii) {
      const Item w = item_of(it, a, s_toff);
      const int b = ii & 1;
      const bool got = tc_wait(&acc_full[b], static_cast<uint32_t>((ii >> 1) & 1), abort_flag);
      // the gate/up epilogue's warps meet at named barriers below: they take the abort
      // decision together, after a barrier that every one of them reaches
      if (GATEUP) named_bar_sync(1, NEPI * 32);
      if (!got || *abort_flag) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll 1
      for (int cg = 0; cg < BT / 16; ++cg) {
        float v[16];
        tmem_ld16(tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(b * BT + 16 * cg), v);
        if (GATEUP) {
          // lanes 0-63: gate rows, 64-127: the same up rows
          const int il = 32 * (q & 1) + lane;
          if (q >= 2) {
#pragma unroll
            for (int c = 0; c < 16; ++c) s_u[il * U_PITCH + 16 * cg + c] = v[c];
          }
          named_bar_sync(1, NEPI * 32);
          if (q < 2) {
            const int i = w.mt * (BM / 2) + il;
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              const int col = 16 * cg + c;
              if (col < w.nrows) {
                const float g = v[c], u = s_u[il * U_PITCH + col];
                const float act = act_mul(a.act_kind, g, u);
                const int pos = w.row0 + col;
                const int z = a.pl.perm[pos];
                a.act[static_cast<size_t>(z) * a.F + i] = act;
                a.act_sorted[static_cast<size_t>(pos) * a.F + i] = __float2bfloat16_rn(act);
              }
            }
          }
          named_bar_sync(1, NEPI * 32);  // s_u is free for the next columns
        } else {
          const int h = w.mt * BM + 32 * q + lane;
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const int col = 16 * cg + c;
            if (col < w.nrows) a.dn[static_cast<size_t>(a.pl.perm[w.row0 + col]) * a.H + h] = v[c];
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[b]);
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// x[t][h] = (add_residual ? x[t][h] : 0) + (sum_j (dn[t k + j][h] ds[e_j]) w[t][j] + sh[t][h] s(sg[t])),
// picks in order (moeAccum; moeSum with the per-expert down scale ds; moeAccumShared with the
// shared expert's row sh and gate logit sg, s the logistic function), picks with a bad id or
// slot left out; ds, sh may be null
__global__ void moe_tc_combine_kernel(const float *__restrict__ dn, const float *__restrict__ wts,
                                      const int32_t *ids, const int32_t *slots, int n_slots, int E, int T, int k,
                                      int H, float *x, int add_residual, const float *__restrict__ ds,
                                      const float *__restrict__ sh, const float *__restrict__ sg) {
  pdl_wait();
  pdl_launch_dependents();
  const int H4 = H / 4;
  const long long total = static_cast<long long>(T) * H4;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int t = static_cast<int>(i / H4), h4 = static_cast<int>(i - static_cast<long long>(t) * H4);
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    // the picks in batches of 8: every dn load of a batch is in flight at once, then the sums
    // in pick order
    for (int j0 = 0; j0 < k; j0 += 8) {
      float4 d[8];
      float wj[8], c[8];
      bool use[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int z = t * k + j0 + u;
        int e = 0;
        use[u] = j0 + u < k && pair_valid(ids, slots, n_slots, E, z, e);
        d[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        wj[u] = 0.f;
        c[u] = 1.f;
        if (use[u]) {
          wj[u] = __ldg(wts + z);
          d[u] = __ldg(reinterpret_cast<const float4 *>(dn + static_cast<size_t>(z) * H) + h4);
          if (ds) c[u] = __ldg(ds + e);
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (!use[u]) continue;
        float4 v = d[u];
        if (ds) v = make_float4(v.x * c[u], v.y * c[u], v.z * c[u], v.w * c[u]);
        s.x = fmaf(wj[u], v.x, s.x);
        s.y = fmaf(wj[u], v.y, s.y);
        s.z = fmaf(wj[u], v.z, s.z);
        s.w = fmaf(wj[u], v.w, s.w);
      }
    }
    if (sh) {
      const float gt = 1.0f / (1.0f + expf(-__ldg(sg + t)));
      const float4 v = __ldg(reinterpret_cast<const float4 *>(sh + static_cast<size_t>(t) * H) + h4);
      s.x += v.x * gt;
      s.y += v.y * gt;
      s.z += v.z * gt;
      s.w += v.w * gt;
    }
    float4 *xp = reinterpret_cast<float4 *>(x + static_cast<size_t>(t) * H) + h4;
    if (add_residual) {
      const float4 o = *xp;
      s.x += o.x;
      s.y += o.y;
      s.z += o.z;
      s.w += o.w;
    }
    *xp = s;
  }
}

// ---- host -------------------------------------------------------------------------------

inline size_t up256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

struct TcLayout {
  size_t cnt, off, toff, perm, xs, acts, total;
};

TcLayout tc_layout(int T, int k, int E, int H, int F) {
  const size_t P = static_cast<size_t>(T) * k;
  TcLayout l;
  l.cnt = 0;
  l.off = up256(static_cast<size_t>(E) * 4);
  l.toff = l.off + up256(static_cast<size_t>(E + 1) * 4);
  l.perm = l.toff + up256(static_cast<size_t>(E + 1) * 4);
  l.xs = l.perm + up256(P * 4);
  l.acts = l.xs + up256(P * H * 2);
  l.total = l.acts + up256(P * F * 2);
  return l;
}

Plan plan_at(void *ws, const TcLayout &l) {
  uint8_t *b = static_cast<uint8_t *>(ws);
  Plan p;
  p.cnt = reinterpret_cast<unsigned int *>(b + l.cnt);
  p.off = reinterpret_cast<int *>(b + l.off);
  p.toff = reinterpret_cast<int *>(b + l.toff);
  p.perm = reinterpret_cast<int *>(b + l.perm);
  return p;
}

// raw Q8_0 expert rows as a 16-bit [n_slots][rows][row_bytes / 2] tensor, boxes of 272 bytes
// x box_rows rows x 1 slot
bool encode_expert_map(CUtensorMap *m, const void *base, long long row_bytes, int rows, int n_slots, long long stride,
                       int box_rows) {
  auto enc = qg::encode_fn();
  if (!enc) return false;
  const cuuint64_t gdim[3] = {static_cast<cuuint64_t>(row_bytes / 2), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(n_slots)};
  const cuuint64_t gstride[2] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(stride)};
  const cuuint32_t box[3] = {RAW_ROW / 2, static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void *>(base), gdim, gstride, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_rows_map(CUtensorMap *m, const __nv_bfloat16 *base, int K, int rows) {
  auto enc = qg::encode_fn();
  if (!enc) return false;
  const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(K) * 2};
  const cuuint32_t box[2] = {BK, BT};
  const cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<__nv_bfloat16 *>(base), gdim, gstride, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

qg_status launch_plan(const int32_t *ids, const int32_t *slots, int n_slots, int E, int P, float *act_zero, int F,
                      const Plan &pl, cudaStream_t s) {
  return qg::launch_pdl(moe_tc_plan_kernel, dim3(1), dim3(1024), 0, s, ids, slots, n_slots, E, P, act_zero, F, pl) ==
                 cudaSuccess
             ? QG_OK
             : QG_ECUDA;
}

template <bool BY_TOKEN>
qg_status launch_gather(const float *src, int K, int k, const Plan &pl, const int *n_valid, __nv_bfloat16 *dst, int P,
                        cudaStream_t s) {
  const qg::DeviceInfo &dev = qg::device_info();
  const long long work = static_cast<long long>(P) * (K / 8);
  const int grid = static_cast<int>(std::max<long long>(1, std::min<long long>(4LL * dev.sms, (work + 255) / 256)));
  return qg::launch_pdl(moe_tc_gather_kernel<BY_TOKEN>, dim3(grid), dim3(256), 0, s, src, K, k,
                        static_cast<const int *>(pl.perm), n_valid, dst, P) == cudaSuccess
             ? QG_OK
             : QG_ECUDA;
}

template <bool GATEUP>
qg_status launch_tc_gemm(const CUtensorMap &ma, const CUtensorMap &mb, const CUtensorMap &mx, const TcArgs &a,
                         cudaStream_t s) {
  const qg::DeviceInfo &dev = qg::device_info();
  auto kern = moe_tc_gemm_kernel<GATEUP>;
  if (!qg::set_smem_attr(reinterpret_cast<const void *>(kern), SMEM_BYTES)) return QG_ECUDA;
  return qg::launch_pdl(kern, dim3(dev.sms), dim3(NTHREADS), SMEM_BYTES, s, ma, mb, mx, a) == cudaSuccess ? QG_OK
                                                                                                         : QG_ECUDA;
}

}  // namespace

namespace qg {

unsigned int read_status_moetc(bool clear) {
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_qg_status_moetc, sizeof(v)) != cudaSuccess) return 0xFFFFFFFFu;
  if (clear) {
    const unsigned int z = 0;
    cudaMemcpyToSymbol(g_qg_status_moetc, &z, sizeof(z));
  }
  return v;
}

bool moe_tc_supported(int type, int H, int F, int E) {
  return type == QG_TYPE_Q8_0 && H % RK == 0 && F % RK == 0 && H % BM == 0 && F % (BM / 2) == 0 && E <= kMaxE;
}

size_t moe_tc_workspace(int T, int k, int E, int H, int F) { return tc_layout(T, k, E, H, F).total; }

qg_status moe_swiglu_tc(const void *w_gate, const void *w_up, int64_t stride, const int32_t *slots, int n_slots,
                        int E, const int32_t *ids, const float *xn, int T, int k, int H, int F, float *act, void *ws,
                        cudaStream_t s, int act_kind) {
  const int P = T * k;
  const TcLayout L = tc_layout(T, k, E, H, F);
  const Plan pl = plan_at(ws, L);
  uint8_t *b = static_cast<uint8_t *>(ws);
  __nv_bfloat16 *xs = reinterpret_cast<__nv_bfloat16 *>(b + L.xs);
  __nv_bfloat16 *acts = reinterpret_cast<__nv_bfloat16 *>(b + L.acts);
  const long long row_bytes = static_cast<long long>(H) / 32 * 34;
  CUtensorMap mg, mu, mx;
  if (!encode_expert_map(&mg, w_gate, row_bytes, F, n_slots, stride, BM / 2) ||
      !encode_expert_map(&mu, w_up, row_bytes, F, n_slots, stride, BM / 2) || !encode_rows_map(&mx, xs, H, P))
    return QG_ECUDA;
  qg_status r = launch_plan(ids, slots, n_slots, E, P, act, F, pl, s);
  if (r != QG_OK) return r;
  r = launch_gather<true>(xn, H, k, pl, pl.off + E, xs, P, s);
  if (r != QG_OK) return r;
  TcArgs a{};
  a.pl = pl;
  a.slots = slots;
  a.E = E;
  a.n_mt = F / (BM / 2);
  a.KS = H / RK;
  a.k = k;
  a.F = F;
  a.H = H;
  a.act = act;
  a.act_sorted = acts;
  a.act_kind = act_kind;
  return launch_tc_gemm<true>(mg, mu, mx, a, s);
}

qg_status moe_launch_combine(const float *dn, const float *weights, const int32_t *ids, const int32_t *slots,
                             int n_slots, int E, int T, int k, int H, float *x_inout, int add_residual,
                             cudaStream_t s, const MoeVar &v) {
  const qg::DeviceInfo &dev = qg::device_info();
  const long long work = static_cast<long long>(T) * (H / 4);
  const int grid = static_cast<int>(std::max<long long>(1, std::min<long long>(4LL * dev.sms, (work + 127) / 128)));
  return qg::launch_pdl(moe_tc_combine_kernel, dim3(grid), dim3(128), 0, s, dn, weights, ids, slots, n_slots, E, T, k,
                        H, x_inout, add_residual, v.ds, v.sh, v.sg) == cudaSuccess
             ? QG_OK
             : QG_ECUDA;
}

qg_status moe_combine_tc(const void *w_down, int64_t stride, const int32_t *slots, int n_slots, int E,
                         const int32_t *ids, const float *weights, const float *act, int T, int k, int H, int F,
                         float *x_inout, int add_residual, float *dn, void *ws, cudaStream_t s,
                         const MoeVar &v, bool sorted_ready) {
  const int P = T * k;
  const TcLayout L = tc_layout(T, k, E, H, F);
  const Plan pl = plan_at(ws, L);
  uint8_t *b = static_cast<uint8_t *>(ws);
  __nv_bfloat16 *acts = reinterpret_cast<__nv_bfloat16 *>(b + L.acts);
  const long long row_bytes = static_cast<long long>(F) / 32 * 34;
  CUtensorMap md, mx;
  if (!encode_expert_map(&md, w_down, row_bytes, H, n_slots, stride, BM) || !encode_rows_map(&mx, acts, F, P))
    return QG_ECUDA;
  qg_status r;
  if (!sorted_ready) {
    // the grouping and the bf16 act rows in expert order; moe_layer's gate/up step has left
    // both in the workspace already (its epilogue writes the sorted rows)
    r = launch_plan(ids, slots, n_slots, E, P, nullptr, F, pl, s);
    if (r != QG_OK) return r;
    r = launch_gather<false>(act, F, k, pl, pl.off + E, acts, P, s);
    if (r != QG_OK) return r;
  }
  TcArgs a{};
  a.pl = pl;
  a.slots = slots;
  a.E = E;
  a.n_mt = H / BM;
  a.KS = F / RK;
  a.k = k;
  a.F = F;
  a.H = H;
  a.dn = dn;
  r = launch_tc_gemm<false>(md, md, mx, a, s);
  if (r != QG_OK) return r;
  return moe_launch_combine(dn, weights, ids, slots, n_slots, E, T, k, H, x_inout, add_residual, s, v);
}

}  // namespace qg
