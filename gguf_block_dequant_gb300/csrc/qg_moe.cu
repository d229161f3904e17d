// qg_moe.cu -- the MoE step on sm_103a: router + top-k, grouped gate/up expert rows with
// SwiGLU, and down expert rows with the weighted combine (the qwen3_moe_ssd.js decode
// sequence on the engine pages: matmulF32 -> topk -> expertQ8 (gate||up) -> siluMulMoe ->
// expertQ8 with inputPerSlot (down) -> moeAccum).
//
// Router: one CTA per expert row of the f32 router matrix (its warps split the row), all
// tokens of a 16-token tile reused against each weight load; the last CTA of a token tile (ticket counter) takes the k
// greedy picks per token (one warp per token) and their renormalised softmax weights.
//
// Expert kernels (persistent, one CTA per SM): every CTA first groups the (token, pick)
// pairs by expert in shared memory (deterministic warp-ballot counting, no atomics), so each
// picked expert forms one "unit" that carries up to TT tokens.  Units are cut into row blocks
// of four weight rows -- {gate i, gate i+1, up i, up i+1} for the gate/up kernel, {down h ..
// h+3} for the down kernel -- and the CTAs take balanced contiguous ranges of row blocks.
// Inside a CTA every warp streams its row blocks through its own ring of shared-memory slots
// with 1-D bulk copies (cp.async.bulk) and decodes the raw blocks in registers exactly as
// the dense GEMV does (qg_decode.cuh), the unit's token activations resident in shared
// memory.  Each expert's weight bytes cross HBM once per call, for all of its tokens.
//
// Gate/up epilogue: act[z][i] = g_i / (1 + exp(-g_i)) * u_i written straight from the warp's
// sums.  Down epilogue: the warp writes the dn values of each pair to the workspace; a small
// combine kernel then forms  x[t][h] = x[t][h] + sum_j w_j * dn_j[h]  in pick order
// (deterministic), launched with programmatic dependent launch so that it starts as the down
// kernel drains.
#include <cuda.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "qg_decode.cuh"
#include "qg_host.h"
#include "qg_pipe.cuh"

__device__ unsigned int g_qg_status_moe;

namespace {

constexpr int kMaxNS = 4;
constexpr int kRouterTB = 16;  // tokens per router CTA
constexpr int kRouterWarps = 4;  // warps per router CTA (one expert per CTA)
constexpr int kMaxE = 256;
constexpr int kMaxK = 32;

QG_DEVICE void moe_status(unsigned int bits) { atomicOr(&g_qg_status_moe, bits); }

// ------------------------------------------------------------------------------------------
// Router and top-k
// ------------------------------------------------------------------------------------------

// k greedy picks over one token's E logits (ties to the lowest expert id), weights
// exp(l_j - l_max) / sum over the picks (softmax restricted to the picks).  One warp.
QG_DEVICE void topk_token(const float *l, int E, int k, int lane, int32_t *ids, float *wts) {
  float v[kMaxE / 32];
  unsigned int avail = 0;
#pragma unroll
  for (int i = 0; i < kMaxE / 32; ++i) {
    const int e = lane + 32 * i;
    v[i] = 0.f;
    if (e < E) {
      v[i] = __ldcg(l + e);
      avail |= 1u << i;
    }
  }
  float lmax = 0.f, den = 0.f, my_ex = 0.f;
  int my_id = 0;
  for (int j = 0; j < k; ++j) {
    float bv = 0.f;
    int bi = INT_MAX;
#pragma unroll
    for (int i = 0; i < kMaxE / 32; ++i)
      if ((avail >> i) & 1u)
        if (bi == INT_MAX || v[i] > bv) {
          bv = v[i];
          bi = lane + 32 * i;
        }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
      const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
      if (oi != INT_MAX && (bi == INT_MAX || ov > bv || (ov == bv && oi < bi))) {
        bv = ov;
        bi = oi;
      }
    }
    if ((bi & 31) == lane) avail &= ~(1u << (bi >> 5));
    if (j == 0) lmax = bv;
    const float ex = expf(bv - lmax);
    den += ex;
    if (lane == j) {
      my_id = bi;
      my_ex = ex;
    }
  }
  if (lane < k) {
    ids[lane] = my_id;
    wts[lane] = my_ex / den;
  }
}

// grid (E, token tiles of kRouterTB); kRouterWarps warps split the H dot of the CTA's expert
__global__ void __launch_bounds__(kRouterWarps * 32) moe_router_kernel(const float *__restrict__ xn,
                                                                        const float *__restrict__ wr, int T, int H,
                                                                        int E, int k, float *logits, int32_t *ids,
                                                                        float *weights, unsigned int *ticket,
                                                                        int do_topk) {
  __shared__ float part[kRouterWarps][kRouterTB];
  __shared__ unsigned int s_last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_wait();
  pdl_launch_dependents();
  const int e = blockIdx.x;
  const int t0 = blockIdx.y * kRouterTB;
  const int nt = min(kRouterTB, T - t0);
  float acc[kRouterTB];
#pragma unroll
  for (int t = 0; t < kRouterTB; ++t) acc[t] = 0.f;
  const float4 *w4 = reinterpret_cast<const float4 *>(wr + static_cast<size_t>(e) * H);
  const float4 *x4 = reinterpret_cast<const float4 *>(xn + static_cast<size_t>(t0) * H);
  const int H4 = H >> 2;
#pragma unroll 4
  for (int h = warp * 32 + lane; h < H4; h += kRouterWarps * 32) {
    const float4 w = __ldg(w4 + h);
#pragma unroll
    for (int t = 0; t < kRouterTB; ++t) {
      if (t < nt) {
        const float4 x = __ldg(x4 + static_cast<size_t>(t) * H4 + h);
        acc[t] = fmaf(w.x, x.x, acc[t]);
        acc[t] = fmaf(w.y, x.y, acc[t]);
        acc[t] = fmaf(w.z, x.z, acc[t]);
        acc[t] = fmaf(w.w, x.w, acc[t]);
      }
    }
  }
#pragma unroll
  for (int t = 0; t < kRouterTB; ++t) {
    const float s = warp_sum(acc[t]);
    if (lane == 0) part[warp][t] = s;
  }
  __syncthreads();
  if (threadIdx.x < nt) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kRouterWarps; ++w) s += part[w][threadIdx.x];
    logits[static_cast<size_t>(t0 + threadIdx.x) * E + e] = s;
  }
  if (!do_topk) return;
  // the last CTA of this token tile to finish takes the picks
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned int old = atomicAdd(&ticket[blockIdx.y], 1u);
    s_last = (old == gridDim.x - 1) ? 1u : 0u;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int t = t0 + warp; t < t0 + nt; t += kRouterWarps)
    topk_token(logits + static_cast<size_t>(t) * E, E, k, lane, ids + static_cast<size_t>(t) * k,
               weights + static_cast<size_t>(t) * k);
  __syncthreads();
  if (threadIdx.x == 0) ticket[blockIdx.y] = 0u;
}

// ------------------------------------------------------------------------------------------
// Expert kernels
// ------------------------------------------------------------------------------------------

struct MoeArgs {
  const uint8_t *wa;  // gate rows (gate/up kernel) or down rows (down kernel)
  const uint8_t *wb;  // up rows (gate/up kernel)
  long long stride;   // bytes between expert slots
  uintptr_t mend_a, mend_b;  // last 16-byte boundary inside each weight tensor's extent
  const int32_t *slots;
  int n_slots, E;
  const int32_t *ids;
  const float *wts;  // combine weights [T][k] (down kernel)
  const float *xin;  // xn [T][H] (gate/up) or act [T*k][F] (down)
  float *out;        // act [T*k][F] (gate/up) or x_inout [T][H] (down)
  float *dn;         // [T*k][H] workspace (down)
  int T, k, H, F;
  int K;             // dot length: H (gate/up) or F (down)
  int R;             // rows of one expert matrix: F (gate/up) or H (down)
  long long row_bytes;
  int nblk;          // row blocks per unit
  int KC, nchunks, NS, stage_bytes, seg_slot;
  int xrow_bytes;    // shared-memory bytes per token slot (whole groups of SG elements)
  int gseg;          // whole-row stages of the gate/up kernel: offset of the up rows in a slot
  int add_residual;
  int box_rows;      // one token: rows (of 32 floats) per activation tensor copy
  // gate/up kernel inside moe_layer: take the top-k picks from the router logits here
  // (every CTA ranks the logits itself; CTA 0 also stores ids and weights)
  int fuse_topk;
  const float *logits;
  int32_t *ids_out;
  float *wts_out;
  uint32_t off_plan, off_x, off_ring;
};

// Pairs grouped by expert.  s_id[z]: expert of pair z, or -1 when its id or slot is out of
// range; s_pairs: pair indices ordered by expert, then by pair index; unit u covers
// s_pairs[u_first[u] .. + u_cnt[u]) of one expert (at most TT pairs), slot u_slot[u].
struct PlanSmem {
  int *s_id, *s_pairs, *u_slot, *u_first, *u_cnt, *s_cnt, *s_start, *s_ustart, *s_kv;
  int32_t *tk_ids;  // fused top-k results [T][k]
  float *tk_w;
};

QG_DEVICE PlanSmem plan_layout(uint8_t *base, int P, int T) {
  PlanSmem p;
  int *q = reinterpret_cast<int *>(base);
  p.s_id = q;
  q += P;
  p.s_pairs = q;
  q += P;
  p.u_slot = q;
  q += P;
  p.u_first = q;
  q += P;
  p.u_cnt = q;
  q += P;
  p.s_cnt = q;
  q += kMaxE;
  p.s_start = q;
  q += kMaxE;
  p.s_ustart = q;
  q += kMaxE + 1;
  p.s_kv = q;
  q += T;
  p.tk_ids = q;
  q += P;
  p.tk_w = reinterpret_cast<float *>(q);
  return p;
}

inline uint32_t plan_bytes(int P, int T) {
  return static_cast<uint32_t>((7 * P + 3 * kMaxE + 1 + T) * 4 + 15) & ~15u;
}

// Builds the grouping; returns the number of units.  Every thread of the CTA takes part.
template <int NW>
QG_DEVICE int build_plan(const MoeArgs &a, int TT, const PlanSmem &p) {
  const int P = a.T * a.k;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (a.fuse_topk) {
    for (int t = warp; t < a.T; t += NW)
      topk_token(a.logits + static_cast<size_t>(t) * a.E, a.E, a.k, lane, p.tk_ids + t * a.k, p.tk_w + t * a.k);
    __syncthreads();
    if (blockIdx.x == 0)
      for (int z = tid; z < P; z += NW * 32) {
        a.ids_out[z] = p.tk_ids[z];
        a.wts_out[z] = p.tk_w[z];
      }
  }
  for (int z = tid; z < P; z += NW * 32) {
    const int e = a.fuse_topk ? p.tk_ids[z] : __ldg(a.ids + z);
    bool ok = e >= 0 && e < a.E;
    if (ok) {
      const int s = a.slots ? __ldg(a.slots + e) : e;
      ok = s >= 0 && s < a.n_slots;
    }
    p.s_id[z] = ok ? e : -1;
    if (!ok && blockIdx.x == 0) moe_status(QG_STATUS_BIT_ID);
  }
  __syncthreads();
  // pairs per expert
  for (int e = warp; e < a.E; e += NW) {
    int c = 0;
    for (int z0 = 0; z0 < P; z0 += 32) {
      const bool m = (z0 + lane < P) && p.s_id[z0 + lane] == e;
      c += __popc(__ballot_sync(0xFFFFFFFFu, m));
    }
    if (lane == 0) p.s_cnt[e] = c;
  }
  // valid picks per token
  for (int t = tid; t < a.T; t += NW * 32) {
    int c = 0;
    for (int j = 0; j < a.k; ++j) c += p.s_id[t * a.k + j] >= 0;
    p.s_kv[t] = c;
  }
  __syncthreads();
  if (warp == 0) {
    // exclusive scans over experts (8 per lane) of the pair counts and unit counts
    constexpr int PER = kMaxE / 32;
    int c[PER], nu[PER], sc = 0, su = 0;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int e = lane * PER + i;
      c[i] = e < a.E ? p.s_cnt[e] : 0;
      nu[i] = (c[i] + TT - 1) / TT;
      sc += c[i];
      su += nu[i];
    }
    int ic = sc, iu = su;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int vc = __shfl_up_sync(0xFFFFFFFFu, ic, o), vu = __shfl_up_sync(0xFFFFFFFFu, iu, o);
      if (lane >= o) {
        ic += vc;
        iu += vu;
      }
    }
    int rc = ic - sc, ru = iu - su;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int e = lane * PER + i;
      if (e < a.E) {
        p.s_start[e] = rc;
        p.s_ustart[e] = ru;
      }
      rc += c[i];
      ru += nu[i];
    }
    if (lane == 31) p.s_ustart[a.E] = iu;
  }
  __syncthreads();
  for (int e = warp; e < a.E; e += NW) {
    const int cnt = p.s_cnt[e];
    if (cnt == 0) continue;
    int pos = p.s_start[e];
    for (int z0 = 0; z0 < P; z0 += 32) {
      const bool m = (z0 + lane < P) && p.s_id[z0 + lane] == e;
      const unsigned int bal = __ballot_sync(0xFFFFFFFFu, m);
      if (m) p.s_pairs[pos + __popc(bal & ((1u << lane) - 1u))] = z0 + lane;
      pos += __popc(bal);
    }
    const int nu = (cnt + TT - 1) / TT, us = p.s_ustart[e];
    const int slot = a.slots ? __ldg(a.slots + e) : e;
    for (int c = lane; c < nu; c += 32) {
      p.u_slot[us + c] = slot;
      p.u_first[us + c] = p.s_start[e] + c * TT;
      p.u_cnt[us + c] = min(TT, cnt - c * TT);
    }
  }
  __syncthreads();
  return p.s_ustart[a.E];
}

// One token (every pick its own unit): each warp builds the identical plan in shared memory
// by itself (the same values land at the same addresses from every warp), so no CTA barrier
// is needed.  With fuse_topk the warp first ranks the router logits.  Returns the units.
QG_DEVICE int warp_plan_one_token(const MoeArgs &a, const PlanSmem &p, int lane) {
  const int P = a.k;  // one token: P = k <= 32
  if (a.fuse_topk) {
    topk_token(a.logits, a.E, a.k, lane, p.tk_ids, p.tk_w);
    __syncwarp();
    if (blockIdx.x == 0 && threadIdx.x < 32 && lane < P) {
      a.ids_out[lane] = p.tk_ids[lane];
      a.wts_out[lane] = p.tk_w[lane];
    }
  }
  bool ok = false;
  int e = -1, slot = -1;
  if (lane < P) {
    e = a.fuse_topk ? p.tk_ids[lane] : __ldg(a.ids + lane);
    ok = e >= 0 && e < a.E;
    if (ok) {
      slot = a.slots ? __ldg(a.slots + e) : e;
      ok = slot >= 0 && slot < a.n_slots;
    }
    p.s_id[lane] = ok ? e : -1;
    if (!ok && blockIdx.x == 0 && threadIdx.x < 32) moe_status(QG_STATUS_BIT_ID);
  }
  const unsigned int mask = __ballot_sync(0xFFFFFFFFu, ok);
  if (ok) {
    const int rank = __popc(mask & ((1u << lane) - 1u));
    p.s_pairs[rank] = lane;
    p.u_slot[rank] = slot;
    p.u_first[rank] = rank;
    p.u_cnt[rank] = 1;
  }
  if (lane == 0) p.s_kv[0] = __popc(mask);
  __syncwarp();
  return __popc(mask);
}

// Row r of row block p of a unit, for blocks of RR rows: a gate/up block is RR/2 gate rows
// then the same RR/2 up rows ({gate p, up p} for RR = 2, {gate 2p, gate 2p+1, up 2p,
// up 2p+1} for RR = 4); a down block is rows RR p .. RR p + RR - 1.
template <bool DOWN, int RR>
QG_DEVICE int block_row(int p, int r) {
  return DOWN ? RR * p + r : (RR / 2) * p + (r % (RR / 2));
}

QG_DEVICE float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

// Token activation rows into shared memory in the 128-byte swizzled layout the decoders read
// (16-byte unit j of 32-float row R at 128 R + 16 (j ^ (R & 7))), as asynchronous 16-byte
// copies; the caller waits with cp_async_wait_all() and a CTA barrier.
QG_DEVICE void copy_x_row(uint8_t *xs, int slot, int xrow_bytes, const float *src, int K, int t0, int nthr) {
  const int K4 = K >> 2;
  const uint32_t base = smem_u32(xs) + static_cast<uint32_t>(slot * xrow_bytes);
  for (int i = t0; i < K4; i += nthr) {
    const int R = i >> 3, j = i & 7;
    cp_async16(base + static_cast<uint32_t>(R * 128 + 16 * (j ^ (R & 7))), src + 4 * i);
  }
}

// rows per block: 2 for one token (so that whole-row stages stay large copies with 16
// warps), 4 when several tokens share every decoded weight
template <int TT>
__host__ __device__ constexpr int moe_rows() {
  return TT == 1 ? 2 : 4;
}

template <int QT, int TT, int NW, bool DOWN>
__global__ void __launch_bounds__(NW * 32, 1) moe_expert_kernel(const __grid_constant__ CUtensorMap xmap,
                                                                const MoeArgs a) {
  using D = Dec<QT>;
  constexpr int RR = moe_rows<TT>(), HALF = RR / 2;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t *wbar = reinterpret_cast<uint64_t *>(smem);  // [NW][kMaxNS]
  uint64_t *xbar = wbar + NW * kMaxNS;                   // one token: activation rows by TMA
  const int P = a.T * a.k;
  const PlanSmem pl = plan_layout(smem + a.off_plan, P, a.T);
  uint8_t *xs = smem + a.off_x;
  uint8_t *ring = smem + a.off_ring;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NW * kMaxNS; ++i) mbar_init(&wbar[i], 1);
    mbar_init(xbar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();
  pdl_launch_dependents();
  int nunits;
  if constexpr (TT == 1)
    nunits = warp_plan_one_token(a, pl, lane);
  else
    nunits = build_plan<NW>(a, TT, pl);

  // pairs with a bad id: their act row is zero (gate/up); tokens without any valid pick keep
  // (or clear) their residual (down)
  if (blockIdx.x == 0) {
    if constexpr (!DOWN) {
      for (int i = threadIdx.x; i < P * a.F; i += NW * 32)
        if (pl.s_id[i / a.F] < 0) a.out[i] = 0.f;
    }
  }

  const long long RB = static_cast<long long>(nunits) * a.nblk;
  const int G = static_cast<int>(gridDim.x);
  const long long rbA = static_cast<long long>(blockIdx.x) * RB / G;
  const long long rbB = static_cast<long long>(blockIdx.x + 1) * RB / G;
  if (rbA >= rbB) return;  // nothing for this CTA (no copies were issued)
  const int uA = static_cast<int>(rbA / a.nblk);
  const int uB = static_cast<int>((rbB - 1) / a.nblk);

  // ---- this warp's row blocks rbA + warp + i * NW, each in nchunks K chunks
  const int nrb = static_cast<int>(rbB - rbA);
  const int my_rbs = warp < nrb ? (nrb - warp + NW - 1) / NW : 0;
  const int n_items = my_rbs * a.nchunks;
  const long long chunk_bytes = static_cast<long long>(a.KC / D::QK) * D::BB;
  uint8_t *wring = ring + warp * a.NS * a.stage_bytes;
  const uint32_t wring_s = smem_u32(wring);

  // Stage of one item: whole rows (seg_slot == 0; one copy of the block's down rows, or one
  // copy of its gate rows and one of its up rows) or one copy per row segment.
  const bool whole = a.seg_slot == 0;
  auto issue = [&](int item, int s) {
    const int i = item / a.nchunks, c = item - i * a.nchunks;
    const long long rb = rbA + warp + static_cast<long long>(i) * NW;
    const int u = static_cast<int>(rb / a.nblk), p = static_cast<int>(rb - static_cast<long long>(u) * a.nblk);
    uint8_t *st = wring + s * a.stage_bytes;
    const uintptr_t slot_off = static_cast<uintptr_t>(pl.u_slot[u]) * static_cast<uintptr_t>(a.stride);
    uintptr_t src = 0;
    uint32_t n = 0;
    uint8_t *dst = st;
    uintptr_t mend = 0;
    if (whole) {
      if (DOWN ? lane == 0 : lane < 2) {
        const int r0 = DOWN ? RR * p : HALF * p;
        const int nr = min(DOWN ? RR : HALF, a.R - r0);
        const bool second = !DOWN && lane == 1;
        if (nr > 0) {
          n = static_cast<uint32_t>(nr) * static_cast<uint32_t>(a.row_bytes);
          src = reinterpret_cast<uintptr_t>(second ? a.wb : a.wa) + slot_off +
                static_cast<uintptr_t>(r0) * static_cast<uintptr_t>(a.row_bytes);
          mend = second ? a.mend_b : a.mend_a;
          dst = st + (second ? a.gseg : 0);
        }
      }
    } else if (lane < RR) {
      const int row = block_row<DOWN, RR>(p, lane);
      if (row < a.R) {
        const int kel = min(a.K - c * a.KC, a.KC);
        n = static_cast<uint32_t>(kel / D::QK) * D::BB;
        const bool second = !DOWN && lane >= HALF;
        src = reinterpret_cast<uintptr_t>(second ? a.wb : a.wa) + slot_off +
              static_cast<uintptr_t>(row) * static_cast<uintptr_t>(a.row_bytes) +
              static_cast<uintptr_t>(c) * static_cast<uintptr_t>(chunk_bytes);
        mend = second ? a.mend_b : a.mend_a;
        dst = st + lane * a.seg_slot;
      }
    }
    warp_bulk_copies(dst, src, n, mend, &wbar[warp * kMaxNS + s], lane);
  };

  int issued = 0;
  for (; issued < a.NS - 1 && issued < n_items; ++issued) issue(issued, issued % a.NS);

  // activations of the tokens this CTA needs (the first weight stages are already in flight)
  bool x_ok = true;
  if constexpr (TT == 1) {
    // one token: tensor copies with the 128-byte swizzle, waited for by each warp
    const int R = a.K / 32;  // 32-float rows per activation row
    if (threadIdx.x == 0) {
      const int nslot = DOWN ? uB - uA + 1 : 1;
      mbar_arrive_expect_tx(xbar, static_cast<uint32_t>(nslot * R) * 128u);
      for (int sl = 0; sl < nslot; ++sl) {
        const int row = DOWN ? pl.s_pairs[pl.u_first[uA + sl]] : 0;
        for (int b = 0; b < R; b += a.box_rows)
          tma_load_2d(xs + static_cast<size_t>(sl) * a.xrow_bytes + b * 128, &xmap, 0, row * R + b, xbar);
      }
    }
    x_ok = mbar_wait(xbar, 0);
  } else {
    if constexpr (!DOWN) {
      for (int t = 0; t < a.T; ++t)
        copy_x_row(xs, t, a.xrow_bytes, a.xin + static_cast<size_t>(t) * a.K, a.K, threadIdx.x, NW * 32);
    } else {
      for (int u = uA; u <= uB; ++u)
        for (int t = 0; t < pl.u_cnt[u]; ++t) {
          const int z = pl.s_pairs[pl.u_first[u] + t];
          copy_x_row(xs, (u - uA) * TT + t, a.xrow_bytes, a.xin + static_cast<size_t>(z) * a.K, a.K, threadIdx.x,
                     NW * 32);
        }
    }
    cp_async_wait_all();
    __syncthreads();
  }

  if (n_items == 0) return;

  const uint32_t wo = static_cast<uint32_t>(D::woff(lane));
  uint32_t xo[D::NCH];
#pragma unroll
  for (int ch = 0; ch < D::NCH; ++ch) xo[ch] = x_lane_off<QT>(lane, ch);
  const int gpc = a.KC / D::SG;
  const uint32_t xs_s = smem_u32(xs);

  bool ok = x_ok;
  float acc1[RR];
  f2 acc2[RR][TT];
  int consumed = 0;
  for (int item = 0; item < n_items; ++item) {
    if (issued < n_items) {
      issue(issued, issued % a.NS);
      ++issued;
    }
    const int i = item / a.nchunks, c = item - i * a.nchunks;
    const long long rb = rbA + warp + static_cast<long long>(i) * NW;
    const int u = static_cast<int>(rb / a.nblk), p = static_cast<int>(rb - static_cast<long long>(u) * a.nblk);
    const int ucnt = pl.u_cnt[u];
    if (c == 0) {
#pragma unroll
      for (int r = 0; r < RR; ++r) {
        acc1[r] = 0.f;
#pragma unroll
        for (int t = 0; t < TT; ++t) acc2[r][t] = mk2(0.f, 0.f);
      }
    }
    const int cs = item % a.NS;
    if (ok && !mbar_wait(&wbar[warp * kMaxNS + cs], (item / a.NS) & 1)) ok = false;
    if (ok) {
      const int kel = min(a.K - c * a.KC, a.KC);
      const int gcount = (kel + D::SG - 1) / D::SG;
      const uint32_t st = wring_s + static_cast<uint32_t>(cs * a.stage_bytes);
      uint32_t wrow[RR];
      {
        // low 32 bits of the global addresses suffice: only their remainder mod 16 matters
        const uint32_t srow = static_cast<uint32_t>(pl.u_slot[u]) * static_cast<uint32_t>(a.stride);
        const uint32_t cb = static_cast<uint32_t>(c) * static_cast<uint32_t>(chunk_bytes);
        const uint32_t rbytes = static_cast<uint32_t>(a.row_bytes);
#pragma unroll
        for (int r = 0; r < RR; ++r) {
          const bool second = !DOWN && r >= HALF;
          const int row = block_row<DOWN, RR>(p, r);
          const uint32_t base = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(second ? a.wb : a.wa));
          if (whole) {
            // rows of one tensor are contiguous in the slot from the copy's first row
            const int r0 = DOWN ? RR * p : HALF * p;
            const uint32_t first = base + srow + static_cast<uint32_t>(r0) * rbytes;
            wrow[r] = st + (second ? static_cast<uint32_t>(a.gseg) : 0u) + (first & 15u) +
                      static_cast<uint32_t>(row - r0) * rbytes + wo;
          } else {
            const uint32_t addr = base + srow + static_cast<uint32_t>(row) * rbytes + cb;
            wrow[r] = st + static_cast<uint32_t>(r * a.seg_slot) + (addr & 15u) + wo;
          }
        }
      }
      // shared-memory offsets of the unit's token rows
      uint32_t toff[TT];
#pragma unroll
      for (int t = 0; t < TT; ++t) {
        const int tslot = t >= ucnt ? 0 : DOWN ? (u - uA) * TT + t : pl.s_pairs[pl.u_first[u] + t] / a.k;
        toff[t] = static_cast<uint32_t>(tslot * a.xrow_bytes);
      }
      const uint32_t xc0 = xs_s + static_cast<uint32_t>(c * gpc * (D::SG * 4));
      for (int g = 0; g < gcount; ++g) {
        if (g * D::SG + D::block_first(lane) >= kel) break;
        const uint32_t goff = static_cast<uint32_t>(g * D::GB);
        const uint32_t xg = xc0 + static_cast<uint32_t>(g * (D::SG * 4));
        if constexpr (TT == 1) {
          const uint32_t xt = xg + toff[0];
          float4 xc[D::NCH];
#pragma unroll
          for (int ch = 0; ch < D::NCH; ++ch) xc[ch] = lds_f4(xt + xo[ch]);
          const float aux = D::xaux(xc);
          typename D::U w[RR];
#pragma unroll
          for (int r = 0; r < RR; ++r) w[r] = D::load(wrow[r] + goff, lane);
#pragma unroll
          for (int r = 0; r < RR; ++r) acc1[r] += D::dot1(w[r], xc, aux);
        } else {
          typename D::U w[RR];
#pragma unroll
          for (int r = 0; r < RR; ++r) w[r] = D::load(wrow[r] + goff, lane);
#pragma unroll
          for (int ch = 0; ch < D::NCH; ++ch) {
            f2 w01[RR], w23[RR];
#pragma unroll
            for (int r = 0; r < RR; ++r) D::weights(w[r], ch, w01[r], w23[r]);
#pragma unroll
            for (int t = 0; t < TT; ++t) {
              if (t < ucnt) {
                const float4 xv = lds_f4(xg + toff[t] + xo[ch]);
                const f2 x01 = mk2(xv.x, xv.y), x23 = mk2(xv.z, xv.w);
#pragma unroll
                for (int r = 0; r < RR; ++r) {
                  acc2[r][t] = fma2(w01[r], x01, acc2[r][t]);
                  acc2[r][t] = fma2(w23[r], x23, acc2[r][t]);
                }
              }
            }
          }
        }
      }
    }
    __syncwarp();  // every lane is done with this slot before it is refilled
    ++consumed;

    if (c == a.nchunks - 1) {
      // the unit's RR x TT row sums, reduce-scattered over the warp
      constexpr int NV = RR * TT;
      constexpr int NH = NV == 64 ? 2 : 1;
      float v[NV];
      if constexpr (!DOWN) {
        // order (t, i, gate/up) so that a lane ends up with g and u of the same output
#pragma unroll
        for (int t = 0; t < TT; ++t)
#pragma unroll
          for (int i = 0; i < HALF; ++i)
#pragma unroll
            for (int gu = 0; gu < 2; ++gu) {
              const int r = HALF * gu + i;
              v[(t * HALF + i) * 2 + gu] = TT == 1 ? acc1[r] : acc2[r][t].x + acc2[r][t].y;
            }
      } else {
#pragma unroll
        for (int t = 0; t < TT; ++t)
#pragma unroll
          for (int r = 0; r < RR; ++r) v[t * RR + r] = TT == 1 ? acc1[r] : acc2[r][t].x + acc2[r][t].y;
      }
      reduce_scatter<NV>(v, lane);
      const int i0 = rs_index<NV>(lane);
      const bool own = rs_owner<NV>(lane);
      if constexpr (!DOWN) {
        float g, uu;
        if constexpr (NV == 64) {
          g = v[0];
          uu = v[1];
        } else {
          g = v[0];
          uu = __shfl_down_sync(0xFFFFFFFFu, v[0], 1 << rs_shift<NV>());
        }
        const int q = i0 >> 1;  // output index t * HALF + i
        const int t = q / HALF, i = HALF * p + (q - (q / HALF) * HALF);
        const bool writer = (NV == 64 || (own && (i0 & 1) == 0));
        if (writer && ok && t < ucnt && i < a.F) {
          const int z = pl.s_pairs[pl.u_first[u] + t];
          a.out[static_cast<size_t>(z) * a.F + i] = silu_mul(g, uu);
        }
      } else {
        const int h0 = RR * p;
#pragma unroll
        for (int hh = 0; hh < NH; ++hh) {
          const int idx = i0 + hh;
          const int t = idx / RR, r = idx - (idx / RR) * RR;
          if (own && ok && t < ucnt && h0 + r < a.H) {
            const int z = pl.s_pairs[pl.u_first[u] + t];
            a.dn[static_cast<size_t>(z) * a.H + h0 + r] = v[hh];
          }
        }
      }
    }
  }
  if (!ok) {
    if (lane == 0) moe_status(QG_STATUS_BIT_TIMEOUT);
    if (lane == 0)
      for (int it = consumed; it < issued; ++it) mbar_wait(&wbar[warp * kMaxNS + (it % a.NS)], (it / a.NS) & 1);
  }
}

// ------------------------------------------------------------------------------------------
// Host side
// ------------------------------------------------------------------------------------------

struct WsLayout {
  size_t logits, ticket, dn, tc, total;
};

inline size_t up256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

WsLayout ws_layout(int T, int k, int E, int H, int F = 0) {
  WsLayout w;
  w.logits = 0;
  w.ticket = up256(static_cast<size_t>(T) * E * 4);
  w.dn = w.ticket + up256(static_cast<size_t>((T + kRouterTB - 1) / kRouterTB) * 4);
  w.tc = w.dn + up256(static_cast<size_t>(T) * k * H * 4);
  w.total = w.tc;
  // grouped tensor-core path (more than 16 tokens): plan, grouped bf16 rows
  if (T > 16 && F > 0) w.total += up256(qg::moe_tc_workspace(T, k, E, H, F));
  return w;
}

bool valid_type(int type) { return type == QG_TYPE_Q8_0 || type == QG_TYPE_Q4_0 || type == QG_TYPE_Q4_K || type == QG_TYPE_Q6_K; }

qg_status check_common(int T, int k, int E, int H, int F) {
  if (T < 1 || k < 1 || k > kMaxK || E < k || E > kMaxE || H < 4 || H % 4 || F < 1) return QG_EINVAL_SHAPE;
  if (static_cast<long long>(T) * k > 1LL << 20 || static_cast<long long>(T) * H > INT32_MAX) return QG_EINVAL_SHAPE;
  return QG_OK;
}

qg_status route_impl(const float *xn, const float *wr, int T, int H, int E, int k, int32_t *ids, float *weights,
                     float *logits_out, void *ws, size_t ws_bytes, cudaStream_t s, int do_topk = 1) {
  if (!xn || !wr || !ids || !weights || !ws) return QG_EINVAL_PTR;
  if (T < 1 || k < 1 || k > kMaxK || E < k || E > kMaxE || H < 4 || H % 4) return QG_EINVAL_SHAPE;
  if (static_cast<long long>(T) * H > INT32_MAX || static_cast<long long>(T) * E > INT32_MAX) return QG_EINVAL_SHAPE;
  if (!qg::aligned16(xn) || !qg::aligned16(wr) || !qg::aligned16(ws)) return QG_EALIGN;
  const WsLayout L = ws_layout(T, 1, E, H);
  if (ws_bytes < L.dn) return QG_EWORKSPACE;
  uint8_t *w = static_cast<uint8_t *>(ws);
  float *logits = logits_out ? logits_out : reinterpret_cast<float *>(w + L.logits);
  const dim3 grid(E, (T + kRouterTB - 1) / kRouterTB);
  if (grid.y > 65535) return QG_EINVAL_SHAPE;
  if (qg::launch_pdl(moe_router_kernel, grid, dim3(kRouterWarps * 32), 0, s, xn, wr, T, H, E, k, logits, ids, weights,
                     reinterpret_cast<unsigned int *>(w + L.ticket), do_topk) != cudaSuccess)
    return QG_ECUDA;
  return cudaGetLastError() == cudaSuccess ? QG_OK : QG_ECUDA;
}

template <int QT, int TT, bool DOWN>
qg_status launch_expert(MoeArgs a, cudaStream_t s) {
  using D = Dec<QT>;
  constexpr int NW = (TT == 1) ? 16 : 8;
  constexpr int RR = moe_rows<TT>(), HALF = RR / 2;
  const qg::DeviceInfo &dev = qg::device_info();
  if (!dev.ok) return QG_ECUDA;
  const int P = a.T * a.k;
  const int ngroups = (a.K + D::SG - 1) / D::SG;
  a.xrow_bytes = ngroups * D::SG * 4;
  a.row_bytes = static_cast<long long>(a.K / D::QK) * D::BB;
  a.nblk = DOWN ? (a.H + RR - 1) / RR : (a.F + HALF - 1) / HALF;
  const int G = dev.sms;
  // token slots: all T tokens (gate/up); the units a CTA's row-block range can touch (down)
  int xslots = a.T;
  if (DOWN) {
    // units: at most one per pair, and at most ceil(pairs of the expert / TT) per expert
    const long long umax = std::min<long long>(P, static_cast<long long>(a.E) + (P + TT - 1) / TT);
    const long long L = (umax * a.nblk + G - 1) / G;
    const long long span = std::min<long long>(umax, (L - 1) / a.nblk + 2);
    xslots = static_cast<int>(span) * TT;
  }
  const uint32_t hdr = 1024;  // mbarriers: NW * kMaxNS + 1 of them
  a.off_plan = hdr;
  a.off_x = (a.off_plan + plan_bytes(P, a.T) + 1023) & ~1023u;
  const long long xbytes = static_cast<long long>(xslots) * a.xrow_bytes;
  const long long budget = dev.smem_optin - 4096;
  const long long ring_avail = budget - a.off_x - xbytes - 1024;
  if (ring_avail <= 0) return QG_EUNSUPPORTED;
  // Whole rows per stage when two such stages per warp fit: one copy of the block's down
  // rows, or one of its gate rows and one of its up rows.  Otherwise one copy per row
  // segment, segments of at least 2 KB (small bulk copies are capped by the copy engine's
  // per-copy rate).
  const long long half_bytes = ((static_cast<long long>(DOWN ? RR : HALF) * a.row_bytes + 15) & ~15LL) + 32;
  const long long whole_stage = DOWN ? half_bytes : 2 * half_bytes;
  if (2LL * NW * whole_stage <= ring_avail) {
    a.seg_slot = 0;
    a.gseg = DOWN ? 0 : static_cast<int>(half_bytes);
    a.stage_bytes = static_cast<int>(whole_stage);
    a.KC = ngroups * D::SG;
    a.nchunks = 1;
  } else {
    const long long target = std::max<long long>(2048, std::min<long long>(16384, ring_avail / (2LL * NW)));
    // the 2 KB floor first; without it when it leaves fewer than two slots per warp
    for (int floor_groups : {std::min(ngroups, (2048 + D::GB - 1) / D::GB), 1}) {
      int gmax = static_cast<int>(std::max<long long>(1, (target / RR - 32) / D::GB));
      gmax = std::max(std::min(gmax, ngroups), floor_groups);
      const int nch = (ngroups + gmax - 1) / gmax;
      const int gpc = (ngroups + nch - 1) / nch;
      a.seg_slot = static_cast<int>(((static_cast<long long>(gpc) * D::GB + 15) & ~15LL) + 32);
      a.gseg = 0;
      a.stage_bytes = RR * a.seg_slot;
      a.KC = gpc * D::SG;
      a.nchunks = nch;
      if (ring_avail / (static_cast<long long>(NW) * a.stage_bytes) >= 2) break;
    }
  }
  a.NS = static_cast<int>(std::min<long long>(kMaxNS, ring_avail / (static_cast<long long>(NW) * a.stage_bytes)));
  if (a.NS < 2) return QG_EUNSUPPORTED;
  a.off_ring = static_cast<uint32_t>(a.off_x + xbytes);
  const uint32_t smem = a.off_ring + static_cast<uint32_t>(NW * a.NS * a.stage_bytes) + 1024 + 64;
  // one token: tensor map over the activation rows ([rows * K / 32][32] f32, 128-byte swizzle)
  CUtensorMap xmap;
  memset(&xmap, 0, sizeof(xmap));
  if (TT == 1) {
    const int R = a.K / 32;  // largest box height <= 256 dividing the rows of one activation row
    a.box_rows = 1;
    for (int d = std::min(R, 256); d >= 1; --d)
      if (R % d == 0) {
        a.box_rows = d;
        break;
      }
    if (!qg::encode_x_map(&xmap, a.xin, DOWN ? P : a.T, a.K, a.box_rows)) return QG_ECUDA;
  }
  auto kern = moe_expert_kernel<QT, TT, NW, DOWN>;
  if (!qg::set_smem_attr(reinterpret_cast<const void *>(kern), smem)) return QG_ECUDA;
  if (qg::launch_pdl(kern, dim3(G), dim3(NW * 32), smem, s, xmap, a) != cudaSuccess) return QG_ECUDA;
  return cudaGetLastError() == cudaSuccess ? QG_OK : QG_ECUDA;
}

template <int QT, bool DOWN>
qg_status launch_expert_t(const MoeArgs &a, cudaStream_t s) {
  if (a.T == 1) return launch_expert<QT, 1, DOWN>(a, s);
  if (a.T <= 2) return launch_expert<QT, 2, DOWN>(a, s);
  if (a.T <= 4) return launch_expert<QT, 4, DOWN>(a, s);
  if (a.T <= 8) return launch_expert<QT, 8, DOWN>(a, s);
  return launch_expert<QT, 16, DOWN>(a, s);
}

template <bool DOWN>
qg_status launch_expert_type(int type, const MoeArgs &a, cudaStream_t s) {
  switch (type) {
    case QG_TYPE_Q8_0: return launch_expert_t<QG_TYPE_Q8_0, DOWN>(a, s);
    case QG_TYPE_Q4_0: return launch_expert_t<QG_TYPE_Q4_0, DOWN>(a, s);
    case QG_TYPE_Q4_K: return launch_expert_t<QG_TYPE_Q4_K, DOWN>(a, s);
    case QG_TYPE_Q6_K: return launch_expert_t<QG_TYPE_Q6_K, DOWN>(a, s);
    default: return QG_EUNSUPPORTED;
  }
}

// last 16-byte boundary of the extent of n_slots expert matrices of rows x row_bytes
uintptr_t tensor_mend(const void *base, long long stride, int n_slots, long long mat_bytes) {
  const uintptr_t end = reinterpret_cast<uintptr_t>(base) + static_cast<uintptr_t>(stride) * (n_slots - 1) +
                        static_cast<uintptr_t>(mat_bytes);
  return end & ~static_cast<uintptr_t>(15);
}

qg_status expert_checks(int type, int T, int k, int E, int H, int F, int n_slots, long long stride) {
  int qk = 0, bb = 0;
  if (!valid_type(type) || qg_block_shape(type, &qk, &bb) != QG_OK) return QG_EUNSUPPORTED;
  const qg_status c = check_common(T, k, E, H, F);
  if (c != QG_OK) return c;
  if (H % qk || F % qk || n_slots < 1 || stride < 0) return QG_EINVAL_SHAPE;
  // more than 16 tokens: the grouped tensor-core path (Q8_0, rows in whole 256-element boxes)
  if (T > 16 && (!qg::moe_tc_supported(type, H, F, E) || stride % 16)) return QG_EUNSUPPORTED;
  if (static_cast<long long>(stride) * n_slots > (1LL << 40)) return QG_EINVAL_SHAPE;
  return QG_OK;
}

qg_status swiglu_impl(int type, const void *w_gate, const void *w_up, int64_t stride, const int32_t *slots,
                      int n_slots, int E, const int32_t *ids, const float *xn, int T, int k, int H, int F,
                      float *act, void *ws, size_t ws_bytes, cudaStream_t s, const float *fused_logits = nullptr,
                      int32_t *ids_out = nullptr, float *wts_out = nullptr) {
  if (!w_gate || !w_up || !ids || !xn || !act) return QG_EINVAL_PTR;
  const qg_status c = expert_checks(type, T, k, E, H, F, n_slots, stride);
  if (c != QG_OK) return c;
  if (!qg::aligned16(xn) || !qg::aligned16(act)) return QG_EALIGN;
  int qk = 0, bb = 0;
  qg_block_shape(type, &qk, &bb);
  const long long mat = static_cast<long long>(F) * (H / qk) * bb;
  if (n_slots > 1 && stride < mat) return QG_EINVAL_SHAPE;
  if (T > 16) {
    if (!ws) return QG_EINVAL_PTR;
    if (!qg::aligned16(ws) || !qg::aligned16(w_gate) || !qg::aligned16(w_up)) return QG_EALIGN;
    const WsLayout L = ws_layout(T, k, E, H, F);
    if (ws_bytes < L.total) return QG_EWORKSPACE;
    return qg::moe_swiglu_tc(w_gate, w_up, stride, slots, n_slots, E, ids, xn, T, k, H, F, act,
                             static_cast<uint8_t *>(ws) + L.tc, s);
  }
  MoeArgs a{};
  a.wa = static_cast<const uint8_t *>(w_gate);
  a.wb = static_cast<const uint8_t *>(w_up);
  a.stride = stride;
  a.mend_a = tensor_mend(w_gate, stride, n_slots, mat);
  a.mend_b = tensor_mend(w_up, stride, n_slots, mat);
  a.slots = slots;
  a.n_slots = n_slots;
  a.E = E;
  a.ids = ids;
  a.xin = xn;
  a.out = act;
  a.T = T;
  a.k = k;
  a.H = H;
  a.F = F;
  a.K = H;
  a.R = F;
  if (fused_logits) {
    a.fuse_topk = 1;
    a.logits = fused_logits;
    a.ids_out = ids_out;
    a.wts_out = wts_out;
  }
  return launch_expert_type<false>(type, a, s);
}

qg_status combine_impl(int type, const void *w_down, int64_t stride, const int32_t *slots, int n_slots, int E,
                       const int32_t *ids, const float *weights, const float *act, int T, int k, int H, int F,
                       float *x_inout, int add_residual, void *ws, size_t ws_bytes, cudaStream_t s) {
  if (!w_down || !ids || !weights || !act || !x_inout || !ws) return QG_EINVAL_PTR;
  const qg_status c = expert_checks(type, T, k, E, H, F, n_slots, stride);
  if (c != QG_OK) return c;
  if (!qg::aligned16(act) || !qg::aligned16(ws)) return QG_EALIGN;
  const WsLayout L = ws_layout(T, k, E, H, F);
  if (ws_bytes < L.total) return QG_EWORKSPACE;
  int qk = 0, bb = 0;
  qg_block_shape(type, &qk, &bb);
  const long long mat = static_cast<long long>(H) * (F / qk) * bb;
  if (n_slots > 1 && stride < mat) return QG_EINVAL_SHAPE;
  uint8_t *w = static_cast<uint8_t *>(ws);
  if (T > 16) {
    if (!qg::aligned16(x_inout) || !qg::aligned16(w_down)) return QG_EALIGN;
    return qg::moe_combine_tc(w_down, stride, slots, n_slots, E, ids, weights, act, T, k, H, F, x_inout,
                              add_residual ? 1 : 0, reinterpret_cast<float *>(w + L.dn), w + L.tc, s);
  }
  MoeArgs a{};
  a.wa = static_cast<const uint8_t *>(w_down);
  a.wb = a.wa;
  a.stride = stride;
  a.mend_a = tensor_mend(w_down, stride, n_slots, mat);
  a.mend_b = a.mend_a;
  a.slots = slots;
  a.n_slots = n_slots;
  a.E = E;
  a.ids = ids;
  a.wts = weights;
  a.xin = act;
  a.out = x_inout;
  a.dn = reinterpret_cast<float *>(w + L.dn);
  a.T = T;
  a.k = k;
  a.H = H;
  a.F = F;
  a.K = F;
  a.R = H;
  a.add_residual = add_residual ? 1 : 0;
  const qg_status r = launch_expert_type<true>(type, a, s);
  if (r != QG_OK) return r;
  if (!qg::aligned16(x_inout) || H % 4) return QG_EALIGN;
  return qg::moe_launch_combine(a.dn, weights, ids, slots, n_slots, E, T, k, H, x_inout, add_residual ? 1 : 0, s);
}

}  // namespace

namespace qg {
unsigned int read_status_moe(bool clear) {
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_qg_status_moe, sizeof(v)) != cudaSuccess) return 0xFFFFFFFFu;
  if (clear) {
    const unsigned int z = 0;
    cudaMemcpyToSymbol(g_qg_status_moe, &z, sizeof(z));
  }
  return v;
}
}  // namespace qg

// ---- router without a caller workspace -----------------------------------------------------
// Fixed device scratch for moe_route_topk_noalloc: the router's logits and its per-tile
// tickets, laid out exactly as the workspace of moe_route_topk.  Sized for T * E <= 16384
// logits and 1024 token tiles (68 KB).
namespace {
constexpr int kNoAllocLogits = 16384;
constexpr int kNoAllocTiles = 1024;
constexpr size_t kNoAllocBytes = static_cast<size_t>(kNoAllocLogits) * 4 + static_cast<size_t>(kNoAllocTiles) * 4;
__device__ __align__(256) unsigned char g_route_scratch[kNoAllocBytes];

std::mutex g_scratch_mu;
void *g_scratch_ptr[64];  // per device, filled on the first call with that device current

void *route_scratch() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}
}  // namespace

extern "C" {

qg_status moe_route_topk_noalloc(const float *xn, const float *wr, int T, int H, int E, int k, int32_t *ids,
                                 float *weights, float *logits_out, qg_stream_t stream) {
  if (T < 1 || E < 1 || static_cast<long long>(T) * E > kNoAllocLogits ||
      (T + kRouterTB - 1) / kRouterTB > kNoAllocTiles)
    return QG_EWORKSPACE;
  void *ws = route_scratch();
  if (!ws) return QG_ECUDA;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const WsLayout L = ws_layout(T, 1, E, H);
  // the tickets must read zero when the router starts: clear them for this shape's layout
  if (cudaMemsetAsync(static_cast<uint8_t *>(ws) + L.ticket, 0,
                      static_cast<size_t>((T + kRouterTB - 1) / kRouterTB) * 4, s) != cudaSuccess)
    return QG_ECUDA;
  return route_impl(xn, wr, T, H, E, k, ids, weights, logits_out, ws, kNoAllocBytes, s);
}

size_t moe_workspace_size(int T, int k, int E, int H, int F) {
  if (check_common(T, k, E, H, F) != QG_OK) return 0;
  return ws_layout(T, k, E, H, F).total;
}

qg_status moe_route_topk(const float *xn, const float *wr, int T, int H, int E, int k, int32_t *ids, float *weights,
                         float *logits_out, void *ws, size_t ws_bytes, qg_stream_t stream) {
  return route_impl(xn, wr, T, H, E, k, ids, weights, logits_out, ws, ws_bytes,
                    reinterpret_cast<cudaStream_t>(stream));
}

qg_status moe_expert_swiglu(int type, const void *w_gate, const void *w_up, int64_t expert_stride,
                            const int32_t *slots, int n_slots, int E, const int32_t *ids, const float *xn, int T,
                            int k, int H, int F, float *act, void *ws, size_t ws_bytes, qg_stream_t stream) {
  return swiglu_impl(type, w_gate, w_up, expert_stride, slots, n_slots, E, ids, xn, T, k, H, F, act, ws, ws_bytes,
                     reinterpret_cast<cudaStream_t>(stream));
}

qg_status moe_combine(int type, const void *w_down, int64_t expert_stride, const int32_t *slots, int n_slots, int E,
                      const int32_t *ids, const float *weights, const float *act, int T, int k, int H, int F,
                      float *x_inout, int add_residual, void *ws, size_t ws_bytes, qg_stream_t stream) {
  return combine_impl(type, w_down, expert_stride, slots, n_slots, E, ids, weights, act, T, k, H, F, x_inout,
                      add_residual, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

qg_status moe_layer(int type, const float *xn, const float *wr, const void *w_gate, const void *w_up,
                    const void *w_down, int64_t expert_stride, const int32_t *slots, int n_slots, int T, int H, int F,
                    int E, int k, int32_t *ids, float *weights, float *act, float *x_inout, void *ws,
                    size_t ws_bytes, qg_stream_t stream) {
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (!xn || !wr || !w_gate || !w_up || !w_down || !ids || !weights || !act || !x_inout || !ws) return QG_EINVAL_PTR;
  const qg_status c = expert_checks(type, T, k, E, H, F, n_slots, expert_stride);
  if (c != QG_OK) return c;
  if (ws_bytes < ws_layout(T, k, E, H, F).total) return QG_EWORKSPACE;
  qg_status r;
  if (T > 16) {
    // prefill-sized batch: router with top-k, then the grouped tensor-core expert steps
    r = route_impl(xn, wr, T, H, E, k, ids, weights, nullptr, ws, ws_bytes, s, 1);
    if (r != QG_OK) return r;
    r = swiglu_impl(type, w_gate, w_up, expert_stride, slots, n_slots, E, ids, xn, T, k, H, F, act, ws, ws_bytes, s);
    if (r != QG_OK) return r;
    return combine_impl(type, w_down, expert_stride, slots, n_slots, E, ids, weights, act, T, k, H, F, x_inout, 1,
                        ws, ws_bytes, s);
  }
  // router logits into the workspace; the gate/up kernel ranks them (every CTA needs the
  // picks for its plan anyway) and stores ids and weights for the combine
  r = route_impl(xn, wr, T, H, E, k, ids, weights, nullptr, ws, ws_bytes, s, 0);
  if (r != QG_OK) return r;
  const float *logits = reinterpret_cast<const float *>(static_cast<uint8_t *>(ws) + ws_layout(T, k, E, H).logits);
  r = swiglu_impl(type, w_gate, w_up, expert_stride, slots, n_slots, E, ids, xn, T, k, H, F, act, ws, ws_bytes, s,
                  logits, ids, weights);
  if (r != QG_OK) return r;
  return combine_impl(type, w_down, expert_stride, slots, n_slots, E, ids, weights, act, T, k, H, F, x_inout, 1, ws,
                      ws_bytes, s);
}

}  // extern "C"
