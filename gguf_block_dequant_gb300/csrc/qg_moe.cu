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

// The same logits for many token tiles: a CTA stages one tile of kRouterTB tokens in shared
// memory once and runs `epc` experts over it (the kernel above reads the tile from L2 again
// for every expert: 128 experts x 512 tokens x 8 KB = 537 MB for a 512-token prefill).  Its 16
// warps are four quads; quad q takes experts eA + q, eA + q + 4, ..., and inside a quad warp w
// does what warp w of the kernel above does for one expert, so every logit is summed in the
// same order (lane partials over h = 32 w + lane + 128 j, the warp sum, then the four warp
// partials in order) and equals that kernel's bit for bit.
constexpr int kRouterTiledWarps = 16;

__global__ void __launch_bounds__(kRouterTiledWarps * 32, 1)
    moe_router_tiled_kernel(const float *__restrict__ xn, const float *__restrict__ wr, int T, int H, int E, int k,
                            int epc, float *logits, int32_t *ids, float *weights, unsigned int *ticket, int do_topk) {
  extern __shared__ __align__(16) float rt_smem[];
  float4 *xs = reinterpret_cast<float4 *>(rt_smem);    // [kRouterTB][H / 4]
  float *part = rt_smem + static_cast<size_t>(kRouterTB) * H;  // [4 quads][kRouterWarps][kRouterTB]
  __shared__ unsigned int s_last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quad = warp >> 2, wq = warp & 3;
  pdl_wait();
  pdl_launch_dependents();
  const int t0 = blockIdx.y * kRouterTB;
  const int nt = min(kRouterTB, T - t0);
  const int H4 = H >> 2;
  const float4 *xg = reinterpret_cast<const float4 *>(xn + static_cast<size_t>(t0) * H);
  for (int i = threadIdx.x; i < nt * H4; i += blockDim.x) xs[i] = __ldg(xg + i);
  __syncthreads();
  const int eA = blockIdx.x * epc, eB = min(E, eA + epc);
  float *qpart = part + quad * (kRouterWarps * kRouterTB);
  for (int e = eA + quad; e < eB; e += 4) {
    float acc[kRouterTB];
#pragma unroll
    for (int t = 0; t < kRouterTB; ++t) acc[t] = 0.f;
    const float4 *w4 = reinterpret_cast<const float4 *>(wr + static_cast<size_t>(e) * H);
#pragma unroll 4
    for (int h = wq * 32 + lane; h < H4; h += kRouterWarps * 32) {
      const float4 w = __ldg(w4 + h);
#pragma unroll
      for (int t = 0; t < kRouterTB; ++t) {
        if (t < nt) {
          const float4 x = xs[t * H4 + h];
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
      if (lane == 0) qpart[wq * kRouterTB + t] = s;
    }
    named_bar_sync(1 + quad, kRouterWarps * 32);
    if (wq == 0 && lane < nt) {
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < kRouterWarps; ++w) s += qpart[w * kRouterTB + lane];
      logits[static_cast<size_t>(t0 + lane) * E + e] = s;
    }
    named_bar_sync(1 + quad, kRouterWarps * 32);  // qpart is free for the quad's next expert
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
  for (int t = t0 + warp; t < t0 + nt; t += kRouterTiledWarps)
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
  int plan_only;  // host side: check that the shapes fit the kernel's shared-memory plan, launch nothing
  int act_kind;   // gate/up: 0 SiLU(g) u (siluMulMoe), 1 GELU-tanh(g) u (geglu)
};

// Pairs grouped by expert.  s_id[z]: expert of pair z, or -1 when its id or slot is out of
// range; s_pairs: pair indices ordered by expert, then by pair index; unit u covers
// s_pairs[u_first[u] .. + u_cnt[u]) of one expert (at most TT pairs), slot u_slot[u].
struct PlanSmem {
  int *s_id, *s_pairs, *u_slot, *u_first, *u_cnt, *s_cnt, *s_start, *s_ustart, *s_kv;
  int32_t *tk_ids;  // fused top-k results [T][k]
  float *tk_w;
  float *tk_lg;     // the router logits being ranked [T][E] (fused top-k, several tokens; lives in
                    // the activation buffer, which is filled only after the plan)
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
  p.tk_lg = nullptr;  // set by the kernel: the activation buffer, still unused while the plan is built
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
    // the k greedy picks of each token (ties to the lowest expert id) are the experts of rank
    // < k, rank(e) = #{e' : l[e'] > l[e] or l[e'] == l[e] and e' < e}: one thread per (token,
    // expert) instead of a warp-serial selection; the weights follow in pick order as in
    // topk_token, so picks and weights equal the standalone router's
    const int TE = a.T * a.E;
    for (int i = tid; i < TE; i += NW * 32) p.tk_lg[i] = __ldcg(a.logits + i);
    // a rank that no expert takes (NaN logits tie with everything) leaves pick -1, which the
    // id check below reports
    for (int z = tid; z < P; z += NW * 32) p.tk_ids[z] = -1;
    __syncthreads();
    for (int i = tid; i < TE; i += NW * 32) {
      const int t = i / a.E, e = i - t * a.E;
      const float *lt = p.tk_lg + t * a.E;
      const float le = lt[e];
      int rank = 0;
      for (int f = 0; f < a.E; ++f) {
        const float lf = lt[f];
        rank += (lf > le || (lf == le && f < e)) ? 1 : 0;
      }
      if (rank < a.k) p.tk_ids[t * a.k + rank] = e;
    }
    __syncthreads();
    for (int t = tid; t < a.T; t += NW * 32) {
      const float *lt = p.tk_lg + t * a.E;
      const int e0 = p.tk_ids[t * a.k];
      const float lmax = e0 >= 0 ? lt[e0] : 0.f;
      float den = 0.f;
      for (int j = 0; j < a.k; ++j) {
        const int ej = p.tk_ids[t * a.k + j];
        const float ex = ej >= 0 ? expf(lt[ej] - lmax) : 0.f;
        den += ex;
        p.tk_w[t * a.k + j] = ex;
      }
      for (int j = 0; j < a.k; ++j) p.tk_w[t * a.k + j] = p.tk_w[t * a.k + j] / den;
    }
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
  PlanSmem pl = plan_layout(smem + a.off_plan, P, a.T);
  uint8_t *xs = smem + a.off_x;
  pl.tk_lg = reinterpret_cast<float *>(xs);
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
      for (int q = 0; q < P; ++q)
        if (pl.s_id[q] < 0)
          for (int i = threadIdx.x; i < a.F; i += NW * 32) a.out[static_cast<size_t>(q) * a.F + i] = 0.f;
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
  // Item cursor: chunk c of row block p of unit u, advanced without divisions (a warp's row
  // blocks are NW apart, so u and p move by whole strides).
  struct ItemCur {
    int c, u, p;
  };
  auto cur_first = [&]() {
    const long long rb = rbA + warp;
    const int u0 = static_cast<int>(rb / a.nblk);
    return ItemCur{0, u0, static_cast<int>(rb - static_cast<long long>(u0) * a.nblk)};
  };
  auto cur_next = [&](ItemCur &q) {
    if (++q.c == a.nchunks) {
      q.c = 0;
      q.p += NW;
      while (q.p >= a.nblk) {
        q.p -= a.nblk;
        ++q.u;
      }
    }
  };
  auto issue = [&](const ItemCur &q, int s) {
    const int c = q.c, u = q.u, p = q.p;
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

  int issued = 0, is = 0;
  ItemCur ic = cur_first();
  for (; issued < a.NS - 1 && issued < n_items; ++issued) {
    issue(ic, is);
    cur_next(ic);
    is = (is + 1 == a.NS) ? 0 : is + 1;
  }

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
  int consumed = 0, cs = 0, cph = 0;
  ItemCur cc = cur_first();
  int toff_u = -1;  // unit whose token offsets toff[] hold
  uint32_t toff[TT];
  for (int item = 0; item < n_items; ++item, cur_next(cc)) {
    if (issued < n_items) {
      issue(ic, is);
      cur_next(ic);
      is = (is + 1 == a.NS) ? 0 : is + 1;
      ++issued;
    }
    const int c = cc.c, u = cc.u, p = cc.p;
    const int ucnt = pl.u_cnt[u];
    if (c == 0) {
#pragma unroll
      for (int r = 0; r < RR; ++r) {
        acc1[r] = 0.f;
#pragma unroll
        for (int t = 0; t < TT; ++t) acc2[r][t] = mk2(0.f, 0.f);
      }
    }
    if (ok && !mbar_wait(&wbar[warp * kMaxNS + cs], static_cast<uint32_t>(cph))) ok = false;
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
      // shared-memory offsets of the unit's token rows (recomputed when the unit changes)
      if (u != toff_u) {
        toff_u = u;
#pragma unroll
        for (int t = 0; t < TT; ++t) {
          const int tslot = t >= ucnt ? 0 : DOWN ? (u - uA) * TT + t : pl.s_pairs[pl.u_first[u] + t] / a.k;
          toff[t] = static_cast<uint32_t>(tslot * a.xrow_bytes);
        }
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
    if (++cs == a.NS) {
      cs = 0;
      cph ^= 1;
    }

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
          a.out[static_cast<size_t>(z) * a.F + i] = act_mul(a.act_kind, g, uu);
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
// One token, the whole layer in one cooperative launch
// ------------------------------------------------------------------------------------------
// With a single token the layer is four short dependent steps (router, gate/up, down,
// combine) around ~40 MB of weights, and separate launches spend most of the time on their
// own start-up and drain.  This kernel runs them as phases of one persistent grid (one CTA
// per SM, all co-resident: cooperative launch):
//   phase 0  router logits, one expert row per CTA (its warps split the row), each published
//            as a word tagged with the call; every CTA polls the E words until all carry the
//            tag (no grid barrier);
//   phase 1  every CTA ranks the logits itself (the same picks everywhere), then streams its
//            share of the {gate i, up i} row pairs of the picked experts and writes
//            act = silu(g) * u; then it requests the down rows it will need next;
//   barrier
//   phase 2  every CTA owns a range of hidden rows h: it dots the down rows h of each picked
//            expert with that expert's act row and adds sum_j w_j dn_j[h] to x[h] in pick
//            order (the combine needs no separate pass).
// The grid barrier is an arrival counter in the caller's workspace that only grows (no reset
// step between calls).  The picks are ranked by the whole CTA at once (a serial warp-level
// selection costs microseconds of shuffle latency).  Every wait is bounded and reports an
// expired wait in the status word.

struct OneArgs {
  const float *xn, *wr;
  const uint8_t *wg, *wu, *wd;
  long long stride;  // bytes between expert slots
  uintptr_t mend_g, mend_u, mend_d;
  const int32_t *slots;
  int n_slots, E, k, H, F;
  int32_t *ids_out;
  float *wts_out;
  float *act;        // [k][F]
  float *x;          // [H], updated in place
  unsigned long long *bar;   // arrivals of the grid barrier (workspace header)
  unsigned long long *gen;   // calls of this kernel on the workspace (header; tags the logits)
  unsigned long long *xlog;  // [E] logits, each tagged with its call (header)
  long long rbh, rbf;  // bytes of an H-long row (gate, up) and of an F-long row (down)
  int NS, stage_bytes, gseg, dseg;
  int hmax;          // most hidden rows of one CTA
  int early_weights;
  uint32_t off_x, off_part, off_ring;
};

QG_DEVICE unsigned long long ld_relaxed_u64(const unsigned long long *p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
QG_DEVICE void st_relaxed_u64(unsigned long long *p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Grid-wide barrier for a cooperative grid: `bar` counts arrivals and only ever grows.  Every
// launch adds exactly G per barrier and launches in a stream do not overlap this part (it comes
// after the wait on the predecessor), so the arrivals of one barrier all return values in
// [n G, n G + G) for the same n, and the barrier is passed once the count reaches (n + 1) G.
// The arrival follows a fence (this CTA's writes before it); the polls are acquire loads, so
// what the other CTAs wrote before arriving is visible after the barrier.  Returns false when
// the wait expired.
QG_DEVICE bool grid_barrier(unsigned long long *bar, unsigned int nctas, unsigned int *s_flag) {
  __syncthreads();
  if (threadIdx.x == 0) {
    // the arrival is a release: this CTA's writes (ordered before it by the CTA barrier) are
    // visible to every CTA whose acquire poll sees the count
    unsigned long long v;
    asm volatile("atom.release.gpu.global.add.u64 %0, [%1], 1;" : "=l"(v) : "l"(bar) : "memory");
    const unsigned long long target = (v / nctas + 1) * nctas;
    unsigned int ok = 1u;
    const uint64_t t0 = global_ns();
    for (unsigned int spin = 1;; ++spin) {
      unsigned long long cur;
      asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(cur) : "l"(bar) : "memory");
      if (cur >= target) break;
      if ((spin & 31u) == 0u && global_ns() - t0 > QG_WAIT_NS) {
        ok = 0u;
        break;
      }
    }
    *s_flag = ok;
  }
  __syncthreads();
  return *s_flag != 0u;
}

template <int QT, int NW>
__global__ void __launch_bounds__(NW * 32, 1) moe_one_token_kernel(const OneArgs a) {
  using D = Dec<QT>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t *wbar = reinterpret_cast<uint64_t *>(smem);                 // [NW][kMaxNS]
  int32_t *s_ids = reinterpret_cast<int32_t *>(smem + 512);            // [kMaxK] picks
  float *s_w = reinterpret_cast<float *>(smem + 640);                  // [kMaxK] weights
  int32_t *s_slot = reinterpret_cast<int32_t *>(smem + 768);           // [kMaxK] slot, -1: bad id
  int32_t *s_vz = reinterpret_cast<int32_t *>(smem + 896);             // [kMaxK] valid picks in order
  float *red = reinterpret_cast<float *>(smem + 1024);                 // [NW] router partials
  unsigned int *s_misc = reinterpret_cast<unsigned int *>(smem + 1024 + 4 * NW);  // flag, valid count, tag
  uintptr_t *s_base = reinterpret_cast<uintptr_t *>(smem + 1152);      // [kMaxK][3] gate, up, down of valid picks
  uint8_t *xs = smem + a.off_x;
  float *part = reinterpret_cast<float *>(smem + a.off_part);          // [hmax][kMaxK]
  uint8_t *ring = smem + a.off_ring;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = static_cast<int>(gridDim.x);
  const int H = a.H, F = a.F, k = a.k;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NW * kMaxNS; ++i) mbar_init(&wbar[i], 1);
    fence_mbar_init();
  }
  // a rank that no expert takes (NaN logits tie with everything) leaves pick -1, an invalid id
  if (threadIdx.x < kMaxK) s_ids[threadIdx.x] = -1;
  __syncthreads();

  // ---- phase 0: router logits of experts blockIdx.x, + G, ..., summed by kRouterWarps warps
  // in exactly the order of moe_router_kernel, so that the logits (and picks and weights) are
  // the ones the standalone router gives.  Each logit is published as one 64-bit word holding
  // this call's tag and the value, so every CTA can gather all of them without a grid barrier:
  // a word carrying the tag is this call's logit.  The tag is the number of earlier calls on
  // the workspace plus one (CTA 0 advances the count once every CTA is past the grid barrier,
  // so every CTA of a call reads the same count).
  pdl_wait();
  if (threadIdx.x == 0) s_misc[2] = static_cast<unsigned int>(ld_relaxed_u64(a.gen)) + 1u;
  // hidden rows of phase 2 for this CTA; their residual values are read now (only this CTA
  // writes them), so that the combine at the end does not wait for them
  const int hA = static_cast<int>(static_cast<long long>(blockIdx.x) * H / G);
  const int hB = static_cast<int>(static_cast<long long>(blockIdx.x + 1) * H / G);
  const float x_pre = threadIdx.x < hB - hA ? a.x[hA + threadIdx.x] : 0.f;
  __syncthreads();
  const unsigned int tag = s_misc[2];
  bool ok = true;
  const int H4 = H >> 2;
  for (int e = blockIdx.x; e < a.E; e += G) {
    if (warp < kRouterWarps) {
      const float4 *w4 = reinterpret_cast<const float4 *>(a.wr + static_cast<size_t>(e) * H);
      const float4 *x4 = reinterpret_cast<const float4 *>(a.xn);
      float acc = 0.f;
#pragma unroll 4
      for (int h = warp * 32 + lane; h < H4; h += kRouterWarps * 32) {
        const float4 w = __ldg(w4 + h);
        const float4 xv = __ldg(x4 + h);
        acc = fmaf(w.x, xv.x, acc);
        acc = fmaf(w.y, xv.y, acc);
        acc = fmaf(w.z, xv.z, acc);
        acc = fmaf(w.w, xv.w, acc);
      }
      const float sw = warp_sum(acc);
      if (lane == 0) red[warp] = sw;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      float t = 0.f;
#pragma unroll
      for (int w = 0; w < kRouterWarps; ++w) t += red[w];
      st_relaxed_u64(a.xlog + e, (static_cast<unsigned long long>(tag) << 32) | __float_as_uint(t));
    }
    __syncthreads();
  }
  // ---- phase 1: picks, then the gate/up row pairs.  The k greedy picks of the logits (ties
  // to the lowest expert id) are the experts of rank < k, rank(e) = #{e' : l[e'] > l[e] or
  // l[e'] == l[e] and e' < e}; the weights follow in pick order as in topk_token.
  // the token's activations into shared memory (128-byte swizzled rows) while the logits
  // arrive (issued before the router instead, these copies measured 1.5 us slower per layer)
  copy_x_row(xs, 0, 0, a.xn, H, threadIdx.x, NW * 32);
  float *s_l = part;  // the logits (part is free until phase 2)
  int late = 0;
  for (int e = threadIdx.x; e < a.E; e += NW * 32) {
    // bounded wait for this call's tag on expert e's word
    unsigned long long v = ld_relaxed_u64(a.xlog + e);
    if (static_cast<unsigned int>(v >> 32) != tag) {
      const uint64_t t0 = global_ns();
      do {
        v = ld_relaxed_u64(a.xlog + e);
      } while (static_cast<unsigned int>(v >> 32) != tag && global_ns() - t0 < QG_WAIT_NS);
      if (static_cast<unsigned int>(v >> 32) != tag) late = 1;
    }
    s_l[e] = __uint_as_float(static_cast<unsigned int>(v));
  }
  if (__syncthreads_or(late)) ok = false;
  {
    // rank(e) in four partial counts over quarters of the experts, so that every warp of the
    // CTA takes a share (the ring is idle until the gate/up stages: it holds the counts)
    int *s_rk = reinterpret_cast<int *>(ring);  // [4][E]
    const int QF = (a.E + 3) >> 2;
    for (int idx = threadIdx.x; idx < 4 * a.E; idx += NW * 32) {
      const int q = idx / a.E, e = idx - q * a.E;
      const float le = s_l[e];
      const int f1 = min(a.E, (q + 1) * QF);
      int r = 0;
      for (int f = q * QF; f < f1; ++f) {
        const float lf = s_l[f];
        r += (lf > le || (lf == le && f < e)) ? 1 : 0;
      }
      s_rk[idx] = r;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < a.E; e += NW * 32) {
      const int rank = s_rk[e] + s_rk[a.E + e] + s_rk[2 * a.E + e] + s_rk[3 * a.E + e];
      if (rank < k) s_ids[rank] = e;
    }
  }
  __syncthreads();
  if (warp == 0) {
    // softmax over the picks: one exponential per lane, the denominator summed in pick order
    // (the router's order, so the weights are the standalone router's bit for bit)
    const int e0 = s_ids[0], el = lane < k ? s_ids[lane] : -1;
    const float lmax = e0 >= 0 ? s_l[e0] : 0.f;
    const float ex = el >= 0 ? expf(s_l[el] - lmax) : 0.f;
    float den = 0.f;
    for (int j = 0; j < k; ++j) den += __shfl_sync(0xFFFFFFFFu, ex, j);
    const float wt = ex / den;
    if (lane < k) s_w[lane] = wt;
    bool valid = false;
    int slot = -1;
    if (lane < k) {
      const int e = s_ids[lane];
      valid = e >= 0 && e < a.E;
      if (valid) {
        slot = a.slots ? __ldg(a.slots + e) : e;
        valid = slot >= 0 && slot < a.n_slots;
      }
      s_slot[lane] = valid ? slot : -1;
      if (blockIdx.x == 0) {
        a.ids_out[lane] = s_ids[lane];
        a.wts_out[lane] = wt;
        if (!valid) moe_status(QG_STATUS_BIT_ID);
      }
    }
    const unsigned int m = __ballot_sync(0xFFFFFFFFu, valid);
    if (valid) s_vz[__popc(m & ((1u << lane) - 1u))] = lane;
    if (lane == 0) s_misc[1] = __popc(m);
    __syncwarp();
    // the valid picks' expert bases (gate, up and down rows of slot s_slot)
    if (lane < static_cast<int>(__popc(m))) {
      const uintptr_t off = static_cast<uintptr_t>(s_slot[s_vz[lane]]) * static_cast<uintptr_t>(a.stride);
      s_base[3 * lane + 0] = reinterpret_cast<uintptr_t>(a.wg) + off;
      s_base[3 * lane + 1] = reinterpret_cast<uintptr_t>(a.wu) + off;
      s_base[3 * lane + 2] = reinterpret_cast<uintptr_t>(a.wd) + off;
    }
  }
  __syncthreads();
  const int kv = static_cast<int>(s_misc[1]);
  // a pick with a bad id has a zero act row
  if (blockIdx.x == 0)
    for (int j = 0; j < k; ++j)
      if (s_slot[j] < 0)
        for (int i = threadIdx.x; i < F; i += NW * 32) a.act[static_cast<size_t>(j) * F + i] = 0.f;

  // the down rows of this CTA's hidden rows are requested right after each warp's gate/up
  // items, into the ring slots the gate/up phase leaves free

  const uint32_t wo = static_cast<uint32_t>(D::woff(lane));
  uint32_t xo[D::NCH];
#pragma unroll
  for (int ch = 0; ch < D::NCH; ++ch) xo[ch] = x_lane_off<QT>(lane, ch);
  uint8_t *wring = ring + warp * a.NS * a.stage_bytes;
  const uint32_t wring_s = smem_u32(wring);
  const uint32_t xs_s = smem_u32(xs);
  const int bfirst = D::block_first(lane);

  // RR rows of one stage against activation row xrow: the dense one-token decode, row r's
  // raw blocks at shared address row[r] (any 2-byte alignment), K elements
  auto dot_rows = [&](auto &acc, const uint32_t *row, int K, uint32_t xrow) {
    constexpr int RR = static_cast<int>(sizeof(acc) / sizeof(acc[0]));
    RowPrep<QT> rp[RR];
#pragma unroll
    for (int r = 0; r < RR; ++r) {
      acc[r] = 0.f;
      rp[r].init(row[r] + wo, lane);
    }
    auto group = [&](int g) {
      const uint32_t goff = static_cast<uint32_t>(g * D::GB);
      const uint32_t xg = xrow + static_cast<uint32_t>(g * (D::SG * 4));
      float4 xc[D::NCH];
#pragma unroll
      for (int ch = 0; ch < D::NCH; ++ch) xc[ch] = lds_f4(xg + xo[ch]);
      const float aux = D::xaux(xc);
      typename D::U w[RR];
#pragma unroll
      for (int r = 0; r < RR; ++r) w[r] = rp[r].load(goff, lane);
#pragma unroll
      for (int r = 0; r < RR; ++r) acc[r] += D::dot1(w[r], xc, aux);
    };
    const int gfull = K / D::SG;
    for (int g = 0; g < gfull; ++g) group(g);
    if (gfull * D::SG < K && gfull * D::SG + bfirst < K) group(gfull);  // the partial last group
  };

  // Streaming through the warp's ring.  Ring positions continue across the phases, so every
  // slot's mbarrier phase stays in step: `issued` copies were requested, `waited` consumed.
  // After an expired wait the warp issues nothing more and waits for what it has in flight
  // before it exits.
  int issued = 0, waited = 0;
  int islot = 0, wslot = 0, wph = 0;  // ring slot of the next issue / wait, and the wait's phase bit
  auto next_slot = [&]() {
    ++issued;
    if (++islot == a.NS) islot = 0;
  };
  auto wait_slot = [&]() {
    if (!mbar_wait(&wbar[warp * kMaxNS + wslot], static_cast<uint32_t>(wph))) return false;
    return true;
  };
  auto release_slot = [&]() {
    __syncwarp();  // every lane is done with the slot before it is refilled
    ++waited;
    if (++wslot == a.NS) {
      wslot = 0;
      wph ^= 1;
    }
  };

  // gate/up: row pairs (pick jv, row i), contiguous balanced ranges per CTA, the warp's pairs
  // NW apart; a stage holds the gate row (lane 0's copy) and the up row (lane 1's copy, at
  // gseg).  Cursors advance by NW rows, with no division in the loop.
  {
    const long long nb = static_cast<long long>(kv) * F;
    const int bA = static_cast<int>(static_cast<long long>(blockIdx.x) * nb / G);
    const int bB = static_cast<int>(static_cast<long long>(blockIdx.x + 1) * nb / G);
    const int nrb = bB - bA;
    const int n_items = warp < nrb ? (nrb - warp + NW - 1) / NW : 0;
    int jvi = (bA + warp) / F, ii = (bA + warp) - jvi * F;  // issue cursor
    int jvc = jvi, ic = ii;                                   // consume cursor
    auto adv = [&](int &jv, int &i) {
      i += NW;
      while (i >= F) {
        i -= F;
        ++jv;
      }
    };
    auto row_src = [&](int jv, int i, int r) {
      return s_base[3 * jv + r] + static_cast<uintptr_t>(i) * static_cast<uintptr_t>(a.rbh);
    };
    auto issue = [&]() {
      uintptr_t src = 0, mend = 0;
      uint32_t n = 0;
      if (lane < 2) {
        src = row_src(jvi, ii, lane);
        n = static_cast<uint32_t>(a.rbh);
        mend = lane ? a.mend_u : a.mend_g;
      }
      warp_bulk_copies<true>(wring + islot * a.stage_bytes + lane * a.gseg, src, n, mend, &wbar[warp * kMaxNS + islot], lane);
      next_slot();
      adv(jvi, ii);
    };
    int n_iss = 0;
    for (; ok && n_iss < n_items && n_iss < a.NS - 1; ++n_iss) issue();
    // the token's activations (copied while the logits arrived) are waited for only now,
    // after the first weight requests of every warp are out
    cp_async_wait_all();
    __syncthreads();
    for (int it = 0; it < n_items && ok; ++it) {
      if (n_iss < n_items) {
        issue();
        ++n_iss;
      }
      if (!wait_slot()) {
        ok = false;
        break;
      }
      const uint32_t st = wring_s + static_cast<uint32_t>(wslot * a.stage_bytes);
      const uint32_t rows[2] = {st + (static_cast<uint32_t>(row_src(jvc, ic, 0)) & 15u),
                                st + static_cast<uint32_t>(a.gseg) + (static_cast<uint32_t>(row_src(jvc, ic, 1)) & 15u)};
      float acc[2];
      dot_rows(acc, rows, H, xs_s);
      // gate sum to lane 0, up sum to lane 16, then the up sum to lane 0 for the SwiGLU
      reduce_scatter<2>(acc, lane);
      const float usum = __shfl_sync(0xFFFFFFFFu, acc[0], 16);
      if (lane == 0) a.act[static_cast<size_t>(s_vz[jvc]) * F + ic] = silu_mul(acc[0], usum);
      release_slot();
      adv(jvc, ic);
    }
  }

  // down: items (pick jv, 4 consecutive hidden rows of this CTA), one copy of the rows (they
  // are contiguous); the ring is filled before the grid barrier (the rows are known), each
  // slot refilled right after it is consumed
  const int nh = hB - hA, nqd = (nh + 3) / 4;
  const int n2 = warp < kv * nqd ? (kv * nqd - warp + NW - 1) / NW : 0;
  int jd_i = nqd > 0 ? warp / nqd : 0, qd_i = warp - jd_i * nqd;  // issue cursor (quad qd of pick jd)
  int jd_c = jd_i, qd_c = qd_i;                                     // consume cursor
  auto adv2 = [&](int &jv, int &q) {
    q += NW;
    while (q >= nqd) {
      q -= nqd;
      ++jv;
    }
  };
  auto down_src = [&](int jv, int q) {
    return s_base[3 * jv + 2] + static_cast<uintptr_t>(hA + 4 * q) * static_cast<uintptr_t>(a.rbf);
  };
  auto issue2 = [&]() {
    uintptr_t src = 0;
    uint32_t n = 0;
    if (lane == 0) {
      src = down_src(jd_i, qd_i);
      n = static_cast<uint32_t>(min(4, nh - 4 * qd_i)) * static_cast<uint32_t>(a.rbf);
    }
    warp_bulk_copies<true>(wring + islot * a.stage_bytes, src, n, a.mend_d, &wbar[warp * kMaxNS + islot], lane);
    next_slot();
    adv2(jd_i, qd_i);
  };
  int n2_iss = 0;
  for (; ok && n2_iss < n2 && n2_iss < a.NS; ++n2_iss) issue2();
  if (!grid_barrier(a.bar, static_cast<unsigned int>(G), s_misc)) ok = false;
  // every CTA has read the call count: advance it for the next call on this workspace
  if (blockIdx.x == 0 && threadIdx.x == 0) st_relaxed_u64(a.gen, tag);
  pdl_launch_dependents();

  // ---- phase 2: the act rows of the valid picks into shared memory, the down dots, and the
  // combine for this CTA's hidden rows
  const int xrow_f = ((F + D::SG - 1) / D::SG) * D::SG * 4;  // bytes per act row in shared memory
  for (int jv = 0; jv < kv; ++jv) copy_x_row(xs, jv, xrow_f, a.act + static_cast<size_t>(s_vz[jv]) * F, F, threadIdx.x, NW * 32);
  cp_async_wait_all();
  __syncthreads();
  for (int it = 0; it < n2 && ok; ++it) {
    if (!wait_slot()) {
      ok = false;
      break;
    }
    const int nr = min(4, nh - 4 * qd_c);
    const uint32_t r0 = wring_s + static_cast<uint32_t>(wslot * a.stage_bytes) +
                        (static_cast<uint32_t>(down_src(jd_c, qd_c)) & 15u);
    const uint32_t rb = static_cast<uint32_t>(a.rbf);
    const uint32_t rows[4] = {r0, r0 + rb, r0 + 2u * rb, r0 + 3u * rb};
    float acc[4];
    dot_rows(acc, rows, F, xs_s + static_cast<uint32_t>(jd_c * xrow_f));
    reduce_scatter<4>(acc, lane);  // row r's sum in lane 8 r
    if ((lane & 7) == 0 && (lane >> 3) < nr) part[(4 * qd_c + (lane >> 3)) * kMaxK + jd_c] = acc[0];
    release_slot();
    adv2(jd_c, qd_c);
    if (n2_iss < n2) {
      issue2();
      ++n2_iss;
    }
  }
  __syncthreads();
  for (int hl = threadIdx.x; hl < nh; hl += NW * 32) {
    float sum = 0.f;
    for (int jv = 0; jv < kv; ++jv) sum = fmaf(s_w[s_vz[jv]], part[hl * kMaxK + jv], sum);
    if (ok) a.x[hA + hl] = (hl == static_cast<int>(threadIdx.x) ? x_pre : a.x[hA + hl]) + sum;
  }
  if (!ok) {
    if (lane == 0) moe_status(QG_STATUS_BIT_TIMEOUT);
    if (lane == 0)
      for (int it = waited; it < issued; ++it) mbar_wait(&wbar[warp * kMaxNS + (it % a.NS)], (it / a.NS) & 1);
  }
}

// ------------------------------------------------------------------------------------------
// Host side
// ------------------------------------------------------------------------------------------

// Workspace layout.  A fixed header comes first, at offsets that do not depend on the shape
// of a call: the one-token layer's grid-barrier counter and call counter (64-bit words that
// only grow) and its tagged logits, then the router's tickets (one word per 16-token tile,
// room for every tile count the router accepts).  Both must read zero in a fresh workspace and keep their meaning from call to
// call, so one workspace sized for the largest shape serves every smaller one.  The scratch
// regions (logits, dn rows, the grouped rows of the T > 16 path) follow the header and are
// rewritten by every call.
constexpr int kMaxRouterTiles = 65535;  // grid.y limit of the router launch
constexpr size_t kWsBar = 0;      // one-token layer: grid-barrier arrivals
constexpr size_t kWsGen = 16;     // one-token layer: calls on this workspace
constexpr size_t kWsXlog = 1024;  // one-token layer: tagged logits, up to 256 experts
constexpr size_t kWsTickets = 4096;
constexpr size_t kWsHeader = (kWsTickets + static_cast<size_t>(kMaxRouterTiles) * 4 + 255) & ~static_cast<size_t>(255);

struct WsLayout {
  size_t logits, dn, tc, total;
};

inline size_t up256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

WsLayout ws_layout(int T, int k, int E, int H, int F = 0) {
  WsLayout w;
  w.logits = kWsHeader;
  w.dn = w.logits + up256(static_cast<size_t>(T) * E * 4);
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

// Argument checks of the router (everything but the workspace), run before anything is
// enqueued.
qg_status route_check(const float *xn, const float *wr, int T, int H, int E, int k, const int32_t *ids,
                      const float *weights) {
  if (!xn || !wr || !ids || !weights) return QG_EINVAL_PTR;
  if (T < 1 || k < 1 || k > kMaxK || E < k || E > kMaxE || H < 4 || H % 4) return QG_EINVAL_SHAPE;
  if (static_cast<long long>(T) * H > INT32_MAX || static_cast<long long>(T) * E > INT32_MAX) return QG_EINVAL_SHAPE;
  if ((T + kRouterTB - 1) / kRouterTB > kMaxRouterTiles) return QG_EINVAL_SHAPE;
  if (!qg::aligned16(xn) || !qg::aligned16(wr)) return QG_EALIGN;
  return QG_OK;
}

// Router launch (route_check passed): logits into `logits` ([T][E]); with do_topk the last
// CTA of each token tile takes the picks, counting arrivals on tickets[tile] (zero on entry,
// zero again on exit).
qg_status route_launch(const float *xn, const float *wr, int T, int H, int E, int k, int32_t *ids, float *weights,
                       float *logits, unsigned int *tickets, int do_topk, cudaStream_t s) {
  const int tiles = (T + kRouterTB - 1) / kRouterTB;
  const qg::DeviceInfo &dev = qg::device_info();
  const size_t tiled_smem = (static_cast<size_t>(kRouterTB) * H + 4 * kRouterWarps * kRouterTB) * 4;
  if (dev.ok && tiles >= 4 && tiled_smem <= static_cast<size_t>(dev.smem_optin) - 1024) {
    // many token tiles: each CTA keeps its tile resident and runs a share of the experts,
    // about one CTA per SM in all
    const int n_eg = std::max(1, std::min((E + 3) / 4, dev.sms / tiles));
    const int epc = (E + n_eg - 1) / n_eg;
    const dim3 grid((E + epc - 1) / epc, tiles);
    if (!qg::set_smem_attr(reinterpret_cast<const void *>(moe_router_tiled_kernel), static_cast<uint32_t>(tiled_smem)))
      return QG_ECUDA;
    if (qg::launch_pdl(moe_router_tiled_kernel, grid, dim3(kRouterTiledWarps * 32), tiled_smem, s, xn, wr, T, H, E, k,
                       epc, logits, ids, weights, tickets, do_topk) != cudaSuccess)
      return QG_ECUDA;
    return cudaGetLastError() == cudaSuccess ? QG_OK : QG_ECUDA;
  }
  const dim3 grid(E, tiles);
  if (qg::launch_pdl(moe_router_kernel, grid, dim3(kRouterWarps * 32), 0, s, xn, wr, T, H, E, k, logits, ids, weights,
                     tickets, do_topk) != cudaSuccess)
    return QG_ECUDA;
  return cudaGetLastError() == cudaSuccess ? QG_OK : QG_ECUDA;
}

qg_status ws_check(const void *ws, size_t ws_bytes, size_t need) {
  if (!ws) return QG_EWORKSPACE;
  if (!qg::aligned16(ws)) return QG_EALIGN;
  return ws_bytes < need ? QG_EWORKSPACE : QG_OK;
}

qg_status route_impl(const float *xn, const float *wr, int T, int H, int E, int k, int32_t *ids, float *weights,
                     float *logits_out, void *ws, size_t ws_bytes, cudaStream_t s, int do_topk = 1) {
  qg_status c = route_check(xn, wr, T, H, E, k, ids, weights);
  if (c != QG_OK) return c;
  const WsLayout L = ws_layout(T, 1, E, H);
  c = ws_check(ws, ws_bytes, L.dn);
  if (c != QG_OK) return c;
  uint8_t *w = static_cast<uint8_t *>(ws);
  float *logits = logits_out ? logits_out : reinterpret_cast<float *>(w + L.logits);
  return route_launch(xn, wr, T, H, E, k, ids, weights, logits, reinterpret_cast<unsigned int *>(w + kWsTickets),
                      do_topk, s);
}

template <int QT, int TT, bool DOWN>
qg_status launch_expert(MoeArgs a, cudaStream_t s) {
  using D = Dec<QT>;
  constexpr int NW = 16;
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
  if (a.plan_only) return QG_OK;
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
  // Units of at most two tokens per expert for any T > 1: an expert with c tokens is read
  // ceil(c / 2) times, but the kernel keeps few accumulators and runs 16 warps per SM.  With
  // random routing of 8 tokens (64 picks over 128 experts) the re-reads are a few percent of
  // the bytes, and the layer ran 1.7x faster than with units of up to 8 tokens at 8 warps
  // per SM (latency-bound: 12 % warp occupancy, 38 % issue).
  if (a.T == 1) return launch_expert<QT, 1, DOWN>(a, s);
  return launch_expert<QT, 2, DOWN>(a, s);
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

// The one-token layer in one cooperative launch; QG_EUNSUPPORTED (nothing launched) when the
// shapes do not fit its shared-memory plan or the grid cannot be co-resident.
template <int QT>
qg_status launch_one_token(OneArgs a, cudaStream_t s) {
  using D = Dec<QT>;
  constexpr int NW = 16;
  const qg::DeviceInfo &dev = qg::device_info();
  if (!dev.ok) return QG_ECUDA;
  if (a.k > kMaxK) return QG_EUNSUPPORTED;
  const int G = dev.sms;
  const uint32_t hdr = 2048;
  const long long xrow_h = static_cast<long long>((a.H + D::SG - 1) / D::SG) * D::SG * 4;
  const long long xrow_f = static_cast<long long>((a.F + D::SG - 1) / D::SG) * D::SG * 4;
  const long long xbytes = ((std::max(xrow_h, a.k * xrow_f) + 1023) / 1024) * 1024;
  a.hmax = (a.H + G - 1) / G;
  // per-row pick dots of phase 2; the logits for the ranking before that
  const long long part = ((std::max<long long>(static_cast<long long>(a.hmax) * kMaxK, kMaxE) * 4 + 1023) / 1024) * 1024;
  a.gseg = static_cast<int>(((a.rbh + 15) & ~15LL) + 32);
  a.dseg = static_cast<int>(((a.rbf + 15) & ~15LL) + 32);
  const long long stage = std::max<long long>(2LL * a.gseg, ((4 * a.rbf + 15) & ~15LL) + 32);
  const long long ring = dev.smem_optin - 1024 - hdr - xbytes - part;
  const int NS = ring > 0 ? static_cast<int>(std::min<long long>(kMaxNS, ring / (NW * stage))) : 0;
  if (NS < 2) return QG_EUNSUPPORTED;
  if (static_cast<long long>(NW) * NS * stage < 16LL * a.E) return QG_EUNSUPPORTED;  // the ranking's counts
  a.NS = NS;
  a.stage_bytes = static_cast<int>(stage);
  a.off_x = hdr;
  a.off_part = static_cast<uint32_t>(hdr + xbytes);
  a.off_ring = static_cast<uint32_t>(hdr + xbytes + part);
  const uint32_t smem = a.off_ring + static_cast<uint32_t>(NW * NS * stage) + 1024;
  auto kern = moe_one_token_kernel<QT, NW>;
  if (!qg::set_smem_attr(reinterpret_cast<const void *>(kern), smem)) return QG_ECUDA;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, NW * 32, smem) != cudaSuccess || per_sm < 1)
    return QG_EUNSUPPORTED;
  a.early_weights = qg::static_weights(s) ? 1 : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(G);
  cfg.blockDim = dim3(NW * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (cudaLaunchKernelEx(&cfg, kern, a) != cudaSuccess) return QG_ECUDA;
  return cudaGetLastError() == cudaSuccess ? QG_OK : QG_ECUDA;
}

qg_status one_token_layer(int type, const float *xn, const float *wr, const void *w_gate, const void *w_up,
                          const void *w_down, int64_t stride, const int32_t *slots, int n_slots, int H, int F, int E,
                          int k, int32_t *ids, float *weights, float *act, float *x_inout, void *ws, cudaStream_t s) {
  int qk = 0, bb = 0;
  qg_block_shape(type, &qk, &bb);
  if (!qg::aligned16(xn) || !qg::aligned16(wr) || !qg::aligned16(act) || !qg::aligned16(ws)) return QG_EUNSUPPORTED;
  if (static_cast<long long>(k) * F > INT32_MAX) return QG_EUNSUPPORTED;  // row pairs are numbered in 32 bits
  OneArgs a{};
  a.xn = xn;
  a.wr = wr;
  a.wg = static_cast<const uint8_t *>(w_gate);
  a.wu = static_cast<const uint8_t *>(w_up);
  a.wd = static_cast<const uint8_t *>(w_down);
  a.stride = stride;
  const long long mat_gu = static_cast<long long>(F) * (H / qk) * bb, mat_d = static_cast<long long>(H) * (F / qk) * bb;
  a.mend_g = tensor_mend(w_gate, stride, n_slots, mat_gu);
  a.mend_u = tensor_mend(w_up, stride, n_slots, mat_gu);
  a.mend_d = tensor_mend(w_down, stride, n_slots, mat_d);
  a.slots = slots;
  a.n_slots = n_slots;
  a.E = E;
  a.k = k;
  a.H = H;
  a.F = F;
  a.ids_out = ids;
  a.wts_out = weights;
  a.act = act;
  a.x = x_inout;
  a.bar = reinterpret_cast<unsigned long long *>(static_cast<uint8_t *>(ws) + kWsBar);
  a.gen = reinterpret_cast<unsigned long long *>(static_cast<uint8_t *>(ws) + kWsGen);
  a.xlog = reinterpret_cast<unsigned long long *>(static_cast<uint8_t *>(ws) + kWsXlog);
  a.rbh = static_cast<long long>(H / qk) * bb;
  a.rbf = static_cast<long long>(F / qk) * bb;
  switch (type) {
    case QG_TYPE_Q8_0: return launch_one_token<QG_TYPE_Q8_0>(a, s);
    case QG_TYPE_Q4_0: return launch_one_token<QG_TYPE_Q4_0>(a, s);
    case QG_TYPE_Q4_K: return launch_one_token<QG_TYPE_Q4_K>(a, s);
    case QG_TYPE_Q6_K: return launch_one_token<QG_TYPE_Q6_K>(a, s);
    default: return QG_EUNSUPPORTED;
  }
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

// Host checks of the gate/up step that need no launch; the shared-memory plan is checked by
// swiglu_plan.  Nothing is enqueued by either.
qg_status swiglu_check(int type, const void *w_gate, const void *w_up, int64_t stride, int n_slots, int E,
                       const int32_t *ids, const float *xn, int T, int k, int H, int F, const float *act,
                       const void *ws, size_t ws_bytes) {
  if (!w_gate || !w_up || !ids || !xn || !act) return QG_EINVAL_PTR;
  const qg_status c = expert_checks(type, T, k, E, H, F, n_slots, stride);
  if (c != QG_OK) return c;
  if (!qg::aligned16(xn) || !qg::aligned16(act)) return QG_EALIGN;
  int qk = 0, bb = 0;
  qg_block_shape(type, &qk, &bb);
  const long long mat = static_cast<long long>(F) * (H / qk) * bb;
  if (n_slots > 1 && stride < mat) return QG_EINVAL_SHAPE;
  if (T > 16) {
    if (!qg::aligned16(w_gate) || !qg::aligned16(w_up)) return QG_EALIGN;
    return ws_check(ws, ws_bytes, ws_layout(T, k, E, H, F).total);
  }
  return QG_OK;
}

MoeArgs swiglu_args(int type, const void *w_gate, const void *w_up, int64_t stride, const int32_t *slots,
                    int n_slots, int E, const int32_t *ids, const float *xn, int T, int k, int H, int F, float *act) {
  int qk = 0, bb = 0;
  qg_block_shape(type, &qk, &bb);
  const long long mat = static_cast<long long>(F) * (H / qk) * bb;
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
  return a;
}

qg_status swiglu_impl(int type, const void *w_gate, const void *w_up, int64_t stride, const int32_t *slots,
                      int n_slots, int E, const int32_t *ids, const float *xn, int T, int k, int H, int F,
                      float *act, void *ws, size_t ws_bytes, cudaStream_t s, const float *fused_logits = nullptr,
                      int32_t *ids_out = nullptr, float *wts_out = nullptr, int plan_only = 0,
                      const qg::MoeVar &v = qg::MoeVar()) {
  const qg_status c = swiglu_check(type, w_gate, w_up, stride, n_slots, E, ids, xn, T, k, H, F, act, ws, ws_bytes);
  if (c != QG_OK) return c;
  if (T > 16) {
    if (plan_only) return QG_OK;
    return qg::moe_swiglu_tc(w_gate, w_up, stride, slots, n_slots, E, ids, xn, T, k, H, F, act,
                             static_cast<uint8_t *>(ws) + ws_layout(T, k, E, H, F).tc, s, v.act);
  }
  MoeArgs a = swiglu_args(type, w_gate, w_up, stride, slots, n_slots, E, ids, xn, T, k, H, F, act);
  a.plan_only = plan_only;
  a.act_kind = v.act;
  if (fused_logits) {
    a.fuse_topk = 1;
    a.logits = fused_logits;
    a.ids_out = ids_out;
    a.wts_out = wts_out;
  }
  return launch_expert_type<false>(type, a, s);
}

qg_status combine_check(int type, const void *w_down, int64_t stride, int n_slots, int E, const int32_t *ids,
                        const float *weights, const float *act, int T, int k, int H, int F, const float *x_inout,
                        const void *ws, size_t ws_bytes) {
  if (!w_down || !ids || !weights || !act || !x_inout) return QG_EINVAL_PTR;
  const qg_status c = expert_checks(type, T, k, E, H, F, n_slots, stride);
  if (c != QG_OK) return c;
  if (!qg::aligned16(act) || !qg::aligned16(x_inout)) return QG_EALIGN;
  if (T > 16 && !qg::aligned16(w_down)) return QG_EALIGN;
  int qk = 0, bb = 0;
  qg_block_shape(type, &qk, &bb);
  const long long mat = static_cast<long long>(H) * (F / qk) * bb;
  if (n_slots > 1 && stride < mat) return QG_EINVAL_SHAPE;
  return ws_check(ws, ws_bytes, ws_layout(T, k, E, H, F).total);
}

qg_status combine_impl(int type, const void *w_down, int64_t stride, const int32_t *slots, int n_slots, int E,
                       const int32_t *ids, const float *weights, const float *act, int T, int k, int H, int F,
                       float *x_inout, int add_residual, void *ws, size_t ws_bytes, cudaStream_t s,
                       int plan_only = 0, const qg::MoeVar &v = qg::MoeVar(), bool sorted_ready = false) {
  const qg_status c =
      combine_check(type, w_down, stride, n_slots, E, ids, weights, act, T, k, H, F, x_inout, ws, ws_bytes);
  if (c != QG_OK) return c;
  const WsLayout L = ws_layout(T, k, E, H, F);
  uint8_t *w = static_cast<uint8_t *>(ws);
  if (T > 16) {
    if (plan_only) return QG_OK;
    return qg::moe_combine_tc(w_down, stride, slots, n_slots, E, ids, weights, act, T, k, H, F, x_inout,
                              add_residual ? 1 : 0, reinterpret_cast<float *>(w + L.dn), w + L.tc, s, v, sorted_ready);
  }
  int qk = 0, bb = 0;
  qg_block_shape(type, &qk, &bb);
  const long long mat = static_cast<long long>(H) * (F / qk) * bb;
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
  a.plan_only = plan_only;
  const qg_status r = launch_expert_type<true>(type, a, s);
  if (r != QG_OK || plan_only) return r;
  return qg::moe_launch_combine(a.dn, weights, ids, slots, n_slots, E, T, k, H, x_inout, add_residual ? 1 : 0, s, v);
}

// The variant of one call: QG_EINVAL_SHAPE for an unknown activation, QG_EINVAL_PTR for a
// shared row without its gate (or the reverse), QG_EALIGN for misaligned vectors.
qg_status variant_check(const qg_moe_variant *v, qg::MoeVar &out) {
  out = qg::MoeVar();
  if (!v) return QG_OK;
  if (v->act != QG_ACT_SILU && v->act != QG_ACT_GELU_TANH) return QG_EINVAL_SHAPE;
  if ((v->shared_out == nullptr) != (v->shared_gate == nullptr)) return QG_EINVAL_PTR;
  if ((v->shared_out && !qg::aligned16(v->shared_out)) || (reinterpret_cast<uintptr_t>(v->shared_gate) & 3u) ||
      (reinterpret_cast<uintptr_t>(v->down_scale) & 3u))
    return QG_EALIGN;
  out.act = v->act;
  out.ds = v->down_scale;
  out.sh = v->shared_out;
  out.sg = v->shared_gate;
  return QG_OK;
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
// Fixed device scratch for moe_route_topk_noalloc: the per-tile tickets (1024 words) and then
// the logits (16384 floats), 68 KB in all.  Every device that loads the library holds one copy
// until the process exits.
namespace {
constexpr int kNoAllocLogits = 16384;
constexpr int kNoAllocTiles = 1024;
constexpr size_t kNoAllocTicketBytes = static_cast<size_t>(kNoAllocTiles) * 4;
constexpr size_t kNoAllocBytes = kNoAllocTicketBytes + static_cast<size_t>(kNoAllocLogits) * 4;
__device__ __align__(256) unsigned char g_route_scratch[kNoAllocBytes];

std::mutex g_scratch_mu;
void *g_scratch_ptr[64];  // per device, filled on the first call with that device current

// Device address of the scratch array on the current device.  In host code the array's name
// is only a stand-in, so the address comes from the runtime, once per device.
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
  // every check before anything is enqueued
  const qg_status c = route_check(xn, wr, T, H, E, k, ids, weights);
  if (c != QG_OK) return c;
  const int tiles = (T + kRouterTB - 1) / kRouterTB;
  if (static_cast<long long>(T) * E > kNoAllocLogits || tiles > kNoAllocTiles) return QG_EWORKSPACE;
  void *ws = route_scratch();
  if (!ws) return QG_ECUDA;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t *w = static_cast<uint8_t *>(ws);
  // the tickets must read zero when the router starts (the previous call may have had another
  // shape, or may not have finished its tiles)
  if (cudaMemsetAsync(w, 0, static_cast<size_t>(tiles) * 4, s) != cudaSuccess) return QG_ECUDA;
  float *logits = logits_out ? logits_out : reinterpret_cast<float *>(w + kNoAllocTicketBytes);
  return route_launch(xn, wr, T, H, E, k, ids, weights, logits, reinterpret_cast<unsigned int *>(w), 1, s);
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

qg_status moe_expert_act(int type, const void *w_gate, const void *w_up, int64_t expert_stride,
                         const int32_t *slots, int n_slots, int E, const int32_t *ids, const float *xn, int T,
                         int k, int H, int F, const qg_moe_variant *variant, float *act, void *ws,
                         size_t ws_bytes, qg_stream_t stream) {
  qg::MoeVar v;
  const qg_status c = variant_check(variant, v);
  if (c != QG_OK) return c;
  return swiglu_impl(type, w_gate, w_up, expert_stride, slots, n_slots, E, ids, xn, T, k, H, F, act, ws, ws_bytes,
                     reinterpret_cast<cudaStream_t>(stream), nullptr, nullptr, nullptr, 0, v);
}

qg_status moe_combine_ex(int type, const void *w_down, int64_t expert_stride, const int32_t *slots, int n_slots,
                         int E, const int32_t *ids, const float *weights, const float *act, int T, int k, int H, int F,
                         const qg_moe_variant *variant, float *x_inout, int add_residual, void *ws, size_t ws_bytes,
                         qg_stream_t stream) {
  qg::MoeVar v;
  const qg_status c = variant_check(variant, v);
  if (c != QG_OK) return c;
  return combine_impl(type, w_down, expert_stride, slots, n_slots, E, ids, weights, act, T, k, H, F, x_inout,
                      add_residual, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream), 0, v);
}

qg_status moe_layer_ex(int type, const float *xn, const float *wr, const void *w_gate, const void *w_up,
                       const void *w_down, int64_t expert_stride, const int32_t *slots, int n_slots, int T, int H,
                       int F, int E, int k, const qg_moe_variant *variant, int32_t *ids, float *weights, float *act,
                       float *x_inout, void *ws, size_t ws_bytes, qg_stream_t stream) {
  qg::MoeVar v;
  qg_status c = variant_check(variant, v);
  if (c != QG_OK) return c;
  if (v.act == 0 && !v.ds && !v.sh)
    return moe_layer(type, xn, wr, w_gate, w_up, w_down, expert_stride, slots, n_slots, T, H, F, E, k, ids, weights,
                     act, x_inout, ws, ws_bytes, stream);
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (!xn || !wr || !w_gate || !w_up || !w_down || !ids || !weights || !act || !x_inout) return QG_EINVAL_PTR;
  c = route_check(xn, wr, T, H, E, k, ids, weights);
  if (c != QG_OK) return c;
  c = swiglu_check(type, w_gate, w_up, expert_stride, n_slots, E, ids, xn, T, k, H, F, act, ws, ws_bytes);
  if (c != QG_OK) return c;
  c = combine_check(type, w_down, expert_stride, n_slots, E, ids, weights, act, T, k, H, F, x_inout, ws, ws_bytes);
  if (c != QG_OK) return c;
  if (T <= 16) {
    // every launch's shared-memory plan before the first launch
    c = swiglu_impl(type, w_gate, w_up, expert_stride, slots, n_slots, E, ids, xn, T, k, H, F, act, ws, ws_bytes, s,
                    nullptr, nullptr, nullptr, 1, v);
    if (c != QG_OK) return c;
    c = combine_impl(type, w_down, expert_stride, slots, n_slots, E, ids, weights, act, T, k, H, F, x_inout, 1, ws,
                     ws_bytes, s, 1, v);
    if (c != QG_OK) return c;
  }
  // the variants run as three steps at every T: router with top-k, expert gate/up with the
  // variant's activation, down rows and the variant's combine
  qg_status r = route_impl(xn, wr, T, H, E, k, ids, weights, nullptr, ws, ws_bytes, s, 1);
  if (r != QG_OK) return r;
  r = swiglu_impl(type, w_gate, w_up, expert_stride, slots, n_slots, E, ids, xn, T, k, H, F, act, ws, ws_bytes, s,
                  nullptr, nullptr, nullptr, 0, v);
  if (r != QG_OK) return r;
  // above 16 tokens the gate/up step left the grouping and the sorted act rows for the down step
  return combine_impl(type, w_down, expert_stride, slots, n_slots, E, ids, weights, act, T, k, H, F, x_inout, 1, ws,
                      ws_bytes, s, 0, v, T > 16);
}

qg_status moe_layer(int type, const float *xn, const float *wr, const void *w_gate, const void *w_up,
                    const void *w_down, int64_t expert_stride, const int32_t *slots, int n_slots, int T, int H, int F,
                    int E, int k, int32_t *ids, float *weights, float *act, float *x_inout, void *ws,
                    size_t ws_bytes, qg_stream_t stream) {
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // every step's checks (and, for T <= 16, its shared-memory plan) before the first launch
  if (!xn || !wr || !w_gate || !w_up || !w_down || !ids || !weights || !act || !x_inout) return QG_EINVAL_PTR;
  qg_status c = route_check(xn, wr, T, H, E, k, ids, weights);
  if (c != QG_OK) return c;
  c = swiglu_check(type, w_gate, w_up, expert_stride, n_slots, E, ids, xn, T, k, H, F, act, ws, ws_bytes);
  if (c != QG_OK) return c;
  c = combine_check(type, w_down, expert_stride, n_slots, E, ids, weights, act, T, k, H, F, x_inout, ws, ws_bytes);
  if (c != QG_OK) return c;
  qg_status r;
  if (T > 16) {
    // prefill-sized batch: router with top-k, then the grouped tensor-core expert steps
    r = route_impl(xn, wr, T, H, E, k, ids, weights, nullptr, ws, ws_bytes, s, 1);
    if (r != QG_OK) return r;
    r = swiglu_impl(type, w_gate, w_up, expert_stride, slots, n_slots, E, ids, xn, T, k, H, F, act, ws, ws_bytes, s);
    if (r != QG_OK) return r;
    return combine_impl(type, w_down, expert_stride, slots, n_slots, E, ids, weights, act, T, k, H, F, x_inout, 1,
                        ws, ws_bytes, s, 0, qg::MoeVar(), true);
  }
  // one token: the whole layer in one cooperative launch when it fits
  if (T == 1) {
    r = one_token_layer(type, xn, wr, w_gate, w_up, w_down, expert_stride, slots, n_slots, H, F, E, k, ids, weights,
                        act, x_inout, ws, s);
    if (r != QG_EUNSUPPORTED) return r;
  }
  // router logits into the workspace; the gate/up kernel ranks them (every CTA needs the
  // picks for its plan anyway) and stores ids and weights for the combine
  const float *logits = reinterpret_cast<const float *>(static_cast<uint8_t *>(ws) + ws_layout(T, k, E, H).logits);
  r = swiglu_impl(type, w_gate, w_up, expert_stride, slots, n_slots, E, ids, xn, T, k, H, F, act, ws, ws_bytes, s,
                  logits, ids, weights, 1);
  if (r != QG_OK) return r;
  r = combine_impl(type, w_down, expert_stride, slots, n_slots, E, ids, weights, act, T, k, H, F, x_inout, 1, ws,
                   ws_bytes, s, 1);
  if (r != QG_OK) return r;
  r = route_impl(xn, wr, T, H, E, k, ids, weights, nullptr, ws, ws_bytes, s, 0);
  if (r != QG_OK) return r;
  r = swiglu_impl(type, w_gate, w_up, expert_stride, slots, n_slots, E, ids, xn, T, k, H, F, act, ws, ws_bytes, s,
                  logits, ids, weights);
  if (r != QG_OK) return r;
  return combine_impl(type, w_down, expert_stride, slots, n_slots, E, ids, weights, act, T, k, H, F, x_inout, 1, ws,
                      ws_bytes, s);
}

}  // extern "C"
