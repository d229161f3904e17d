// qg_gemv.cu -- dense quantized GEMV over 1..16 token columns on sm_103a.
//
// Y[t][m] = sum_k W[m][k] * X[t][k] with W in raw GGUF blocks (matmulQ8 / matmulQ4 /
// matmulQ6K for one token, matmulQ8T for a token batch, in the engine pages of the
// diskformer package), f32 activations and f32 accumulation.
//
// Design (persistent CTAs, one per SM; every warp runs its own pipeline):
//   - each warp owns row blocks (2 rows for one token, 4 when several token columns share
//     every decoded weight) and NS shared-memory slots with one mbarrier each.  The warp
//     issues its next stages ahead with 1-D bulk copies (the TMA engine, cp.async.bulk): a
//     stage is the block's whole rows in one copy (they are contiguous in the raw layout)
//     or one copy per row segment of at least 2 KB.  Copies that small stream at full
//     speed; much smaller ones are capped by the copy engine's per-copy rate.  No producer
//     warp: a single issuing thread caps a CTA's bulk-copy rate well below HBM speed, while
//     per-warp issue streams at full bandwidth.
//   - the warp decodes its rows straight from the raw blocks in shared memory
//     (qg_decode.cuh), reusing every activation load for the block's rows, and keeps the
//     accumulators in registers across the row's chunks.
//   - activations: when all T rows fit in shared memory they are loaded once (2-D tensor
//     copies with the 128-byte swizzle); otherwise they come in double-buffered K chunks
//     that every warp walks in step, chunk partial sums kept in shared memory.
//   - with few rows, KW warps split a row block's chunks and meet at a named barrier to sum
//     their partials in a fixed order (deterministic).
//   - every weight byte crosses HBM once per call, whatever T is.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "qg_decode.cuh"
#include "qg_host.h"
#include "qg_pipe.cuh"

__device__ unsigned int g_qg_status_gemv;

namespace {

constexpr int kMaxNS = 4;  // slots per warp

constexpr int kMaxMats = 4;  // matrices that one launch may cover (sharing x)

struct GemvArgs {
  // up to kMaxMats matrices of the same type and row length over the same activations: their
  // row blocks are numbered one after another (matrix j owns [rb0[j], rb0[j + 1]))
  const uint8_t *w[kMaxMats];
  float *y[kMaxMats];
  int Mj[kMaxMats];
  long long rb0[kMaxMats + 1];
  int nmat;
  long long row_bytes;
  int N, T;
  int mode;          // 0: activations resident; 1: activations in K chunks (one per weight chunk)
  int KC;            // elements per weight chunk (multiple of SG)
  int nchunks;       // chunks per row
  int xR;            // activation rows (32 floats) per token in one buffer
  int rblocks;       // row blocks (2 rows for one token, else 4)
  int max_kw;        // most warps that may split one row block (mode 0; <= nchunks)
  int NS;            // slots per warp
  int stage_bytes;   // bytes per slot
  int seg_slot;      // bytes per row segment inside a slot; 0: the block's whole rows in one copy
  int box_rows;      // rows per activation tensor copy
  int maxq;          // most row blocks of one warp (mode 1 partial sums)
  int early_weights;  // weights are static: issue the first weight stages before the wait on the predecessor
  uint32_t off_x, off_ring, off_red, off_part;
  uint32_t xbuf_bytes;
};

QG_DEVICE void set_status(unsigned int bits) { atomicOr(&g_qg_status_gemv, bits); }

// The matrix that owns row block rb, and the block's index within it.
struct RowBlock {
  const uint8_t *w;
  float *y;
  int M;
  long long lrb;
  uintptr_t mend;  // last 16-byte boundary of the matrix
};

QG_DEVICE RowBlock row_block(const GemvArgs &a, long long rb) {
  int j = 0;
#pragma unroll
  for (int q = 1; q < kMaxMats; ++q)
    if (q < a.nmat && rb >= a.rb0[q]) j = q;
  RowBlock b;
  b.w = a.w[j];
  b.y = a.y[j];
  b.M = a.Mj[j];
  b.lrb = rb - a.rb0[j];
  b.mend = (reinterpret_cast<uintptr_t>(b.w) + static_cast<uintptr_t>(static_cast<long long>(b.M) * a.row_bytes)) &
           ~static_cast<uintptr_t>(15);
  return b;
}

// Item cursor of one warp: tile index q (within the CTA) and chunk c.
struct Cursor {
  int q, c;
};

// Rows per row block: 2 for one token (so that a stage of whole rows stays one large copy
// with 16 warps), 4 when several token columns share every decoded weight.
template <int TT>
__host__ __device__ constexpr int rows_per_block() {
  return TT == 1 ? 2 : 4;
}

template <int QT, int TT, int NW>
__global__ void __launch_bounds__(NW * 32, (TT == 1 && NW == 8) ? 2 : 1) qgemv_kernel(const __grid_constant__ CUtensorMap xmap, const GemvArgs a) {
  using D = Dec<QT>;
  constexpr int RR = rows_per_block<TT>();
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t *wbar = reinterpret_cast<uint64_t *>(smem);  // [NW][kMaxNS]
  uint64_t *xfull = wbar + NW * kMaxNS;                  // [2]
  float *red = reinterpret_cast<float *>(smem + a.off_red);    // [2][NW][RR][TT]
  float *part = reinterpret_cast<float *>(smem + a.off_part);  // [NW][maxq][RR][TT] (mode 1)
  uint8_t *xs = smem + a.off_x;
  uint8_t *ring = smem + a.off_ring;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = static_cast<int>(gridDim.x);
  // this CTA's contiguous, balanced range of row blocks
  const long long rbA = static_cast<long long>(blockIdx.x) * a.rblocks / G;
  const long long rbB = static_cast<long long>(blockIdx.x + 1) * a.rblocks / G;
  const int nrb = static_cast<int>(rbB - rbA);
  // warps per row block: 1 when the CTA has at least NW row blocks, else the CTA's warps
  // split each row block's chunks (mode 0 only)
  int KW = 1;
  if (a.mode == 0 && nrb < NW) KW = max(1, min(NW / max(nrb, 1), a.max_kw));
  const int kw = warp % KW, rbl = warp / KW;
  const int nslots = NW / KW;                       // row-block lanes in this CTA
  const bool active = rbl < nslots && (nrb >= NW || rbl < nrb);
  const int my_rbs = active ? (nrb - rbl + nslots - 1) / nslots : 0;  // row blocks rbA + rbl + i * nslots
  const int xbytes_token = a.xR * 128;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NW * kMaxNS; ++i) mbar_init(&wbar[i], 1);
    mbar_init(&xfull[0], 1);
    mbar_init(&xfull[1], 1);
    fence_mbar_init();
  }
  __syncthreads();

  // ---- this warp's item sequence: (i-th row block of this warp, chunk c)
  auto first = [&]() { return Cursor{0, a.mode == 0 ? kw : 0}; };
  auto next = [&](Cursor u) {
    if (a.mode == 0) {
      u.c += KW;
      if (u.c >= a.nchunks) {
        u.c = kw;
        ++u.q;
      }
    } else if (++u.q >= my_rbs) {
      u.q = 0;
      ++u.c;
    }
    return u;
  };
  // mode 1 walks every chunk (with my_rbs == 0 the warp only joins the chunk barriers)
  auto valid = [&](Cursor u) { return a.mode == 0 ? u.q < my_rbs : u.c < a.nchunks; };
  auto rb_of = [&](Cursor u) { return rbA + rbl + static_cast<long long>(u.q) * nslots; };

  const long long chunk_bytes = static_cast<long long>(a.KC / D::QK) * D::BB;
  uint8_t *wring = ring + warp * a.NS * a.stage_bytes;
  const uint32_t wring_s = smem_u32(wring);

  // Issue the stage of item u into slot s: lane r copies row r's segment (lane 0 copies 4
  // whole rows at once when the stage holds whole rows); the byte count goes to the slot's
  // mbarrier before any copy starts.
  const bool pad_rows = a.seg_slot != 0;
  auto issue = [&](Cursor u, int s) {
    const RowBlock b = row_block(a, rb_of(u));
    const uintptr_t wbase = reinterpret_cast<uintptr_t>(b.w);
    const long long rb = b.lrb;
    const int nr = (my_rbs == 0) ? 0 : static_cast<int>(max(0LL, min(static_cast<long long>(RR), b.M - rb * RR)));
    uint8_t *st = wring + s * a.stage_bytes;
    uintptr_t src = 0;
    uint32_t n = 0;
    uint8_t *dst = st;
    if (!pad_rows) {
      if (lane == 0) {
        src = wbase + static_cast<uintptr_t>(rb * RR * a.row_bytes);
        n = static_cast<uint32_t>(nr * a.row_bytes);
      }
    } else if (lane < nr) {
      const int kel = min(a.N - u.c * a.KC, a.KC);
      n = static_cast<uint32_t>(kel / D::QK) * D::BB;
      src = wbase + static_cast<uintptr_t>((rb * RR + lane) * a.row_bytes + u.c * chunk_bytes);
      dst = st + lane * a.seg_slot;
    }
    warp_bulk_copies<true>(dst, src, n, b.mend, &wbar[warp * kMaxNS + s], lane);
  };

  // Prologue: the first NS - 1 items.  Normally issued after the wait on the preceding kernel
  // and after the activations; with static weights (the caller guarantees that no kernel
  // writes them) they are issued as soon as the CTA is resident, while the preceding kernel
  // drains, and only the activations and outputs wait.
  Cursor ic = first();
  int is = 0, issued = 0;
  auto prologue = [&]() {
    for (int i = 0; i < a.NS - 1 && valid(ic); ++i) {
      issue(ic, is);
      ic = next(ic);
      is = (is + 1 == a.NS) ? 0 : is + 1;
      ++issued;
    }
  };
  if (a.early_weights) prologue();
  pdl_wait();
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    load_x(xs, &xmap, a.T, a.N, 0, a.xR, a.box_rows, &xfull[0]);
    if (a.mode == 1 && a.nchunks > 1) load_x(xs + a.xbuf_bytes, &xmap, a.T, a.N, 1, a.xR, a.box_rows, &xfull[1]);
  }
  if (!a.early_weights) prologue();

  const uint32_t wo = static_cast<uint32_t>(D::woff(lane));
  uint32_t xo[D::NCH];
#pragma unroll
  for (int ch = 0; ch < D::NCH; ++ch) xo[ch] = x_lane_off<QT>(lane, ch);
  const int gpc = a.KC / D::SG;

  bool ok = true;
  if (!mbar_wait(&xfull[0], 0)) ok = false;
  float acc1[RR];
  f2 acc2[RR][TT];
  Cursor cc = first();
  int cs = 0, cround = 0, consumed = 0;
  int cur_xc = 0;  // activation chunk the warp is on (mode 1)
  while (valid(cc)) {
    // keep NS - 1 stages in flight ahead of this one
    if (valid(ic)) {
      issue(ic, is);
      ic = next(ic);
      is = (is + 1 == a.NS) ? 0 : is + 1;
      ++issued;
    }
    if (a.mode == 1 && cc.c != cur_xc) {  // every warp is done with chunk cur_xc
      named_bar_sync(1, NW * 32);
      if (threadIdx.x == 0 && cur_xc + 2 < a.nchunks)
        load_x(xs + (cur_xc & 1) * a.xbuf_bytes, &xmap, a.T, a.N, cur_xc + 2, a.xR, a.box_rows, &xfull[cur_xc & 1]);
      cur_xc = cc.c;
      if (ok && !mbar_wait(&xfull[cur_xc & 1], (cur_xc >> 1) & 1)) ok = false;
    }
    const RowBlock blk = row_block(a, rb_of(cc));
    const bool first_chunk = (a.mode == 1) || (cc.c == kw);
    const bool last_chunk = (a.mode == 1) || (cc.c + KW >= a.nchunks);
    if (first_chunk) {
#pragma unroll
      for (int r = 0; r < RR; ++r) {
        acc1[r] = 0.f;
#pragma unroll
        for (int t = 0; t < TT; ++t) acc2[r][t] = mk2(0.f, 0.f);
      }
    }
    if (ok && !mbar_wait(&wbar[warp * kMaxNS + cs], cround & 1)) ok = false;
    if (ok) {
      const int kel = min(a.N - cc.c * a.KC, a.KC);
      const int gcount = (kel + D::SG - 1) / D::SG;
      const uint32_t st = wring_s + static_cast<uint32_t>(cs * a.stage_bytes);
      uint32_t wrow[RR];
      {
        // low 32 bits suffice: only the address modulo 16 matters
        const uint32_t r0 = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(blk.w)) +
                            static_cast<uint32_t>(blk.lrb * RR) * static_cast<uint32_t>(a.row_bytes);
        const uint32_t cb = static_cast<uint32_t>(cc.c) * static_cast<uint32_t>(chunk_bytes);
#pragma unroll
        for (int r = 0; r < RR; ++r) {
          if (!pad_rows)
            wrow[r] = st + (r0 & 15u) + static_cast<uint32_t>(r) * static_cast<uint32_t>(a.row_bytes) + wo;
          else
            wrow[r] = st + static_cast<uint32_t>(r * a.seg_slot) +
                      ((r0 + static_cast<uint32_t>(r) * static_cast<uint32_t>(a.row_bytes) + cb) & 15u) + wo;
        }
      }
      // activation base of this chunk's first group
      const uint32_t xg0 = smem_u32(xs) + (a.mode == 0 ? static_cast<uint32_t>(cc.c * gpc * (D::SG * 4))
                                                        : static_cast<uint32_t>(cc.c & 1) * a.xbuf_bytes);
      // one token: the groups in which every lane's unit is in range, then the last, partial
      // group with a per-lane check (several tokens keep the per-group check)
      const int gfull = kel / D::SG;
      RowPrep<QT> rp[RR];
#pragma unroll
      for (int r = 0; r < RR; ++r) rp[r].init(wrow[r], lane);
      auto group = [&](int g) {
        const uint32_t goff = static_cast<uint32_t>(g * D::GB);
        const uint32_t xg = xg0 + static_cast<uint32_t>(g * (D::SG * 4));
        if constexpr (TT == 1) {
          float4 xc[D::NCH];
#pragma unroll
          for (int ch = 0; ch < D::NCH; ++ch) xc[ch] = lds_f4(xg + xo[ch]);
          const float aux = D::xaux(xc);
          typename D::U u[RR];
#pragma unroll
          for (int r = 0; r < RR; ++r) u[r] = rp[r].load(goff, lane);
#pragma unroll
          for (int r = 0; r < RR; ++r) acc1[r] += D::dot1(u[r], xc, aux);
        } else {
          typename D::U u[RR];
#pragma unroll
          for (int r = 0; r < RR; ++r) u[r] = D::load(wrow[r] + goff, lane);
#pragma unroll
          for (int ch = 0; ch < D::NCH; ++ch) {
            f2 w01[RR], w23[RR];
#pragma unroll
            for (int r = 0; r < RR; ++r) D::weights(u[r], ch, w01[r], w23[r]);
#pragma unroll
            for (int t = 0; t < TT; ++t) {
              if (t < a.T) {
                const float4 xv = lds_f4(xg + static_cast<uint32_t>(t * xbytes_token) + xo[ch]);
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
      };
      if constexpr (TT == 1) {
        for (int g = 0; g < gfull; ++g) group(g);
        if (gfull < gcount && gfull * D::SG + D::block_first(lane) < kel) group(gfull);
      } else {
        for (int g = 0; g < gcount; ++g) {
          if (g * D::SG + D::block_first(lane) >= kel) break;
          group(g);
        }
      }
    }
    __syncwarp();  // every lane is done reading this slot before lane 0 refills it
    ++consumed;
    if (++cs == a.NS) {
      cs = 0;
      ++cround;
    }

    if (last_chunk && my_rbs > 0) {
      // the 4 x TT row sums, reduce-scattered over the warp (each lane ends up owning one or
      // two of them)
      constexpr int NV = RR * TT;
      constexpr int NH = NV == 64 ? 2 : 1;
      float v[NV];
#pragma unroll
      for (int r = 0; r < RR; ++r)
#pragma unroll
        for (int t = 0; t < TT; ++t) v[r * TT + t] = (TT == 1) ? acc1[r] : acc2[r][t].x + acc2[r][t].y;
      reduce_scatter<NV>(v, lane);
      const int i0 = rs_index<NV>(lane);
      const bool own = rs_owner<NV>(lane);
      if (KW == 1) {
        // mode 1: partial sums of the row block's K chunks stay in shared memory, added in
        // chunk order; y is written once, after the last chunk
        float *pacc = part + (warp * a.maxq + cc.q) * NV;
        const bool final_chunk = (a.mode == 0) || (cc.c + 1 == a.nchunks);
#pragma unroll
        for (int h = 0; h < NH; ++h) {
          const int idx = i0 + h;
          const int r = idx / TT, t = idx - r * TT;
          float val = v[h];
          if (own && a.mode == 1) {
            if (cc.c > 0) val += pacc[idx];
            if (!final_chunk) pacc[idx] = val;
          }
          const long long row = blk.lrb * RR + r;
          if (own && final_chunk && ok && t < a.T && row < blk.M) blk.y[static_cast<long long>(t) * blk.M + row] = val;
        }
      } else {
        float *myred = red + ((cc.q & 1) * NW + warp) * NV;  // double-buffered by row block
#pragma unroll
        for (int h = 0; h < NH; ++h)
          if (own) myred[i0 + h] = v[h];
        named_bar_sync(2 + rbl, KW * 32);
        if (kw == 0) {
          const float *base = red + ((cc.q & 1) * NW + rbl * KW) * NV;
          for (int idx = lane; idx < NV; idx += 32) {
            const int r = idx / TT, t = idx - r * TT;
            float sum = 0.f;
            for (int k = 0; k < KW; ++k) sum += base[k * NV + idx];
            const long long row = blk.lrb * RR + r;
            if (ok && t < a.T && row < blk.M) blk.y[static_cast<long long>(t) * blk.M + row] = sum;
          }
        }
      }
    }
    cc = next(cc);
  }
  if (!ok) {
    if (lane == 0) set_status(QG_STATUS_BIT_TIMEOUT);
    // never leave this warp's copies in flight
    if (lane == 0)
      for (int i = consumed; i < issued; ++i) mbar_wait(&wbar[warp * kMaxNS + (i % a.NS)], (i / a.NS) & 1);
  }
}

// ------------------------------------------------------------------------------------------
// Host side
// ------------------------------------------------------------------------------------------

template <int QT, int TT, int NW, int CPS>
qg_status launch_cfg(int nmat, const void *const *w, const float *x, float *const *y, const int64_t *Ms, int64_t N,
                     int T, cudaStream_t stream) {
  using D = Dec<QT>;
  const qg::DeviceInfo &dev = qg::device_info();
  if (!dev.ok) return QG_ECUDA;
  const int ngroups = static_cast<int>((N + D::SG - 1) / D::SG);
  const long long row_bytes = N / D::QK * D::BB;
  const long long budget = (CPS == 1) ? dev.smem_optin - 4096 : dev.smem_per_sm / CPS - 4096;
  const uint32_t hdr = 1024;
  constexpr int RR = rows_per_block<TT>();
  const uint32_t red_bytes = 2 * NW * RR * TT * 4;
  const long long xres = ((static_cast<long long>(T) * ngroups * D::SG * 4 + 1023) / 1024) * 1024;

  GemvArgs a{};
  long long rblocks = 0;
  for (int j = 0; j < nmat; ++j) {
    a.w[j] = static_cast<const uint8_t *>(w[j]);
    a.y[j] = y[j];
    a.Mj[j] = static_cast<int>(Ms[j]);
    a.rb0[j] = rblocks;
    rblocks += (Ms[j] + RR - 1) / RR;
  }
  for (int j = nmat; j <= kMaxMats; ++j) a.rb0[j] = rblocks;
  a.nmat = nmat;
  const long long grid_ctas = std::min<long long>(rblocks, static_cast<long long>(CPS) * dev.sms);
  const long long rb_per_cta = (rblocks + grid_ctas - 1) / grid_ctas;
  // activations resident (mode 0) when that still leaves the warps a ring of >= 48 KB
  int mode = (xres + 48 * 1024 <= budget - hdr - red_bytes - 1024) ? 0 : 1;
  int gpc = 0, NS = 0, seg_slot = 0;
  long long stage = 0, part_bytes = 0;
  uint32_t xbuf = 0;
  // Bulk copies of 2 KB or more stream at full speed; much smaller ones are limited by the
  // copy engine's per-copy rate.  One token: stages of whole rows (one copy) when two fit in
  // a warp's share of the ring, else row segments of at least 2 KB.  Several tokens: stages
  // of ~2-6 KB with three or more slots per warp.
  const int gpc_floor = (TT == 1) ? std::min(ngroups, (2048 + D::GB - 1) / D::GB) : 1;
  auto seg_for = [&](int g) { return static_cast<int>(((static_cast<long long>(g) * D::GB + 15) & ~15LL) + 32); };
  auto plan_ring = [&](long long ring_avail) {
    const long long tmax = (TT == 1) ? 16384 : 6144;
    const long long target = std::max<long long>(2048, std::min<long long>(tmax, ring_avail / ((TT == 1 ? 2LL : 3LL) * NW)));
    const long long whole = ((RR * row_bytes + 15) & ~15LL) + 32;
    if (mode == 0 && whole <= target) {
      gpc = ngroups;
      seg_slot = 0;
      stage = whole;
    } else {
      int gmax = static_cast<int>(std::max<long long>(1, (target / RR - 32) / D::GB));
      gmax = std::max(std::min(gmax, ngroups), gpc_floor);
      const int nch = (ngroups + gmax - 1) / gmax;
      gpc = (ngroups + nch - 1) / nch;  // even chunks
      seg_slot = seg_for(gpc);
      stage = static_cast<long long>(RR) * seg_slot;
    }
    NS = static_cast<int>(std::min<long long>(kMaxNS, ring_avail / (static_cast<long long>(NW) * stage)));
  };
  if (mode == 0) {
    xbuf = static_cast<uint32_t>(xres);
    plan_ring(budget - hdr - red_bytes - xbuf - 1024);
    if (NS < 2) mode = 1;
  }
  if (mode == 1) {
    // activation chunks double-buffered: each chunk is gpc groups of every token
    const long long per_group = static_cast<long long>(T) * D::SG * 4;
    int g = static_cast<int>(std::max<long long>(1, (40 * 1024) / per_group));
    g = std::min(g, ngroups);
    // per-warp partial sums of its row blocks across chunks
    part_bytes = ((static_cast<long long>(NW) * ((rb_per_cta + NW - 1) / NW) * RR * TT * 4) + 1023) & ~1023LL;
    while (true) {
      xbuf = static_cast<uint32_t>(((per_group * g + 1023) / 1024) * 1024);
      const long long ring_avail = budget - hdr - red_bytes - 2LL * xbuf - part_bytes - 1024;
      gpc = g;
      seg_slot = seg_for(gpc);
      stage = static_cast<long long>(RR) * seg_slot;
      NS = ring_avail > 0 ? static_cast<int>(std::min<long long>(kMaxNS, ring_avail / (static_cast<long long>(NW) * stage)))
                          : 0;
      if (NS >= 3 || g == 1) break;
      g = std::max(1, g / 2);
    }
    if (NS < 2) return QG_EUNSUPPORTED;
  }
  int nchunks = (ngroups + gpc - 1) / gpc;
  // when a CTA gets fewer row blocks than warps its warps split K: make sure there are
  // enough chunks for that (but keep segments at the copy-size floor)
  if (mode == 0 && rb_per_cta < NW) {
    const int want_kw = static_cast<int>(std::min<long long>(NW, NW / std::max<long long>(1, rb_per_cta)));
    while (gpc > gpc_floor && (ngroups + gpc - 1) / gpc < want_kw) {
      gpc = std::max(gpc_floor, gpc / 2);
      seg_slot = seg_for(gpc);
      stage = static_cast<long long>(RR) * seg_slot;
    }
    nchunks = (ngroups + gpc - 1) / gpc;
    NS = static_cast<int>(std::min<long long>(kMaxNS, (budget - hdr - red_bytes - xbuf - 1024) / (static_cast<long long>(NW) * stage)));
    if (NS < 2) return QG_EUNSUPPORTED;
  }
  a.row_bytes = row_bytes;
  a.N = static_cast<int>(N);
  a.T = T;
  a.mode = mode;
  a.KC = gpc * D::SG;
  a.nchunks = nchunks;
  a.xR = (mode == 0 ? ngroups * D::SG : a.KC) / 32;
  a.rblocks = static_cast<int>(rblocks);
  a.max_kw = nchunks;
  a.NS = NS;
  a.stage_bytes = static_cast<int>(stage);
  a.seg_slot = seg_slot;
  a.xbuf_bytes = xbuf;
  int box = 8;
  for (int d = 8; d <= 256; d += 8)
    if (a.xR % d == 0) box = d;
  a.box_rows = box;
  a.off_red = hdr;
  a.off_x = (hdr + red_bytes + 1023) & ~1023u;
  a.maxq = static_cast<int>((rb_per_cta + NW - 1) / NW);
  a.off_part = a.off_x + (mode == 0 ? 1u : 2u) * xbuf;
  a.off_ring = a.off_part + static_cast<uint32_t>(part_bytes);
  const uint32_t smem = a.off_ring + static_cast<uint32_t>(NW * NS * stage) + 1024 + 64;

  // activation tensor map: [T*N/32 rows][32 f32], 128-byte swizzle, box [box][32]
  auto enc = qg::encode_fn();
  if (!enc) return QG_ECUDA;
  CUtensorMap map;
  const cuuint64_t gdim[2] = {32, static_cast<cuuint64_t>(T) * static_cast<cuuint64_t>(N / 32)};
  const cuuint64_t gstride[1] = {128};
  const cuuint32_t boxd[2] = {32, static_cast<cuuint32_t>(box)};
  const cuuint32_t estr[2] = {1, 1};
  if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(x), gdim, gstride, boxd, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return QG_ECUDA;

  auto kern = qgemv_kernel<QT, TT, NW>;
  if (!qg::set_smem_attr(reinterpret_cast<const void *>(kern), smem)) return QG_ECUDA;
  const int grid = static_cast<int>(grid_ctas);
  a.early_weights = qg::static_weights(stream) ? 1 : 0;
  if (qg::launch_pdl(kern, dim3(grid), dim3(NW * 32), smem, stream, map, a) != cudaSuccess) return QG_ECUDA;
  return cudaGetLastError() == cudaSuccess ? QG_OK : QG_ECUDA;
}

// CTA shape per launch.  One token: CTAs of 8 warps, two per SM (half the shared memory each),
// so that the next kernel's CTAs can already sit on an SM while this kernel's last CTAs drain.
// Q4_K rows whose activations would not stay resident in half an SM (above 56 KB) take one
// 16-warp CTA per SM instead, which holds them once beside a large ring (measured: 36 -> 27 us
// on 5120 x 17408; the same shape is slower for Q6_K and for the Q8_0 rows of 9728).  Several
// tokens: one 8-warp CTA per SM.
template <int QT, int TT>
qg_status launch_t(int nmat, const void *const *w, const float *x, float *const *y, const int64_t *Ms, int64_t N,
                   int T, cudaStream_t stream) {
  // several tokens: rows across lanes (qg_gemv_mt.cu) when the launch has at least two
  // 16-row groups per SM; with fewer, a CTA's single group leaves its warps short of work and
  // the lean kernel's 2-row blocks win (2560 x 4096 at T = 4: 7.9 vs 9.2 us)
  long long groups = 0;
  for (int j = 0; j < nmat; ++j) groups += (Ms[j] + 15) / 16;
  const bool mt_first = TT > 1 && groups >= 2LL * qg::device_info().sms;
  if constexpr (TT > 1) {
    if (mt_first) {
      const qg_status r0 = qg::gemv_mt_launch<QT>(nmat, w, x, y, Ms, N, T, stream);
      if (r0 != QG_EUNSUPPORTED) return r0;
    }
  }
  const qg_status r = qg::gemv1_launch<QT>(nmat, w, x, y, Ms, N, T, stream);
  if (r != QG_EUNSUPPORTED) return r;
  if constexpr (TT > 1) {
    // activations too long to stay resident in one CTA: K split over a cluster
    if (!mt_first) {
      const qg_status r2 = qg::gemv_mt_launch<QT>(nmat, w, x, y, Ms, N, T, stream);
      if (r2 != QG_EUNSUPPORTED) return r2;
    }
  }
  if constexpr (TT == 1) {
    if constexpr (QT == QG_TYPE_Q4_K) {
      using D = Dec<QT>;
      const long long xres = (N + D::SG - 1) / D::SG * D::SG * 4;
      if (xres > 56 * 1024) return launch_cfg<QT, 1, 16, 1>(nmat, w, x, y, Ms, N, T, stream);
    }
    return launch_cfg<QT, 1, 8, 2>(nmat, w, x, y, Ms, N, T, stream);
  } else {
    return launch_cfg<QT, TT, 8, 1>(nmat, w, x, y, Ms, N, T, stream);
  }
}

template <int QT>
qg_status launch_type(int n, const void *const *w, const float *x, float *const *y, const int64_t *M, int64_t N, int T,
                      cudaStream_t s) {
  if (T == 1) return launch_t<QT, 1>(n, w, x, y, M, N, T, s);
  if (T <= 2) return launch_t<QT, 2>(n, w, x, y, M, N, T, s);
  if (T <= 4) return launch_t<QT, 4>(n, w, x, y, M, N, T, s);
  if (T <= 8) return launch_t<QT, 8>(n, w, x, y, M, N, T, s);
  return launch_t<QT, 16>(n, w, x, y, M, N, T, s);
}

}  // namespace

namespace qg {

qg_status gemv_multi_dispatch(int type, int n, const void *const *w, const float *x, float *const *y,
                              const int64_t *M, int64_t N, int T, cudaStream_t s) {
  int qk = 0, bb = 0;
  if (qg_block_shape(type, &qk, &bb) != QG_OK) return QG_EUNSUPPORTED;
  if (n < 1 || n > kMaxMats) return QG_EINVAL_SHAPE;
  if (!w || !y || !M || !x) return QG_EINVAL_PTR;
  if (N <= 0 || N % qk || T < 1 || T > 16 || N > INT32_MAX) return QG_EINVAL_SHAPE;
  if (static_cast<long long>(T) * N > INT32_MAX) return QG_EINVAL_SHAPE;
  if (!aligned16(x)) return QG_EALIGN;
  // matrices with no rows are dropped; the rest keep their order
  const void *ww[kMaxMats];
  float *yy[kMaxMats];
  int64_t mm[kMaxMats];
  int k = 0;
  long long rows = 0;
  for (int j = 0; j < n; ++j) {
    if (M[j] < 0 || M[j] > INT32_MAX) return QG_EINVAL_SHAPE;
    if (M[j] == 0) continue;
    if (!w[j] || !y[j]) return QG_EINVAL_PTR;
    if (!aligned16(w[j]) || !aligned16(y[j])) return QG_EALIGN;
    ww[k] = w[j];
    yy[k] = y[j];
    mm[k] = M[j];
    rows += M[j];
    ++k;
  }
  if (k == 0) return QG_OK;
  if (rows > INT32_MAX) return QG_EINVAL_SHAPE;
  switch (type) {
    case QG_TYPE_Q8_0: return launch_type<QG_TYPE_Q8_0>(k, ww, x, yy, mm, N, T, s);
    case QG_TYPE_Q4_0: return launch_type<QG_TYPE_Q4_0>(k, ww, x, yy, mm, N, T, s);
    case QG_TYPE_Q4_K: return launch_type<QG_TYPE_Q4_K>(k, ww, x, yy, mm, N, T, s);
    case QG_TYPE_Q6_K: return launch_type<QG_TYPE_Q6_K>(k, ww, x, yy, mm, N, T, s);
    default: return QG_EUNSUPPORTED;
  }
}

qg_status gemv_dispatch(int type, const void *w, const float *x, float *y, int64_t M, int64_t N, int T,
                        cudaStream_t s) {
  int qk = 0, bb = 0;
  if (qg_block_shape(type, &qk, &bb) != QG_OK) return QG_EUNSUPPORTED;
  if (!w || !x || !y) return QG_EINVAL_PTR;
  if (M < 0 || N <= 0 || N % qk || T < 1 || T > 16 || M > INT32_MAX || N > INT32_MAX) return QG_EINVAL_SHAPE;
  if (static_cast<long long>(T) * N > INT32_MAX) return QG_EINVAL_SHAPE;
  if (!aligned16(w) || !aligned16(x) || !aligned16(y)) return QG_EALIGN;
  if (M == 0) return QG_OK;
  return gemv_multi_dispatch(type, 1, &w, x, &y, &M, N, T, s);
}

unsigned int read_status_gemv(bool clear) {
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_qg_status_gemv, sizeof(v)) != cudaSuccess) return 0xFFFFFFFFu;
  if (clear) {
    const unsigned int z = 0;
    cudaMemcpyToSymbol(g_qg_status_gemv, &z, sizeof(z));
  }
  return v;
}

}  // namespace qg

extern "C" {

qg_status qgemv_q8_0(const void *w, const float *x, float *y, int64_t M, int64_t N, qg_stream_t s) {
  return qg::gemv_dispatch(QG_TYPE_Q8_0, w, x, y, M, N, 1, reinterpret_cast<cudaStream_t>(s));
}
qg_status qgemv_q4_0(const void *w, const float *x, float *y, int64_t M, int64_t N, qg_stream_t s) {
  return qg::gemv_dispatch(QG_TYPE_Q4_0, w, x, y, M, N, 1, reinterpret_cast<cudaStream_t>(s));
}
qg_status qgemv_q4_k(const void *w, const float *x, float *y, int64_t M, int64_t N, qg_stream_t s) {
  return qg::gemv_dispatch(QG_TYPE_Q4_K, w, x, y, M, N, 1, reinterpret_cast<cudaStream_t>(s));
}
qg_status qgemv_q6_k(const void *w, const float *x, float *y, int64_t M, int64_t N, qg_stream_t s) {
  return qg::gemv_dispatch(QG_TYPE_Q6_K, w, x, y, M, N, 1, reinterpret_cast<cudaStream_t>(s));
}
qg_status qgemv_t(int type, const void *w, const float *x, float *y, int64_t M, int64_t N, int T, qg_stream_t s) {
  return qg::gemv_dispatch(type, w, x, y, M, N, T, reinterpret_cast<cudaStream_t>(s));
}
qg_status qgemv_multi(int type, int n, const void *const *w, float *const *y, const int64_t *M, int64_t N,
                      const float *x, int T, qg_stream_t s) {
  return qg::gemv_multi_dispatch(type, n, w, x, y, M, N, T, reinterpret_cast<cudaStream_t>(s));
}

}  // extern "C"
