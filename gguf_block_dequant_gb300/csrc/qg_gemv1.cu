// qg_gemv1.cu -- one-token quantized GEMV (T = 1), the lean pipeline for the shapes that
// dominate a decode step: row blocks whose byte length is a multiple of 16 (every row block
// then starts on a 16-byte boundary; rows of Q6_K's 210-byte blocks start 2-byte aligned inside
// them) and activations that stay resident in shared memory.
//
// y[m] = sum_k W[m][k] * x[k]  (matmulQ8 / matmulQ4 / the Q4_K row dot of WG_GEMM_Q4K on the
// engine pages), raw GGUF blocks decoded in registers, f32 accumulation.
//
// Work mapping: persistent CTAs with a balanced contiguous range of RR-row blocks each; a row
// block is cut into K chunks when its rows do not fit a stage (or to give every warp work), and
// the CTA's (row block, chunk) items are dealt to its warps in contiguous ranges equal to
// within one item, so that no warp streams more than its share when the CTA's row blocks do
// not divide among its warps.  Every warp streams its items through a private ring of
// shared-memory slots with bulk copies and decodes them with the lane decoders of
// qg_decode.cuh (two lanes per block, sixteen blocks per 512-element group); a row block whose
// chunks span two warps' ranges is summed from their parts in shared memory, in chunk order.
// What is specialised away, because it cost instruction issue in every stage:
//   - 32-bit row and byte offsets (every matrix < 4 GiB), matrix bounds precomputed;
//   - a stage of whole rows is one copy issued by lane 0 alone (rows are contiguous);
//   - no tail handling of unaligned row blocks (they start 16-byte aligned by construction);
//   - the item cursor is two counters, the ring slot and phase are counters too.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "qg_decode.cuh"
#include "qg_host.h"
#include "qg_pipe.cuh"

__device__ unsigned int g_qg_status_gemv1;  // this translation unit's device status word

namespace {

constexpr int kNS = 4;    // most slots per warp
constexpr int kMats = 4;  // matrices per launch (sharing x)

struct G1Args {
  const uint8_t *w[kMats];
  float *y[kMats];
  uint32_t rb0[kMats + 1];  // matrix j owns row blocks [rb0[j], rb0[j + 1])
  uint32_t M[kMats];
  int nmat;
  uint32_t row_bytes;    // multiple of 16
  uint32_t rblocks;      // row blocks of the launch
  int nchunks;           // K chunks per row (1: a stage holds the block's whole rows)
  int gpc;               // full groups per chunk
  int gtail;             // groups of the last chunk (the last one may be partial)
  int last_full;         // the last chunk's groups are all full (N % SG == 0)
  uint32_t chunk_bytes;  // bytes of one row's chunk (all chunks but the last)
  uint32_t seg;          // slot bytes per row of a chunked stage
  uint32_t stage_bytes;  // bytes per slot
  int NS;
  int N;
  int T;                 // token columns (<= TT of the kernel)
  uint32_t xtok;         // shared-memory bytes of one token's activations
  int xR, box_rows;
  uint32_t off_x, off_red, off_ring;
  int early_weights;
  int unal;                  // rows not 16-byte multiples, in chunks: each row's chunk is copied
                             // from the 16-byte boundary below it and read at its own offset
  uintptr_t mend[kMats];     // unal: last 16-byte boundary inside each matrix
};

QG_DEVICE void g1_status(unsigned int bits) { atomicOr(&g_qg_status_gemv1, bits); }

// QT block type, NW warps per CTA, CPS CTAs per SM, RR rows per row block, GU groups per
// chunk when known at compile time (0: a runtime loop), TT token columns (a.T <= TT of them
// are used).  With GU the group loop is unrolled: every group's shared-memory offsets become
// immediates of the loads.  One token takes the fused dot (Dec::dot1); several tokens decode
// each weight once and multiply it into every token column.
template <int QT, int NW, int CPS, int RR, int GU, int TT, bool XREG = false>
__global__ void __launch_bounds__(NW * 32, CPS) qgemv1_kernel(const __grid_constant__ CUtensorMap xmap, const G1Args a) {
  using D = Dec<QT>;
  constexpr bool kUnal = QT == QG_TYPE_Q6_K;  // the only type whose chunked rows may start unaligned
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t *wbar = reinterpret_cast<uint64_t *>(smem);  // [NW][kNS]
  uint64_t *xfull = wbar + NW * kNS;
  float *red = reinterpret_cast<float *>(smem + a.off_red);  // [2 NW][RR * TT] parts of split row blocks
  uint8_t *xs = smem + a.off_x;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t G = gridDim.x;
  const uint32_t rbA = static_cast<uint32_t>(static_cast<unsigned long long>(blockIdx.x) * a.rblocks / G);
  const uint32_t rbB = static_cast<uint32_t>(static_cast<unsigned long long>(blockIdx.x + 1) * a.rblocks / G);
  const int nrb = static_cast<int>(rbB - rbA);
  const int nc = a.nchunks;
  // The CTA's items are its (row block, chunk) pairs in row-block-major order.  Whole rows
  // (nc == 1): warp w takes row blocks w, w + NW, ... (the CTA streams neighbouring blocks at
  // any time).  Chunked rows: the first NWa warps take contiguous ranges of items, equal to
  // within one item, every range non-empty.
  const int n_items = nrb * nc;
  const int NWa = max(1, min(NW, n_items));
  auto kb = [&](int w) { return w * n_items / NWa; };
  const int k0 = nc == 1 ? warp : (warp < NWa ? kb(warp) : 0);
  const int items = nc == 1 ? (warp < n_items ? (n_items - warp + NW - 1) / NW : 0) : (warp < NWa ? kb(warp + 1) - k0 : 0);
  const int istep = nc == 1 ? NW : 1;  // row blocks from one whole-row item to the next

  if (threadIdx.x == 0) {
    for (int i = 0; i < NW * kNS; ++i) mbar_init(&wbar[i], 1);
    mbar_init(xfull, 1);
    fence_mbar_init();
  }
  __syncthreads();

  uint64_t *mybar = wbar + warp * kNS;
  const uint32_t ring_s = smem_u32(smem + a.off_ring) + static_cast<uint32_t>(warp * a.NS) * a.stage_bytes;
  uint8_t *ring = smem + a.off_ring + static_cast<uint32_t>(warp * a.NS) * a.stage_bytes;

  // matrix of row block rb: j and the block's first row within the matrix
  auto locate = [&](uint32_t rb, int &j, uint32_t &row) {
    j = 0;
#pragma unroll
    for (int q = 1; q < kMats; ++q)
      if (q < a.nmat && rb >= a.rb0[q]) j = q;
    row = (rb - a.rb0[j]) * RR;
  };

  // issue chunk c of the CTA's row block i into slot s
  auto issue = [&](int i, int c, int s) {
    const uint32_t rb = rbA + static_cast<uint32_t>(i);
    int j;
    uint32_t row;
    locate(rb, j, row);
    const uint32_t nr = min(static_cast<uint32_t>(RR), a.M[j] - row);
    const uint8_t *src = a.w[j] + row * a.row_bytes;
    if (nc == 1) {
      if (lane == 0) {
        const uint32_t bytes = nr * a.row_bytes;
        mbar_arrive_expect_tx(&mybar[s], bytes);
        bulk_g2s<true>(ring + s * a.stage_bytes, src, bytes, &mybar[s]);
      }
    } else {
      const uint32_t cb = (c == nc - 1) ? a.row_bytes - static_cast<uint32_t>(c) * a.chunk_bytes : a.chunk_bytes;
      if (kUnal && a.unal) {
        const uintptr_t sl = reinterpret_cast<uintptr_t>(src) + lane * a.row_bytes + static_cast<uint32_t>(c) * a.chunk_bytes;
        warp_bulk_copies<true>(ring + s * a.stage_bytes + lane * a.seg, sl, static_cast<uint32_t>(lane) < nr ? cb : 0u,
                               a.mend[j], &mybar[s], lane);
      } else {
        if (lane == 0) mbar_arrive_expect_tx(&mybar[s], nr * cb);
        __syncwarp();
        if (static_cast<uint32_t>(lane) < nr)
          bulk_g2s<true>(ring + s * a.stage_bytes + lane * a.seg, src + lane * a.row_bytes + static_cast<uint32_t>(c) * a.chunk_bytes,
                   cb, &mybar[s]);
      }
    }
  };

  // prologue: the first NS - 1 items.  With static weights the first item of every warp is
  // requested before the wait on the predecessor and the rest after the activations' copy
  // (more weight requests in flight at the wait only delay the activations).
  int ii = k0 / nc, ic = k0 - (k0 / nc) * nc, is = 0, issued = 0;
  auto advance_issue = [&]() {
    if (++ic == nc) {
      ic = 0;
      ii += istep;
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
  if (a.early_weights) prologue(1);
  pdl_wait();
  pdl_launch_dependents();
  if (threadIdx.x == 0) load_x(xs, &xmap, a.T, a.N, 0, a.xR, a.box_rows, xfull);
  prologue(a.NS - 1);

  const uint32_t wo = static_cast<uint32_t>(D::woff(lane));
  const uint32_t xs_s = smem_u32(xs);
  uint32_t xo[D::NCH];
#pragma unroll
  for (int ch = 0; ch < D::NCH; ++ch) xo[ch] = x_lane_off<QT>(lane, ch);
  const int bfirst = D::block_first(lane);

  bool ok = mbar_wait(xfull, 0);
  // XREG (one token, whole rows of GU groups): a lane multiplies the same activations in every
  // row, so they are read from shared memory once and kept in registers
  float4 xr[XREG ? GU : 1][D::NCH];
  if constexpr (XREG) {
#pragma unroll
    for (int g = 0; g < GU; ++g)
#pragma unroll
      for (int ch = 0; ch < D::NCH; ++ch) xr[g][ch] = lds_f4(xs_s + static_cast<uint32_t>(g * (D::SG * 4)) + xo[ch]);
  }
  constexpr int NV = RR * TT;
  float acc[RR];
  f2 acc2[RR][TT];
  int i = k0 / nc, c = k0 - (k0 / nc) * nc, cs = 0, done = 0;  // the compute cursor
  int c_first = c;  // first chunk of the current segment (the items of one row block in a row)
  uint32_t phase = 0;
  for (int it = 0; it < items; ++it) {
    if (ok && issued < items) {
      issue(ii, ic, is);
      advance_issue();
    }
    if (c == 0 || it == 0) {
      c_first = c;
#pragma unroll
      for (int r = 0; r < RR; ++r) {
        acc[r] = 0.f;
#pragma unroll
        for (int t = 0; t < TT; ++t) acc2[r][t] = mk2(0.f, 0.f);
      }
    }
    if (ok && !mbar_wait(&mybar[cs], phase)) ok = false;
    if (ok) {
      ++done;
      const uint32_t st = ring_s + static_cast<uint32_t>(cs) * a.stage_bytes + wo;
      const uint32_t pitch = (nc == 1) ? a.row_bytes : a.seg;
      uint32_t ro[RR];  // each row's offset from the 16-byte boundary its chunk was copied from
#pragma unroll
      for (int r = 0; r < RR; ++r) ro[r] = 0u;
      if (kUnal && a.unal) {
        int j;
        uint32_t row;
        locate(rbA + static_cast<uint32_t>(i), j, row);
        const uintptr_t b0 = reinterpret_cast<uintptr_t>(a.w[j]);
#pragma unroll
        for (int r = 0; r < RR; ++r) ro[r] = static_cast<uint32_t>((b0 + (row + r) * static_cast<uintptr_t>(a.row_bytes)) & 15u);
      }
      RowPrep<QT> rp[RR];
#pragma unroll
      for (int r = 0; r < RR; ++r) rp[r].init(st + static_cast<uint32_t>(r) * pitch + ro[r], lane);
      const uint32_t xg0 = xs_s + static_cast<uint32_t>(c * a.gpc) * (D::SG * 4);
      auto group = [&](int g) {
        const uint32_t goff = static_cast<uint32_t>(g * D::GB);
        const uint32_t xg = xg0 + static_cast<uint32_t>(g * (D::SG * 4));
        typename D::U u[RR];
        if constexpr (TT == 1) {
          float4 xc[D::NCH];
#pragma unroll
          for (int ch = 0; ch < D::NCH; ++ch) xc[ch] = XREG ? xr[XREG ? g : 0][ch] : lds_f4(xg + xo[ch]);
          const float aux = D::xaux(xc);
#pragma unroll
          for (int r = 0; r < RR; ++r) u[r] = rp[r].load(goff, lane);
#pragma unroll
          for (int r = 0; r < RR; ++r) acc[r] += D::dot1(u[r], xc, aux);
        } else {
#pragma unroll
          for (int r = 0; r < RR; ++r) u[r] = rp[r].load(goff, lane);
#pragma unroll
          for (int ch = 0; ch < D::NCH; ++ch) {
            f2 w01[RR], w23[RR];
#pragma unroll
            for (int r = 0; r < RR; ++r) D::weights(u[r], ch, w01[r], w23[r]);
#pragma unroll
            for (int t = 0; t < TT; ++t) {
              if (t < a.T) {
                const float4 xv = lds_f4(xg + static_cast<uint32_t>(t) * a.xtok + xo[ch]);
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
      if constexpr (GU > 0) {
        // a chunk has GU groups, the last one gtail (<= GU); a partial group only at the end
        const int gl = (c < nc - 1) ? GU : (a.last_full ? a.gtail : a.gtail - 1);
#pragma unroll
        for (int g = 0; g < GU; ++g)
          if (g < gl) group(g);
        if (c == nc - 1 && !a.last_full && gl * D::SG + bfirst < a.N - c * a.gpc * D::SG) {
          if constexpr (XREG) {
            // xr is indexed by constants only, or it would live in local memory
#pragma unroll
            for (int g = 0; g < GU; ++g)
              if (g == gl) group(g);
          } else {
            group(gl);
          }
        }
      } else if (c < nc - 1) {
        for (int g = 0; g < a.gpc; ++g) group(g);
      } else {
        const int gl = a.last_full ? a.gtail : a.gtail - 1;
        for (int g = 0; g < gl; ++g) group(g);
        if (!a.last_full && gl * D::SG + bfirst < a.N - c * a.gpc * D::SG) group(gl);
      }
    }
    __syncwarp();  // every lane is done reading this slot before lane 0 refills it
    if (++cs == a.NS) {
      cs = 0;
      phase ^= 1u;
    }
    if (c == nc - 1 || it == items - 1) {
      // end of a segment (this warp's items of row block i): the RR x TT sums (row r, token t
      // at r * TT + t), reduce-scattered over the warp so that each lane owns one of them (two
      // when there are 64).  A whole row block goes to y; a part of one split between warps
      // goes to its slot of red: the part that starts at chunk 0 to slot 2 (w + 1), w its
      // warp, the part that starts at a later chunk (at its warp's first item) to slot 2 w + 1.
      constexpr int NH = NV == 64 ? 2 : 1;
      static_assert(NV <= 64, "at most two sums per lane");
      float v[NV];
#pragma unroll
      for (int r = 0; r < RR; ++r)
#pragma unroll
        for (int t = 0; t < TT; ++t) v[r * TT + t] = (TT == 1) ? acc[r] : acc2[r][t].x + acc2[r][t].y;
      reduce_scatter<NV>(v, lane);
      const int i0 = rs_index<NV>(lane);
      const bool own = rs_owner<NV>(lane);
      if (c_first == 0 && c == nc - 1) {
        int j;
        uint32_t row;
        locate(rbA + static_cast<uint32_t>(i), j, row);
        const uint32_t M = a.M[j];
#pragma unroll
        for (int h = 0; h < NH; ++h) {
          const int r0 = (i0 + h) / TT, t0 = (i0 + h) - r0 * TT;
          if (own && ok && t0 < a.T && row + r0 < M) a.y[j][static_cast<size_t>(t0) * M + row + r0] = v[h];
        }
      } else {
        float *slot = red + (c_first == 0 ? 2 * (warp + 1) : 2 * warp + 1) * NV;
#pragma unroll
        for (int h = 0; h < NH; ++h)
          if (own) slot[i0 + h] = v[h];
      }
    }
    if (++c == nc) {
      c = 0;
      i += istep;
    }
  }
  if (nc > 1) {
    // row blocks split between warps: warp w, the first boundary inside such a block, sums its
    // parts in chunk order (deterministic) and writes y
    __syncthreads();
    if (warp >= 1 && warp < NWa) {
      const int b = kb(warp);
      const int rbl = b / nc, lo = rbl * nc;
      if (b != lo && kb(warp - 1) <= lo) {
        int j;
        uint32_t row;
        locate(rbA + static_cast<uint32_t>(rbl), j, row);
        const uint32_t M = a.M[j];
        for (int idx = lane; idx < NV; idx += 32) {
          float sum = red[2 * warp * NV + idx];
          for (int w = warp; w < NWa && kb(w) < lo + nc; ++w) sum += red[(2 * w + 1) * NV + idx];
          const int rr = idx / TT, tt = idx - rr * TT;
          if (ok && tt < a.T && row + rr < M) a.y[j][static_cast<size_t>(tt) * M + row + rr] = sum;
        }
      }
    }
  }
  if (!ok) {
    if (lane == 0) g1_status(QG_STATUS_BIT_TIMEOUT);
    // never leave this warp's copies in flight
    if (lane == 0)
      for (int k = done; k < issued; ++k) mbar_wait(&mybar[k % a.NS], (k / a.NS) & 1);
  }
}

}  // namespace

namespace qg {

struct G1Plan {
  G1Args a;
  CUtensorMap map;
  unsigned grid;
  uint32_t smem;
};

// Plans the lean one-token kernel in one CTA shape; QG_EUNSUPPORTED when the shape is outside
// its scope (the caller then takes the general kernel).  Enqueues nothing.
template <int QT, int NW, int CPS, int RR, int TT>
qg_status gemv1_plan(int nmat, const void *const *w, const float *x, float *const *y, const int64_t *Ms, int64_t N,
                     int T, cudaStream_t stream, G1Plan &P) {
  using D = Dec<QT>;
  const DeviceInfo &dev = device_info();
  if (!dev.ok) return QG_ECUDA;
  const long long row_bytes = N / D::QK * D::BB;
  // rows of a 16-byte multiple, or (Q6_K's 210-byte blocks) row blocks of one: then every
  // stage holds whole row blocks (one copy from a 16-byte boundary) and every matrix has whole
  // row blocks, and the decoders read each row at its own 2-byte alignment
  const bool rows16 = row_bytes % 16 == 0;
  const int ngroups = static_cast<int>((N + D::SG - 1) / D::SG);
  const long long xtok = static_cast<long long>(ngroups) * D::SG * 4;
  const long long xres = ((static_cast<long long>(T) * xtok + 1023) / 1024) * 1024;
  const long long budget = (CPS == 1 ? dev.smem_optin : dev.smem_per_sm / CPS) - 4096;
  const uint32_t hdr = 1024;
  const uint32_t red_bytes = 2 * NW * RR * TT * 4;  // two part slots per warp
  G1Args a{};
  unsigned long long rblocks = 0;
  for (int j = 0; j < nmat; ++j) {
    if (static_cast<unsigned long long>(Ms[j]) * row_bytes >= (1ull << 32)) return QG_EUNSUPPORTED;
    a.w[j] = static_cast<const uint8_t *>(w[j]);
    a.y[j] = y[j];
    a.M[j] = static_cast<uint32_t>(Ms[j]);
    a.rb0[j] = static_cast<uint32_t>(rblocks);
    rblocks += (Ms[j] + RR - 1) / RR;
  }
  if (rblocks >= (1ull << 31)) return QG_EUNSUPPORTED;
  for (int j = nmat; j <= kMats; ++j) a.rb0[j] = static_cast<uint32_t>(rblocks);
  a.nmat = nmat;
  const long long ring_avail = budget - hdr - red_bytes - 1024 - xres - 1024;
  if (ring_avail < 2LL * NW * 2048) return QG_EUNSUPPORTED;  // activations too long to stay resident
  const long long grid = std::min<long long>(static_cast<long long>(rblocks), static_cast<long long>(CPS) * dev.sms);
  const long long rb_per_cta = (static_cast<long long>(rblocks) + grid - 1) / grid;
  // Whole rows per stage when two such stages per warp fit (one copy each); otherwise chunks
  // of whole groups, at least 2 KB per row, each chunk a multiple of 16 bytes.
  const long long whole = RR * row_bytes;
  int gpc, nchunks, NS;
  long long stage, seg = 0;
  if (2LL * NW * whole <= ring_avail) {
    gpc = ngroups;
    nchunks = 1;
    stage = whole;
  } else {
    const long long target = std::max<long long>(2048, std::min<long long>(16384, ring_avail / (2LL * NW)));
    int gmax = static_cast<int>(std::max<long long>(1, (target / RR) / D::GB));
    const int floor_g = std::min(ngroups, (2048 + D::GB - 1) / D::GB);
    gmax = std::max(std::min(gmax, ngroups), floor_g);
    int nch = (ngroups + gmax - 1) / gmax;
    gpc = (ngroups + nch - 1) / nch;
    while ((static_cast<long long>(gpc) * D::GB) % 16) ++gpc;  // chunks stay 16-byte multiples
    nchunks = (ngroups + gpc - 1) / gpc;
    seg = static_cast<long long>(gpc) * D::GB;
    stage = RR * seg;
  }
  // when the CTAs have fewer row blocks than warps, cut the rows into chunks so that every
  // warp gets items
  if (rb_per_cta < NW) {
    const int want_kw = static_cast<int>(std::min<long long>(NW, (NW + rb_per_cta - 1) / std::max<long long>(1, rb_per_cta)));
    const int floor_g = std::min(ngroups, (2048 + D::GB - 1) / D::GB);
    while (gpc > floor_g && (ngroups + gpc - 1) / gpc < want_kw) {
      int g2 = std::max(floor_g, gpc / 2);
      while ((static_cast<long long>(g2) * D::GB) % 16) ++g2;
      if (g2 >= gpc) break;
      gpc = g2;
    }
    nchunks = (ngroups + gpc - 1) / gpc;
    if (nchunks > 1) {
      seg = static_cast<long long>(gpc) * D::GB;
      stage = RR * seg;
    }
  }
  if (!rows16) {
    if (nchunks == 1) {
      // whole rows: one copy of each row block, which must then be a 16-byte multiple
      // (rows that do not make one take the general kernel: cutting short Q6_K rows into
      // realigned chunks made the 262144 x 2816 head 1.6x slower)
      if ((RR * row_bytes) % 16 != 0) return QG_EUNSUPPORTED;
      for (int j = 0; j < nmat; ++j)
        if (Ms[j] % RR != 0) return QG_EUNSUPPORTED;
    } else {
      // chunks of rows that start anywhere (Q6_K): 16 bytes of slack per row segment, chunks
      // kept 16-byte multiples, made smaller until two stages per warp fit
      if (QT != QG_TYPE_Q6_K) return QG_EUNSUPPORTED;
      a.unal = 1;
      auto fits = [&]() { return ring_avail / (static_cast<long long>(NW) * RR * (static_cast<long long>(gpc) * D::GB + 16)) >= 2; };
      while (!fits()) {
        int g2 = gpc - 1;
        while (g2 > 0 && (static_cast<long long>(g2) * D::GB) % 16) --g2;
        if (g2 < 1) return QG_EUNSUPPORTED;
        gpc = g2;
      }
      nchunks = (ngroups + gpc - 1) / gpc;
      if (nchunks < 2) return QG_EUNSUPPORTED;
      seg = static_cast<long long>(gpc) * D::GB + 16;
      stage = RR * seg;
      for (int j = 0; j < nmat; ++j)
        a.mend[j] = (reinterpret_cast<uintptr_t>(w[j]) + static_cast<uintptr_t>(Ms[j] * row_bytes)) & ~static_cast<uintptr_t>(15);
    }
  }
  NS = static_cast<int>(std::min<long long>(kNS, ring_avail / (static_cast<long long>(NW) * stage)));
  if (NS < 2) return QG_EUNSUPPORTED;
  a.row_bytes = static_cast<uint32_t>(row_bytes);
  a.rblocks = static_cast<uint32_t>(rblocks);
  a.nchunks = nchunks;
  a.gpc = gpc;
  a.gtail = ngroups - (nchunks - 1) * gpc;
  a.last_full = (N % D::SG) == 0 ? 1 : 0;
  a.chunk_bytes = static_cast<uint32_t>(static_cast<long long>(gpc) * D::GB);
  a.seg = static_cast<uint32_t>(seg);
  a.stage_bytes = static_cast<uint32_t>(stage);
  a.NS = NS;
  a.N = static_cast<int>(N);
  a.T = T;
  a.xtok = static_cast<uint32_t>(xtok);
  a.xR = ngroups * D::SG / 32;
  a.box_rows = box_rows_for(a.xR);
  a.off_red = hdr;
  a.off_x = (hdr + red_bytes + 1023) & ~1023u;
  a.off_ring = a.off_x + static_cast<uint32_t>(xres);
  const uint32_t smem = a.off_ring + static_cast<uint32_t>(NW * NS * stage) + 1024;
  if (!encode_x_map(&P.map, x, T, N, a.box_rows)) return QG_ECUDA;
  a.early_weights = static_weights(stream) ? 1 : 0;
  P.a = a;
  P.grid = static_cast<unsigned>(grid);
  P.smem = smem;
  return QG_OK;
}

template <int QT, int NW, int CPS, int RR, int GU, int TT, bool XREG = false>
qg_status gemv1_run(const G1Plan &P, cudaStream_t stream) {
  auto kern = qgemv1_kernel<QT, NW, CPS, RR, GU, TT, XREG>;
  if (!set_smem_attr(reinterpret_cast<const void *>(kern), P.smem)) return QG_ECUDA;
  if (launch_pdl(kern, dim3(P.grid), dim3(NW * 32), P.smem, stream, P.map, P.a) != cudaSuccess) return QG_ECUDA;
  return cudaGetLastError() == cudaSuccess ? QG_OK : QG_ECUDA;
}

// One CTA shape, its group loop unrolled for the chunk sizes of the common row lengths
// (2560 -> 5 groups, 4096 and 9728 -> chunks of 4, 1024 -> 2), a runtime loop otherwise.
template <int QT, int NW, int CPS, int RR, int TT, bool XREG = false>
qg_status gemv1_cfg(int nmat, const void *const *w, const float *x, float *const *y, const int64_t *Ms, int64_t N,
                    int T, cudaStream_t stream) {
  G1Plan P;
  const qg_status r = gemv1_plan<QT, NW, CPS, RR, TT>(nmat, w, x, y, Ms, N, T, stream, P);
  if (r != QG_OK) return r;
  if constexpr (TT == 1 && XREG) {
    if (P.a.nchunks != 1) return QG_EUNSUPPORTED;
    switch (P.a.gpc) {
      case 5: return gemv1_run<QT, NW, CPS, RR, 5, TT, true>(P, stream);
      case 4: return gemv1_run<QT, NW, CPS, RR, 4, TT, true>(P, stream);
      case 2: return gemv1_run<QT, NW, CPS, RR, 2, TT, true>(P, stream);
      default: return QG_EUNSUPPORTED;
    }
  } else if constexpr (TT == 1) {
    switch (P.a.gpc) {
      case 5: return gemv1_run<QT, NW, CPS, RR, 5, TT>(P, stream);
      case 4: return gemv1_run<QT, NW, CPS, RR, 4, TT>(P, stream);
      case 2: return gemv1_run<QT, NW, CPS, RR, 2, TT>(P, stream);
      default: break;
    }
  }
  return gemv1_run<QT, NW, CPS, RR, 0, TT>(P, stream);
}

// CTA shape per token count: two 8-warp CTAs per SM while the activations leave them room,
// else one 8-warp CTA per SM (more shared memory and registers per warp).  One token over a
// very tall matrix (an output head) takes one 8-warp CTA per SM with 4-row blocks and the
// activations in registers: every activation value then serves four rows and is read from
// shared memory once per launch (151936 x 2560: 75 -> 71 us); the other shapes lose with it.
template <int QT>
qg_status gemv1_launch(int nmat, const void *const *w, const float *x, float *const *y, const int64_t *Ms, int64_t N,
                       int T, cudaStream_t stream) {
  if (T == 1) {
    long long rows = 0;
    for (int j = 0; j < nmat; ++j) rows += Ms[j];
    if constexpr (Dec<QT>::QK == 32) {
      if (rows >= 65536) {
        const qg_status r = gemv1_cfg<QT, 8, 1, 4, 1, true>(nmat, w, x, y, Ms, N, T, stream);
        if (r != QG_EUNSUPPORTED) return r;
      }
    }
    if constexpr (QT == QG_TYPE_Q6_K) {
      // Q6_K rows (210-byte blocks) take one 8-warp CTA per SM: its room holds two whole 2-row
      // blocks per warp where two CTAs per SM would cut the rows into chunks (17408 x 5120:
      // 24.1 vs 25.9 us), and longer rows go in realigned chunks
      const qg_status r6 = gemv1_cfg<QT, 8, 1, 2, 1>(nmat, w, x, y, Ms, N, T, stream);
      if (r6 != QG_EUNSUPPORTED) return r6;
    }
    const qg_status r = gemv1_cfg<QT, 8, 2, 2, 1>(nmat, w, x, y, Ms, N, T, stream);
    if (r != QG_EUNSUPPORTED) return r;
    // long rows whose activations leave half an SM too small a ring: one 16-warp CTA per SM
    // holds them once beside a full ring
    return gemv1_cfg<QT, 16, 1, 2, 1>(nmat, w, x, y, Ms, N, T, stream);
  }
  // several tokens: the 32-element types (the K-quants' lane state is too large to keep TT
  // accumulators beside it; they take the general kernel)
  if constexpr (QT != QG_TYPE_Q8_0 && QT != QG_TYPE_Q4_0) {
    return QG_EUNSUPPORTED;
  } else {
    qg_status r = QG_EUNSUPPORTED;
    if (T == 2) r = gemv1_cfg<QT, 8, 2, 2, 2>(nmat, w, x, y, Ms, N, T, stream);
    else if (T <= 4) r = gemv1_cfg<QT, 8, 2, 2, 4>(nmat, w, x, y, Ms, N, T, stream);
    if (r != QG_EUNSUPPORTED || T <= 2) return r;
    if (T <= 4) return gemv1_cfg<QT, 8, 1, 2, 4>(nmat, w, x, y, Ms, N, T, stream);
    // 8 and 16 tokens: 2-row blocks (4-row blocks measured 15-20 % slower on the decode step)
    if (T <= 8) return gemv1_cfg<QT, 8, 1, 2, 8>(nmat, w, x, y, Ms, N, T, stream);
    return gemv1_cfg<QT, 8, 1, 2, 16>(nmat, w, x, y, Ms, N, T, stream);
  }
}

unsigned int read_status_gemv1(bool clear) {
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_qg_status_gemv1, sizeof(v)) != cudaSuccess) return 0xFFFFFFFFu;
  if (clear) {
    const unsigned int z = 0;
    cudaMemcpyToSymbol(g_qg_status_gemv1, &z, sizeof(z));
  }
  return v;
}

template qg_status gemv1_launch<QG_TYPE_Q8_0>(int, const void *const *, const float *, float *const *, const int64_t *,
                                              int64_t, int, cudaStream_t);
template qg_status gemv1_launch<QG_TYPE_Q4_0>(int, const void *const *, const float *, float *const *, const int64_t *,
                                              int64_t, int, cudaStream_t);
template qg_status gemv1_launch<QG_TYPE_Q4_K>(int, const void *const *, const float *, float *const *, const int64_t *,
                                              int64_t, int, cudaStream_t);
template qg_status gemv1_launch<QG_TYPE_Q6_K>(int, const void *const *, const float *, float *const *, const int64_t *,
                                              int64_t, int, cudaStream_t);

}  // namespace qg
