// qg_gemv1.cu -- one-token quantized GEMV (T = 1), the lean pipeline for the shapes that
// dominate a decode step: rows whose byte length is a multiple of 16 (every row then starts
// on a 16-byte boundary) and activations that stay resident in shared memory.
//
// y[m] = sum_k W[m][k] * x[k]  (matmulQ8 / matmulQ4 / the Q4_K row dot of WG_GEMM_Q4K on the
// engine pages), raw GGUF blocks decoded in registers, f32 accumulation.
//
// Same work mapping as the general kernel (qg_gemv.cu): persistent CTAs with a balanced
// contiguous range of RR-row blocks each; every warp streams its own row blocks through a
// private ring of shared-memory slots with bulk copies and decodes them with the lane decoders
// of qg_decode.cuh (two lanes per block, sixteen blocks per 512-element group); when a CTA
// has fewer row blocks than warps, KW warps split each row block's K chunks and meet at a
// named barrier.  What is specialised away, because it cost instruction issue in every stage:
//   - 32-bit row and byte offsets (every matrix < 4 GiB), matrix bounds precomputed;
//   - a stage of whole rows is one copy issued by lane 0 alone (rows are contiguous);
//   - no tail handling of unaligned rows (rows start 16-byte aligned by construction);
//   - the item cursor is two counters, the ring slot and phase are counters too.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "qg_decode.cuh"
#include "qg_host.h"
#include "qg_pipe.cuh"

extern __device__ unsigned int g_qg_status_gemv;

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
  int max_kw;
  int N;
  int xR, box_rows;
  uint32_t off_x, off_red, off_ring;
  int early_weights;
};

QG_DEVICE void g1_status(unsigned int bits) { atomicOr(&g_qg_status_gemv, bits); }

// QT block type, NW warps per CTA, CPS CTAs per SM, RR rows per row block
template <int QT, int NW, int CPS, int RR>
__global__ void __launch_bounds__(NW * 32, CPS) qgemv1_kernel(const __grid_constant__ CUtensorMap xmap, const G1Args a) {
  using D = Dec<QT>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t *wbar = reinterpret_cast<uint64_t *>(smem);  // [NW][kNS]
  uint64_t *xfull = wbar + NW * kNS;
  float *red = reinterpret_cast<float *>(smem + a.off_red);  // [NW][RR] (K-split partial sums)
  uint8_t *xs = smem + a.off_x;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t G = gridDim.x;
  const uint32_t rbA = static_cast<uint32_t>(static_cast<unsigned long long>(blockIdx.x) * a.rblocks / G);
  const uint32_t rbB = static_cast<uint32_t>(static_cast<unsigned long long>(blockIdx.x + 1) * a.rblocks / G);
  const int nrb = static_cast<int>(rbB - rbA);
  int KW = 1;
  if (nrb < NW) KW = max(1, min(NW / max(nrb, 1), a.max_kw));
  const int kw = warp % KW, rbl = warp / KW;
  const int lanes_rb = NW / KW;  // row-block lanes of the CTA
  const int my_n = (rbl < lanes_rb && rbl < nrb) ? (nrb - rbl + lanes_rb - 1) / lanes_rb : 0;
  const int nc = a.nchunks;
  const int my_c = (nc - kw + KW - 1) / KW;  // chunks kw, kw + KW, ... of each row block
  const int items = my_n * my_c;

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

  // issue item (i, ci) -- the i-th row block of this warp, its ci-th chunk -- into slot s
  auto issue = [&](int i, int ci, int s) {
    const uint32_t rb = rbA + static_cast<uint32_t>(rbl + i * lanes_rb);
    int j;
    uint32_t row;
    locate(rb, j, row);
    const uint32_t nr = min(static_cast<uint32_t>(RR), a.M[j] - row);
    const uint8_t *src = a.w[j] + row * a.row_bytes;
    if (nc == 1) {
      if (lane == 0) {
        const uint32_t bytes = nr * a.row_bytes;
        mbar_arrive_expect_tx(&mybar[s], bytes);
        bulk_g2s(ring + s * a.stage_bytes, src, bytes, &mybar[s]);
      }
    } else {
      const int c = kw + ci * KW;
      const uint32_t cb = (c == nc - 1) ? a.row_bytes - static_cast<uint32_t>(c) * a.chunk_bytes : a.chunk_bytes;
      if (lane == 0) mbar_arrive_expect_tx(&mybar[s], nr * cb);
      __syncwarp();
      if (static_cast<uint32_t>(lane) < nr)
        bulk_g2s(ring + s * a.stage_bytes + lane * a.seg, src + lane * a.row_bytes + static_cast<uint32_t>(c) * a.chunk_bytes,
                 cb, &mybar[s]);
    }
  };

  // prologue: the first NS - 1 items (before the wait on the predecessor with static weights)
  int ii = 0, ic = 0, is = 0, issued = 0;
  auto advance_issue = [&]() {
    if (++ic == my_c) {
      ic = 0;
      ++ii;
    }
    is = (is + 1 == a.NS) ? 0 : is + 1;
    ++issued;
  };
  auto prologue = [&]() {
    for (int k = 0; k < a.NS - 1 && issued < items; ++k) {
      issue(ii, ic, is);
      advance_issue();
    }
  };
  if (a.early_weights) prologue();
  pdl_wait();
  pdl_launch_dependents();
  if (threadIdx.x == 0) load_x(xs, &xmap, 1, a.N, 0, a.xR, a.box_rows, xfull);
  if (!a.early_weights) prologue();

  const uint32_t wo = static_cast<uint32_t>(D::woff(lane));
  const uint32_t xs_s = smem_u32(xs);
  uint32_t xo[D::NCH];
#pragma unroll
  for (int ch = 0; ch < D::NCH; ++ch) xo[ch] = x_lane_off<QT>(lane, ch);
  const int bfirst = D::block_first(lane);

  bool ok = mbar_wait(xfull, 0);
  float acc[RR];
  int ci = 0, i = 0, cs = 0, done = 0;
  uint32_t phase = 0;
  for (int t = 0; t < items; ++t) {
    if (ok && issued < items) {
      issue(ii, ic, is);
      advance_issue();
    }
    const int c = kw + ci * KW;
    if (ci == 0) {
#pragma unroll
      for (int r = 0; r < RR; ++r) acc[r] = 0.f;
    }
    if (ok && !mbar_wait(&mybar[cs], phase)) ok = false;
    if (ok) {
      ++done;
      const uint32_t st = ring_s + static_cast<uint32_t>(cs) * a.stage_bytes + wo;
      const uint32_t pitch = (nc == 1) ? a.row_bytes : a.seg;
      RowPrep<QT> rp[RR];
#pragma unroll
      for (int r = 0; r < RR; ++r) rp[r].init(st + static_cast<uint32_t>(r) * pitch, lane);
      const uint32_t xg0 = xs_s + static_cast<uint32_t>(c * a.gpc) * (D::SG * 4);
      auto group = [&](int g) {
        const uint32_t goff = static_cast<uint32_t>(g * D::GB);
        const uint32_t xg = xg0 + static_cast<uint32_t>(g * (D::SG * 4));
        float4 xc[D::NCH];
#pragma unroll
        for (int ch = 0; ch < D::NCH; ++ch) xc[ch] = lds_f4(xg + xo[ch]);
        const float aux = D::xaux(xc);
        typename D::U u[RR];
#pragma unroll
        for (int r = 0; r < RR; ++r) u[r] = rp[r].load(goff, lane);
#pragma unroll
        for (int r = 0; r < RR; ++r) acc[r] += D::dot1(u[r], xc, aux);
      };
      if (c < nc - 1) {
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
    if (++ci == my_c) {
      // row block done: the RR row sums, reduce-scattered over the warp
      float v[RR];
#pragma unroll
      for (int r = 0; r < RR; ++r) v[r] = acc[r];
      reduce_scatter<RR>(v, lane);
      const int r0 = rs_index<RR>(lane);
      const bool own = rs_owner<RR>(lane);
      const uint32_t rb = rbA + static_cast<uint32_t>(rbl + i * lanes_rb);
      int j;
      uint32_t row;
      locate(rb, j, row);
      if (KW == 1) {
        if (own && ok && row + r0 < a.M[j]) a.y[j][row + r0] = v[0];
      } else {
        float *myred = red + warp * RR;
        if (own) myred[r0] = v[0];
        named_bar_sync(1 + rbl, KW * 32);
        if (kw == 0 && lane < RR) {
          float s = 0.f;
          for (int q = 0; q < KW; ++q) s += red[(rbl * KW + q) * RR + lane];
          if (ok && row + lane < a.M[j]) a.y[j][row + lane] = s;
        }
        named_bar_sync(1 + rbl, KW * 32);  // red is reused by the next row block
      }
      ci = 0;
      ++i;
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

// Plans and launches the lean one-token kernel in one CTA shape; QG_EUNSUPPORTED (nothing
// launched) when the shape is outside its scope, so the caller takes the general kernel.
template <int QT, int NW, int CPS, int RR>
qg_status gemv1_cfg(int nmat, const void *const *w, const float *x, float *const *y, const int64_t *Ms, int64_t N,
                    cudaStream_t stream) {
  using D = Dec<QT>;
  const DeviceInfo &dev = device_info();
  if (!dev.ok) return QG_ECUDA;
  const long long row_bytes = N / D::QK * D::BB;
  if (row_bytes % 16 != 0) return QG_EUNSUPPORTED;
  const int ngroups = static_cast<int>((N + D::SG - 1) / D::SG);
  const long long xres = ((static_cast<long long>(ngroups) * D::SG * 4 + 1023) / 1024) * 1024;
  const long long budget = (CPS == 1 ? dev.smem_optin : dev.smem_per_sm / CPS) - 4096;
  const uint32_t hdr = 1024;
  const uint32_t red_bytes = NW * RR * 4;
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
  // when the CTAs have fewer row blocks than warps, the warps split K: give them chunks
  if (rb_per_cta < NW) {
    const int want_kw = static_cast<int>(std::min<long long>(NW, NW / std::max<long long>(1, rb_per_cta)));
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
  a.max_kw = nchunks;
  a.N = static_cast<int>(N);
  a.xR = ngroups * D::SG / 32;
  a.box_rows = box_rows_for(a.xR);
  a.off_red = hdr;
  a.off_x = (hdr + red_bytes + 1023) & ~1023u;
  a.off_ring = a.off_x + static_cast<uint32_t>(xres);
  const uint32_t smem = a.off_ring + static_cast<uint32_t>(NW * NS * stage) + 1024;
  CUtensorMap map;
  if (!encode_x_map(&map, x, 1, N, a.box_rows)) return QG_ECUDA;
  auto kern = qgemv1_kernel<QT, NW, CPS, RR>;
  if (!set_smem_attr(reinterpret_cast<const void *>(kern), smem)) return QG_ECUDA;
  a.early_weights = static_weights(stream) ? 1 : 0;
  if (launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(NW * 32), smem, stream, map, a) != cudaSuccess)
    return QG_ECUDA;
  return cudaGetLastError() == cudaSuccess ? QG_OK : QG_ECUDA;
}

template <int QT>
qg_status gemv1_launch(int nmat, const void *const *w, const float *x, float *const *y, const int64_t *Ms, int64_t N,
                       cudaStream_t stream) {
  return gemv1_cfg<QT, 8, 2, 2>(nmat, w, x, y, Ms, N, stream);
}

template qg_status gemv1_launch<QG_TYPE_Q8_0>(int, const void *const *, const float *, float *const *, const int64_t *,
                                              int64_t, cudaStream_t);
template qg_status gemv1_launch<QG_TYPE_Q4_0>(int, const void *const *, const float *, float *const *, const int64_t *,
                                              int64_t, cudaStream_t);
template qg_status gemv1_launch<QG_TYPE_Q4_K>(int, const void *const *, const float *, float *const *, const int64_t *,
                                              int64_t, cudaStream_t);
template qg_status gemv1_launch<QG_TYPE_Q6_K>(int, const void *const *, const float *, float *const *, const int64_t *,
                                              int64_t, cudaStream_t);

}  // namespace qg
