// qg_head.cu -- the steps on either side of a GEMV chain: embedding row gathers (embedQ8 /
// embedQ6K), RMSNorm (rmsnorm / rmsnormB), the per-row argmax that ends a greedy decode step
// (argmax / argmaxRows), and the tied head with its argmax in one call.
//
// The gather decodes with the GEMV's lane decoders (qg_decode.cuh): a warp stages one group
// of a row's raw blocks in shared memory, each lane decodes its unit and writes its values,
// so every dequantized value is the one the GEMV multiplies.
#include <cuda.h>
#include <math.h>

#include "qg_decode.cuh"
#include "qg_host.h"

__device__ unsigned int g_qg_status_head;  // this translation unit's device status word

namespace {

constexpr int kEmbedWarps = 8;

// out[i][k] = w(ids[i], k) * scale: one warp per (row i, group g) unit, grid-strided.
template <int QT>
__global__ void __launch_bounds__(kEmbedWarps * 32) embed_kernel(const uint8_t *__restrict__ table, long long V,
                                                                 int N, const int32_t *__restrict__ ids, int n,
                                                                 float scale, float *__restrict__ out) {
  using D = Dec<QT>;
  // a group's bytes plus 16 of alignment slack and 16 of decoder over-read, per warp; every
  // slot starts on a 16-byte boundary (the 16-byte stores below need it)
  constexpr int SLOT = (D::GB + 32 + 15) / 16 * 16;
  __shared__ __align__(16) uint8_t buf[kEmbedWarps][SLOT];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_wait();
  pdl_launch_dependents();
  const int groups = (N + D::SG - 1) / D::SG;
  const long long row_bytes = static_cast<long long>(N / D::QK) * D::BB;
  const uintptr_t tend = reinterpret_cast<uintptr_t>(table) + static_cast<uintptr_t>(V * row_bytes);
  const uintptr_t mend = tend & ~static_cast<uintptr_t>(15);  // last 16-byte boundary of the table
  const long long units = static_cast<long long>(n) * groups;
  uint8_t *slot = buf[warp];
  for (long long u = static_cast<long long>(blockIdx.x) * kEmbedWarps + warp; u < units;
       u += static_cast<long long>(gridDim.x) * kEmbedWarps) {
    const int i = static_cast<int>(u / groups), g = static_cast<int>(u - static_cast<long long>(i) * groups);
    const int id = __ldg(ids + i);
    const int ne = min(D::SG, N - g * D::SG);  // elements of this group
    float *o = out + static_cast<size_t>(i) * N + static_cast<size_t>(g) * D::SG;
    if (id < 0 || id >= V) {
      // an id outside the table: the row is zeros and the device status records it
      for (int k = 4 * lane; k < ne; k += 128) *reinterpret_cast<float4 *>(o + k) = make_float4(0.f, 0.f, 0.f, 0.f);
      if (lane == 0) atomicOr(&g_qg_status_head, QG_STATUS_BIT_ID);
      continue;
    }
    const uintptr_t src = reinterpret_cast<uintptr_t>(table) + static_cast<uintptr_t>(id) * row_bytes +
                          static_cast<uintptr_t>(g) * D::GB;
    const uint32_t nb = static_cast<uint32_t>(ne / D::QK * D::BB);
    // [src & ~15, src + nb) into the slot: 16-byte words below the table's last 16-byte
    // boundary, single bytes past it (the table pointer is 16-byte aligned)
    const uintptr_t a0 = src & ~static_cast<uintptr_t>(15);
    const uint32_t span = static_cast<uint32_t>(src + nb - a0);
    for (uint32_t off = 16u * lane; off < span; off += 512u) {
      const uintptr_t p = a0 + off;
      if (p + 16 <= mend) {
        *reinterpret_cast<uint4 *>(slot + off) = __ldg(reinterpret_cast<const uint4 *>(p));
      } else {
        for (uint32_t b = 0; b < 16u && p + b < tend; ++b) slot[off + b] = *reinterpret_cast<const uint8_t *>(p + b);
      }
    }
    __syncwarp();
    if (D::block_first(lane) < ne) {
      const uint32_t base = smem_u32(slot) + static_cast<uint32_t>(src - a0);
      const typename D::U w = D::load(base + static_cast<uint32_t>(D::woff(lane)), lane);
#pragma unroll
      for (int ch = 0; ch < D::NCH; ++ch) {
        f2 w01, w23;
        D::weights(w, ch, w01, w23);
        const int e = 32 * D::xrow(lane, ch) + 4 * D::xunit(lane, ch);
        if (e < ne)
          *reinterpret_cast<float4 *>(o + e) = make_float4(w01.x * scale, w01.y * scale, w23.x * scale, w23.y * scale);
      }
    }
    __syncwarp();  // the slot is refilled for the next unit
  }
}

// y[t][i] = ((x[t][i] * s_t) * k) * w[i], s_t = 1 / sqrt(mean_i x[t][i]^2 + eps): one CTA per row.
__global__ void __launch_bounds__(256) rmsnorm_kernel(const float *__restrict__ x, const float *__restrict__ w, int N,
                                                      float eps, float kf, float *__restrict__ y) {
  __shared__ float part[8];
  const int t = blockIdx.x;
  pdl_wait();
  pdl_launch_dependents();
  const float4 *xr = reinterpret_cast<const float4 *>(x + static_cast<size_t>(t) * N);
  const int n4 = N / 4;
  float ss = 0.f;
  for (int i = threadIdx.x; i < n4; i += 256) {
    const float4 v = xr[i];
    ss = fmaf(v.x, v.x, ss);
    ss = fmaf(v.y, v.y, ss);
    ss = fmaf(v.z, v.z, ss);
    ss = fmaf(v.w, v.w, ss);
  }
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int q = 0; q < 8; ++q) tot += part[q];
  const float s = 1.0f / sqrtf(tot / static_cast<float>(N) + eps);
  const float4 *wr = reinterpret_cast<const float4 *>(w);
  float4 *yr = reinterpret_cast<float4 *>(y + static_cast<size_t>(t) * N);
  for (int i = threadIdx.x; i < n4; i += 256) {
    const float4 v = xr[i], g = wr[i];
    yr[i] = make_float4(((v.x * s) * kf) * g.x, ((v.y * s) * kf) * g.y, ((v.z * s) * kf) * g.z, ((v.w * s) * kf) * g.w);
  }
}

// (value, index) that wins: the larger value, the lower index on ties; index < 0 is empty
QG_DEVICE void am_take(float &bv, int &bi, float v, int i) {
  if (i >= 0 && (bi < 0 || v > bv || (v == bv && i < bi))) {
    bv = v;
    bi = i;
  }
}

constexpr int kArgmaxCluster = 8;  // CTAs per row

QG_DEVICE uint32_t am_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
QG_DEVICE void am_cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ids[t] = the lowest index of the largest value of row t (NaN never picked; a row with no
// value other than NaN gives 0).  A cluster of kArgmaxCluster CTAs per row: rank r scans the
// r-th slice, reduces it over its warps, and rank 0 takes the best of the ranks' pairs from
// their shared memory (the slices are in index order, so ties still go to the lowest index).
__global__ void __launch_bounds__(256) argmax_kernel(const float *__restrict__ l, long long n, int vec4,
                                                     int32_t *__restrict__ ids) {
  __shared__ float sv[8];
  __shared__ int si[8];
  const uint32_t rank = am_rank();
  const int t = static_cast<int>(blockIdx.x / kArgmaxCluster);
  pdl_wait();
  pdl_launch_dependents();
  const float *r = l + static_cast<size_t>(t) * static_cast<size_t>(n);
  const long long lo = static_cast<long long>(rank) * n / kArgmaxCluster;
  const long long hi = static_cast<long long>(rank + 1) * n / kArgmaxCluster;
  float bv = 0.f;
  int bi = -1;
  auto take = [&](float v, long long i) {
    if (!isnan(v) && (bi < 0 || v > bv)) {  // a thread's indices rise: strict > keeps the lowest
      bv = v;
      bi = static_cast<int>(i);
    }
  };
  if (vec4) {
    // 16-byte loads over the slice's whole quads, single loads at its two ends
    const long long q0 = (lo + 3) / 4, q1 = hi / 4;
    if (q0 >= q1) {
      for (long long i = lo + threadIdx.x; i < hi; i += 256) take(r[i], i);
    } else {
      for (long long i = lo + threadIdx.x; i < 4 * q0; i += 256) take(r[i], i);
      const float4 *r4 = reinterpret_cast<const float4 *>(r);
      for (long long q = q0 + threadIdx.x; q < q1; q += 256) {
        const float4 v = r4[q];
        take(v.x, 4 * q);
        take(v.y, 4 * q + 1);
        take(v.z, 4 * q + 2);
        take(v.w, 4 * q + 3);
      }
      for (long long i = 4 * q1 + threadIdx.x; i < hi; i += 256) take(r[i], i);
    }
  } else {
    for (long long i = lo + threadIdx.x; i < hi; i += 256) take(r[i], i);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
    const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
    am_take(bv, bi, ov, oi);
  }
  if ((threadIdx.x & 31) == 0) {
    sv[threadIdx.x >> 5] = bv;
    si[threadIdx.x >> 5] = bi;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int q = 1; q < 8; ++q) am_take(sv[0], si[0], sv[q], si[q]);
  }
  am_cluster_sync();  // every rank's pair is in its shared memory
  if (rank == 0 && threadIdx.x == 0) {
    float v = sv[0];
    int i = si[0];
    for (uint32_t q = 1; q < kArgmaxCluster; ++q) {
      uint32_t av, ai;
      asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(av) : "r"(smem_u32(&sv[0])), "r"(q));
      asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ai) : "r"(smem_u32(&si[0])), "r"(q));
      float ov;
      int oi;
      asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(ov) : "r"(av) : "memory");
      asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(oi) : "r"(ai) : "memory");
      am_take(v, i, ov, oi);
    }
    ids[t] = i < 0 ? 0 : i;
  }
  am_cluster_sync();  // no rank leaves while rank 0 reads it
}

}  // namespace

namespace qg {

template <int QT>
static qg_status embed_launch(const void *table, int64_t V, int64_t N, const int32_t *ids, int n, float scale,
                              float *out, cudaStream_t s) {
  using D = Dec<QT>;
  const DeviceInfo &dev = device_info();
  if (!dev.ok) return QG_ECUDA;
  const long long units = static_cast<long long>(n) * ((N + D::SG - 1) / D::SG);
  const long long grid = std::max<long long>(1, std::min<long long>((units + kEmbedWarps - 1) / kEmbedWarps,
                                                                    8LL * dev.sms));
  if (launch_pdl(embed_kernel<QT>, dim3(static_cast<unsigned>(grid)), dim3(kEmbedWarps * 32), 0, s,
                 static_cast<const uint8_t *>(table), static_cast<long long>(V), static_cast<int>(N), ids, n, scale,
                 out) != cudaSuccess)
    return QG_ECUDA;
  return cudaGetLastError() == cudaSuccess ? QG_OK : QG_ECUDA;
}

static qg_status argmax_launch(const float *logits, int T, int64_t n, int32_t *ids, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(T * kArgmaxCluster));
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = kArgmaxCluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const int vec4 = (n % 4 == 0 && aligned16(logits)) ? 1 : 0;
  if (cudaLaunchKernelEx(&cfg, argmax_kernel, logits, static_cast<long long>(n), vec4, ids) != cudaSuccess)
    return QG_ECUDA;
  return cudaGetLastError() == cudaSuccess ? QG_OK : QG_ECUDA;
}

unsigned int read_status_head(bool clear) {
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_qg_status_head, sizeof(v)) != cudaSuccess) return 0xFFFFFFFFu;
  if (clear) {
    const unsigned int z = 0;
    cudaMemcpyToSymbol(g_qg_status_head, &z, sizeof(z));
  }
  return v;
}

}  // namespace qg

extern "C" {

qg_status qg_embed_rows(int type, const void *table, int64_t V, int64_t N, const int32_t *ids, int n, float scale,
                        float *out, qg_stream_t stream) {
  int qk = 0, bb = 0;
  if (qg_block_shape(type, &qk, &bb) != QG_OK) return QG_EUNSUPPORTED;
  if (!table || !ids || !out) return QG_EINVAL_PTR;
  if (V < 1 || N <= 0 || N % qk || n < 0 || N > INT32_MAX || V > INT32_MAX) return QG_EINVAL_SHAPE;
  if (static_cast<long long>(n) * N > (1LL << 40)) return QG_EINVAL_SHAPE;
  if (!qg::aligned16(table) || !qg::aligned16(out) || (reinterpret_cast<uintptr_t>(ids) & 3u)) return QG_EALIGN;
  if (n == 0) return QG_OK;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  switch (type) {
    case QG_TYPE_Q8_0: return qg::embed_launch<QG_TYPE_Q8_0>(table, V, N, ids, n, scale, out, s);
    case QG_TYPE_Q4_0: return qg::embed_launch<QG_TYPE_Q4_0>(table, V, N, ids, n, scale, out, s);
    case QG_TYPE_Q4_K: return qg::embed_launch<QG_TYPE_Q4_K>(table, V, N, ids, n, scale, out, s);
    default: return qg::embed_launch<QG_TYPE_Q6_K>(table, V, N, ids, n, scale, out, s);
  }
}

qg_status qg_rmsnorm(const float *x, const float *w, int T, int64_t N, float eps, float k, float *y,
                     qg_stream_t stream) {
  if (!x || !w || !y) return QG_EINVAL_PTR;
  if (T < 0 || T > 65535 || N <= 0 || N % 4 || N > INT32_MAX || !(eps >= 0.f) || !isfinite(k)) return QG_EINVAL_SHAPE;
  if (!qg::aligned16(x) || !qg::aligned16(w) || !qg::aligned16(y)) return QG_EALIGN;
  if (T == 0) return QG_OK;
  if (qg::launch_pdl(rmsnorm_kernel, dim3(static_cast<unsigned>(T)), dim3(256), 0,
                     reinterpret_cast<cudaStream_t>(stream), x, w, static_cast<int>(N), eps, k, y) != cudaSuccess)
    return QG_ECUDA;
  return cudaGetLastError() == cudaSuccess ? QG_OK : QG_ECUDA;
}

qg_status qg_argmax_rows(const float *logits, int T, int64_t n, int32_t *ids, qg_stream_t stream) {
  if (!logits || !ids) return QG_EINVAL_PTR;
  if (T < 0 || T > 8191 || n <= 0 || n > INT32_MAX) return QG_EINVAL_SHAPE;
  if ((reinterpret_cast<uintptr_t>(logits) & 3u) || (reinterpret_cast<uintptr_t>(ids) & 3u)) return QG_EALIGN;
  if (T == 0) return QG_OK;
  return qg::argmax_launch(logits, T, n, ids, reinterpret_cast<cudaStream_t>(stream));
}

qg_status qg_head_argmax(int type, const void *w, int64_t M, int64_t N, const float *x, int T, float *logits,
                         int32_t *ids, qg_stream_t stream) {
  int qk = 0, bb = 0;
  if (qg_block_shape(type, &qk, &bb) != QG_OK) return QG_EUNSUPPORTED;
  if (!w || !x || !logits || !ids) return QG_EINVAL_PTR;
  if (M < 1 || N <= 0 || N % qk || T < 1 || T > 16 || M > INT32_MAX || N > INT32_MAX) return QG_EINVAL_SHAPE;
  if (static_cast<long long>(T) * N > INT32_MAX) return QG_EINVAL_SHAPE;
  if (!qg::aligned16(w) || !qg::aligned16(x) || !qg::aligned16(logits) || (reinterpret_cast<uintptr_t>(ids) & 3u))
    return QG_EALIGN;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const qg_status r = qg::gemv_dispatch(type, w, x, logits, M, N, T, s);
  if (r != QG_OK) return r;
  return qg::argmax_launch(logits, T, M, ids, s);
}

}  // extern "C"
