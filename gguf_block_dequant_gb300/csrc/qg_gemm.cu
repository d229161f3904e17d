// qg_gemm.cu -- prefill dequant-GEMM (placeholder until the tensor-core kernel lands).
#include "qg_host.h"

__device__ unsigned int g_qg_status_gemm;

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
size_t qgemm_workspace_size(int, int64_t, int64_t, int64_t) { return 0; }
qg_status qgemm(int type, const void *w, const float *x, float *y, int64_t M, int64_t N, int64_t T, void *, size_t,
                qg_stream_t s) {
  if (T >= 1 && T <= 16) return qg::gemv_dispatch(type, w, x, y, M, N, static_cast<int>(T), reinterpret_cast<cudaStream_t>(s));
  return QG_EUNSUPPORTED;
}
}
