// qg_moe.cu -- MoE router, expert and combine kernels (placeholder).
#include "qg_host.h"

__device__ unsigned int g_qg_status_moe;

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

extern "C" {
size_t moe_workspace_size(int, int, int, int, int) { return 0; }
qg_status moe_route_topk(const float *, const float *, int, int, int, int, int32_t *, float *, float *, void *, size_t,
                         qg_stream_t) {
  return QG_EUNSUPPORTED;
}
qg_status moe_expert_swiglu(int, const void *, const void *, int64_t, const int32_t *, int, int, const int32_t *,
                            const float *, int, int, int, int, float *, void *, size_t, qg_stream_t) {
  return QG_EUNSUPPORTED;
}
qg_status moe_combine(int, const void *, int64_t, const int32_t *, int, int, const int32_t *, const float *,
                      const float *, int, int, int, int, float *, int, void *, size_t, qg_stream_t) {
  return QG_EUNSUPPORTED;
}
qg_status moe_layer(int, const float *, const float *, const void *, const void *, const void *, int64_t,
                    const int32_t *, int, int, int, int, int, int, int32_t *, float *, float *, float *, void *, size_t,
                    qg_stream_t) {
  return QG_EUNSUPPORTED;
}
}
