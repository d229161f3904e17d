// qg_host.h -- host-side helpers shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/ggufdq.h"

namespace qg {

// The MoE variants of one call (the header's qg_moe_variant, resolved): expert activation
// kind, per-expert down scale, sigmoid-gated shared expert.
struct MoeVar {
  int act = 0;
  const float *ds = nullptr;
  const float *sh = nullptr;
  const float *sg = nullptr;
};

struct DeviceInfo {
  bool ok = false;
  int sms = 0;         // streaming multiprocessors
  int smem_optin = 0;  // max dynamic shared memory per block (opt-in)
  int smem_per_sm = 0; // shared memory per SM
  int l2_bytes = 0;
};

// Properties of the current device (queried once per device).
const DeviceInfo &device_info();

// Raise a kernel's dynamic shared-memory limit on the current device (cached).
bool set_smem_attr(const void *func, uint32_t bytes);

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Launch with programmatic stream serialization allowed: the kernel may begin while its
// predecessor in the stream drains; it synchronises with griddepcontrol.wait (pdl_wait).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// whether the caller declared the weights read by launches on stream s (on the current
// device) immutable (qg_set_static_weights)
bool static_weights(cudaStream_t s);

// dense GEMV entry shared by qgemv_* / qgemv_t / qgemm (small T) / MoE helpers
qg_status gemv_dispatch(int type, const void *w, const float *x, float *y, int64_t M, int64_t N, int T,
                        cudaStream_t s);

// grouped tensor-core MoE expert steps for more than 16 tokens (qg_moe_tc.cu)
bool moe_tc_supported(int type, int H, int F, int E);
size_t moe_tc_workspace(int T, int k, int E, int H, int F);
qg_status moe_swiglu_tc(const void *w_gate, const void *w_up, int64_t stride, const int32_t *slots, int n_slots,
                        int E, const int32_t *ids, const float *xn, int T, int k, int H, int F, float *act, void *ws,
                        cudaStream_t s, int act_kind = 0);
// x[t] = (add_residual ? x[t] : 0) + [sum_j (dn[t k + j] ds[e_j]) w[t][j] in pick order
// + sh[t] sigmoid(sg[t])], from dn rows in memory (both MoE paths; ds, sh from v, optional)
qg_status moe_launch_combine(const float *dn, const float *weights, const int32_t *ids, const int32_t *slots,
                             int n_slots, int E, int T, int k, int H, float *x_inout, int add_residual,
                             cudaStream_t s, const MoeVar &v = MoeVar());
qg_status moe_combine_tc(const void *w_down, int64_t stride, const int32_t *slots, int n_slots, int E,
                         const int32_t *ids, const float *weights, const float *act, int T, int k, int H, int F,
                         float *x_inout, int add_residual, float *dn, void *ws, cudaStream_t s,
                         const MoeVar &v = MoeVar(), bool sorted_ready = false);

// GEMV over T <= 16 token columns, lean kernel for rows of 16-byte multiples with resident
// activations (qg_gemv1.cu); QG_EUNSUPPORTED with nothing launched for other shapes
template <int QT>
qg_status gemv1_launch(int nmat, const void *const *w, const float *x, float *const *y, const int64_t *Ms, int64_t N,
                       int T, cudaStream_t stream);

// GEMV over 2..16 token columns, Q8_0 / Q4_0 rows of whole 256-element units, rows across
// lanes (qg_gemv_mt.cu); QG_EUNSUPPORTED with nothing launched for other shapes
template <int QT>
qg_status gemv_mt_launch(int nmat, const void *const *w, const float *x, float *const *y, const int64_t *Ms,
                         int64_t N, int T, cudaStream_t stream);

qg_status gemv_multi_dispatch(int type, int n, const void *const *w, const float *x, float *const *y,
                              const int64_t *M, int64_t N, int T, cudaStream_t s);
unsigned int read_status_gemv(bool clear);
unsigned int read_status_gemv1(bool clear);
unsigned int read_status_mt(bool clear);
unsigned int read_status_head(bool clear);
unsigned int read_status_moetc(bool clear);
unsigned int read_status_moe(bool clear);
unsigned int read_status_gemm(bool clear);

}  // namespace qg
