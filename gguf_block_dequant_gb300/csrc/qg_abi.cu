// qg_abi.cu -- library-wide entry points: version, status strings, block shapes, device
// status word, and the per-device property cache.
#include <mutex>

#include "qg_host.h"

namespace qg {

namespace {
constexpr int kMaxDevices = 64;
DeviceInfo g_info[kMaxDevices];
std::once_flag g_once[kMaxDevices];

struct AttrEntry {
  const void *func;
  int device;
  uint32_t bytes;
};
std::mutex g_attr_mu;
AttrEntry g_attr[256];
int g_attr_n = 0;
}  // namespace

const DeviceInfo &device_info() {
  static DeviceInfo bad;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return bad;
  std::call_once(g_once[dev], [dev] {
    DeviceInfo &d = g_info[dev];
    d.ok = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
           cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) == cudaSuccess &&
           cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) == cudaSuccess &&
           cudaDeviceGetAttribute(&d.l2_bytes, cudaDevAttrL2CacheSize, dev) == cudaSuccess;
  });
  return g_info[dev];
}

namespace {
// Streams whose callers declared their weights immutable (qg_set_static_weights), per device.
// A small table searched per launch: a process holds a handful of streams.
constexpr int kMaxStaticStreams = 256;
struct StaticEntry {
  cudaStream_t s;
  int device;
};
std::mutex g_static_mu;
StaticEntry g_static[kMaxStaticStreams];
int g_static_n = 0;

int find_static(cudaStream_t s, int dev) {
  for (int i = 0; i < g_static_n; ++i)
    if (g_static[i].s == s && g_static[i].device == dev) return i;
  return -1;
}
}  // namespace

bool static_weights(cudaStream_t s) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
  std::lock_guard<std::mutex> lk(g_static_mu);
  return find_static(s, dev) >= 0;
}

bool set_smem_attr(const void *func, uint32_t bytes) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  std::lock_guard<std::mutex> lk(g_attr_mu);
  for (int i = 0; i < g_attr_n; ++i)
    if (g_attr[i].func == func && g_attr[i].device == dev) {
      if (g_attr[i].bytes >= bytes) return true;
      if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes)) !=
          cudaSuccess)
        return false;
      g_attr[i].bytes = bytes;
      return true;
    }
  if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes)) != cudaSuccess)
    return false;
  // the whole unified L1/shared array as shared memory: every kernel here stages its operands
  // there, and two-CTA-per-SM launches need the full carveout
  cudaFuncSetAttribute(func, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (g_attr_n < 256) g_attr[g_attr_n++] = AttrEntry{func, dev, bytes};
  return true;
}

}  // namespace qg

extern "C" {

int qg_version(void) { return 3; }

const char *qg_strerror(int status) {
  switch (status) {
    case QG_OK: return "ok";
    case QG_EINVAL_SHAPE: return "invalid shape (size out of range or not a multiple of the block size)";
    case QG_EINVAL_PTR: return "a required pointer is NULL";
    case QG_EALIGN: return "a pointer or stride is not 16-byte aligned";
    case QG_EUNSUPPORTED: return "block type or configuration not supported by this call";
    case QG_ECUDA: return "a CUDA call or kernel launch failed";
    case QG_EDEVICE_ID: return "device status: an expert id or slot was out of range";
    case QG_ETIMEOUT: return "device status: a bounded wait inside a kernel expired";
    case QG_EWORKSPACE: return "workspace missing or too small";
    default: return "unknown status";
  }
}

qg_status qg_block_shape(int type, int *qk, int *block_bytes) {
  int a, b;
  switch (type) {
    case QG_TYPE_Q8_0: a = 32; b = 34; break;
    case QG_TYPE_Q4_0: a = 32; b = 18; break;
    case QG_TYPE_Q4_K: a = 256; b = 144; break;
    case QG_TYPE_Q6_K: a = 256; b = 210; break;
    default: return QG_EUNSUPPORTED;
  }
  if (qk) *qk = a;
  if (block_bytes) *block_bytes = b;
  return QG_OK;
}

int qg_set_static_weights(qg_stream_t stream, int enable) {
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;  // no device: the handle alone is the key
  std::lock_guard<std::mutex> lk(qg::g_static_mu);
  const int i = qg::find_static(s, dev);
  const int prev = i >= 0 ? 1 : 0;
  if (enable && i < 0) {
    if (qg::g_static_n >= qg::kMaxStaticStreams) return -1;
    qg::g_static[qg::g_static_n++] = qg::StaticEntry{s, dev};
  } else if (!enable && i >= 0) {
    qg::g_static[i] = qg::g_static[--qg::g_static_n];
  }
  return prev;
}

qg_status qg_device_status(uint32_t *status_out, int clear) {
  if (!status_out) return QG_EINVAL_PTR;
  if (cudaDeviceSynchronize() != cudaSuccess) return QG_ECUDA;
  // one status word per translation unit (device variables are not shared across units)
  const unsigned int w[] = {qg::read_status_gemv(clear != 0), qg::read_status_gemv1(clear != 0),
                            qg::read_status_mt(clear != 0),   qg::read_status_head(clear != 0),
                            qg::read_status_moe(clear != 0),  qg::read_status_gemm(clear != 0),
                            qg::read_status_moetc(clear != 0)};
  unsigned int all = 0;
  for (const unsigned int v : w) {
    if (v == 0xFFFFFFFFu) return QG_ECUDA;
    all |= v;
  }
  *status_out = all;
  return QG_OK;
}

}  // extern "C"
