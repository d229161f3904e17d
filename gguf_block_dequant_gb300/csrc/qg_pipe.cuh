// qg_pipe.cuh -- pieces of the warp-autonomous streaming pipeline shared by the GEMV and
// MoE kernels: activation tensor copies, unaligned bulk-copy sizing and the host-side
// tensor-map encoder.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "qg_decode.cuh"

QG_DEVICE void tma_load_2d(void *dst, const CUtensorMap *map, int c0, int c1, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

QG_DEVICE void tma_load_3d(void *dst, const CUtensorMap *map, int c0, int c1, int c2, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

// T activation rows blocks [row0(t), row0(t) + xR) into the buffer at dst (1024-byte aligned),
// with expect_tx on bar
QG_DEVICE void load_x(uint8_t *dst, const CUtensorMap *map, int T, int N, int c, int xR, int box_rows,
                      uint64_t *bar) {
  mbar_arrive_expect_tx(bar, static_cast<uint32_t>(T * xR) * 128u);
  for (int t = 0; t < T; ++t)
    for (int b = 0; b < xR; b += box_rows) tma_load_2d(dst + (t * xR + b) * 128, map, 0, t * (N / 32) + c * xR + b, bar);
}

// Bytes to bulk-copy for [src, src + n) where src may be unaligned: the copy starts at the
// 16-byte boundary below src (dst receives src at dst + (src & 15)); bytes past the
// tensor's last 16-byte boundary `mend` are written here with plain loads instead.
QG_DEVICE uint32_t stage_copy(uint8_t *dst, uintptr_t src, uint32_t n, uintptr_t mend) {
  const uintptr_t al = src & ~static_cast<uintptr_t>(15);
  const uintptr_t want = (src + n + 15) & ~static_cast<uintptr_t>(15);
  if (want <= mend) return static_cast<uint32_t>(want - al);  // the usual case
  const uint32_t nb = mend > al ? static_cast<uint32_t>(mend - al) : 0u;
  for (uintptr_t p = al + nb; p < src + n; ++p) dst[p - al] = *reinterpret_cast<const uint8_t *>(p);
  return nb;
}

// One bulk copy per active lane (each lane's own segment), all on one mbarrier: the byte
// count of every segment is added to the barrier's transaction count before any copy starts.
// ONCE as for bulk_g2s.
template <bool ONCE = false>
QG_DEVICE void warp_bulk_copies(uint8_t *dst, uintptr_t src, uint32_t n, uintptr_t mend, uint64_t *bar, int lane) {
  uint32_t nb = 0;
  if (n) nb = stage_copy(dst, src, n, mend);
  const uint32_t tx = __reduce_add_sync(0xFFFFFFFFu, nb);
  if (lane == 0) mbar_arrive_expect_tx(bar, tx);
  __syncwarp();
  if (nb) {
    fence_proxy_async_smem();  // the slot's previous bytes were read through the generic proxy
    bulk_g2s<ONCE>(dst, reinterpret_cast<const void *>(src & ~static_cast<uintptr_t>(15)), nb, bar);
  }
}

namespace qg {
inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}


// Tensor map over a token-major f32 [rows][K] activation matrix viewed as [rows * K / 32]
// rows of 32 floats, 128-byte swizzle, boxes of box_rows rows.  K % 32 == 0.
inline bool encode_x_map(CUtensorMap *map, const float *x, long long rows, long long K, int box_rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t gdim[2] = {32, static_cast<cuuint64_t>(rows) * static_cast<cuuint64_t>(K / 32)};
  const cuuint64_t gstride[1] = {128};
  const cuuint32_t boxd[2] = {32, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(x), gdim, gstride, boxd, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor map over a token-major f32 [T][K] activation matrix seen as K/32 rows of tt token
// slots of 32 floats: a box (32 floats, tt tokens, box_rows rows) lands as [row][token][32]
// (row r, token t at 32-float row r * tt + t of the box), with the 128-byte swizzle; token
// slots >= T read as zero.  K % 32 == 0, tt <= 256, box_rows <= 256.
inline bool encode_x_map_tok(CUtensorMap *map, const float *x, long long T, long long K, int tt, int box_rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t gdim[3] = {32, static_cast<cuuint64_t>(T), static_cast<cuuint64_t>(K / 32)};
  const cuuint64_t gstride[2] = {static_cast<cuuint64_t>(K) * 4u, 128};
  const cuuint32_t boxd[3] = {32, static_cast<cuuint32_t>(tt), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(x), gdim, gstride, boxd, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Largest box height (multiple of 8, <= 256) dividing rows.
inline int box_rows_for(int rows) {
  int box = 8;
  for (int d = 8; d <= 256; d += 8)
    if (rows % d == 0) box = d;
  return box;
}

}  // namespace qg
