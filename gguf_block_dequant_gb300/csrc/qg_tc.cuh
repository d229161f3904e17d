// qg_tc.cuh -- tcgen05 (5th-generation tensor core) helpers shared by the prefill GEMM and
// the grouped MoE GEMM: TMEM allocation, MMA issue and commit, TMEM loads, the shared-memory
// matrix descriptor of K-major 128-byte-swizzled bf16 tiles, the kind::f16 instruction
// descriptor, abort-aware bounded waits, and the Q8_0 -> bf16 converter that fills A tiles.
#pragma once

#include <cuda_bf16.h>

#include "qg_common.cuh"

QG_DEVICE void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
QG_DEVICE void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
QG_DEVICE void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
QG_DEVICE void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

QG_DEVICE void tc_mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accum)
      : "memory");
}
// arrives once on `bar` when every MMA this thread issued before it has completed
QG_DEVICE void tc_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// 32 consecutive f32 columns of this thread's TMEM lane
QG_DEVICE void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 16 consecutive f32 columns of this thread's TMEM lane
QG_DEVICE void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor of a K-major operand tile in the 128-byte swizzled
// layout: rows of 128 bytes, 8-row (1024-byte) swizzle atoms stacked along M/N.
//   bits  0-13  start address >> 4        bits 16-29  leading byte offset >> 4 (unused here)
//   bits 32-45  stride byte offset >> 4 (1024: next 8-row group)
//   bits 46-47  descriptor version 1      bits 61-63  layout: 2 = 128-byte swizzle
QG_DEVICE uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>(1u) << 16;
  d |= static_cast<uint64_t>((1024u >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}

// Instruction descriptor, kind::f16: f32 accumulator, bf16 A and B, both K-major.
__host__ __device__ constexpr uint32_t make_idesc(int m, int n) {
  return (1u << 4)                                 // D format f32
         | (1u << 7)                               // A format bf16
         | (1u << 10)                              // B format bf16
         | (static_cast<uint32_t>(n >> 3) << 17)   // N / 8
         | (static_cast<uint32_t>(m >> 4) << 24);  // M / 16
}

// ---- abort-aware bounded waits -------------------------------------------------------------
// A wait that gives up when another role of the CTA has aborted, or after QG_WAIT_NS; an
// expired wait raises the CTA's abort flag and records QG_ETIMEOUT in *status.
QG_DEVICE bool wait_or_abort(uint64_t *bar, uint32_t parity, volatile int *abort_flag, unsigned int *status) {
  if (mbar_try_wait_sleep(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (true) {
    if (mbar_try_wait_sleep(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_ns() - t0 > QG_WAIT_NS) break;
  }
  *abort_flag = 1;
  atomicOr(status, QG_STATUS_BIT_TIMEOUT);
  return false;
}

// short bounded wait used only while shutting down
QG_DEVICE void cleanup_wait(uint64_t *bar, uint32_t parity) {
  for (uint32_t i = 0; i < (1u << 16); ++i)
    if (mbar_try_wait(bar, parity)) return;
}

// Decode 16 Q8_0 weights (half hb & 1 of block hb >> 1 of the 64-k stage `sub`) of one row
// from the raw stage into the A slot.  raw_row: shared address of the row's 272 raw bytes;
// a_row: shared address of the row in the A slot (128 bytes, 16-byte chunks swizzled by
// row & 7).  The 16 code bytes start 2-byte aligned; they come from five aligned words.
QG_DEVICE void convert_half(uint32_t raw_row, int sub, int hb, uint32_t a_row, int row) {
  const uint32_t blk = raw_row + 68u * static_cast<uint32_t>(sub) + 34u * static_cast<uint32_t>(hb >> 1);
  uint32_t d16;
  QG_LDS16(blk, 0, d16);
  const float d = h2f(d16);
  // the 16 codes start 2-byte aligned: five aligned words and four funnel shifts
  const uint32_t o = blk + 2u + 16u * static_cast<uint32_t>(hb & 1);
  const uint32_t wb = o & ~3u, sh = (o & 3u) * 8u;
  const uint32_t w0 = lds_u32(wb), w1 = lds_u32(wb + 4u), w2 = lds_u32(wb + 8u), w3 = lds_u32(wb + 12u),
                 w4 = lds_u32(wb + 16u);
  const uint32_t cw[4] = {__funnelshift_r(w0, w1, sh), __funnelshift_r(w1, w2, sh), __funnelshift_r(w2, w3, sh),
                          __funnelshift_r(w3, w4, sh)};
  const f2 d2 = mk2(d, d);
  const f2 bias = mk2(-8388736.0f, -8388736.0f);  // -(2^23 + 128)
#pragma unroll
  for (int c = 0; c < 2; ++c) {  // two 16-byte chunks of 8 weights
    uint32_t outw[4];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t word = cw[2 * c + h] ^ 0x80808080u;
      const f2 w01 = mul2(add2(mk2(magic_byte(word, 0), magic_byte(word, 1)), bias), d2);
      const f2 w23 = mul2(add2(mk2(magic_byte(word, 2), magic_byte(word, 3)), bias), d2);
      const __nv_bfloat162 b01 = __floats2bfloat162_rn(w01.x, w01.y);
      const __nv_bfloat162 b23 = __floats2bfloat162_rn(w23.x, w23.y);
      outw[2 * h] = *reinterpret_cast<const uint32_t *>(&b01);
      outw[2 * h + 1] = *reinterpret_cast<const uint32_t *>(&b23);
    }
    const uint32_t chunk = static_cast<uint32_t>((2 * hb + c) ^ (row & 7));
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a_row + chunk * 16u), "r"(outw[0]), "r"(outw[1]),
                 "r"(outw[2]), "r"(outw[3])
                 : "memory");
  }
}

