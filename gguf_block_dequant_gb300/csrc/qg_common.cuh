// qg_common.cuh -- shared device helpers for the sm_103a kernels: mbarrier and bulk-copy
// (TMA) wrappers with bounded waits, the device status word, and exact in-register decode
// helpers for the block formats.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ggufdq.h"

#define QG_DEVICE __device__ __forceinline__

// ---------------------------------------------------------------------------------------
// Device status word (one per translation unit; qg_device_status ORs them).
// ---------------------------------------------------------------------------------------
#define QG_STATUS_BIT_ID (1u << QG_EDEVICE_ID)
#define QG_STATUS_BIT_TIMEOUT (1u << QG_ETIMEOUT)

// Time after which a wait on an mbarrier is declared expired (nanoseconds of the GPU's
// global timer).  Far above any healthy pipeline's wait, far below a watchdog's patience.
#define QG_WAIT_NS 200000000ull
// Suspend-time hint of one mbarrier.try_wait (nanoseconds): a waiting thread sleeps until the
// phase completes or this much time has passed, instead of spinning on the issue slots the
// working warps need.
#define QG_TRY_WAIT_HINT_NS 1000000u

// ---------------------------------------------------------------------------------------
// Shared-memory addressing and mbarriers
// ---------------------------------------------------------------------------------------
QG_DEVICE uint32_t smem_u32(const void *p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

QG_DEVICE void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

QG_DEVICE void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

QG_DEVICE void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Arrive once and add `bytes` to the transaction count of the current phase.
QG_DEVICE void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

QG_DEVICE void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

QG_DEVICE bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

QG_DEVICE uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// try_wait that lets the hardware suspend the thread (up to the hint) while the phase is
// incomplete
QG_DEVICE bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(QG_TRY_WAIT_HINT_NS)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity to complete.  Returns false (and the
// caller must abandon its work) once QG_WAIT_NS has passed.
QG_DEVICE bool mbar_wait(uint64_t *bar, uint32_t parity) {
  if (mbar_try_wait_sleep(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (true) {
    if (mbar_try_wait_sleep(bar, parity)) return true;
    if (global_ns() - t0 > QG_WAIT_NS) return false;
  }
}

// ---------------------------------------------------------------------------------------
// Bulk copies global -> shared (the TMA engine's non-tensor form).  Both addresses must be
// 16-byte aligned and the size a multiple of 16; completion is signalled on `bar` as
// transaction bytes.  ONCE: the bytes are read once per launch (a weight stream), so their
// L2 lines are the first to be evicted and the activations and outputs that the neighbouring
// launches read stay resident.
// ---------------------------------------------------------------------------------------
template <bool ONCE = false>
QG_DEVICE void bulk_g2s(void *dst_smem, const void *src_gmem, uint32_t bytes, uint64_t *bar) {
  if constexpr (ONCE) {
    asm volatile(
        "{\n\t.reg .b64 pol;\n\t"
        "createpolicy.fractional.L2::evict_first.b64 pol, 1.0;\n\t"
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], pol;\n\t}" ::"r"(
            smem_u32(dst_smem)),
        "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
  } else {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst_smem)),
        "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
  }
}

// 16-byte asynchronous global -> shared copy (both addresses 16-byte aligned); completes at
// cp_async_wait_all()
QG_DEVICE void cp_async16(uint32_t dst_smem, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst_smem), "l"(src) : "memory");
}
QG_DEVICE void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// one arrival on `bar` once every cp.async this thread issued before it has landed (the
// barrier's expected count covers these arrivals)
QG_DEVICE void cp_async_mbar_arrive(uint64_t *bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Programmatic dependent launch: wait until the preceding kernel in the stream has completed
// and its memory is visible (a no-op when the launch did not allow the overlap), and let the
// next kernel start its prologue early.  Kernels call wait before touching any input or
// output, and launch_dependents only after their wait, so every kernel that has started can
// rely on all kernels two or more launches back having completed.
QG_DEVICE void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
QG_DEVICE void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Named barrier among `nthreads` threads (multiple of 32) on barrier id `id` (1..15).
QG_DEVICE void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------------------------------
// Shared-memory loads used by the decoders: 32-bit shared-window addresses with the
// offset folded into the instruction.  Not volatile, but ordered after the mbarrier
// waits by their "memory" clobber dependency on the address-producing code.
// ---------------------------------------------------------------------------------------
#define QG_LDS32(addr, off, out) asm("ld.shared.b32 %0, [%1+" #off "];" : "=r"(out) : "r"(addr) : "memory")
#define QG_LDS16(addr, off, out)                                                        \
  do {                                                                                  \
    uint16_t qg_t16_;                                                                   \
    asm("ld.shared.b16 %0, [%1+" #off "];" : "=h"(qg_t16_) : "r"(addr) : "memory");     \
    (out) = qg_t16_;                                                                    \
  } while (0)
#define QG_LDS128(addr, off, o0, o1, o2, o3) \
  asm("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4+" #off "];" : "=r"(o0), "=r"(o1), "=r"(o2), "=r"(o3) : "r"(addr) : "memory")
#define QG_LDSF4(addr, off, v)                                                                  \
  asm("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4+" #off "];" : "=f"((v).x), "=f"((v).y), "=f"((v).z), \
      "=f"((v).w)                                                                               \
      : "r"(addr)                                                                               \
      : "memory")

QG_DEVICE uint32_t lds_u32(uint32_t addr) {
  uint32_t v;
  QG_LDS32(addr, 0, v);
  return v;
}
QG_DEVICE uint32_t lds_u16(uint32_t addr) {
  uint32_t v;
  QG_LDS16(addr, 0, v);
  return v;
}
QG_DEVICE uint4 lds_v4(uint32_t addr) {
  uint4 v;
  QG_LDS128(addr, 0, v.x, v.y, v.z, v.w);
  return v;
}
QG_DEVICE float4 lds_f4(uint32_t addr) {
  float4 v;
  QG_LDSF4(addr, 0, v);
  return v;
}

// ---------------------------------------------------------------------------------------
// Exact small-integer -> f32 conversion.  A byte u placed in the low mantissa bits of the
// float 2^23 (bit pattern 0x4B0000uu) is the float 2^23 + u exactly; subtracting 2^23 + c
// gives u - c exactly.  This uses the integer byte-permute unit instead of the slower
// integer-to-float conversion path.
// ---------------------------------------------------------------------------------------
QG_DEVICE float magic_byte(uint32_t word, uint32_t byte_idx) {
  // result bytes (LSB first): word[byte_idx], 0x00, 0x00, 0x4B
  return __uint_as_float(__byte_perm(word, 0x4B000000u, 0x7440u | byte_idx));
}

// Packed f32x2 arithmetic (sm_100+): two IEEE f32 operations per instruction, operands in
// register pairs.  The flush-to-zero forms are used: a denormal f32 operand (|v| < 2^-126)
// counts as zero.  The packed unit takes a slow path on denormal operands without it (about
// 40x slower in a micro-benchmark), so activations with many denormals would slow every
// product down.  Every weight the decoders produce is 0 or at least 2^-24 in magnitude (f16
// scales times small integers), so only products with a denormal activation and denormal
// partial sums are affected: each error is below 2^-126 * 2^23 (the largest decoded weight is
// about 65504 * 127), far inside the 1e-6 absolute term of the output bound.
using f2 = float2;
QG_DEVICE f2 mk2(float a, float b) { return make_float2(a, b); }
QG_DEVICE unsigned long long pack2(f2 v) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(v.x), "f"(v.y));
  return r;
}
QG_DEVICE f2 unpack2(unsigned long long r) {
  f2 v;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(v.x), "=f"(v.y) : "l"(r));
  return v;
}
QG_DEVICE f2 add2(f2 a, f2 b) {
  unsigned long long d;
  asm("add.rn.ftz.f32x2 %0, %1, %2;" : "=l"(d) : "l"(pack2(a)), "l"(pack2(b)));
  return unpack2(d);
}
QG_DEVICE f2 mul2(f2 a, f2 b) {
  unsigned long long d;
  asm("mul.rn.ftz.f32x2 %0, %1, %2;" : "=l"(d) : "l"(pack2(a)), "l"(pack2(b)));
  return unpack2(d);
}
QG_DEVICE f2 fma2(f2 a, f2 b, f2 c) {
  unsigned long long d;
  asm("fma.rn.ftz.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(pack2(a)), "l"(pack2(b)), "l"(pack2(c)));
  return unpack2(d);
}

// f16 bits -> f32 (exact; hardware conversion).
QG_DEVICE float h2f(uint32_t bits16) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(bits16 & 0xFFFFu)));
}

// Expert activations of gate g and up u: SiLU(g) u (siluMulMoe) and GELU(g) u with the tanh
// form, its argument clamped to [-10, 10] as the geglu preamble does.
QG_DEVICE float act_silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }
QG_DEVICE float act_gelu_mul(float g, float u) {
  const float a = fminf(fmaxf(0.7978845608f * g * (1.0f + 0.044715f * g * g), -10.0f), 10.0f);
  return 0.5f * g * (1.0f + tanhf(a)) * u;
}
QG_DEVICE float act_mul(int kind, float g, float u) { return kind ? act_gelu_mul(g, u) : act_silu_mul(g, u); }

QG_DEVICE float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// Butterfly reduce-scatter of N per-lane partial values (N a power of two, N <= 64): at each
// step a lane keeps half of its values and adds the partner's copy of that half, so the
// warp needs N - 1 + (5 - log2 N) shuffles instead of 5 N.  Afterwards v[0] holds the full
// sum of value rs_index(lane) (N <= 32; lanes that differ only in their low 5 - log2 N bits
// hold the same value), or v[0], v[1] hold values 2 lane and 2 lane + 1 (N = 64).
template <int N>
QG_DEVICE void reduce_scatter(float (&v)[N], int lane) {
  static_assert(N >= 1 && N <= 64 && (N & (N - 1)) == 0, "power of two up to 64");
#pragma unroll
  for (int s = 0; s < 5; ++s) {
    const int o = 16 >> s;
    const int m = N >> s;  // values held before this step
    if (m >= 2) {
      const bool hi = (lane & o) != 0;
#pragma unroll
      for (int i = 0; i < (N + 1) / 2; ++i) {
        if (i < m / 2) {
          const float send = hi ? v[i] : v[i + m / 2];
          const float keep = hi ? v[i + m / 2] : v[i];
          v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, o);
        }
      }
    } else {
      v[0] += __shfl_xor_sync(0xFFFFFFFFu, v[0], o);
    }
  }
}

template <int N>
QG_DEVICE constexpr int rs_shift() {
  return N >= 32 ? 0 : N >= 16 ? 1 : N >= 8 ? 2 : N >= 4 ? 3 : N >= 2 ? 4 : 5;
}
// value index held in v[0] by this lane, and whether this lane is the one that owns it
template <int N>
QG_DEVICE int rs_index(int lane) {
  return N == 64 ? 2 * lane : (lane >> rs_shift<N>());
}
template <int N>
QG_DEVICE bool rs_owner(int lane) {
  return (lane & ((1 << rs_shift<N>()) - 1)) == 0;
}
