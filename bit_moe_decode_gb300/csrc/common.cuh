// common.cuh -- device helpers shared by the kernels of libmoe.so (sm_103a only).
// PTX wrappers for mbarriers, 1-D bulk copies (TMA engine, no tensor map), legacy-path tensor-core MMA used for
// the mat-vec work, conversions, and bounded waits that report a timeout instead of hanging.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>

#include "../../include/moe.h"

namespace moe {

// ------------------------------------------------------------------ workspace header (device scratch)
// Every FFN workspace starts with this header; the rest is carved out by the host (ffn.cu).
struct WsHeader {
  int32_t status;        // MOE_OK or a device error code
  uint32_t done;         // CTAs finished (the last one clears the per-call counters)
  uint32_t gbar;         // grid-wide barrier arrivals
  uint32_t pad[61];      // keep the counters on their own 256-byte line
};

// A device-side wait gives up after this many nanoseconds (2 s) unless a caller passes its own limit. On giving
// up it records MOE_ERR_DEVICE_TIMEOUT and the kernel unwinds without touching memory it does not own.
constexpr long long kDefaultWaitNs = 2000000000LL;

__device__ __forceinline__ long long globaltimer_ns() {
  long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void record_error(int32_t* status, int32_t code) {
  atomicCAS(status, 0, code);
}

// ------------------------------------------------------------------ shared-memory addresses, barriers
__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_u32(b)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(b)) : "memory");
}
// `n` arrivals at once
__device__ __forceinline__ void mbar_arrive_n(uint64_t* b, uint32_t n) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_u32(b)), "r"(n)
               : "memory");
}
// Arrive without release semantics: for a consumer handing back a buffer it only read through TMEM or that only
// the async proxy touched. A default (release) arrive would first wait until every global store the thread has in
// flight is performed, which under a saturated memory system costs about a microsecond.
__device__ __forceinline__ void mbar_arrive_relaxed(uint64_t* b) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.relaxed.cta.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(b))
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
// The same with a suspend-time hint: the thread sleeps until the phase completes or about `hint_ns` passed, so a
// waiting warp takes neither issue slots nor shared-memory bandwidth from the warps that work meanwhile.
__device__ __forceinline__ bool mbar_try_wait_hint(uint64_t* b, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(b)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}
// Non-blocking test of an mbarrier phase (mbarrier.test_wait never suspends the thread).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait on an mbarrier phase. Returns false if `limit_ns` nanoseconds passed first.
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity, long long limit_ns) {
  if (mbar_try_wait(b, parity)) return true;
  long long t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(b, parity)) return true;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// L2 policy: stream the expert weights through L2 with evict-first so small, reused data stays resident.
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 1-D bulk copy global -> shared through the TMA engine, completion counted on an mbarrier (bytes).
// dst, src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// Named barrier among `nthreads` threads (multiple of 32) with id `id` (1..15; 0 is __syncthreads).
__device__ __forceinline__ void named_bar(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Arrive at named barrier `id` without waiting (the waiting threads use bar.sync with the same count); the
// arriving threads' earlier memory accesses are ordered before the waiters' later ones.
__device__ __forceinline__ void named_bar_arrive(int id, int nthreads) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ------------------------------------------------------------------ global-memory flag helpers
__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Release add: the caller's earlier writes, and those ordered before it by a CTA or warp barrier, are visible to
// any thread that reads the counter with acquire semantics and sees the addition. Much cheaper under load than a
// full fence (__threadfence) followed by a relaxed atomic.
__device__ __forceinline__ void red_release_add(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t atom_acq_rel_add(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
// Wait until *p >= target; false on timeout.
__device__ __forceinline__ bool wait_counter(const uint32_t* p, uint32_t target, long long limit_ns) {
  if (ld_acquire_u32(p) >= target) return true;
  long long t0 = globaltimer_ns();
  while (true) {
    __nanosleep(32);
    if (ld_acquire_u32(p) >= target) return true;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// ------------------------------------------------------------------ tensor-core mat-vec primitive
// D = A(16x16, row) * B(16x8, col) + C, fp16 inputs, fp32 accumulate. Fragment ownership per lane l:
//   A: a0 = (row l/4, k 2(l%4)..+1), a1 = (row l/4+8, same k), a2 = (row l/4, k+8..+9), a3 = (row l/4+8, k+8..+9)
//   B: b0 = (k 2(l%4)..+1, col l/4), b1 = (k 2(l%4)+8..+9, col l/4)
//   C: c0,c1 = (row l/4, cols 2(l%4), 2(l%4)+1), c2,c3 = (row l/4+8, same cols)
// Each 32-bit register holds two fp16 values, the lower k (or lower column) in the low half.
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1, const float (&c)[4]) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%11,%12,%13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]), "f"(c[3]));
}

// Two E2M1 codes (low nibble = lower k) -> fp16x2 with the exact E2M1 values (hardware conversion).
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t word, int byte) {
  uint32_t d;
  switch (byte) {
    case 0: asm("{\n\t.reg .b8 a,b,c,e;\n\tmov.b32 {a,b,c,e}, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, a;\n\t}" : "=r"(d) : "r"(word)); break;
    case 1: asm("{\n\t.reg .b8 a,b,c,e;\n\tmov.b32 {a,b,c,e}, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b;\n\t}" : "=r"(d) : "r"(word)); break;
    case 2: asm("{\n\t.reg .b8 a,b,c,e;\n\tmov.b32 {a,b,c,e}, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, c;\n\t}" : "=r"(d) : "r"(word)); break;
    default: asm("{\n\t.reg .b8 a,b,c,e;\n\tmov.b32 {a,b,c,e}, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, e;\n\t}" : "=r"(d) : "r"(word)); break;
  }
  return d;
}

__device__ __forceinline__ uint32_t lop3_and_xor(uint32_t a, uint32_t mask, uint32_t x) {
  // (a & mask) ^ x
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0x6a;" : "=r"(d) : "r"(a), "r"(mask), "r"(x));
  return d;
}
__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Power-of-two rescale exponent: sigma such that amax * 2^sigma lies in [2^14, 2^15) for normal amax, clamped
// to [-126, 126] so both 2^sigma and 2^-sigma are representable fp32 values.
__device__ __forceinline__ int rescale_exponent(float amax) {
  uint32_t b = __float_as_uint(amax) & 0x7FFFFFFFu;
  int ef = (int)(b >> 23);                 // biased exponent; 0 for zero/subnormal, 255 for inf/nan
  int s = 141 - ef;                        // 14 - (ef - 127)
  if (ef == 0) s = 126;
  if (s > 126) s = 126;
  if (s < -126) s = -126;
  return s;
}
__device__ __forceinline__ float exp2i(int e) {  // 2^e for e in [-126, 127]
  return __uint_as_float((uint32_t)(e + 127) << 23);
}
__device__ __forceinline__ float exp2i_neg(int s) {  // 2^-s for s in [-126, 126]; s = 126 -> 2^-126 normal
  return __uint_as_float((uint32_t)(127 - s) << 23);
}

}  // namespace moe
