// qb_device.cuh -- device-side building blocks of libqb (sm_103a).
//
// Pinned logistic function, BF16 rounding and the order-preserving key,
// inline-PTX wrappers for mbarriers and bulk async copies, and the device
// status word that bounded waits report into.
//
// Sources, cited by page title and section:
//   "[Dev] Add global-batch quantile balancing" (Megatron-LM PR 6637),
//     "Quantile estimator": s = raw sigmoid score, alpha = (k+1)-th largest of
//     s + b, r = alpha - s, quantile at k/E, mean-centering.
//   "Exact Quantile Balancing and Load-Error Injection for Mixture-of-Experts",
//     EQB paragraph: order-preserving BF16 bit patterns, hi-byte then lo-byte
//     256-bin histograms.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace qb {

// Device status word (one int in device memory, owned by the library's API
// translation unit and passed to kernels by pointer): bit flags that kernels
// set instead of trapping.
enum : int {
  kDevTimeout = 1,  // a bounded wait on an mbarrier gave up
};

// ---------------------------------------------------------------------------
// Pinned logistic function.
//
// One fixed sequence of IEEE-754 binary32 operations (round to nearest even,
// no flush to zero), so that every score -- and with it every margin and
// every histogram count -- is reproducible bit for bit:
//   a = min(|x|, 104);  z = -a
//   t = fma(z, log2e, 1.5*2^23);  n = t - 1.5*2^23        (n = rint(z*log2e))
//   u = fma(n, -ln2_hi, z);  u = fma(n, -ln2_lo, u)       (Cody & Waite 1980)
//   p = degree-7 Taylor polynomial of exp(u), Horner form with fma,
//       coefficients RN(1/i!)
//   e = RN(p * 2^n)           (exact exponent add; one rounding if subnormal)
//   s = RN(num / RN(1 + e)),  num = 1 for x >= 0, e otherwise.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float exp_neg_abs(float x) {
  constexpr float kL2E = 0x1.715476p+0f;
  constexpr float kMagic = 0x1.8p+23f;
  constexpr float kLn2Hi = 0x1.62e4p-1f;
  constexpr float kLn2Lo = 0x1.7f7d1cp-20f;
  float a = fabsf(x);
  a = a > 104.0f ? 104.0f : a;
  const float z = -a;
  const float t = __fmaf_rn(z, kL2E, kMagic);
  const float n = __fsub_rn(t, kMagic);
  float u = __fmaf_rn(n, -kLn2Hi, z);
  u = __fmaf_rn(n, -kLn2Lo, u);
  float p = 0x1.a01a02p-13f;          // 1/7!
  p = __fmaf_rn(p, u, 0x1.6c16c2p-10f);  // 1/6!
  p = __fmaf_rn(p, u, 0x1.111112p-7f);   // 1/5!
  p = __fmaf_rn(p, u, 0x1.555556p-5f);   // 1/4!
  p = __fmaf_rn(p, u, 0x1.555556p-3f);   // 1/3!
  p = __fmaf_rn(p, u, 0x1.0p-1f);        // 1/2!
  p = __fmaf_rn(p, u, 1.0f);             // 1/1!
  p = __fmaf_rn(p, u, 1.0f);             // 1/0!
  const int ni = __float2int_rz(n);   // exact: n is an integer in [-151, 0]
  if (ni >= -125) return __int_as_float(__float_as_int(p) + (ni << 23));
  // Result may be subnormal: scale exactly into the normal range, then apply
  // the remaining power of two with one correctly rounded multiply.
  const float q = __int_as_float(__float_as_int(p) + ((ni + 64) << 23));
  return __fmul_rn(q, 0x1.0p-64f);
}

__device__ __forceinline__ float sigmoid_pinned(float x) {
  const float e = exp_neg_abs(x);
  const float d = __fadd_rn(1.0f, e);
  const float num = (x >= 0.0f) ? 1.0f : e;
  return __fdiv_rn(num, d);
}

// ---------------------------------------------------------------------------
// BF16 rounding and the order-preserving key.
// ---------------------------------------------------------------------------

// Two fp32 values -> packed bf16x2 (round to nearest even): lo in bits 0-15.
__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Packed bf16x2 -> packed key pair.  Each 16-bit half h becomes
//   h == 0x8000 (-0) -> 0x8000 (same key as +0)
//   sign clear       -> h ^ 0x8000
//   sign set         -> h ^ 0xFFFF
// so that unsigned key order is numeric order.
__device__ __forceinline__ uint32_t keys_from_bf16x2(uint32_t w) {
  // bit 15 of each half is set iff that half's magnitude is non-zero
  const uint32_t nz = (w & 0x7FFF7FFFu) + 0x7FFF7FFFu;
  w &= (nz | 0x7FFF7FFFu);                  // -0 -> +0
  const uint32_t sgn = prmt(w, 0u, 0xBB99u);  // 0xFFFF per negative half
  return w ^ (sgn | 0x80008000u);
}

__device__ __forceinline__ uint32_t key_of(float r) {
  return keys_from_bf16x2(bf16x2_rn(r, 0.0f)) & 0xFFFFu;
}

// ---------------------------------------------------------------------------
// mbarrier / bulk-copy wrappers (inline PTX).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// One try_wait on the given phase parity; true once that phase has completed.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
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

// Bounded wait: gives up after ~2^24 polls (well over a second), records
// kDevTimeout in the device status word and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, int* status) {
  for (uint32_t it = 0; it < (1u << 24); ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if (it > 64) __nanosleep(64);
  }
  atomicOr(status, kDevTimeout);
  return false;
}

// Global -> shared bulk copy (no tensor map), completion counted on `bar`.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src_gmem, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst_smem)),
      "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ int lane_id() { return threadIdx.x & 31; }

}  // namespace qb
