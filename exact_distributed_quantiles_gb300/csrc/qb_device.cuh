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
//   x = clamp(x, -104, 104)
//   t = fma(x, -log2e, 1.5*2^23);  n = t - 1.5*2^23       (n = rint(-x*log2e))
//   w = fma(n, ln2_hi, x);  w = fma(n, ln2_lo, w)         (Cody & Waite 1980;
//                                                          w = x + n*ln2)
//   p = sum_{i<=7} (-w)^i/i!, Horner in w with fma, coefficients RN((-1)^i/i!)
//   e = RN(p * 2^n)                      (+inf on overflow)
//   s = RN(1 / RN(1 + e))                (correctly rounded reciprocal)
// so s = 1/(1+exp(-x)).  Two implementations of the same function follow:
// a packed fast path for |x| <= 86 (no over/underflow in the scaling) and an
// exact scalar path for any input.
// ---------------------------------------------------------------------------
constexpr float kL2E = 0x1.715476p+0f;
constexpr float kMagic = 0x1.8p+23f;
constexpr float kLn2Hi = 0x1.62e4p-1f;
constexpr float kLn2Lo = 0x1.7f7d1cp-20f;
constexpr float kC0 = 0x1.0p+0f, kC1 = -0x1.0p+0f, kC2 = 0x1.0p-1f, kC3 = -0x1.555556p-3f,
                kC4 = 0x1.555556p-5f, kC5 = -0x1.111112p-7f, kC6 = 0x1.6c16c2p-10f,
                kC7 = -0x1.a01a02p-13f;
constexpr float kFastAbsX = 86.0f;  // |x| <= this: 2^n stays normal, p*2^n exact
// |x| <= this: every score is above 2^-100, so no margin can round to bf16 -0
constexpr float kFoldAbsX = 75.0f;

__device__ __forceinline__ float sigmoid_pinned(float x) {
  float xc = x > 104.0f ? 104.0f : x;
  xc = xc < -104.0f ? -104.0f : xc;
  const float t = __fmaf_rn(xc, -kL2E, kMagic);
  const float n = __fsub_rn(t, kMagic);
  float w = __fmaf_rn(n, kLn2Hi, xc);
  w = __fmaf_rn(n, kLn2Lo, w);
  float p = kC7;
  p = __fmaf_rn(p, w, kC6);
  p = __fmaf_rn(p, w, kC5);
  p = __fmaf_rn(p, w, kC4);
  p = __fmaf_rn(p, w, kC3);
  p = __fmaf_rn(p, w, kC2);
  p = __fmaf_rn(p, w, kC1);
  p = __fmaf_rn(p, w, kC0);
  const int ni = __float2int_rz(n);  // exact: n is an integer in [-151, 151]
  float e;
  if (ni >= -125 && ni <= 126) {
    e = __uint_as_float(__float_as_uint(p) + ((unsigned)ni << 23));
  } else if (ni > 126) {  // exact scale into range, then one rounding (may overflow)
    e = __fmul_rn(__uint_as_float(__float_as_uint(p) + ((unsigned)(ni - 64) << 23)), 0x1.0p+64f);
  } else {  // may be subnormal: one rounding
    e = __fmul_rn(__uint_as_float(__float_as_uint(p) + ((unsigned)(ni + 64) << 23)), 0x1.0p-64f);
  }
  return __frcp_rn(__fadd_rn(1.0f, e));
}

// ---- packed binary32 pairs (sm_100+ f32x2 instructions; same IEEE results
// as the scalar operations, two lanes per instruction)
typedef unsigned long long f2_t;

__device__ __forceinline__ f2_t f2_pack(float lo, float hi) {
  f2_t r;
  asm("mov.b64 %0, {%1,%2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(f2_t r, float& lo, float& hi) {
  asm("mov.b64 {%0,%1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ f2_t f2_fma(f2_t a, f2_t b, f2_t c) {
  f2_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ f2_t f2_add(f2_t a, f2_t b) {
  f2_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f2_t f2_sub(f2_t a, f2_t b) {
  f2_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f2_t f2_mul(f2_t a, f2_t b) {
  f2_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// Cluster barrier in two halves: every thread of every CTA of the cluster
// arrives, and waits until all have arrived.  arrive_relaxed orders nothing
// (it only records that the CTA is running); arrive_release makes this
// thread's earlier writes, distributed shared memory included, visible to
// the threads that then pass wait.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// round toward zero (used to truncate by adding 2^23)
__device__ __forceinline__ f2_t f2_add_rz(f2_t a, f2_t b) {
  f2_t d;
  asm("add.rz.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f2_t f2_splat(float v) { return f2_pack(v, v); }

// Hardware reciprocal estimate.  The .ftz form is the bare estimate; the
// callers only pass d in [1, 2^125), where input and result are normal and
// flushing never applies.
__device__ __forceinline__ float rcp_approx(float d) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(d));
  return y;
}

// -sigmoid of two inputs with |x| <= kFastAbsX, by the pinned sequence.
//  * 2^n is built from t's bit pattern: t = 1.5*2^23 + n and
//    (bits(1.5*2^23) << 23) == 0 mod 2^32, so bits(t)*2^23 + bits(1.0f) is
//    the pattern of 2^n (|n| <= 124 here, so 2^n is normal);
//  * d = fma(p, 2^n, 1) = RN(1 + e): e = p*2^n is exact (a power-of-two
//    scaling of a normal number), so this is the sequence's RN(1 + RN(e));
//  * the reciprocal RN(1/d) is the hardware estimate refined by one Newton
//    step (Markstein's method), taken on -d so that the sign folds in:
//    y' = est(1/(-d)) = -y, r = fma(d, y', 1) = RN(1 - d*y) and
//    fma(r, y', y') = -RN(y + r*y).
// That the result equals the correctly rounded reciprocal of the pinned d for
// every input (and that the estimate is odd in its argument) is checked by
// running qb_sigmoid, which uses this function, on every binary32 input
// against the oracle.
__device__ __forceinline__ f2_t neg_sigmoid2_fast(f2_t X) {
  const f2_t T = f2_fma(X, f2_splat(-kL2E), f2_splat(kMagic));
  const f2_t N = f2_sub(T, f2_splat(kMagic));
  f2_t W = f2_fma(N, f2_splat(kLn2Hi), X);
  W = f2_fma(N, f2_splat(kLn2Lo), W);
  f2_t P = f2_fma(f2_splat(kC7), W, f2_splat(kC6));
  P = f2_fma(P, W, f2_splat(kC5));
  P = f2_fma(P, W, f2_splat(kC4));
  P = f2_fma(P, W, f2_splat(kC3));
  P = f2_fma(P, W, f2_splat(kC2));
  P = f2_fma(P, W, f2_splat(kC1));
  P = f2_fma(P, W, f2_splat(kC0));
  float t0, t1;
  f2_unpack(T, t0, t1);
  const float s0 = __uint_as_float(__float_as_uint(t0) * 0x800000u + 0x3F800000u);
  const float s1 = __uint_as_float(__float_as_uint(t1) * 0x800000u + 0x3F800000u);
  const f2_t D = f2_fma(P, f2_pack(s0, s1), f2_splat(1.0f));
  float d0, d1;
  f2_unpack(D, d0, d1);
  const f2_t YN = f2_pack(rcp_approx(-d0), rcp_approx(-d1));
  const f2_t R = f2_fma(D, YN, f2_splat(1.0f));
  return f2_fma(R, YN, YN);
}

// sigmoid of two inputs with |x| <= kFastAbsX (the negation is exact).
__device__ __forceinline__ f2_t sigmoid2_fast(f2_t X) {
  return f2_sub(f2_splat(0.0f), neg_sigmoid2_fast(X));
}

__device__ __forceinline__ float max_abs8(const float (&x)[8]) {
  const float m = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
  return fmaxf(m, fmaxf(fmaxf(fabsf(x[4]), fabsf(x[5])), fmaxf(fabsf(x[6]), fabsf(x[7]))));
}

// Eight inputs in registers -> eight scores; the fast path when all |x| are
// small enough, the exact scalar path otherwise.  Returns max |x|.
__device__ __forceinline__ float sigmoid8(const float (&x)[8], float (&s)[8]) {
  const float m = max_abs8(x);
  if (m <= kFastAbsX) {
#pragma unroll
    for (int i = 0; i < 4; ++i) f2_unpack(sigmoid2_fast(f2_pack(x[2 * i], x[2 * i + 1])),
                                          s[2 * i], s[2 * i + 1]);
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) s[i] = sigmoid_pinned(x[i]);
  }
  return m;
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

// Plain arrive (count one) on a CTA-local mbarrier.
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
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

// Bounded wait: gives up after `polls` polls (by default 2^24, well over a
// second), records kDevTimeout in the device status word and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, int* status,
                                                  uint32_t polls = 1u << 24) {
  for (uint32_t it = 0; it < polls; ++it) {
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
