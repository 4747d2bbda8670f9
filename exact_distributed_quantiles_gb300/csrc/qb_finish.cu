// qb_finish.cu -- the EQB second pass from stored keys, the rank selects, the
// bias finalizers (EQB and K3), and small utility kernels.
//
// "Exact Quantile Balancing and Load-Error Injection for Mixture-of-Experts",
//   EQB paragraph: locate the hi-byte bin holding the r-th smallest value,
//   histogram the low byte within that bin, concatenate the two bytes.
// "[Dev] Add global-batch quantile balancing", "Quantile estimator" (quantile
//   at k/E, subtract the mean; K3 range [min b - 1, max b + 1]) and
//   "Implementation" (update bias and bounds once, reset the histogram in
//   place).
#include "qb_device.cuh"
#include "qb_internal.h"

namespace qb {
namespace {

// ------------------------------------------------------------------------
// Lo-byte histogram from stored keys.
//
// Each lane owns 8 consecutive experts (one 16-byte chunk of a key row); the
// selected hi byte of those experts sits in registers.  Matching keys are
// counted in a per-CTA shared histogram of 16-bit counters packed in pairs
// (two experts per 32-bit word), flushed with one global atomic per non-zero
// counter.  A CTA flushes at least every 65535 rows so no counter wraps.
// Pair-word layout: word(lo, p) = lo * (E/2) + (p & 3) * (E/8) + (p >> 2) with
// p = e/2, so for a fixed element index the 32 lanes hit 32 distinct banks.
// ------------------------------------------------------------------------
constexpr int kLoThreads = 1024;
constexpr int kLoEpochRows = 65535;

template <int E>
__device__ __forceinline__ int lo_word(int lo, int e) {
  const int p = e >> 1;
  return lo * (E / 2) + (p & 3) * (E / 8) + (p >> 2);
}

template <int E>
__global__ void __launch_bounds__(kLoThreads, 1)
    keys_hist_lo_kernel(const uint16_t* __restrict__ keys, int64_t N,
                        const int32_t* __restrict__ sel, int32_t* __restrict__ hist_lo,
                        int64_t rows_per_cta) {
  static_assert(E <= 256, "shared lo histogram sized for E <= 256");
  extern __shared__ __align__(16) uint32_t h[];
  constexpr int kWords = 256 * E / 2;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  constexpr int kWarps = kLoThreads / 32;
  // 32 chunks of 8 keys = 256 elements per warp step; E <= 256 divides it.
  const int e0 = (8 * lane) % E;
  uint32_t pat[4], valid[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int s0 = sel[e0 + 2 * i], s1 = sel[e0 + 2 * i + 1];
    pat[i] = ((uint32_t)(s0 & 0xFF) << 8) | ((uint32_t)(s1 & 0xFF) << 24);
    valid[i] = (s0 >= 0 ? 1u : 0u) | (s1 >= 0 ? 2u : 0u);
  }
  const int64_t r_begin = (int64_t)blockIdx.x * rows_per_cta;
  int64_t r_end = r_begin + rows_per_cta;
  if (r_end > N) r_end = N;
  constexpr int kRowsPerStep = 256 / E;
  for (int64_t ep = r_begin; ep < r_end; ep += kLoEpochRows) {
    const int64_t ep_end = (ep + kLoEpochRows < r_end) ? ep + kLoEpochRows : r_end;
    for (int i = threadIdx.x; i < kWords; i += kLoThreads) h[i] = 0;
    __syncthreads();
    // flat element range of this epoch, in 256-element warp steps
    const int64_t f_begin = ep * E, f_end = ep_end * E;
    const int64_t steps = (f_end - f_begin + 255) / 256;
    constexpr int kU = 4;  // 16-byte chunks in flight per lane
    for (int64_t st0 = (int64_t)warp * kU; st0 < steps; st0 += (int64_t)kWarps * kU) {
      uint4 u[kU];
#pragma unroll
      for (int q = 0; q < kU; ++q) {
        const int64_t f = f_begin + (st0 + q) * 256 + 8 * lane;
        u[q] = (f < f_end) ? __ldcs(reinterpret_cast<const uint4*>(keys + f))
                           : make_uint4(0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu);
      }
#pragma unroll
      for (int q = 0; q < kU; ++q) {
        const int64_t f = f_begin + (st0 + q) * 256 + 8 * lane;
        if (f >= f_end) continue;
        const uint32_t w[4] = {u[q].x, u[q].y, u[q].z, u[q].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t x = w[i] ^ pat[i];
          const bool m0 = ((x & 0x0000FF00u) == 0u) && (valid[i] & 1u);
          const bool m1 = ((x & 0xFF000000u) == 0u) && (valid[i] & 2u);
          if (m0) atomicAdd(&h[lo_word<E>(w[i] & 0xFF, e0 + 2 * i)], 1u);
          if (m1) atomicAdd(&h[lo_word<E>((w[i] >> 16) & 0xFF, e0 + 2 * i + 1)], 0x10000u);
        }
      }
    }
    (void)kRowsPerStep;
    __syncthreads();
    for (int i = threadIdx.x; i < kWords; i += kLoThreads) {
      const uint32_t c = h[i];
      if (c) {
        const int lo = i / (E / 2);
        const int q = i % (E / 2);
        const int p = (q % (E / 8)) * 4 + q / (E / 8);  // inverse of the pair permutation
        if (c & 0xFFFFu) atomicAdd(hist_lo + (int64_t)(2 * p) * 256 + lo, (int)(c & 0xFFFFu));
        if (c >> 16) atomicAdd(hist_lo + (int64_t)(2 * p + 1) * 256 + lo, (int)(c >> 16));
      }
    }
    __syncthreads();
  }
}

// E = 512: no shared privatisation (the packed histogram would need 256 KB).
__global__ void keys_hist_lo_global_kernel(const uint16_t* __restrict__ keys, int64_t N, int E,
                                           const int32_t* __restrict__ sel,
                                           int32_t* __restrict__ hist_lo) {
  const int64_t total = N * (int64_t)E;
  for (int64_t f = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; f < total;
       f += (int64_t)gridDim.x * blockDim.x) {
    const int e = (int)(f % E);
    const uint32_t key = keys[f];
    if ((int32_t)(key >> 8) == sel[e]) atomicAdd(hist_lo + (int64_t)e * 256 + (key & 0xFF), 1);
  }
}

// ------------------------------------------------------------------------
// Hi-byte rank select: one CTA (256 threads) per expert, inclusive scan.
// ------------------------------------------------------------------------
__device__ __forceinline__ long long block_inclusive_scan256(long long v, long long* tmp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
  if (lane == 31) tmp[warp] = v;
  __syncthreads();
  long long add = 0;
  for (int w = 0; w < warp; ++w) add += tmp[w];
  return v + add;
}

__global__ void __launch_bounds__(256) select_hi_kernel(const int32_t* __restrict__ hist_hi,
                                                        long long r, int32_t* __restrict__ sel,
                                                        int32_t* __restrict__ r_lo) {
  __shared__ long long tmp[8];
  __shared__ long long cum_s[256];
  const int j = blockIdx.x;
  const int b = threadIdx.x;
  const long long c = hist_hi[(int64_t)j * 256 + b];
  const long long cum = block_inclusive_scan256(c, tmp);
  cum_s[b] = cum;
  __syncthreads();
  const long long before = cum - c;
  if (cum >= r && before < r) {
    sel[j] = b;
    r_lo[j] = (int32_t)(r - before);
  }
  if (b == 255 && cum < r) {
    sel[j] = -1;
    r_lo[j] = 0;
  }
}

// ------------------------------------------------------------------------
// EQB finalize, two kernels.
// eqb_lo_select_kernel: one CTA (256 threads) per expert.  Block scan of the
//   lo histogram row, first bin reaching r_lo, key -> bf16 value q_j written
//   to bias_out[j] (a staging slot), key to qkey_out; with reset the CTA then
//   zeroes its own hist_hi and hist_lo rows in place.
// eqb_center_kernel: one CTA.  mu = (sum_j q_j in fp64, ascending j) / E,
//   bias_out[j] = RN32(q_j - mu).
// ------------------------------------------------------------------------
__device__ __forceinline__ float key_decode(uint32_t key) {
  const uint32_t h = (key & 0x8000u) ? (key ^ 0x8000u) : (key ^ 0xFFFFu);
  return __uint_as_float((h & 0xFFFFu) << 16);
}

__global__ void __launch_bounds__(256) eqb_lo_select_kernel(
    int32_t* __restrict__ hist_hi, int32_t* __restrict__ hist_lo, const int32_t* __restrict__ sel,
    const int32_t* __restrict__ r_lo, float* __restrict__ bias_out,
    uint16_t* __restrict__ qkey_out, int reset) {
  __shared__ long long tmp[8];
  __shared__ int lo_s;
  const int j = blockIdx.x;
  const int b = threadIdx.x;
  const int sj = sel[j];
  const long long target = r_lo[j];
  const long long c = hist_lo[(int64_t)j * 256 + b];
  if (b == 0) lo_s = -1;
  const long long cum = block_inclusive_scan256(c, tmp);  // contains __syncthreads
  if (cum >= target && cum - c < target) lo_s = b;
  __syncthreads();
  if (b == 0) {
    const int lo = lo_s;
    if (sj >= 0 && lo >= 0) {
      const uint32_t key = ((uint32_t)sj << 8) | (uint32_t)lo;
      bias_out[j] = key_decode(key);
      if (qkey_out) qkey_out[j] = (uint16_t)key;
    } else {
      bias_out[j] = __int_as_float(0x7FC00000);  // rank beyond the pooled count
      if (qkey_out) qkey_out[j] = 0;
    }
  }
  if (reset) {
    hist_lo[(int64_t)j * 256 + b] = 0;
    hist_hi[(int64_t)j * 256 + b] = 0;
  }
}

__global__ void __launch_bounds__(512) eqb_center_kernel(float* __restrict__ bias_out, int E) {
  __shared__ float q_s[512];
  __shared__ double mu_s;
  for (int j = threadIdx.x; j < E; j += blockDim.x) q_s[j] = bias_out[j];
  __syncthreads();
  if (threadIdx.x == 0) {
    double sum = 0.0;
    for (int j = 0; j < E; ++j) sum = __dadd_rn(sum, (double)q_s[j]);
    mu_s = __ddiv_rn(sum, (double)E);
  }
  __syncthreads();
  for (int j = threadIdx.x; j < E; j += blockDim.x)
    bias_out[j] = __double2float_rn(__dsub_rn((double)q_s[j], mu_s));
}

// First index where the inclusive prefix sum of the row reaches `target`, or
// -1; `before` receives the sum of the bins below it.  One warp.
__device__ int warp_first_reaching(const int32_t* __restrict__ row, int nbins, long long target,
                                   long long* before_out) {
  const int lane = threadIdx.x & 31;
  long long base = 0;
  for (int c0 = 0; c0 < nbins; c0 += 32) {
    const int b = c0 + lane;
    const long long c = (b < nbins) ? row[b] : 0;
    long long v = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += y;
    }
    const long long cum = base + v;
    const unsigned hit = __ballot_sync(0xffffffffu, b < nbins && cum >= target);
    if (hit) {
      const int src = __ffs(hit) - 1;
      const long long cum_at = __shfl_sync(0xffffffffu, cum, src);
      const long long c_at = __shfl_sync(0xffffffffu, c, src);
      *before_out = cum_at - c_at;
      return c0 + src;
    }
    base = __shfl_sync(0xffffffffu, cum, 31);
  }
  *before_out = base;
  return -1;
}

// ------------------------------------------------------------------------
// K3 finalize: one CTA of 1024 threads, warp per expert for the bin search,
// then serial fp64 centering and the new bounds.
// ------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) k3_finalize_kernel(const int32_t* __restrict__ hist, int E,
                                                          int nbins, long long r,
                                                          float* __restrict__ bounds,
                                                          float* __restrict__ bias_out) {
  __shared__ double q_s[512];
  __shared__ double mu_s;
  __shared__ float lo_s, hi_s;
  if (threadIdx.x == 0) {
    lo_s = bounds[0];
    hi_s = bounds[1];
  }
  __syncthreads();
  const double dlo = (double)lo_s;
  const double width = __ddiv_rn(__dsub_rn((double)hi_s, dlo), (double)nbins);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int j = warp; j < E; j += 32) {
    long long before = 0;
    const int32_t* row = hist + (int64_t)j * nbins;
    const int b = warp_first_reaching(row, nbins, r, &before);
    if (lane == 0) {
      if (b < 0) {
        q_s[j] = (double)hi_s;
      } else {
        const double edge = __dadd_rn(dlo, __dmul_rn((double)b, width));
        const double frac = __ddiv_rn((double)(r - before), (double)row[b]);
        q_s[j] = __dadd_rn(edge, __dmul_rn(width, frac));
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double sum = 0.0;
    for (int j = 0; j < E; ++j) sum = __dadd_rn(sum, q_s[j]);
    mu_s = __ddiv_rn(sum, (double)E);
  }
  __syncthreads();
  for (int j = threadIdx.x; j < E; j += blockDim.x)
    bias_out[j] = __double2float_rn(__dsub_rn(q_s[j], mu_s));
  __syncthreads();
  if (threadIdx.x == 0) {
    float mn = bias_out[0], mx = bias_out[0];
    for (int j = 1; j < E; ++j) {
      const float v = bias_out[j];
      mn = v < mn ? v : mn;
      mx = v > mx ? v : mx;
    }
    bounds[0] = __fsub_rn(mn, 1.0f);
    bounds[1] = __fadd_rn(mx, 1.0f);
  }
}

// ------------------------------------------------------------------------
// Utilities.
// ------------------------------------------------------------------------
__global__ void zero_i32_kernel(int32_t* __restrict__ p, int64_t n) {
  const int64_t n4 = n / 4;
  const bool al = (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (al) {
    for (int64_t i = tid; i < n4; i += stride) reinterpret_cast<int4*>(p)[i] = make_int4(0, 0, 0, 0);
    for (int64_t i = 4 * n4 + tid; i < n; i += stride) p[i] = 0;
  } else {
    for (int64_t i = tid; i < n; i += stride) p[i] = 0;
  }
}

// The pinned sigmoid through the same code the routing kernels run: chunks
// of 8 go through sigmoid8 (packed fast path when every |x| <= 86, the exact
// scalar path otherwise); a tail shorter than 8 uses the scalar path.
__global__ void sigmoid_kernel(const float* __restrict__ x, float* __restrict__ s, int64_t n) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t n8 = n / 8;
  for (int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c < n8; c += stride) {
    float xv[8], sv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) xv[i] = x[8 * c + i];
    sigmoid8(xv, sv);
#pragma unroll
    for (int i = 0; i < 8; ++i) s[8 * c + i] = sv[i];
  }
  for (int64_t i = 8 * n8 + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
    s[i] = sigmoid_pinned(x[i]);
}

}  // namespace

int launch_keys_hist_lo(const uint16_t* keys, int64_t N, int E, const int32_t* sel,
                        int32_t* hist_lo, cudaStream_t stream) {
  if (E == 512) {
    int64_t grid = (int64_t)sm_count() * 8;
    keys_hist_lo_global_kernel<<<(unsigned)grid, 256, 0, stream>>>(keys, N, E, sel, hist_lo);
    return launch_status();
  }
  const int64_t ctas_max = sm_count();
  // at least 32 rows per CTA so that flush work stays small against the pass
  int64_t ctas = (N + 31) / 32;
  if (ctas > ctas_max) ctas = ctas_max;
  if (ctas < 1) ctas = 1;
  const int64_t rows_per_cta = (N + ctas - 1) / ctas;
#define QB_LO(EE)                                                                            \
  case EE: {                                                                                 \
    const int smem = 256 * EE / 2 * 4;                                                       \
    static bool attr = false;                                                                \
    if (!attr) {                                                                             \
      if (cudaFuncSetAttribute(keys_hist_lo_kernel<EE>,                                      \
                               cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) \
        return launch_status();                                                              \
      attr = true;                                                                           \
    }                                                                                        \
    keys_hist_lo_kernel<EE><<<(unsigned)ctas, kLoThreads, smem, stream>>>(keys, N, sel, hist_lo, \
                                                                          rows_per_cta);     \
    return launch_status();                                                                  \
  }
  switch (E) {
    QB_LO(32)
    QB_LO(64)
    QB_LO(128)
    QB_LO(256)
    default:
      return QB_EUNSUPPORTED;
  }
#undef QB_LO
}

int launch_select_hi(const int32_t* hist_hi, int E, int64_t r, int32_t* sel, int32_t* r_lo,
                     cudaStream_t stream) {
  select_hi_kernel<<<E, 256, 0, stream>>>(hist_hi, (long long)r, sel, r_lo);
  return launch_status();
}

int launch_zero_i32(int32_t* p, int64_t n, cudaStream_t stream) {
  if (n <= 0) return QB_OK;
  int64_t grid = (n / 4 + 255) / 256;
  const int64_t gmax = (int64_t)sm_count() * 4;
  if (grid > gmax) grid = gmax;
  if (grid < 1) grid = 1;
  zero_i32_kernel<<<(unsigned)grid, 256, 0, stream>>>(p, n);
  return launch_status();
}

int launch_finalize(int32_t* hist_hi, int32_t* hist_lo, const int32_t* sel, const int32_t* r_lo,
                    int E, float* bias_out, uint16_t* qkey_out, int reset, cudaStream_t stream) {
  eqb_lo_select_kernel<<<E, 256, 0, stream>>>(hist_hi, hist_lo, sel, r_lo, bias_out, qkey_out,
                                              reset);
  int st = launch_status();
  if (st != QB_OK) return st;
  eqb_center_kernel<<<1, 512, 0, stream>>>(bias_out, E);
  return launch_status();
}

int launch_k3_finalize(int32_t* hist, int E, int nbins, int64_t r, float* bounds,
                       float* bias_out, int reset, cudaStream_t stream) {
  k3_finalize_kernel<<<1, 1024, 0, stream>>>(hist, E, nbins, (long long)r, bounds, bias_out);
  int st = launch_status();
  if (st != QB_OK || !reset) return st;
  return launch_zero_i32(hist, (int64_t)E * nbins, stream);
}

int launch_sigmoid(const float* x, float* s, int64_t n, cudaStream_t stream) {
  if (n <= 0) return QB_OK;
  int64_t grid = (n / 8 + 255) / 256 + 1;
  const int64_t gmax = (int64_t)sm_count() * 16;
  if (grid > gmax) grid = gmax;
  sigmoid_kernel<<<(unsigned)grid, 256, 0, stream>>>(x, s, n);
  return launch_status();
}

}  // namespace qb
