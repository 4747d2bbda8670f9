// qb_finish.cu -- the EQB second pass from stored keys, the hi-byte select,
// the EQB bias finalizer, rank-averaged QB, and small utility kernels (the
// K3 finalizer is in qb_k3.cu).
//
// "Exact Quantile Balancing and Load-Error Injection for Mixture-of-Experts",
//   EQB paragraph: locate the hi-byte bin holding the r-th smallest value,
//   histogram the low byte within that bin, concatenate the two bytes.
// "[Dev] Add global-batch quantile balancing", "Quantile estimator" (quantile
//   at k/E, subtract the mean; K3 range [min b - 1, max b + 1]) and
//   "Implementation" (update bias and bounds once, reset the histogram in
//   place).
#include <cooperative_groups.h>

#include "qb_device.cuh"
#include "qb_internal.h"

namespace qb {
namespace {

namespace cg = cooperative_groups;

// ------------------------------------------------------------------------
// Lo-byte histogram from stored keys.
//
// Work split: a CTA owns a column slice of 32 experts (64 bytes of every key
// row) over a range of tokens, so its shared histogram is only 32 x 256 int32
// counters and the flush issues few global atomics (merging 152 full
// per-SM histograms through L2 atomics would cost more than the pass itself).
// Four lanes cover one row slice (16 bytes = 8 keys each), a warp covers 8
// rows per load.  Loads run one iteration ahead in two register sets used in
// turn (no copies); iterations whose rows are all in range need no bounds
// checks.  Every key issues one shared increment without branching: with
// t = key ^ (sel << 8) the low byte is the key's, the high byte zero exactly
// when the key is in the selected bin, so min(t, 256) is the counter's index,
// or 256 -- the 257th word of the expert's row, never flushed -- for every
// other key.  Layout: counter (e, lo) at word e * 257 + lo (257 spreads the
// experts over the banks).
// ------------------------------------------------------------------------
constexpr int kLoThreads = 256;
constexpr int kLoEG = 32;                // experts per CTA slice
constexpr int kLoRowW = 257;             // words per expert row in shared memory
constexpr int kLoSmemWords = kLoEG * kLoRowW;

// No "memory" clobber: nothing reads the counters before the __syncthreads
// that precedes the flush, and without it the compiler may schedule the
// next loads ahead of the increments.
__device__ __forceinline__ void red_shared1(uint32_t addr) {
  asm volatile("red.shared.add.u32 [%0], 1;" ::"r"(addr));
}

// 16 key bytes through the read-only path, with a 256-byte L2 prefetch: the
// eight CTAs of a row range each read a 64-byte slice of the same 512-byte
// rows, and the prefetch brings a row's neighbouring slices into L2 ahead of
// them (4% faster than streaming 16-byte loads over 524288 x 256 keys).
__device__ __forceinline__ uint4 ld_keys16(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__global__ void __launch_bounds__(kLoThreads, 4)
    keys_hist_lo_kernel(const uint16_t* __restrict__ keys, int64_t N, int E,
                        const int32_t* __restrict__ sel, int32_t* __restrict__ hist_lo,
                        int64_t rows_per_cta) {
  __shared__ uint32_t h[kLoSmemWords];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  constexpr int kWarps = kLoThreads / 32;
  const int n_eg = E / kLoEG;
  const int eg = blockIdx.x % n_eg;
  const int64_t r_begin = (int64_t)(blockIdx.x / n_eg) * rows_per_cta;
  int64_t r_end = r_begin + rows_per_cta;
  if (r_end > N) r_end = N;
  const int c4 = lane & 3;    // which 8-key chunk of the 32-expert slice
  const int rsub = lane >> 2; // row within the warp's 8 rows
  const int el0 = 8 * c4;     // first local expert of this lane
  for (int i = threadIdx.x; i < kLoSmemWords; i += kLoThreads) h[i] = 0;
  // selected hi byte of each key pair, at the pair's hi-byte positions
  uint32_t spat[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    spat[i] = ((uint32_t)(sel[eg * kLoEG + el0 + 2 * i] & 0xFF) << 8) |
              ((uint32_t)(sel[eg * kLoEG + el0 + 2 * i + 1] & 0xFF) << 24);
  const uint32_t hb = (uint32_t)__cvta_generic_to_shared(h);
  uint32_t ebase[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) ebase[j] = hb + 4u * (uint32_t)((el0 + j) * kLoRowW);
  __syncthreads();

  const int64_t n_rows = r_end > r_begin ? r_end - r_begin : 0;
  const uint16_t* base = keys + r_begin * E + eg * kLoEG + el0;
  constexpr int kU = 4;                           // 8-row blocks per warp in flight
  const int64_t stride = (int64_t)kWarps * 8 * kU;  // rows per CTA iteration
  // rows r_first + it * stride + 8 q; in the first n_full iterations all kU
  // rows are in range (no checks, loads two iterations deep without copies)
  const int64_t r_first = (int64_t)warp * 8 * kU + rsub;
  const int64_t last_need = r_first + 8 * (kU - 1);
  const int64_t n_full = n_rows > last_need ? (n_rows - 1 - last_need) / stride + 1 : 0;
  const uint4* p4 = reinterpret_cast<const uint4*>(base + r_first * E);
  const int64_t q4 = E;                 // uint4 between q blocks (8 rows x E/8)
  const int64_t it4 = stride * (E / 8);  // uint4 per iteration
  auto load = [&](uint4 (&v)[kU], const uint4* p) {
#pragma unroll
    for (int q = 0; q < kU; ++q) v[q] = ld_keys16(p + q * q4);
  };
  auto count = [&](const uint4 (&v)[kU]) {
#pragma unroll
    for (int q = 0; q < kU; ++q) {
      const uint32_t w[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t x = w[i] ^ spat[i];  // selected hi bytes become 0
        red_shared1(ebase[2 * i] + 4u * min(x & 0xFFFFu, 256u));
        red_shared1(ebase[2 * i + 1] + 4u * min(x >> 16, 256u));
      }
    }
  };
  uint4 va[kU], vb[kU];
  int64_t it = 0;
  if (n_full > 0) load(va, p4);
  for (; it + 1 < n_full; it += 2) {
    load(vb, p4 + (it + 1) * it4);
    count(va);
    if (it + 2 < n_full) load(va, p4 + (it + 2) * it4);
    count(vb);
  }
  if (it < n_full) {
    count(va);
    ++it;
  }
  // the partial last iteration
  const int64_t r0 = r_first + it * stride;
#pragma unroll
  for (int q = 0; q < kU; ++q) {
    if (r0 + 8 * q < n_rows) {
      const uint4 v = ld_keys16(reinterpret_cast<const uint4*>(base + (r0 + 8 * q) * E));
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t x = w[i] ^ spat[i];
        red_shared1(ebase[2 * i] + 4u * min(x & 0xFFFFu, 256u));
        red_shared1(ebase[2 * i + 1] + 4u * min(x >> 16, 256u));
      }
    }
  }
  __syncthreads();
  // an expert without a selected bin (sel outside [0, 256)) counted the keys
  // of bin sel & 0xFF; its counts are dropped here
  for (int i = threadIdx.x; i < kLoEG * 256; i += kLoThreads) {
    const int el = i >> 8, lo = i & 255;
    const uint32_t c = h[el * kLoRowW + lo];
    const int se = sel[eg * kLoEG + el];
    if (c && se >= 0 && se < 256) atomicAdd(hist_lo + (int64_t)(eg * kLoEG + el) * 256 + lo, (int)c);
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
  const int j = blockIdx.x;
  const int b = threadIdx.x;
  const long long c = hist_hi[(int64_t)j * 256 + b];
  const long long cum = block_inclusive_scan256(c, tmp);
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
// EQB finalize: one cluster of 8 CTAs (1024 threads each), CTA c owning the
// experts [c*E/8, (c+1)*E/8), one warp per expert:
//   the warp scans the expert's lo histogram (8 consecutive bins per lane, a
//   shuffle scan over the lanes) for the first bin reaching r_lo, decodes the
//   key (sel << 8) | lo to the fp32 value q_j of its bf16 number, and with
//   reset zeroes the expert's hist_hi and hist_lo rows in place;
//   mu = (sum_j q_j in fp64) / E.  A bf16 number is m * 2^(e - 134) with an
//   8-bit m (e the biased exponent, 1 for subnormals), so when the non-zero
//   q_j's exponents span at most 36 (none inf or NaN) the sum is the integer
//   S = sum_j +-m_j * 2^(e_j - e_min) < 2^53 times 2^(e_min - 134), the
//   exact value of the ascending serial fp64 sum (which is then exact too),
//   and mu = RN(S * 2^(e_min - 134) / E) (a product by 2^-log2(E) when E is
//   a power of two).  Otherwise the ascending serial fp64 sum is taken.  Every CTA writes its q_j into every CTA's
//   shared memory (one cluster barrier), so each derives mu from all E
//   values by itself, the same way;
//   bias_out[j] = RN32(q_j - mu).
// ------------------------------------------------------------------------
constexpr int kFinCluster = 8;
constexpr int kFinThreads = 1024;
constexpr int kNoExp = 1 << 20;  // exponent-range sentinel of a CTA without non-zero q

__device__ __forceinline__ float key_decode(uint32_t key) {
  const uint32_t h = (key & 0x8000u) ? (key ^ 0x8000u) : (key ^ 0xFFFFu);
  return __uint_as_float((h & 0xFFFFu) << 16);
}

__global__ void __cluster_dims__(kFinCluster, 1, 1) __launch_bounds__(kFinThreads)
    eqb_finalize_kernel(int32_t* __restrict__ hist_hi, int32_t* __restrict__ hist_lo,
                        const int32_t* __restrict__ sel, const int32_t* __restrict__ r_lo, int E,
                        int log2E, float* __restrict__ bias_out, uint16_t* __restrict__ qkey_out,
                        int reset) {
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  __shared__ float q_s[kMaxE / kFinCluster];  // this CTA's quantiles
  __shared__ float q_all[kMaxE];              // every CTA's, pushed by their owners
  __shared__ double mu_s;
  // this CTA is running: other CTAs may write into its shared memory once
  // the matching wait has passed
  cluster_arrive_relaxed();
  const int per = E / kFinCluster;  // experts of this CTA (4 .. 128)
  const int j0 = rank * per;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int jl = warp; jl < per; jl += kFinThreads / 32) {
    const int j = j0 + jl;
    int32_t* row = hist_lo + (int64_t)j * 256;
    int c[8];
    int t = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      c[i] = row[8 * lane + i];
      t += c[i];
    }
    int incl = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const int target = r_lo[j];
    const unsigned hit = __ballot_sync(0xffffffffu, target >= 1 && incl >= target);
    int lo = -1;
    if (hit) {
      const int src = __ffs((int)hit) - 1;
      int off = 7, cum = incl - t;
#pragma unroll
      for (int i = 0, found = 0; i < 8; ++i) {  // the first i with cum + c[0..i] >= target
        cum += c[i];
        if (!found && cum >= target) {
          off = i;
          found = 1;
        }
      }
      lo = __shfl_sync(0xffffffffu, 8 * src + off, src);
    }
    if (lane == 0) {
      const int sj = sel[j];
      if (sj >= 0 && sj < 256 && lo >= 0) {
        const uint32_t key = ((uint32_t)sj << 8) | (uint32_t)lo;
        q_s[jl] = key_decode(key);
        if (qkey_out) qkey_out[j] = (uint16_t)key;
      } else {
        q_s[jl] = __int_as_float(0x7FC00000);  // rank beyond the pooled count
        if (qkey_out) qkey_out[j] = 0;
      }
    }
    if (reset) {
      int32_t* rh = hist_hi + (int64_t)j * 256;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        row[32 * i + lane] = 0;
        rh[32 * i + lane] = 0;
      }
    }
  }
  __syncthreads();
  // every CTA has started: push this CTA's quantiles into every CTA, then
  // one cluster barrier makes them visible everywhere
  cluster_wait();
  for (int t = threadIdx.x; t < per * kFinCluster; t += kFinThreads) {
    const int c = t / per, jl = t - c * per;
    *cluster.map_shared_rank(q_all + j0 + jl, c) = q_s[jl];
  }
  cluster_arrive_release();
  cluster_wait();
  // every CTA derives the same mean from all E quantiles
  if (warp == 0) {
    uint32_t u[kMaxE / 32];
    int bad = 0, emin = kNoExp, emax = -kNoExp;
#pragma unroll
    for (int h = 0; h < kMaxE / 32; ++h) {
      const int j = lane + 32 * h;
      u[h] = j < E ? __float_as_uint(q_all[j]) : 0u;
      const int ex = (int)((u[h] >> 23) & 0xFFu);
      bad |= ex == 0xFF;
      if (u[h] & 0x7FFFFFFFu) {
        emin = min(emin, ex);
        emax = max(emax, ex);
      }
    }
    bad = __reduce_or_sync(0xffffffffu, bad);
    emin = (int)__reduce_min_sync(0xffffffffu, (unsigned)emin);
    emax = __reduce_max_sync(0xffffffffu, emax);
    double mu;
    if (!bad && emin == kNoExp) {
      mu = 0.0;  // every q_j is zero
    } else if (!bad && emax - emin <= 36) {
      const int base_e = max(emin, 1);
      long long S = 0;
#pragma unroll
      for (int h = 0; h < kMaxE / 32; ++h) {
        if (u[h] & 0x7FFFFFFFu) {
          const int ex = (int)((u[h] >> 23) & 0xFFu);
          const long long m = (long long)(((u[h] >> 16) & 0x7Fu) | (ex ? 0x80u : 0u));
          const long long term = m << (max(ex, 1) - base_e);
          S += (u[h] >> 31) ? -term : term;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) S += __shfl_xor_sync(0xffffffffu, S, o);
      if (log2E >= 0) {
        // 2^(base_e - 134 - log2 E) as a double (a normal number for every base_e)
        const double scale = __longlong_as_double((long long)(base_e - 134 - log2E + 1023) << 52);
        mu = __dmul_rn((double)S, scale);
      } else {
        // the exact sum S * 2^(base_e - 134) (a normal double), divided once
        const double scale = __longlong_as_double((long long)(base_e - 134 + 1023) << 52);
        mu = __ddiv_rn(__dmul_rn((double)S, scale), (double)E);
      }
    } else {
      double sum = 0.0;
      if (lane == 0)
        for (int j = 0; j < E; ++j) sum = __dadd_rn(sum, (double)q_all[j]);
      mu = __ddiv_rn(sum, (double)E);
    }
    if (lane == 0) mu_s = mu;
  }
  __syncthreads();
  const double mu = mu_s;
  for (int jl = threadIdx.x; jl < per; jl += kFinThreads)
    bias_out[j0 + jl] = __double2float_rn(__dsub_rn((double)q_s[jl], mu));
}

// ------------------------------------------------------------------------
// Rank-averaged QB: each rank's selected key (qb_finalize's qkey_out) decoded,
// averaged over the ranks in rank order in fp64, then centred like the pooled
// method (serial ascending fp64 mean, as the plain definition does it; one
// call per global batch).
// ------------------------------------------------------------------------
__global__ void __launch_bounds__(512) rank_average_kernel(const uint16_t* __restrict__ qkeys,
                                                           int P, int E,
                                                           float* __restrict__ bias_out) {
  __shared__ double avg_s[kMaxE];
  __shared__ double mu_s;
  for (int j = threadIdx.x; j < E; j += blockDim.x) {
    double s = 0.0;
    for (int p = 0; p < P; ++p) s = __dadd_rn(s, (double)key_decode(qkeys[(int64_t)p * E + j]));
    avg_s[j] = __ddiv_rn(s, (double)P);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double sum = 0.0;
    for (int j = 0; j < E; ++j) sum = __dadd_rn(sum, avg_s[j]);
    mu_s = __ddiv_rn(sum, (double)E);
  }
  __syncthreads();
  for (int j = threadIdx.x; j < E; j += blockDim.x)
    bias_out[j] = __double2float_rn(__dsub_rn(avg_s[j], mu_s));
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
// scalar path otherwise); a tail shorter than 8 uses the scalar path.  With
// `scalar` set every element takes the exact scalar path, which the routing
// kernels run for a whole warp-chunk as soon as one of its inputs is large.
__global__ void sigmoid_kernel(const float* __restrict__ x, float* __restrict__ s, int64_t n,
                               int scalar) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t n8 = n / 8;
  for (int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c < n8; c += stride) {
    float xv[8], sv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) xv[i] = x[8 * c + i];
    if (scalar) {
#pragma unroll
      for (int i = 0; i < 8; ++i) sv[i] = sigmoid_pinned(xv[i]);
    } else {
      sigmoid8(xv, sv);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) s[8 * c + i] = sv[i];
  }
  for (int64_t i = 8 * n8 + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
    s[i] = sigmoid_pinned(x[i]);
}

// The bounded-wait path on demand: one warp waits on an mbarrier that
// nothing completes (no arrival, no copy issued against it) with a short poll
// limit, so the wait gives up, sets kDevTimeout and the kernel returns.
__global__ void wait_timeout_selftest_kernel(int* status, uint32_t polls) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncwarp();
  (void)mbar_wait_bounded(&bar, 0u, status, polls);
}

}  // namespace

int launch_wait_timeout_selftest(uint32_t polls, cudaStream_t stream) {
  int* status = device_status_ptr();
  if (!status) return QB_ECUDA;
  wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(status, polls);
  return launch_status();
}

int launch_keys_hist_lo(const uint16_t* keys, int64_t N, int E, const int32_t* sel,
                        int32_t* hist_lo, cudaStream_t stream) {
  if (E < kLoEG) {  // E = 32 is one slice already; smaller E is not supported
    if (E != 32) return QB_EUNSUPPORTED;
  }
  const int n_eg = E / kLoEG;
  // about four CTAs per SM, at least 64 rows per CTA
  int64_t n_tr = ((int64_t)sm_count() * 4 + n_eg - 1) / n_eg;
  const int64_t max_tr = (N + 63) / 64;
  if (n_tr > max_tr) n_tr = max_tr;
  if (n_tr < 1) n_tr = 1;
  const int64_t rows_per_cta = (N + n_tr - 1) / n_tr;
  keys_hist_lo_kernel<<<(unsigned)(n_tr * n_eg), kLoThreads, 0, stream>>>(keys, N, E, sel, hist_lo,
                                                                        rows_per_cta);
  return launch_status();
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
  if (E % kFinCluster != 0 || E > kMaxE) return QB_EUNSUPPORTED;
  int log2E = 0;
  while ((1 << log2E) < E) ++log2E;
  if ((1 << log2E) != E) log2E = -1;  // not a power of two: the mean divides
  eqb_finalize_kernel<<<kFinCluster, kFinThreads, 0, stream>>>(hist_hi, hist_lo, sel, r_lo, E, log2E,
                                                               bias_out, qkey_out, reset);
  return launch_status();
}

int launch_rank_average(const uint16_t* qkeys, int P, int E, float* bias_out,
                        cudaStream_t stream) {
  rank_average_kernel<<<1, 512, 0, stream>>>(qkeys, P, E, bias_out);
  return launch_status();
}

int launch_sigmoid(const float* x, float* s, int64_t n, int scalar, cudaStream_t stream) {
  if (n <= 0) return QB_OK;
  int64_t grid = (n / 8 + 255) / 256 + 1;
  const int64_t gmax = (int64_t)sm_count() * 16;
  if (grid > gmax) grid = gmax;
  sigmoid_kernel<<<(unsigned)grid, 256, 0, stream>>>(x, s, n, scalar);
  return launch_status();
}

}  // namespace qb
