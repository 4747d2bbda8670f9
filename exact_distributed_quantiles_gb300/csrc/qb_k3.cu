// qb_k3.cu -- K3 histogram mode: counting the stored bin indices, and the
// finalize (interpolated quantile, centering, next bounds).
//
// "[Dev] Add global-batch quantile balancing", "Quantile estimator": a uniform
// histogram of nbins (1000) bins per expert over [min(b) - 1, max(b) + 1]; the
// quantile is read off the bin where the cumulative count reaches the rank
// and interpolated inside it; the new bias is centred and the next bounds
// follow it.  "Implementation": the counts accumulate over the microbatches
// of a global batch in one persistent histogram that is reset in place.
//
// Counting.  The route pass in K3 mode stores one uint16 bin index per
// (token, expert) in a caller workspace.  A [E, nbins] histogram (1 MB at
// E = 256, nbins = 1000) does not fit in shared memory, so a CTA owns a
// slice of EG experts over a range of tokens (EG x nbins int32 counters in
// shared memory) and adds each non-zero counter to the global histogram once
// at the end.  The flush costs one L2 atomic per non-zero counter per CTA, so
// the grid is one CTA per SM: fewer, longer CTAs mean fewer flushed counters.
//
// Finalize.  One cluster of 8 CTAs: a warp per expert finds the bin (blocks
// of 128 bins, coalesced loads, a warp scan per block), the
// fp64 quantiles are summed per CTA and the 8 partial sums are combined
// through distributed shared memory in rank order, so every CTA derives the
// same mean; min and max of the new bias go through the cluster the same way.
#include <cooperative_groups.h>

#include "qb_device.cuh"
#include "qb_internal.h"

namespace cg = cooperative_groups;

namespace qb {
namespace {

constexpr int kCountThreads = 1024;
constexpr int kCountSmemMax = 200 * 1024;

// No "memory" clobber: the counters are read only after a __syncthreads.
__device__ __forceinline__ void red_shared_u32(uint32_t addr, uint32_t v) {
  asm volatile("red.shared.add.u32 [%0], %1;" ::"r"(addr), "r"(v));
}

// EG experts per CTA (8 or 16): EG / 8 lanes per row, each lane reads 8
// consecutive indices (16 bytes) of its row.  Counter (e, b) sits at word
// e * row_w + b, row_w odd so that equal bins of different experts fall in
// different banks.
template <int EG>
__global__ void __launch_bounds__(kCountThreads, 1)
    k3_count_kernel(const uint16_t* __restrict__ bins, int64_t N, int E, int nbins, int row_w,
                    int32_t* __restrict__ hist, int64_t rows_per_cta) {
  extern __shared__ uint32_t h[];
  constexpr int LPR = EG / 8;
  constexpr int RPW = 32 / LPR;  // rows per warp per load
  constexpr int kWarps = kCountThreads / 32;
  constexpr int kU = 4;          // loads in flight per lane
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int n_eg = E / EG;
  const int eg = blockIdx.x % n_eg;
  const int64_t r_begin = (int64_t)(blockIdx.x / n_eg) * rows_per_cta;
  int64_t r_end = r_begin + rows_per_cta;
  if (r_end > N) r_end = N;
  const uint32_t last = (uint32_t)(nbins - 1);
  const int chunk = lane % LPR;
  const int rsub = lane / LPR;
  for (int i = threadIdx.x; i < EG * row_w; i += kCountThreads) h[i] = 0;
  const uint32_t hb = (uint32_t)__cvta_generic_to_shared(h);
  uint32_t ebase[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) ebase[j] = hb + 4u * (uint32_t)((8 * chunk + j) * row_w);
  __syncthreads();

  const int64_t n_rows = r_end > r_begin ? r_end - r_begin : 0;
  const uint16_t* base = bins + r_begin * E + eg * EG + 8 * chunk;
  const int64_t stride = (int64_t)kWarps * RPW * kU;
  int64_t r0 = (int64_t)warp * RPW * kU + rsub;
  uint4 cur[kU];
#pragma unroll
  for (int q = 0; q < kU; ++q) {
    const int64_t r = r0 + RPW * q;
    cur[q] = r < n_rows ? __ldcs(reinterpret_cast<const uint4*>(base + r * E))
                        : make_uint4(0u, 0u, 0u, 0u);
  }
  for (; r0 < n_rows; r0 += stride) {
    uint4 nxt[kU];
#pragma unroll
    for (int q = 0; q < kU; ++q) {
      const int64_t r = r0 + stride + RPW * q;
      nxt[q] = r < n_rows ? __ldcs(reinterpret_cast<const uint4*>(base + r * E))
                          : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int q = 0; q < kU; ++q) {
      if (r0 + RPW * q < n_rows) {
        const uint32_t w[4] = {cur[q].x, cur[q].y, cur[q].z, cur[q].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {  // min() keeps a stray index inside the slice
          red_shared_u32(ebase[2 * i] + 4u * min(w[i] & 0xFFFFu, last), 1u);
          red_shared_u32(ebase[2 * i + 1] + 4u * min(w[i] >> 16, last), 1u);
        }
      }
      cur[q] = nxt[q];
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < EG * nbins; i += kCountThreads) {
    const int el = i / nbins, b = i - el * nbins;
    const uint32_t c = h[el * row_w + b];
    if (c) atomicAdd(hist + (int64_t)(eg * EG + el) * nbins + b, (int)c);
  }
}

// Bins too many for a shared slice of 8 experts: one global atomic per index.
__global__ void k3_count_global_kernel(const uint16_t* __restrict__ bins, int64_t n_elem, int E,
                                       int nbins, int32_t* __restrict__ hist) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_elem; i += stride) {
    const int e = (int)(i % E);
    atomicAdd(hist + (int64_t)e * nbins + min((int)bins[i], nbins - 1), 1);
  }
}

// ---- finalize -------------------------------------------------------------
constexpr int kFinCluster = 8;
constexpr int kFinThreads = 1024;

// First bin whose cumulative count reaches `target` (-1 if none) and the
// count below it.  The row goes in pieces of 8 blocks of 128 bins; lane l
// holds bins 4l..4l+3 of every block (coalesced 16-byte loads, all eight
// issued before any is used), a warp scan per block finds the block and the
// lane that hold the bin, and that lane checks its four counts.
__device__ int warp_find_bin(const int32_t* __restrict__ row, int nbins, long long target,
                             long long* before_out) {
  const int lane = threadIdx.x & 31;
  const bool vec = (reinterpret_cast<uintptr_t>(row) & 15u) == 0;
  unsigned long long base = 0;
  for (int p0 = 0; p0 < nbins; p0 += 8 * 128) {
    int4 v[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int b = p0 + q * 128 + 4 * lane;
      if (vec && b + 3 < nbins) {
        v[q] = *reinterpret_cast<const int4*>(row + b);
      } else {
        v[q].x = b < nbins ? row[b] : 0;
        v[q].y = b + 1 < nbins ? row[b + 1] : 0;
        v[q].z = b + 2 < nbins ? row[b + 2] : 0;
        v[q].w = b + 3 < nbins ? row[b + 3] : 0;
      }
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const unsigned s = (unsigned)v[q].x + (unsigned)v[q].y + (unsigned)v[q].z + (unsigned)v[q].w;
      unsigned incl = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const unsigned long long cum = base + incl;
      const unsigned hit = __ballot_sync(0xffffffffu, (long long)cum >= target);
      if (hit) {
        const int src = __ffs(hit) - 1;
        const unsigned long long r0 = cum - s;
        const unsigned long long r1 = r0 + (unsigned)v[q].x;
        const unsigned long long r2 = r1 + (unsigned)v[q].y;
        const unsigned long long r3 = r2 + (unsigned)v[q].z;
        const int b = p0 + q * 128 + 4 * lane;
        int off;
        unsigned long long before;
        if ((long long)r1 >= target) {
          off = 0; before = r0;
        } else if ((long long)r2 >= target) {
          off = 1; before = r1;
        } else if ((long long)r3 >= target) {
          off = 2; before = r2;
        } else {
          off = 3; before = r3;
        }
        *before_out = (long long)__shfl_sync(0xffffffffu, before, src);
        return __shfl_sync(0xffffffffu, b + off, src);
      }
      base += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  *before_out = (long long)base;
  return -1;
}

__global__ void __cluster_dims__(kFinCluster, 1, 1) __launch_bounds__(kFinThreads)
    k3_finalize_kernel(int32_t* __restrict__ hist, int E, int nbins, double inv_nbins, long long r,
                       float* __restrict__ bounds, float* __restrict__ bias_out, int reset) {
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  __shared__ double q_s[64];
  __shared__ float b_s[64];
  __shared__ double part_s;
  __shared__ float min_s, max_s;
  const int per = E / kFinCluster;  // experts of this CTA (4 .. 64)
  const int j0 = rank * per;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float lo = bounds[0], hi = bounds[1];
  const double dlo = (double)lo;
  // No fp64 division on this path (each costs microseconds of dependent fp64
  // latency here): width uses the host's RN(1/nbins) and the in-bin fraction
  // is an fp32 quotient; either differs from the divided form by far less
  // than the mode's tolerance (the fraction is scaled by width, ~1e-3).
  const double width = __dmul_rn(__dsub_rn((double)hi, dlo), inv_nbins);
  for (int jl = warp; jl < per; jl += kFinThreads / 32) {
    int32_t* row = hist + (int64_t)(j0 + jl) * nbins;
    long long before = 0;
    const int b = warp_find_bin(row, nbins, r, &before);
    if (lane == 0) {
      if (b < 0) {
        q_s[jl] = (double)hi;
      } else {
        const double edge = __dadd_rn(dlo, __dmul_rn((double)b, width));
        const double frac = (double)__fdiv_rn((float)(r - before), (float)row[b]);
        q_s[jl] = __dadd_rn(edge, __dmul_rn(width, frac));
      }
    }
    __syncwarp();
    if (reset)
      for (int i = lane; i < nbins; i += 32) row[i] = 0;
  }
  __syncthreads();
  if (warp == 0) {
    double v = lane < per ? q_s[lane] : 0.0;
    if (lane + 32 < per) v = __dadd_rn(v, q_s[lane + 32]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = __dadd_rn(v, __shfl_down_sync(0xffffffffu, v, o));
    if (lane == 0) part_s = v;
  }
  cluster.sync();
  // every CTA adds the eight partial sums in rank order: the same mean everywhere
  double sum = 0.0;
#pragma unroll
  for (int c = 0; c < kFinCluster; ++c) sum = __dadd_rn(sum, *cluster.map_shared_rank(&part_s, c));
  const double mu = __dmul_rn(sum, 1.0 / (double)E);  // E is a power of two: exact
  for (int jl = threadIdx.x; jl < per; jl += kFinThreads) {
    const float b = __double2float_rn(__dsub_rn(q_s[jl], mu));
    b_s[jl] = b;
    bias_out[j0 + jl] = b;
  }
  __syncthreads();
  if (warp == 0) {
    float mn = lane < per ? b_s[lane] : INFINITY;
    float mx = lane < per ? b_s[lane] : -INFINITY;
    if (lane + 32 < per) {
      mn = fminf(mn, b_s[lane + 32]);
      mx = fmaxf(mx, b_s[lane + 32]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    if (lane == 0) {
      min_s = mn;
      max_s = mx;
    }
  }
  // every CTA has read the old bounds (above) before rank 0 writes new ones
  cluster.sync();
  if (rank == 0 && threadIdx.x == 0) {
    float mn = min_s, mx = max_s;
    for (int c = 1; c < kFinCluster; ++c) {
      mn = fminf(mn, *cluster.map_shared_rank(&min_s, c));
      mx = fmaxf(mx, *cluster.map_shared_rank(&max_s, c));
    }
    bounds[0] = __fsub_rn(mn, 1.0f);
    bounds[1] = __fadd_rn(mx, 1.0f);
  }
  cluster.sync();  // keep every CTA's shared memory alive until rank 0 has read it
}

template <int EG>
int launch_count(const uint16_t* bins, int64_t N, int E, int nbins, int row_w, int32_t* hist,
                 cudaStream_t stream) {
  const int smem = EG * row_w * 4;
  static int attr_bytes = 0;  // per instantiation; benign race (idempotent)
  if (smem > attr_bytes) {
    if (cudaFuncSetAttribute(k3_count_kernel<EG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem) != cudaSuccess)
      return launch_status();
    attr_bytes = smem;
  }
  const int n_eg = E / EG;
  int64_t n_tr = sm_count() / n_eg;
  const int64_t max_tr = (N + 255) / 256;  // at least 256 rows per CTA
  if (n_tr > max_tr) n_tr = max_tr;
  if (n_tr < 1) n_tr = 1;
  const int64_t rows_per_cta = (N + n_tr - 1) / n_tr;
  k3_count_kernel<EG><<<(unsigned)(n_tr * n_eg), kCountThreads, smem, stream>>>(
      bins, N, E, nbins, row_w, hist, rows_per_cta);
  return launch_status();
}

}  // namespace

int launch_k3_count(const uint16_t* bins, int64_t N, int E, int nbins, int32_t* hist,
                    cudaStream_t stream) {
  const int row_w = nbins | 1;
  if (16 * row_w * 4 <= kCountSmemMax) return launch_count<16>(bins, N, E, nbins, row_w, hist, stream);
  if (8 * row_w * 4 <= kCountSmemMax) return launch_count<8>(bins, N, E, nbins, row_w, hist, stream);
  const int64_t n_elem = N * E;
  int64_t grid = (n_elem + 255) / 256;
  const int64_t gmax = (int64_t)sm_count() * 8;
  if (grid > gmax) grid = gmax;
  k3_count_global_kernel<<<(unsigned)grid, 256, 0, stream>>>(bins, n_elem, E, nbins, hist);
  return launch_status();
}

int launch_k3_finalize(int32_t* hist, int E, int nbins, int64_t r, float* bounds, float* bias_out,
                       int reset, cudaStream_t stream) {
  if (E % kFinCluster != 0 || E / kFinCluster > 64) return QB_EUNSUPPORTED;
  k3_finalize_kernel<<<kFinCluster, kFinThreads, 0, stream>>>(hist, E, nbins, 1.0 / (double)nbins,
                                                              (long long)r, bounds, bias_out, reset);
  return launch_status();
}

}  // namespace qb
