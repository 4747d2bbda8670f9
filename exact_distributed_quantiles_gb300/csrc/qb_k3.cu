// qb_k3.cu -- K3 histogram mode: the counts, and the finalize (interpolated
// quantile, centering, next bounds).
//
// "[Dev] Add global-batch quantile balancing", "Quantile estimator": a uniform
// histogram of nbins (1000) bins per expert over [min(b) - 1, max(b) + 1]; the
// quantile is read off the bin where the cumulative count reaches the rank
// and interpolated inside it; the new bias is centred and the next bounds
// follow it.  "Implementation": the counts accumulate over the microbatches
// of a global batch in one persistent histogram that is reset in place.
//
// Counting.  A [E, nbins] histogram (1 MB at E = 256, nbins = 1000) does not
// fit in one SM's shared memory, and spreading it over a cluster does not pay
// on this GPU: shared-memory reductions into another CTA of the cluster ran
// 23 times slower than into the CTA's own (52 against 1198 G/s over the whole
// GPU), and global atomics per element are slower still.  So the routing pass
// (first launch) stops after alpha, and this kernel -- a CTA per expert slice
// and token range -- recomputes the scores of its slice from the logits (the
// same pinned function, bit for bit), forms the margins and their bins and
// counts them in shared memory.  The logits of a 65536-token microbatch
// (32 MiB of bf16) are still in L2 from the first launch.  Non-zero counters
// are added to the global histogram once per CTA.
//
// Finalize.  One cluster of 8 CTAs: a warp per expert finds the bin (blocks
// of 128 bins, coalesced loads, a warp scan per block) and resets the row;
// each CTA then writes its fp64 quantiles into every CTA's shared memory
// (one cluster barrier), so that every CTA holds all E of them and derives
// the same mean -- per-CTA partial sums by a fixed shuffle tree, added in
// rank order -- and rank 0 the min and max of the new bias for the bounds.
#include <cooperative_groups.h>
#include <cuda_bf16.h>

#include "qb_device.cuh"
#include "qb_internal.h"

namespace cg = cooperative_groups;

namespace qb {
namespace {

constexpr int kCountThreads = 1024;
constexpr int kCountSmemMax = 200 * 1024;
constexpr int kEW = 32;  // experts per counting CTA

// No "memory" clobber: the counters are read only after a __syncthreads.
__device__ __forceinline__ void red_shared_inc(uint32_t addr) {
  asm volatile("red.shared.add.u32 [%0], 1;" ::"r"(addr));
}

// Eight logits of a row (fp32 or bf16) as fp32.
__device__ __forceinline__ void load8x(const float* p, float (&x)[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(p));
  const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
  x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}
__device__ __forceinline__ void load8x(const __nv_bfloat16* p, float (&x)[8]) {
  const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// The K3 counts from the logits and alpha (written by the first launch).
// A CTA owns a slice of kEW experts over a range of tokens; a lane takes 8
// consecutive experts of a row (4 lanes per row, 8 rows per warp), recomputes
// their pinned scores -- the routing pass's function, negated, bit for bit --
// the margins r = alpha + sn (= alpha - s) and the bins
//   idx = clamp(floor(RN(RN(r - lo) * scale)), 0, nbins - 1)
// (a float-to-int conversion truncates, saturates and sends NaN to 0, so the
// clamp covers t < 0, t >= nbins and NaN as the definition does), and counts
// them in shared memory: kEW rows of `pitch` int32 (pitch odd, so that equal
// bins of different experts fall in different banks).  GLOBAL: the slice
// would not fit shared memory, so every count is a global atomic.  Non-zero
// shared counters are added to the global histogram once at the end.
// alpha is the output of the kernel this one depends on: read with a plain
// load issued after the dependency wait (an asm statement, so that the
// compiler cannot treat it as read-only data and hoist it above the wait).
__device__ __forceinline__ float ld_after_wait(const float* p) {
  float v;
  asm volatile("ld.global.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
  return v;
}

template <typename T, bool GLOBAL>
__global__ void __launch_bounds__(kCountThreads, 1)
    k3_count_kernel(const T* __restrict__ logits, const float* alpha, int64_t N, int E,
                    const float* bounds, int nbins, int pitch, int bulk,
                    int32_t* __restrict__ hist, int64_t rows_per_cta) {
  extern __shared__ __align__(16) int32_t h[];
  constexpr int kWarps = kCountThreads / 32;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int n_eg = E / kEW;
  const int eg = blockIdx.x % n_eg;
  const int64_t r_begin = (int64_t)(blockIdx.x / n_eg) * rows_per_cta;
  int64_t r_end = r_begin + rows_per_cta;
  if (r_end > N) r_end = N;
  if constexpr (!GLOBAL) {
    for (int i = threadIdx.x; i < kEW * pitch; i += kCountThreads) h[i] = 0;
  }
  // Launched as a programmatic dependent of the alpha pass: this CTA may have
  // cleared its counters while that pass still ran; wait for it (and its
  // memory) before the first global read.  Then the next microbatch's alpha
  // pass, if chained (k3_route_hist_next), may start on the SMs this grid
  // leaves: it writes another alpha buffer and reads nothing this kernel
  // writes.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const float lo = ld_after_wait(bounds);
  const float hi = ld_after_wait(bounds + 1);
  const float scale = __fdiv_rn((float)nbins, __fsub_rn(hi, lo));
  const int last = nbins - 1;
  const int chunk = lane & 3;   // experts 8*chunk .. 8*chunk+7 of the slice
  const int rsub = lane >> 2;   // row of the warp's 8
  const int e0 = eg * kEW + 8 * chunk;
  const uint32_t hb = (uint32_t)__cvta_generic_to_shared(h) + 4u * (uint32_t)(8 * chunk * pitch);
  __syncthreads();

  const f2_t LO = f2_splat(lo), SC = f2_splat(scale);
  // Bins from t = RN(RN(r - lo) * scale) without a float-to-int conversion:
  // u = RZ(t + 2^23) is 2^23 + trunc(t) for 0 <= t < 2^23 (the sum is below
  // 2^24, where float spacing is 1, and rounding toward zero truncates), and
  // below 2^23 for t < 0; clamped to [2^23, 2^23 + nbins - 1] by fmax/fmin
  // (which return the number for a NaN t, i.e. bin 0, as a truncating
  // conversion would) its bit pattern is 0x4B000000 + the bin.
  const f2_t M23 = f2_splat(8388608.0f);
  const float u_last = 8388608.0f + (float)last;  // exact: nbins < 2^23
  const T* base = logits + e0;
  const int64_t stride = (int64_t)kWarps * 8;
  // counter address of bin pattern u for element i: hb + 4 (i pitch) + 4 (u - 0x4B000000)
  const uint32_t hb0 = hb - 4u * 0x4B000000u;
  // Three row buffers used in turn (the compiler keeps them in registers
  // without copies): a row is counted from one while the next two rows'
  // loads are in flight, and the freed buffer loads the row three strides on.
  float x0[8], x1[8], x2[8];
  float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) x0[i] = x1[i] = x2[i] = 0.0f;
  const int64_t w0 = r_begin + warp * 8;   // this warp's first row
  const int64_t n_it = w0 < r_end ? (r_end - w0 + stride - 1) / stride : 0;
  // this lane's rows are w0 + rsub + j * stride, j = 0, 1, ...: n_mine of them
  // are in range; the loads and the counts each walk them with a pointer
  // and a countdown
  const int64_t r_mine = w0 + rsub;
  const int n_mine = r_mine < r_end ? (int)((r_end - 1 - r_mine) / stride) + 1 : 0;
  const T* pl = base + r_mine * E;
  const float* pa = alpha + r_mine;
  const int64_t step_l = stride * E;
  int left_l = n_mine, left_c = n_mine;
  auto load = [&](float (&x)[8], float& a) {
    if (left_l > 0) {
      load8x(pl, x);
      a = ld_after_wait(pa);
    }
    --left_l;
    pl += step_l;
    pa += stride;
  };
  auto count = [&](const float (&x)[8], float a) {
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(x[i]));
    float sn[8];
    if (__all_sync(0xffffffffu, m <= kFastAbsX)) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        f2_unpack(neg_sigmoid2_fast(f2_pack(x[2 * i], x[2 * i + 1])), sn[2 * i], sn[2 * i + 1]);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) sn[i] = -sigmoid_pinned(x[i]);
    }
    const f2_t A = f2_splat(a);
    float u[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      // t = RN(RN(r - lo) * scale) with r = RN(alpha + sn)
      const f2_t R = f2_add(A, f2_pack(sn[2 * i], sn[2 * i + 1]));
      f2_unpack(f2_add_rz(f2_mul(f2_sub(R, LO), SC), M23), u[2 * i], u[2 * i + 1]);
    }
    if (left_c > 0) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t ub = __float_as_uint(fminf(fmaxf(u[i], 8388608.0f), u_last));
        if constexpr (GLOBAL)
          atomicAdd(hist + (int64_t)(e0 + i) * nbins + (int)(ub - 0x4B000000u), 1);
        else
          red_shared_inc(hb0 + 4u * (uint32_t)(i * pitch) + 4u * ub);
      }
    }
    --left_c;
  };
  load(x0, a0);
  load(x1, a1);
  load(x2, a2);
  for (int64_t it = 0; it < n_it; it += 3) {
    count(x0, a0);
    load(x0, a0);
    if (it + 1 >= n_it) break;
    count(x1, a1);
    load(x1, a1);
    if (it + 2 >= n_it) break;
    count(x2, a2);
    load(x2, a2);
  }
  if constexpr (!GLOBAL) {
    if (bulk) {
      // rows 16-byte aligned in shared memory and in the histogram: one bulk
      // reduction per expert row, added in L2 (warp w: row w)
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncthreads();
      if (lane == 0) {
        for (int el = warp; el < kEW; el += kWarps) {
          asm volatile(
              "cp.reduce.async.bulk.global.shared::cta.bulk_group.add.u32 [%0], [%1], %2;" ::"l"(
                  hist + (int64_t)(eg * kEW + el) * nbins),
              "r"((uint32_t)__cvta_generic_to_shared(h + el * pitch)), "r"((uint32_t)(nbins * 4))
              : "memory");
        }
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
      }
    } else {
      __syncthreads();
      for (int el = warp; el < kEW; el += kWarps) {
        for (int b = lane; b < nbins; b += 32) {
          const int c = h[el * pitch + b];
          if (c) atomicAdd(hist + (int64_t)(eg * kEW + el) * nbins + b, c);
        }
      }
    }
  }
}

template <typename T, bool GLOBAL>
int launch_count_t(const T* logits, const float* alpha, int64_t N, int E, const float* bounds,
                   int nbins, int32_t* hist, cudaStream_t stream) {
  // Rows of 16-byte multiples (and an odd multiple of 4 words, so that equal
  // bins of different experts spread over the banks) when every histogram row
  // starts on a 16-byte boundary: they are then flushed by bulk reductions.
  const bool bulk = (nbins % 4 == 0) && (reinterpret_cast<uintptr_t>(hist) % 16 == 0);
  const int pitch = bulk ? ((nbins + 3) & ~3) + ((((nbins + 3) / 4) % 2 == 0) ? 4 : 0) : (nbins | 1);
  const int smem = GLOBAL ? 0 : kEW * pitch * 4;
  static int attr_bytes = 0;  // per instantiation; benign race (idempotent)
  if (smem > attr_bytes) {
    if (cudaFuncSetAttribute(k3_count_kernel<T, GLOBAL>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return launch_status();
    attr_bytes = smem;
  }
  const int n_eg = E / kEW;
  int64_t n_tr = sm_count() / n_eg;
  const int64_t max_tr = (N + 255) / 256;  // at least 256 rows per CTA
  if (n_tr > max_tr) n_tr = max_tr;
  if (n_tr < 1) n_tr = 1;
  const int64_t rows_per_cta = (N + n_tr - 1) / n_tr;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(n_tr * n_eg));
  cfg.blockDim = dim3(kCountThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, k3_count_kernel<T, GLOBAL>, logits, alpha, N, E, bounds, nbins,
                         pitch, bulk ? 1 : 0, hist, rows_per_cta) != cudaSuccess) {
    (void)cudaGetLastError();
    return QB_ECUDA;
  }
  return launch_status();
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
  __shared__ double q_s[kMaxE / kFinCluster];  // this CTA's quantiles
  __shared__ double q_all[kMaxE];              // every CTA's, pushed by their owners
  __shared__ double part_s[kFinCluster];
  __shared__ float mn_s[32], mx_s[32];
  __shared__ double mu_s;
  // (1) this CTA is running: other CTAs may write into its shared memory
  // once the matching wait has passed
  cluster_arrive_relaxed();
  const int per = E / kFinCluster;  // experts of this CTA (4 .. 128)
  const int j0 = rank * per;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float lo = bounds[0], hi = bounds[1];
  const double dlo = (double)lo;
  // No fp64 division on this path (each costs microseconds of dependent fp64
  // latency here): width uses the host's RN(1/nbins) and the in-bin fraction
  // is an fp32 quotient; either differs from the divided form by far less
  // than the mode's tolerance (the fraction is scaled by width, ~1e-3).
  const double width = __dmul_rn(__dsub_rn((double)hi, dlo), inv_nbins);
  const bool vec = (nbins % 4 == 0) && (reinterpret_cast<uintptr_t>(hist) % 16 == 0);
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
    if (reset) {
      if (vec) {
        int4* row4 = reinterpret_cast<int4*>(row);
        for (int i = lane; i < nbins / 4; i += 32) row4[i] = make_int4(0, 0, 0, 0);
      } else {
        for (int i = lane; i < nbins; i += 32) row[i] = 0;
      }
    }
  }
  __syncthreads();
  // (2) every CTA has started: push this CTA's quantiles into every CTA
  cluster_wait();
  for (int t = threadIdx.x; t < per * kFinCluster; t += kFinThreads) {
    const int c = t / per, jl = t - c * per;
    *cluster.map_shared_rank(q_all + j0 + jl, c) = q_s[jl];
  }
  cluster_arrive_release();
  cluster_wait();
  // (3) every CTA now holds all E quantiles and derives the same mean: the
  // per-CTA partial sums (a shuffle tree over each CTA's experts), added in
  // rank order
  if (warp < kFinCluster) {
    const double* qc = q_all + warp * per;
    double v = lane < per ? qc[lane] : 0.0;
    for (int i = lane + 32; i < per; i += 32) v = __dadd_rn(v, qc[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = __dadd_rn(v, __shfl_down_sync(0xffffffffu, v, o));
    if (lane == 0) part_s[warp] = v;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double sum = 0.0;
#pragma unroll
    for (int c = 0; c < kFinCluster; ++c) sum = __dadd_rn(sum, part_s[c]);
    // E a power of two: the product is the quotient; otherwise divide
    mu_s = (E & (E - 1)) == 0 ? __dmul_rn(sum, 1.0 / (double)E) : __ddiv_rn(sum, (double)E);
  }
  __syncthreads();
  const double mu = mu_s;
  // every new bias (this CTA writes its own), and their min and max for the
  // next bounds (rank 0 writes them; every CTA read the old ones above)
  float mn = INFINITY, mx = -INFINITY;
  for (int j = threadIdx.x; j < E; j += kFinThreads) {
    const float b = __double2float_rn(__dsub_rn(q_all[j], mu));
    if (j >= j0 && j < j0 + per) bias_out[j] = b;
    mn = fminf(mn, b);
    mx = fmaxf(mx, b);
  }
  if (rank == 0) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    if (lane == 0) {
      mn_s[warp] = mn;
      mx_s[warp] = mx;
    }
    __syncthreads();
    if (warp == 0) {
      mn = mn_s[lane];
      mx = mx_s[lane];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      }
      if (lane == 0) {
        bounds[0] = __fsub_rn(mn, 1.0f);
        bounds[1] = __fadd_rn(mx, 1.0f);
      }
    }
  }
}

}  // namespace

int launch_k3_count(const void* logits, int dtype, const float* alpha, int64_t N, int E,
                    const float* bounds, int nbins, int32_t* hist, cudaStream_t stream) {
  const bool fits = kEW * (((nbins + 3) & ~3) + 4) * 4 <= kCountSmemMax;
  if (dtype == QB_F32) {
    const float* x = static_cast<const float*>(logits);
    return fits ? launch_count_t<float, false>(x, alpha, N, E, bounds, nbins, hist, stream)
                : launch_count_t<float, true>(x, alpha, N, E, bounds, nbins, hist, stream);
  }
  const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(logits);
  return fits ? launch_count_t<__nv_bfloat16, false>(x, alpha, N, E, bounds, nbins, hist, stream)
              : launch_count_t<__nv_bfloat16, true>(x, alpha, N, E, bounds, nbins, hist, stream);
}

int launch_k3_finalize(int32_t* hist, int E, int nbins, int64_t r, float* bounds, float* bias_out,
                       int reset, cudaStream_t stream) {
  if (E % kFinCluster != 0 || E > kMaxE) return QB_EUNSUPPORTED;
  k3_finalize_kernel<<<kFinCluster, kFinThreads, 0, stream>>>(hist, E, nbins, 1.0 / (double)nbins,
                                                              (long long)r, bounds, bias_out, reset);
  return launch_status();
}

}  // namespace qb
