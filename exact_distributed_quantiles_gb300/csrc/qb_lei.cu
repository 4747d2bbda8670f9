// qb_lei.cu -- load-error injection (LEI).
//
// "Exact Quantile Balancing and Load-Error Injection for Mixture-of-Experts",
// LEI paragraph: with the batch-mean raw sigmoid score as surrogate, the
// correction collapses to adding eta * rho_e to the score gradient of expert e
// for every token of the local batch, rho_e being that expert's relative load
// error, bounded by a tanh rescale that keeps its direction and its zero mean.
// Reading used here: rho_raw = (load_e - T)/T with T = n*k/E, and
// rho = tanh(rho_raw) - mean_e tanh(rho_raw).
//
// Kernels:
//   lei_rho_kernel         one 8-CTA cluster per local batch: load counts in
//                          shared memory, reduced over the cluster, rho in
//                          fp32, c_e = eta * rho_e into the caller's
//                          workspace [num_batches, E] (lei_rho);
//   lei_apply_kernel       grad += c_e of the row's batch, streamed in 16-byte
//                          chunks by small CTAs that each own a run of rows
//                          (lei_apply, lei_inject);
//   lei_apply_bulk_kernel  the same update done by the bulk-copy unit's
//                          reductions into L2, one warp per SM, launched to
//                          run beside the preceding kernel (lei_apply_overlap).
//   load_count_kernel and maxvio_kernel (qb_maxvio) share the counting.
#include <cooperative_groups.h>

#include "qb_device.cuh"
#include "qb_internal.h"

namespace cg = cooperative_groups;

namespace qb {
namespace {

constexpr int kRhoCluster = 8;  // CTAs per local batch (one thread-block cluster)
constexpr int kRhoThreads = 512;
constexpr int kRhoWarps = kRhoThreads / 32;

// One cluster of 8 CTAs per local batch.  Each CTA counts one eighth of the
// batch's top-k entries (16-byte loads, four in flight per thread) into
// per-warp shared histograms and reduces them to its own count row; after a
// cluster barrier, CTA 0 sums the eight rows through distributed shared
// memory, computes rho in fp32 and writes c_e = eta * rho_e.  A second
// cluster barrier keeps every row alive until CTA 0 has read it.
// Count one eighth (this CTA's rank in the cluster) of local batch b's top-k
// entries into cnt[E]: per-warp shared histograms (sub, [kRhoWarps][E]),
// then one row per CTA.  Returns the batch's token range through i0/i1.
__device__ void count_batch_loads(const int32_t* __restrict__ topk, int64_t N, int E, int k,
                                  int64_t batch_tokens, int64_t b, int rank, int32_t* sub,
                                  int32_t* cnt, int64_t& i0, int64_t& i1) {
  const int warp = threadIdx.x >> 5;
  i0 = b * batch_tokens;
  i1 = i0 + batch_tokens;
  if (i1 > N) i1 = N;
  for (int q = threadIdx.x; q < kRhoWarps * E; q += blockDim.x) sub[q] = 0;
  __syncthreads();
  int32_t* mine = sub + warp * E;
  const int64_t n_all = (i1 - i0) * k;
  const int64_t per = ((n_all + kRhoCluster - 1) / kRhoCluster + 3) & ~(int64_t)3;
  const int64_t s0 = rank * per < n_all ? rank * per : n_all;
  const int64_t s1 = s0 + per < n_all ? s0 + per : n_all;
  const int32_t* t = topk + i0 * k + s0;
  const int64_t n_idx = s1 - s0;
  // scalar head until 16-byte alignment, then int4 body, then scalar tail
  const int64_t head = ((16 - (reinterpret_cast<uintptr_t>(t) & 15)) & 15) / 4;
  const int64_t hd = head < n_idx ? head : n_idx;
  for (int64_t q = threadIdx.x; q < hd; q += blockDim.x) {
    const int32_t e = t[q];
    if ((unsigned)e < (unsigned)E) atomicAdd(&mine[e], 1);
  }
  const int4* t4 = reinterpret_cast<const int4*>(t + hd);
  const int64_t n4 = (n_idx - hd) / 4;
  constexpr int kU = 4;
  for (int64_t q0 = threadIdx.x; q0 < n4; q0 += (int64_t)blockDim.x * kU) {
    int4 v[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int64_t q = q0 + (int64_t)u * blockDim.x;
      v[u] = q < n4 ? __ldcs(t4 + q) : make_int4(-1, -1, -1, -1);
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int32_t ev[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
      for (int c = 0; c < 4; ++c)
        if ((unsigned)ev[c] < (unsigned)E) atomicAdd(&mine[ev[c]], 1);
    }
  }
  for (int64_t q = hd + 4 * n4 + threadIdx.x; q < n_idx; q += blockDim.x) {
    const int32_t e = t[q];
    if ((unsigned)e < (unsigned)E) atomicAdd(&mine[e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int32_t c = 0;
    for (int w = 0; w < kRhoWarps; ++w) c += sub[w * E + e];
    cnt[e] = c;
  }
}

__global__ void __cluster_dims__(kRhoCluster, 1, 1) __launch_bounds__(kRhoThreads)
    lei_rho_kernel(const int32_t* __restrict__ topk, int64_t N, int E, int k, float eta,
                   int64_t batch_tokens, float* __restrict__ ws) {
  cg::cluster_group cluster = cg::this_cluster();
  extern __shared__ int32_t sub[];  // [kRhoWarps][E]
  __shared__ int32_t cnt[kMaxE];
  __shared__ float red[kRhoWarps];
  __shared__ float t_s[kMaxE];
  const int warp = threadIdx.x >> 5;
  const int rank = (int)cluster.block_rank();
  const int64_t b = blockIdx.x / kRhoCluster;
  int64_t i0, i1;
  count_batch_loads(topk, N, E, k, batch_tokens, b, rank, sub, cnt, i0, i1);
  cluster.sync();
  if (rank == 0) {
    // fp32 throughout: the fp64 pipe of this part costs ~150 cycles per
    // dependent operation, and the result only needs eta * rho to 1e-6
    // absolute (fp32 keeps it within ~1e-11).  Loads are exact integers.
    const float T = __fdiv_rn((float)((i1 - i0) * (int64_t)k), (float)E);
    float part = 0.0f;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      int32_t load = 0;
#pragma unroll
      for (int r = 0; r < kRhoCluster; ++r) load += cluster.map_shared_rank(cnt, r)[e];
      t_s[e] = tanhf(__fdiv_rn(__fsub_rn((float)load, T), T));
      part = __fadd_rn(part, t_s[e]);
    }
    // mean of tanh over experts: a fixed-shape tree
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) part = __fadd_rn(part, __shfl_xor_sync(0xffffffffu, part, o));
    if ((threadIdx.x & 31) == 0) red[warp] = part;
    __syncthreads();
    float sum = 0.0f;
#pragma unroll
    for (int w = 0; w < kRhoWarps; ++w) sum = __fadd_rn(sum, red[w]);
    const float mean = __fdiv_rn(sum, (float)E);
    for (int e = threadIdx.x; e < E; e += blockDim.x)
      ws[b * E + e] = __fmul_rn(eta, __fsub_rn(t_s[e], mean));
  }
  cluster.sync();
}

// MaxVio, pass 1: the load counts of every local batch (one 8-CTA cluster
// per batch, the same counting as the LEI rho kernel) into loads[nb, E].
__global__ void __cluster_dims__(kRhoCluster, 1, 1) __launch_bounds__(kRhoThreads)
    load_count_kernel(const int32_t* __restrict__ topk, int64_t N, int E, int k,
                      int64_t batch_tokens, int32_t* __restrict__ loads) {
  cg::cluster_group cluster = cg::this_cluster();
  extern __shared__ int32_t sub[];  // [kRhoWarps][E]
  __shared__ int32_t cnt[kMaxE];
  const int rank = (int)cluster.block_rank();
  const int64_t b = blockIdx.x / kRhoCluster;
  int64_t i0, i1;
  count_batch_loads(topk, N, E, k, batch_tokens, b, rank, sub, cnt, i0, i1);
  cluster.sync();
  if (rank == 0) {
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      int32_t load = 0;
#pragma unroll
      for (int r = 0; r < kRhoCluster; ++r) load += cluster.map_shared_rank(cnt, r)[e];
      loads[b * E + e] = load;
    }
  }
  cluster.sync();  // keep every CTA's row alive until rank 0 has read it
}

// MaxVio, pass 2 (one CTA): T = n*k/E; global (max_e sum_b loads - T)/T over
// all tokens, local = mean over batches of (max_e loads_b - T_b)/T_b, in fp64
// with the batch terms added in batch order (the plain definition's order).
// Each warp computes whole batch terms (max over experts, then the fp64
// quotient, independently of the other batches); only the ordered sum of the
// terms is serial.
constexpr int kMaxvioThreads = 512;
constexpr int kMaxvioWarps = kMaxvioThreads / 32;

__global__ void __launch_bounds__(kMaxvioThreads) maxvio_kernel(
    const int32_t* __restrict__ loads, int64_t nb, int64_t N, int E, int k, int64_t batch_tokens,
    double* __restrict__ out) {
  __shared__ double term_s[kMaxvioWarps];
  __shared__ long long gmax_s[kMaxvioWarps];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  double local = 0.0;
  for (int64_t b0 = 0; b0 < nb; b0 += kMaxvioWarps) {
    const int64_t b = b0 + warp;
    if (b < nb) {
      int mx = -1;
      for (int e = lane; e < E; e += 32) mx = max(mx, loads[b * E + e]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const int64_t i0 = b * batch_tokens;
      const int64_t n = i0 + batch_tokens < N ? batch_tokens : N - i0;
      const double Tb = __ddiv_rn((double)(n * k), (double)E);
      if (lane == 0) term_s[warp] = __ddiv_rn(__dsub_rn((double)mx, Tb), Tb);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      const int cnt = nb - b0 < kMaxvioWarps ? (int)(nb - b0) : kMaxvioWarps;
      for (int w = 0; w < cnt; ++w) local = __dadd_rn(local, term_s[w]);
    }
    __syncthreads();
  }
  long long mine = -1;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    long long s = 0;
    for (int64_t b = 0; b < nb; ++b) s += loads[b * E + e];
    mine = s > mine ? s : mine;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const long long y = __shfl_xor_sync(0xffffffffu, mine, o);
    mine = y > mine ? y : mine;
  }
  if (lane == 0) gmax_s[warp] = mine;
  __syncthreads();
  if (threadIdx.x == 0) {
    long long tot = gmax_s[0];
    for (int w = 1; w < kMaxvioWarps; ++w) tot = gmax_s[w] > tot ? gmax_s[w] : tot;
    const double T = __ddiv_rn((double)(N * k), (double)E);
    out[0] = __ddiv_rn(__dsub_rn((double)tot, T), T);
    out[1] = __ddiv_rn(local, (double)nb);
  }
}

// grad += c[batch(row)] streamed in 16-byte chunks.  Each CTA owns a fixed
// run of kApplyIters blocks of rows; in a block every thread has kApplyU
// loads in flight.  The CTAs are small (128 threads, at most 72 registers)
// so that one fits on an SM beside a resident routing CTA, and the grid
// drains through whatever room the other kernels of the step leave.
constexpr int kApplyThreads = 128;
constexpr int kApplyU = 8;
constexpr int kApplyIters = 4;

__global__ void __launch_bounds__(kApplyThreads, 7)
    lei_apply_kernel(float* __restrict__ grad, int N, int e4, int lanes_log2, int batch_tokens,
                     const float* __restrict__ ws) {
  // e4 16-byte chunks per row; 2^lanes_log2 lanes per row (<= e4, <= 128),
  // each taking the row's chunks col, col + lanes, ...
  const int lanes_per_row = 1 << lanes_log2;
  const int rows_per_pass = kApplyThreads >> lanes_log2;
  const int r_in = threadIdx.x >> lanes_log2;
  const int c_in = threadIdx.x & (lanes_per_row - 1);
  const int block_rows = rows_per_pass * kApplyU;
  float4* g4 = reinterpret_cast<float4*>(grad);
  const float4* c4 = reinterpret_cast<const float4*>(ws);
  int64_t rb = (int64_t)blockIdx.x * block_rows * kApplyIters;
  for (int it = 0; it < kApplyIters && rb < N; ++it, rb += block_rows) {
    const int r0 = (int)rb;
    const int last = (int)(rb + block_rows < N ? rb + block_rows : N) - 1;
    const int b0 = r0 / batch_tokens;
    const bool one_batch = last / batch_tokens == b0;  // almost always
    for (int col = c_in; col < e4; col += lanes_per_row) {
      float4 g[kApplyU];
#pragma unroll
      for (int u = 0; u < kApplyU; ++u) {
        const int rr = r0 + u * rows_per_pass + r_in;
        if (rr <= last) g[u] = __ldcs(g4 + (int64_t)rr * e4 + col);
      }
      float4 c = __ldg(c4 + (int64_t)b0 * e4 + col);
#pragma unroll
      for (int u = 0; u < kApplyU; ++u) {
        const int rr = r0 + u * rows_per_pass + r_in;
        if (rr <= last) {
          if (!one_batch) c = __ldg(c4 + (int64_t)(rr / batch_tokens) * e4 + col);
          float4 o;
          o.x = __fadd_rn(g[u].x, c.x);
          o.y = __fadd_rn(g[u].y, c.y);
          o.z = __fadd_rn(g[u].z, c.z);
          o.w = __fadd_rn(g[u].w, c.w);
          __stcs(g4 + (int64_t)rr * e4 + col, o);
        }
      }
    }
  }
}

// The same update done by the bulk-copy unit: a cp.reduce.async.bulk .add.f32
// from a 4 KB shared block holding the batch's c repeated over `rep` rows adds
// c to `rep` rows of grad in L2 per instruction.  No registers or SM load /
// store bandwidth are spent on grad, and a CTA (one warp, 4 KB of shared
// memory) fits beside a resident routing CTA.  One CTA per SM, each over an
// even share of the row groups; the last step waits for the kernel this one
// was launched behind (a no-op without a programmatic launch), so that its
// completion implies that kernel's.
constexpr int kBulkBytes = 4096;

// At most 32 registers (1024 per warp): a routing CTA of 20 warps at 96
// registers leaves exactly that much in each SM sub-partition, and a guest
// that does not fit there waits until the routing CTAs exit and then piles
// onto the few SMs freed first (measured: 2.3 ms instead of 0.33 ms for a
// layer's routing pass plus this update).
__global__ void __maxnreg__(32) lei_apply_bulk_kernel(float* __restrict__ grad, int N, int E,
                                                            int batch_tokens,
                                                            const float* __restrict__ ws) {
  __shared__ __align__(128) float buf[kBulkBytes / 4];
  const int lane = threadIdx.x;
  const int rep = kBulkBytes / (E * 4);  // rows per bulk op (E <= 512: at least 2)
  const int e4 = E >> 2;
  const int fill = rep * e4;             // 16-byte chunks of the block in use
  const int64_t groups = ((int64_t)N + rep - 1) / rep;
  const int64_t g0 = groups * blockIdx.x / gridDim.x;
  const int64_t g1 = groups * (blockIdx.x + 1) / gridDim.x;
  int64_t r = g0 * rep;
  const int64_t r_end = g1 * rep < N ? g1 * rep : N;
  const uint32_t src = (uint32_t)__cvta_generic_to_shared(buf);
  while (r < r_end) {
    const int64_t b = r / batch_tokens;
    const int64_t seg_end = (b + 1) * batch_tokens < r_end ? (b + 1) * batch_tokens : r_end;
    // refill only after the ops issued from the old contents have read them
    if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
    __syncwarp();
    const float4* c4 = reinterpret_cast<const float4*>(ws + b * E);
    float4* b4 = reinterpret_cast<float4*>(buf);
    for (int i = lane; i < fill; i += 32) b4[i] = __ldg(c4 + i % e4);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) {
      for (int64_t q = r; q < seg_end; q += rep) {
        const int64_t nr = seg_end - q < rep ? seg_end - q : rep;
        asm volatile(
            "cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;" ::"l"(
                grad + q * E),
            "r"(src), "r"((uint32_t)(nr * E * 4))
            : "memory");
      }
      asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    }
    r = seg_end;
  }
  if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
  __syncwarp();
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace

// The per-warp count rows take kRhoWarps * E int32 of dynamic shared memory,
// 64 KB at E = 1024: above the default 48 KB, so the kernels opt in once.
template <typename K>
bool rho_smem_attr(K kern, bool& done) {
  if (done) return true;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kRhoWarps * kMaxE * (int)sizeof(int32_t)) != cudaSuccess)
    return false;
  done = true;
  return true;
}

int launch_maxvio(const int32_t* topk, int64_t N, int E, int k, int64_t batch_tokens,
                  int32_t* loads, double* out, cudaStream_t stream) {
  const int64_t nb = (N + batch_tokens - 1) / batch_tokens;
  const int smem = kRhoWarps * E * (int)sizeof(int32_t);
  static bool attr = false;  // benign race (idempotent)
  if (!rho_smem_attr(load_count_kernel, attr)) return launch_status();
  load_count_kernel<<<(unsigned)(nb * kRhoCluster), kRhoThreads, smem, stream>>>(
      topk, N, E, k, batch_tokens, loads);
  int st = launch_status();
  if (st != QB_OK) return st;
  maxvio_kernel<<<1, kMaxvioThreads, 0, stream>>>(loads, nb, N, E, k, batch_tokens, out);
  return launch_status();
}

int launch_lei_rho(const int32_t* topk, int64_t N, int E, int k, float eta,
                   int64_t batch_tokens, float* workspace, cudaStream_t stream) {
  const int64_t nb = (N + batch_tokens - 1) / batch_tokens;
  const int smem = kRhoWarps * E * (int)sizeof(int32_t);
  static bool attr = false;  // benign race (idempotent)
  if (!rho_smem_attr(lei_rho_kernel, attr)) return launch_status();
  lei_rho_kernel<<<(unsigned)(nb * kRhoCluster), kRhoThreads, smem, stream>>>(
      topk, N, E, k, eta, batch_tokens, workspace);
  return launch_status();
}

int launch_lei_apply(float* grad, int64_t N, int E, int64_t batch_tokens, const float* workspace,
                     cudaStream_t stream) {
  const int e4 = E / 4;
  int lanes_log2 = 0;  // the largest power of two <= min(e4, 128)
  while (lanes_log2 < 7 && (2 << lanes_log2) <= e4) ++lanes_log2;
  const int64_t cta_rows = (int64_t)(kApplyThreads >> lanes_log2) * kApplyU * kApplyIters;
  const int64_t grid = (N + cta_rows - 1) / cta_rows;
  lei_apply_kernel<<<(unsigned)grid, kApplyThreads, 0, stream>>>(grad, (int)N, e4, lanes_log2,
                                                                (int)batch_tokens, workspace);
  return launch_status();
}

int launch_lei_apply_overlap(float* grad, int64_t N, int E, int64_t batch_tokens,
                             const float* workspace, cudaStream_t stream) {
  const int64_t groups = (N + kBulkBytes / (E * 4) - 1) / (kBulkBytes / (E * 4));
  int64_t grid = sm_count();
  if (grid > groups) grid = groups;
  if (grid < 1) grid = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, lei_apply_bulk_kernel, grad, (int)N, E, (int)batch_tokens,
                         workspace) != cudaSuccess) {
    (void)cudaGetLastError();
    return QB_ECUDA;
  }
  return launch_status();
}

int launch_lei(float* grad, const int32_t* topk, int64_t N, int E, int k, float eta,
               int64_t batch_tokens, float* workspace, cudaStream_t stream) {
  const int st = launch_lei_rho(topk, N, E, k, eta, batch_tokens, workspace, stream);
  if (st != QB_OK) return st;
  return launch_lei_apply(grad, N, E, batch_tokens, workspace, stream);
}

}  // namespace qb
