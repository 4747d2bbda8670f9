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
// Two kernels:
//   lei_rho_kernel    one CTA per local batch: load counts in shared memory,
//                     rho in fp64, c_e = RN32(eta * rho_e) into the caller's
//                     workspace [num_batches, E];
//   lei_apply_kernel  grid-stride stream over grad in 16-byte chunks:
//                     grad += c_e of the chunk's batch (c rows stay in L1/L2).
#include "qb_device.cuh"
#include "qb_internal.h"

namespace qb {
namespace {

constexpr int kRhoThreads = 1024;

__global__ void __launch_bounds__(kRhoThreads) lei_rho_kernel(const int32_t* __restrict__ topk,
                                                              int64_t N, int E, int k, float eta,
                                                              int64_t batch_tokens,
                                                              float* __restrict__ ws) {
  __shared__ int32_t load_s[512];
  __shared__ double t_s[512];
  __shared__ double mean_s;
  const int64_t b = blockIdx.x;
  const int64_t i0 = b * batch_tokens;
  int64_t i1 = i0 + batch_tokens;
  if (i1 > N) i1 = N;
  for (int e = threadIdx.x; e < E; e += blockDim.x) load_s[e] = 0;
  __syncthreads();
  const int64_t n_idx = (i1 - i0) * k;
  const int32_t* t = topk + i0 * k;
  for (int64_t q = threadIdx.x; q < n_idx; q += blockDim.x) {
    const int32_t e = __ldcs(t + q);
    if ((unsigned)e < (unsigned)E) atomicAdd(&load_s[e], 1);
  }
  __syncthreads();
  const double T = __ddiv_rn((double)((i1 - i0) * (int64_t)k), (double)E);
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    t_s[e] = tanh(__ddiv_rn(__dsub_rn((double)load_s[e], T), T));
  __syncthreads();
  if (threadIdx.x == 0) {
    double sum = 0.0;
    for (int e = 0; e < E; ++e) sum = __dadd_rn(sum, t_s[e]);
    mean_s = __ddiv_rn(sum, (double)E);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    ws[b * E + e] = __double2float_rn(__dmul_rn((double)eta, __dsub_rn(t_s[e], mean_s)));
}

__global__ void __launch_bounds__(256) lei_apply_kernel(float* __restrict__ grad, int64_t N,
                                                        int E, int64_t batch_tokens,
                                                        const float* __restrict__ ws) {
  const int64_t n4 = N * (int64_t)E / 4;
  const int e4 = E / 4;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  float4* g4 = reinterpret_cast<float4*>(grad);
  const float4* c4 = reinterpret_cast<const float4*>(ws);
  for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < n4; q += stride) {
    const int64_t row = q / e4;
    const int col = (int)(q - row * e4);
    const float4 c = __ldg(c4 + (row / batch_tokens) * e4 + col);
    float4 g = __ldcs(g4 + q);
    g.x = __fadd_rn(g.x, c.x);
    g.y = __fadd_rn(g.y, c.y);
    g.z = __fadd_rn(g.z, c.z);
    g.w = __fadd_rn(g.w, c.w);
    __stcs(g4 + q, g);
  }
}

}  // namespace

int launch_lei(float* grad, const int32_t* topk, int64_t N, int E, int k, float eta,
               int64_t batch_tokens, float* workspace, cudaStream_t stream) {
  const int64_t nb = (N + batch_tokens - 1) / batch_tokens;
  lei_rho_kernel<<<(unsigned)nb, kRhoThreads, 0, stream>>>(topk, N, E, k, eta, batch_tokens,
                                                          workspace);
  int st = launch_status();
  if (st != QB_OK) return st;
  const int64_t n4 = N * (int64_t)E / 4;
  int64_t grid = (n4 + 255) / 256;
  const int64_t gmax = (int64_t)sm_count() * 8;
  if (grid > gmax) grid = gmax;
  if (grid < 1) grid = 1;
  lei_apply_kernel<<<(unsigned)grid, 256, 0, stream>>>(grad, N, E, batch_tokens, workspace);
  return launch_status();
}

}  // namespace qb
