// qb_internal.h -- host-side helpers shared by the libqb translation units.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/qb.h"

namespace qb {

// Device pointer to the library's device status word for the current device
// (set up on first use per device); nullptr if CUDA fails.
int* device_status_ptr();

// Streaming multiprocessor count of the current device (cached per device).
int sm_count();

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Expert counts the kernels take: multiples of 32 from 32 to kMaxE.
constexpr int kMaxE = 1024;
inline bool supported_E(int E) { return E >= 32 && E <= kMaxE && E % 32 == 0; }

inline int launch_status() {
  return cudaPeekAtLastError() == cudaSuccess ? QB_OK : (cudaGetLastError(), QB_ECUDA);
}

// Launchers implemented in the kernel translation units.
int launch_route_hi(const void* logits, int dtype, const float* bias, int64_t N, int E, int k,
                    int32_t* hist, uint16_t* keys_out, int32_t* topk_out, float* alpha_out,
                    const int32_t* sel, const float* bounds, int nbins, cudaStream_t stream);
int launch_route_lo(const void* logits, int dtype, const float* bias, int64_t N, int E, int k,
                    int32_t* hist, uint16_t* keys_out, int32_t* topk_out, float* alpha_out,
                    const int32_t* sel, const float* bounds, int nbins, cudaStream_t stream);
int launch_route_k3(const void* logits, int dtype, const float* bias, int64_t N, int E, int k,
                    int32_t* hist, uint16_t* keys_out, int32_t* topk_out, float* alpha_out,
                    const int32_t* sel, const float* bounds, int nbins, cudaStream_t stream);
// EQB hi pass specialised to E = 256 (qb_route256.cuh), per input type;
// chained: a further microbatch right after another such call on the stream
// (qb_route_hist_hi_next).
int launch_route256_hi_f32(const void* logits, const float* bias, int64_t N, int k,
                           int32_t* hist, uint16_t* keys_out, int32_t* topk_out,
                           float* alpha_out, cudaStream_t stream, bool chained = false);
int launch_route256_hi_bf16(const void* logits, const float* bias, int64_t N, int k,
                            int32_t* hist, uint16_t* keys_out, int32_t* topk_out,
                            float* alpha_out, cudaStream_t stream, bool chained = false);
// alpha per token only (the first half of the K3 pass), E = 256; chained: a
// further microbatch right after another K3 call on the stream
// (k3_route_hist_next).
int launch_route256_alpha_f32(const void* logits, const float* bias, int64_t N, int k,
                              float* alpha_out, cudaStream_t stream, bool chained = false);
int launch_route256_alpha_bf16(const void* logits, const float* bias, int64_t N, int k,
                               float* alpha_out, cudaStream_t stream, bool chained = false);
int launch_keys_hist_lo(const uint16_t* keys, int64_t N, int E, const int32_t* sel,
                        int32_t* hist_lo, cudaStream_t stream);
int launch_select_hi(const int32_t* hist_hi, int E, int64_t r, int32_t* sel, int32_t* r_lo,
                     cudaStream_t stream);
int launch_finalize(int32_t* hist_hi, int32_t* hist_lo, const int32_t* sel, const int32_t* r_lo,
                    int E, float* bias_out, uint16_t* qkey_out, int reset, cudaStream_t stream);
int launch_k3_finalize(int32_t* hist, int E, int nbins, int64_t r, float* bounds,
                       float* bias_out, int reset, cudaStream_t stream);
int launch_k3_count(const void* logits, int dtype, const float* alpha, int64_t N, int E,
                    const float* bounds, int nbins, int32_t* hist, cudaStream_t stream);
int launch_zero_i32(int32_t* p, int64_t n, cudaStream_t stream);
int launch_wait_timeout_selftest(uint32_t polls, cudaStream_t stream);
int launch_router_gemm_route(const void* hidden, const void* w_t, int64_t M, int K, int k,
                             const float* bias, int32_t* hist, uint16_t* keys_out,
                             int32_t* topk_out, float* alpha_out, float* logits_out,
                             cudaStream_t stream, bool chained = false);
int launch_rank_average(const uint16_t* qkeys, int P, int E, float* bias_out,
                        cudaStream_t stream);
int launch_maxvio(const int32_t* topk, int64_t N, int E, int k, int64_t batch_tokens,
                  int32_t* loads, double* out, cudaStream_t stream);
int launch_sigmoid(const float* x, float* s, int64_t n, int scalar, cudaStream_t stream);
int launch_lei(float* grad, const int32_t* topk, int64_t N, int E, int k, float eta,
               int64_t batch_tokens, float* workspace, cudaStream_t stream);
int launch_lei_rho(const int32_t* topk, int64_t N, int E, int k, float eta,
                   int64_t batch_tokens, float* workspace, cudaStream_t stream);
int launch_lei_apply(float* grad, int64_t N, int E, int64_t batch_tokens, const float* workspace,
                     cudaStream_t stream);
int launch_lei_apply_overlap(float* grad, int64_t N, int E, int64_t batch_tokens,
                             const float* workspace, cudaStream_t stream);

int launch_router_gemm(const void* hidden, const void* w_t, int64_t M, int K, int E,
                       float* logits, cudaStream_t stream);

enum RouteMode { kModeHi = 0, kModeLo = 1, kModeK3 = 2 };

}  // namespace qb
