// qb_route256_bf16.cu -- instantiates the E = 256 router pass for __nv_bfloat16 logits
// (a translation unit of its own so that the variants compile in parallel).
#include "qb_route256.cuh"

namespace qb {
int launch_route256_hi_bf16(const void* logits, const float* bias, int64_t N, int k,
                            int32_t* hist, uint16_t* keys_out, int32_t* topk_out,
                            float* alpha_out, cudaStream_t stream, bool chained) {
  return r256::launch_hi_t<__nv_bfloat16>(logits, bias, N, k, hist, keys_out, topk_out, alpha_out, stream,
                                          chained);
}
int launch_route256_alpha_bf16(const void* logits, const float* bias, int64_t N, int k,
                               float* alpha_out, cudaStream_t stream, bool chained) {
  return r256::launch_alpha_t<__nv_bfloat16>(logits, bias, N, k, alpha_out, stream, chained);
}
}  // namespace qb
