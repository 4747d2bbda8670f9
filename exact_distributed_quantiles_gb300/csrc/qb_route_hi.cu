// qb_route_hi.cu -- instantiates the fused router pass in mode kModeHi (E = 256
// goes to the specialised pass of qb_route256.cuh).
#include "qb_route.cuh"

namespace qb {
int launch_route_hi(const void* logits, int dtype, const float* bias, int64_t N, int E, int k,
                    int32_t* hist, uint16_t* keys_out, int32_t* topk_out, float* alpha_out,
                    const int32_t* sel, const float* bounds, int nbins, cudaStream_t stream) {
  if (E == 256 && dtype == QB_F32)
    return launch_route256_hi_f32(logits, bias, N, k, hist, keys_out, topk_out, alpha_out, stream);
  if (E == 256)
    return launch_route256_hi_bf16(logits, bias, N, k, hist, keys_out, topk_out, alpha_out, stream);
  return route::launch_mode<kModeHi>(logits, dtype, bias, N, E, k, hist, keys_out, topk_out,
                                alpha_out, sel, bounds, nbins, stream);
}
}  // namespace qb
