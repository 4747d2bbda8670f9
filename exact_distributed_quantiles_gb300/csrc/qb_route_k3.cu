// qb_route_k3.cu -- instantiates the fused router pass in mode kModeK3.
#include "qb_route.cuh"

namespace qb {
int launch_route_k3(const void* logits, int dtype, const float* bias, int64_t N, int E, int k,
                    int32_t* hist, uint16_t* keys_out, int32_t* topk_out, float* alpha_out,
                    const int32_t* sel, const float* bounds, int nbins, cudaStream_t stream) {
  return route::launch_mode<kModeK3>(logits, dtype, bias, N, E, k, hist, keys_out, topk_out,
                                alpha_out, sel, bounds, nbins, stream);
}
}  // namespace qb
