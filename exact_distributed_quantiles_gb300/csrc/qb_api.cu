// qb_api.cu -- the extern "C" entry points of libqb: argument validation on
// the host, then one or more kernel launches on the caller's stream.  No
// entry point allocates memory or synchronises (except qb_device_status).
#include <mutex>

#include "qb_internal.h"

namespace qb {
namespace {

constexpr int kMaxDevices = 64;

// The device status word, one per device that loads the module.
__device__ int g_status_word;

struct PerDevice {
  std::once_flag once;
  int* status = nullptr;
  int sms = 0;
  bool ok = false;
};
PerDevice g_dev[kMaxDevices];

PerDevice* current() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  PerDevice* d = &g_dev[dev];
  std::call_once(d->once, [d, dev] {
    void* p = nullptr;
    int sms = 0;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return;
    d->status = static_cast<int*>(p);
    d->sms = sms;
    d->ok = true;
  });
  return d->ok ? d : nullptr;
}

}  // namespace

int* device_status_ptr() {
  PerDevice* d = current();
  return d ? d->status : nullptr;
}

int sm_count() {
  PerDevice* d = current();
  return d ? d->sms : 1;
}

}  // namespace qb

using namespace qb;

namespace {

int check_route_args(const void* logits, int dtype, const float* bias, int64_t N, int E, int k) {
  if (!logits || !bias) return QB_EINVAL;
  if (dtype != QB_F32 && dtype != QB_BF16) return QB_EINVAL;
  if (!aligned16(logits)) return QB_EINVAL;
  if (N < 0) return QB_EINVAL;
  if (N > INT32_MAX) return QB_EOVERFLOW;
  if (!supported_E(E)) return QB_EUNSUPPORTED;
  if (k < 1 || k >= E) return QB_EINVAL;
  if (k > 15) return QB_EUNSUPPORTED;
  return QB_OK;
}

int router_gemm_hist_hi(const void* hidden, const void* w_t, int64_t M, int H, int E, int k,
                        const float* bias, float* logits_out, int32_t* hist_hi,
                        uint16_t* keys_out, int32_t* topk_out, float* alpha_out, void* stream,
                        bool chained) {
  if (!hidden || !w_t || !bias || !hist_hi) return QB_EINVAL;
  if (!aligned16(hidden) || !aligned16(w_t)) return QB_EINVAL;
  if ((logits_out && !aligned16(logits_out)) || (keys_out && !aligned16(keys_out)))
    return QB_EINVAL;
  if (M < 0) return QB_EINVAL;
  if (M > INT32_MAX) return QB_EOVERFLOW;
  if (E < 32 || E > 256 || E % 32 != 0 || H < 64 || H % 64 != 0) return QB_EUNSUPPORTED;
  if (k < 1 || k >= E) return QB_EINVAL;
  if (k > 15) return QB_EUNSUPPORTED;
  if (E != 256 && !logits_out) return QB_EUNSUPPORTED;
  if (M == 0) return QB_OK;
  if (E == 256)
    return launch_router_gemm_route(hidden, w_t, M, H, k, bias, hist_hi, keys_out, topk_out,
                                    alpha_out, logits_out, as_stream(stream), chained);
  // Other expert counts: the plain GEMM into logits_out, then the routing
  // pass on those logits (two launches; the fused epilogue is built for 256
  // experts).  The results are the same: the fused kernel equals the routing
  // pass run on its own logits.
  int st = launch_router_gemm(hidden, w_t, M, H, E, logits_out, as_stream(stream));
  if (st != QB_OK) return st;
  return launch_route_hi(logits_out, QB_F32, bias, M, E, k, hist_hi, keys_out, topk_out,
                         alpha_out, nullptr, nullptr, 0, as_stream(stream));
}

int k3_route_hist_impl(const void* logits, int dtype, const float* bias, int64_t N, int E, int k,
                       const float* bounds, int nbins, int32_t* hist, float* alpha_out,
                       void* stream, bool chained) {
  int st = check_route_args(logits, dtype, bias, N, E, k);
  if (st != QB_OK) return st;
  if (!bounds || !hist || !alpha_out) return QB_EINVAL;
  if ((reinterpret_cast<uintptr_t>(alpha_out) & 3u) != 0) return QB_EINVAL;
  if (nbins < 1 || nbins > 65536) return QB_EINVAL;
  if (N == 0) return QB_OK;
  cudaStream_t s = as_stream(stream);
  if (E == 256)
    st = dtype == QB_F32 ? launch_route256_alpha_f32(logits, bias, N, k, alpha_out, s, chained)
                         : launch_route256_alpha_bf16(logits, bias, N, k, alpha_out, s, chained);
  else
    st = launch_route_k3(logits, dtype, bias, N, E, k, nullptr, nullptr, nullptr, alpha_out,
                         nullptr, bounds, nbins, s);
  if (st != QB_OK) return st;
  return launch_k3_count(logits, dtype, alpha_out, N, E, bounds, nbins, hist, s);
}
}  // namespace

extern "C" {

const char* qb_status_string(int status) {
  switch (status) {
    case QB_OK:
      return "ok";
    case QB_EINVAL:
      return "invalid argument (null or misaligned pointer, bad size or rank)";
    case QB_EUNSUPPORTED:
      return "unsupported E or k (E a multiple of 32 up to 1024, 1 <= k <= 15, k < E)";
    case QB_ECUDA:
      return "CUDA launch or runtime error";
    case QB_EOVERFLOW:
      return "count would overflow its int32 counter";
    case QB_EDEVICE:
      return "a kernel reported a device-side error (bounded wait timed out)";
    default:
      return "unknown status";
  }
}

const char* qb_version(void) { return "libqb 0.1 (sm_103a)"; }

int64_t qb_rank(int64_t n_pool, int E, int k) {
  if (n_pool < 1 || E < 1 || k < 1 || k >= E) return QB_EINVAL;
  if (n_pool > INT64_MAX / 64) return QB_EOVERFLOW;
  return ((int64_t)k * n_pool + E - 1) / E;
}

int qb_sigmoid(const float* x, float* s, int64_t n, void* stream) {
  if (n < 0 || (n > 0 && (!x || !s))) return QB_EINVAL;
  return launch_sigmoid(x, s, n, 0, as_stream(stream));
}

int qb_sigmoid_scalar(const float* x, float* s, int64_t n, void* stream) {
  if (n < 0 || (n > 0 && (!x || !s))) return QB_EINVAL;
  return launch_sigmoid(x, s, n, 1, as_stream(stream));
}

int qb_selftest_wait_timeout(int64_t polls, void* stream) {
  if (polls < 1 || polls > (int64_t)1 << 24) return QB_EINVAL;
  return launch_wait_timeout_selftest((uint32_t)polls, as_stream(stream));
}

int qb_zero_i32(int32_t* p, int64_t n, void* stream) {
  if (n < 0 || (n > 0 && !p)) return QB_EINVAL;
  return launch_zero_i32(p, n, as_stream(stream));
}

int qb_route_hist_hi(const void* logits, int dtype, const float* bias, int64_t N, int E, int k,
                     int32_t* hist_hi, uint16_t* keys_out, int32_t* topk_out, float* alpha_out,
                     void* stream) {
  int st = check_route_args(logits, dtype, bias, N, E, k);
  if (st != QB_OK) return st;
  if (!hist_hi) return QB_EINVAL;
  if (keys_out && !aligned16(keys_out)) return QB_EINVAL;
  if (N == 0) return QB_OK;
  return launch_route_hi(logits, dtype, bias, N, E, k, hist_hi, keys_out, topk_out, alpha_out,
                         nullptr, nullptr, 0, as_stream(stream));
}

int qb_route_hist_hi_next(const void* logits, int dtype, const float* bias, int64_t N, int E,
                          int k, int32_t* hist_hi, uint16_t* keys_out, int32_t* topk_out,
                          float* alpha_out, void* stream) {
  int st = check_route_args(logits, dtype, bias, N, E, k);
  if (st != QB_OK) return st;
  if (!hist_hi) return QB_EINVAL;
  if (keys_out && !aligned16(keys_out)) return QB_EINVAL;
  if (N == 0) return QB_OK;
  if (E == 256 && dtype == QB_F32)
    return launch_route256_hi_f32(logits, bias, N, k, hist_hi, keys_out, topk_out, alpha_out,
                                  as_stream(stream), true);
  if (E == 256)
    return launch_route256_hi_bf16(logits, bias, N, k, hist_hi, keys_out, topk_out, alpha_out,
                                   as_stream(stream), true);
  return launch_route_hi(logits, dtype, bias, N, E, k, hist_hi, keys_out, topk_out, alpha_out,
                         nullptr, nullptr, 0, as_stream(stream));
}

int qb_select_hi(const int32_t* hist_hi, int E, int64_t r, int32_t* sel, int32_t* r_lo,
                 void* stream) {
  if (!hist_hi || !sel || !r_lo) return QB_EINVAL;
  if (!supported_E(E)) return QB_EUNSUPPORTED;
  if (r < 1) return QB_EINVAL;
  if (r > INT32_MAX) return QB_EOVERFLOW;
  return launch_select_hi(hist_hi, E, r, sel, r_lo, as_stream(stream));
}

int qb_keys_hist_lo(const uint16_t* keys, int64_t N, int E, const int32_t* sel,
                    int32_t* hist_lo, void* stream) {
  if (!keys || !sel || !hist_lo) return QB_EINVAL;
  if (!aligned16(keys)) return QB_EINVAL;
  if (N < 0) return QB_EINVAL;
  if (N > INT32_MAX) return QB_EOVERFLOW;
  if (!supported_E(E)) return QB_EUNSUPPORTED;
  if (N == 0) return QB_OK;
  return launch_keys_hist_lo(keys, N, E, sel, hist_lo, as_stream(stream));
}

int qb_route_hist_lo(const void* logits, int dtype, const float* bias, int64_t N, int E, int k,
                     const int32_t* sel, int32_t* hist_lo, void* stream) {
  int st = check_route_args(logits, dtype, bias, N, E, k);
  if (st != QB_OK) return st;
  if (!sel || !hist_lo) return QB_EINVAL;
  if (N == 0) return QB_OK;
  return launch_route_lo(logits, dtype, bias, N, E, k, hist_lo, nullptr, nullptr, nullptr, sel,
                         nullptr, 0, as_stream(stream));
}

int qb_finalize(int32_t* hist_hi, int32_t* hist_lo, const int32_t* sel, const int32_t* r_lo,
                int E, float* bias_out, uint16_t* qkey_out, int reset, void* stream) {
  if (!hist_lo || !sel || !r_lo || !bias_out) return QB_EINVAL;
  if (reset && !hist_hi) return QB_EINVAL;
  if (!supported_E(E)) return QB_EUNSUPPORTED;
  return launch_finalize(hist_hi, hist_lo, sel, r_lo, E, bias_out, qkey_out, reset,
                         as_stream(stream));
}

int k3_route_hist(const void* logits, int dtype, const float* bias, int64_t N, int E, int k,
                  const float* bounds, int nbins, int32_t* hist, float* alpha_out,
                  void* stream) {
  return k3_route_hist_impl(logits, dtype, bias, N, E, k, bounds, nbins, hist, alpha_out, stream,
                            false);
}

int k3_route_hist_next(const void* logits, int dtype, const float* bias, int64_t N, int E,
                       int k, const float* bounds, int nbins, int32_t* hist, float* alpha_out,
                       void* stream) {
  return k3_route_hist_impl(logits, dtype, bias, N, E, k, bounds, nbins, hist, alpha_out, stream,
                            true);
}

int k3_finalize(int32_t* hist, int E, int nbins, int64_t r, float* bounds, float* bias_out,
                int reset, void* stream) {
  if (!hist || !bounds || !bias_out) return QB_EINVAL;
  if (!supported_E(E)) return QB_EUNSUPPORTED;
  if (nbins < 1 || nbins > 65536) return QB_EINVAL;
  if (r < 1) return QB_EINVAL;
  if (r > INT32_MAX) return QB_EOVERFLOW;
  return launch_k3_finalize(hist, E, nbins, r, bounds, bias_out, reset, as_stream(stream));
}

int lei_inject(float* grad, const int32_t* topk_idx, int64_t N, int E, int k, float eta,
               int64_t batch_tokens, float* workspace, void* stream) {
  if (!grad || !topk_idx || !workspace) return QB_EINVAL;
  if (!aligned16(grad) || !aligned16(workspace)) return QB_EINVAL;
  if (N < 0 || batch_tokens < 0) return QB_EINVAL;
  if (!supported_E(E)) return QB_EUNSUPPORTED;
  if (k < 1 || k >= E) return QB_EINVAL;
  if (N == 0) return QB_OK;
  if (batch_tokens == 0 || batch_tokens > N) batch_tokens = N;
  if (N > INT32_MAX) return QB_EOVERFLOW;
  const int64_t nb = (N + batch_tokens - 1) / batch_tokens;
  if (nb > INT32_MAX) return QB_EINVAL;
  return launch_lei(grad, topk_idx, N, E, k, eta, batch_tokens, workspace, as_stream(stream));
}

int lei_rho(const int32_t* topk_idx, int64_t N, int E, int k, float eta, int64_t batch_tokens,
            float* workspace, void* stream) {
  if (!topk_idx || !workspace) return QB_EINVAL;
  if (!aligned16(workspace)) return QB_EINVAL;
  if (N < 0 || batch_tokens < 0) return QB_EINVAL;
  if (!supported_E(E)) return QB_EUNSUPPORTED;
  if (k < 1 || k >= E) return QB_EINVAL;
  if (N == 0) return QB_OK;
  if (batch_tokens == 0 || batch_tokens > N) batch_tokens = N;
  if (N > INT32_MAX) return QB_EOVERFLOW;
  const int64_t nb = (N + batch_tokens - 1) / batch_tokens;
  if (nb > INT32_MAX) return QB_EINVAL;
  return launch_lei_rho(topk_idx, N, E, k, eta, batch_tokens, workspace, as_stream(stream));
}

int lei_apply(float* grad, int64_t N, int E, int64_t batch_tokens, const float* workspace,
              void* stream) {
  if (!grad || !workspace) return QB_EINVAL;
  if (!aligned16(grad) || !aligned16(workspace)) return QB_EINVAL;
  if (N < 0 || batch_tokens < 0) return QB_EINVAL;
  if (!supported_E(E)) return QB_EUNSUPPORTED;
  if (N == 0) return QB_OK;
  if (batch_tokens == 0 || batch_tokens > N) batch_tokens = N;
  if (N > INT32_MAX) return QB_EOVERFLOW;
  return launch_lei_apply(grad, N, E, batch_tokens, workspace, as_stream(stream));
}

int lei_apply_overlap(float* grad, int64_t N, int E, int64_t batch_tokens, const float* workspace,
                      void* stream) {
  if (!grad || !workspace) return QB_EINVAL;
  if (!aligned16(grad) || !aligned16(workspace)) return QB_EINVAL;
  if (N < 0 || batch_tokens < 0) return QB_EINVAL;
  if (!supported_E(E)) return QB_EUNSUPPORTED;
  if (N == 0) return QB_OK;
  if (batch_tokens == 0 || batch_tokens > N) batch_tokens = N;
  if (N > INT32_MAX) return QB_EOVERFLOW;
  return launch_lei_apply_overlap(grad, N, E, batch_tokens, workspace, as_stream(stream));
}

int qb_router_gemm(const void* hidden, const void* w_t, int64_t M, int H, int E, float* logits_out,
                   void* stream) {
  if (!hidden || !w_t || !logits_out) return QB_EINVAL;
  if (!aligned16(hidden) || !aligned16(w_t) || !aligned16(logits_out)) return QB_EINVAL;
  if (M < 0) return QB_EINVAL;
  if (M > INT32_MAX) return QB_EOVERFLOW;
  if (E < 32 || E > 256 || E % 32 != 0 || H < 64 || H % 64 != 0) return QB_EUNSUPPORTED;
  if (M == 0) return QB_OK;
  return launch_router_gemm(hidden, w_t, M, H, E, logits_out, as_stream(stream));
}

int qb_router_gemm_hist_hi(const void* hidden, const void* w_t, int64_t M, int H, int E, int k,
                           const float* bias, float* logits_out, int32_t* hist_hi,
                           uint16_t* keys_out, int32_t* topk_out, float* alpha_out,
                           void* stream) {
  return router_gemm_hist_hi(hidden, w_t, M, H, E, k, bias, logits_out, hist_hi, keys_out,
                             topk_out, alpha_out, stream, false);
}

int qb_router_gemm_hist_hi_next(const void* hidden, const void* w_t, int64_t M, int H, int E,
                                int k, const float* bias, float* logits_out, int32_t* hist_hi,
                                uint16_t* keys_out, int32_t* topk_out, float* alpha_out,
                                void* stream) {
  return router_gemm_hist_hi(hidden, w_t, M, H, E, k, bias, logits_out, hist_hi, keys_out,
                             topk_out, alpha_out, stream, true);
}

int qb_rank_average(const uint16_t* qkeys, int P, int E, float* bias_out, void* stream) {
  if (!qkeys || !bias_out || P < 1) return QB_EINVAL;
  if (!supported_E(E)) return QB_EUNSUPPORTED;
  return launch_rank_average(qkeys, P, E, bias_out, as_stream(stream));
}

int qb_maxvio(const int32_t* topk_idx, int64_t N, int E, int k, int64_t batch_tokens,
              int32_t* loads_out, double* maxvio_out, void* stream) {
  if (!topk_idx || !loads_out || !maxvio_out) return QB_EINVAL;
  if (!aligned16(topk_idx)) return QB_EINVAL;
  if (N < 1 || batch_tokens < 0) return QB_EINVAL;
  if (!supported_E(E)) return QB_EUNSUPPORTED;
  if (k < 1 || k >= E) return QB_EINVAL;
  if (batch_tokens == 0 || batch_tokens > N) batch_tokens = N;
  if (N > INT32_MAX) return QB_EOVERFLOW;
  return launch_maxvio(topk_idx, N, E, k, batch_tokens, loads_out, maxvio_out,
                       as_stream(stream));
}

int qb_device_status(int* flags_out) {
  int* p = device_status_ptr();
  if (!p) return QB_ECUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_status_word, sizeof(int)) != cudaSuccess) return QB_ECUDA;
  const int zero = 0;
  if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof(int)) != cudaSuccess) return QB_ECUDA;
  if (flags_out) *flags_out = v;
  return v ? QB_EDEVICE : QB_OK;
}

}  // extern "C"
