/*
 * qb.h -- C ABI of libqb: the data-parallel hot path of bias-based quantile
 * balancing (QB) for Mixture-of-Experts routers, on one NVIDIA GB300 (sm_103a).
 *
 * Sources (web pages, cited by title and section):
 *   [QB-PR] "[Dev] Add global-batch quantile balancing" (Megatron-LM pull
 *           request 6637).  "Quantile estimator": s[i,j] is the raw sigmoid
 *           router score, alpha[i] the (k+1)-th largest value of s[i,:] + b,
 *           r[i,j] = alpha[i] - s[i,j], b_next[j] = quantile(r[:,j], k/E),
 *           then b_next -= mean(b_next); the K3 histogram spans
 *           [min(b_next)-1, max(b_next)+1] with 1000 uniform bins per expert.
 *           "Implementation": one persistent-address int32 histogram
 *           [num_experts, num_bins] accumulated over every microbatch; bias and
 *           bounds updated in place once; histogram reset without changing
 *           its address.
 *   [EQB]   "Exact Quantile Balancing and Load-Error Injection for Mixture-of-
 *           Experts".  EQB paragraph: histogram the high byte of the BF16
 *           margins (256 bins per expert), locate the bin holding the r-th
 *           smallest value, histogram the low byte within that bin,
 *           concatenate the bytes.  LEI paragraph: add eta * rho_e to the
 *           score gradient of expert e for every token of the local batch.
 *
 * Conventions common to every entry point
 *   - Pointers marked "device" are CUDA device pointers; the caller owns every
 *     buffer.  The library allocates nothing and keeps no host state.
 *   - Every call is asynchronous on `stream` (a cudaStream_t passed as void*;
 *     NULL is the legacy default stream).  Argument errors are detected on the
 *     host and returned before anything is launched; nothing is written then.
 *   - Layouts are row-major.  logits / scores / grads are [N, E] with the
 *     expert index contiguous.  EQB histograms are int32 [E, 256]; K3
 *     histograms are int32 [E, nbins].
 *   - Histograms accumulate (+=).  Zero them once before the first microbatch
 *     of a global batch (qb_zero_i32), or let the finalize call reset them in
 *     place.  Counts are int32: the pooled token count must stay below 2^31.
 *   - Inputs must be finite; results on NaN logits are unspecified.
 *   - Supported expert counts: any multiple of 32 from 32 to 1024 (rows of
 *     a count that is not a power of two are processed in the tile of the
 *     next power of two, the extra experts masked).  The router GEMM takes
 *     E = 256 only.  Supported k: 1 <= k <= 15 and k < E.
 *   - Return value: QB_OK (0) or a negative qb_status.
 */
#ifndef QB_H
#define QB_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  QB_OK = 0,
  QB_EINVAL = -1,        /* null / misaligned pointer, bad size, bad rank  */
  QB_EUNSUPPORTED = -2,  /* E or k outside the compiled variants           */
  QB_ECUDA = -3,         /* a CUDA launch or runtime call failed           */
  QB_EOVERFLOW = -4,     /* a count would not fit its int32 counter        */
  QB_EDEVICE = -5        /* a kernel reported a device-side error          */
} qb_status;

typedef enum { QB_F32 = 0, QB_BF16 = 1 } qb_dtype;

/* Human-readable text for a status code (static storage). */
const char* qb_status_string(int status);

/* Library version string. */
const char* qb_version(void);

/* Rank of the k/E quantile among n_pool pooled samples, 1-based:
 * r = ceil(k * n_pool / E) in integer arithmetic.  This is the type-1
 * (inverse-CDF) reading of "quantile(r[:,j], k/E)" ([QB-PR] "Quantile
 * estimator") that makes the two-byte radix select of [EQB] return one
 * element.  Returns a negative qb_status on bad arguments. */
int64_t qb_rank(int64_t n_pool, int E, int k);

/* Pinned logistic function, element-wise: s[i] = sigma(x[i]) as the fixed
 * binary32 operation sequence the routing kernels use ([QB-PR] "raw sigmoid
 * router score"):  s = RN(1 / RN(1 + RN(p(w) * 2^n))) with n = rint(-x*log2 e),
 * w = x + n*ln2 (Cody-Waite, two fma), p = degree-7 Taylor polynomial of
 * exp(-w) in Horner/fma form; x clamped to [-104, 104].  Computed by the same
 * device code as the routing kernels (chunks of 8).  x, s: device fp32 [n];
 * may alias. */
int qb_sigmoid(const float* x, float* s, int64_t n, void* stream);

/* The same function through the routing kernels' exact scalar sequence only
 * (the packed fast path covers |x| <= 86; the kernels switch a whole chunk
 * to this sequence when any input of it is larger).  Results equal
 * qb_sigmoid's bit for bit; a diagnostic for checking both sequences.
 * x, s: device fp32 [n]; may alias. */
int qb_sigmoid_scalar(const float* x, float* s, int64_t n, void* stream);

/* Fill n int32 values with zero (a convenience for histograms). */
int qb_zero_i32(int32_t* p, int64_t n, void* stream);

/* ---------------------------------------------------------------- EQB ---- */

/* Route one microbatch and accumulate the EQB hi-byte histogram.
 * ([QB-PR] "Quantile estimator"; [EQB] EQB paragraph, first pass.)
 *   logits   device [N, E], fp32 (dtype QB_F32) or bf16 (QB_BF16); 16-byte
 *            aligned.
 *   bias     device fp32 [E], the selection bias used by this forward pass.
 *   hist_hi  device int32 [E, 256]; hist_hi[j][key>>8] += 1 for every token,
 *            where key is the order-preserving key of RN_bf16(r[i,j])
 *            (-0 folded to +0; key = bits ^ (sign ? 0xFFFF : 0x8000)).
 *   keys_out optional device uint16 [N, E] (16-byte aligned): the keys, for
 *            qb_keys_hist_lo.  NULL to skip.
 *   topk_out optional device int32 [N, k]: the k experts of largest s + b
 *            (ties to the lower index), ascending expert index.  NULL to skip.
 *   alpha_out optional device fp32 [N]: alpha per token.  NULL to skip.
 * Several calls (one per microbatch) accumulate into the same hist_hi. */
int qb_route_hist_hi(const void* logits, int dtype, const float* bias, int64_t N, int E, int k,
                     int32_t* hist_hi, uint16_t* keys_out, int32_t* topk_out, float* alpha_out,
                     void* stream);

/* A further microbatch of the same global batch: the same operation and
 * arguments as qb_route_hist_hi, for a call issued on `stream` directly after
 * a qb_route_hist_hi or qb_route_hist_hi_next call of the same batch (same
 * bias and hist_hi; [QB-PR] "Implementation": the histogram accumulates over
 * every microbatch).  At E = 256 the call may start while the one before it
 * still runs (its counts only add to hist_hi), so back-to-back microbatch
 * calls overlap instead of each waiting for the last one to finish.
 * Ownership and ordering: nothing between the two calls on the stream, and no
 * other stream, may write this call's logits, bias or hist_hi while it runs,
 * nor read its outputs before the stream reaches a later operation (which
 * orders after both calls).  Other E: the same as qb_route_hist_hi. */
int qb_route_hist_hi_next(const void* logits, int dtype, const float* bias, int64_t N, int E,
                          int k, int32_t* hist_hi, uint16_t* keys_out, int32_t* topk_out,
                          float* alpha_out, void* stream);

/* Select the hi-byte bin that holds the rank-r value of every expert
 * ([EQB] EQB paragraph: "locate the bin holding the r-th smallest value").
 *   hist_hi  device int32 [E, 256], pooled over the whole global batch.
 *   r        1-based rank, from qb_rank(N_pool, E, k).
 *   sel      device int32 [E]: first bin b with sum_{b'<=b} hist_hi[j][b'] >= r.
 *   r_lo     device int32 [E]: r minus the count of the bins below sel.
 * A row holding fewer than r samples yields sel = -1, r_lo = 0. */
int qb_select_hi(const int32_t* hist_hi, int E, int64_t r, int32_t* sel, int32_t* r_lo,
                 void* stream);

/* Second pass from stored keys ([EQB] EQB paragraph, "a second pass
 * histograms the low byte within that bin"):
 *   hist_lo[j][key & 0xFF] += 1 for every key of expert j with key>>8 == sel[j].
 *   keys device uint16 [N, E] as written by qb_route_hist_hi; 16-byte aligned.
 * N may cover any number of microbatches (keys stored contiguously). */
int qb_keys_hist_lo(const uint16_t* keys, int64_t N, int E, const int32_t* sel,
                    int32_t* hist_lo, void* stream);

/* Second pass recomputed from the logits (same result as qb_keys_hist_lo on
 * the keys of the same logits and bias, without storing keys). */
int qb_route_hist_lo(const void* logits, int dtype, const float* bias, int64_t N, int E, int k,
                     const int32_t* sel, int32_t* hist_lo, void* stream);

/* Finish the select and update the bias ([EQB] "concatenating the two bytes
 * recovers the exact global quantile"; [QB-PR] "Quantile estimator",
 * mean-centering; "Implementation", in-place update and reset):
 *   lo_j  = first bin l with sum_{l'<=l} hist_lo[j][l'] >= r_lo[j]
 *   q_j   = fp32 value of the bf16 number whose key is (sel_j << 8) | lo_j
 *   mu    = (sum_j q_j in fp64, ascending j) / E
 *   bias_out[j] = RN32(q_j - mu)
 * bias_out (device fp32 [E]) may alias the bias used for routing.
 * qkey_out optional device uint16 [E] receives the selected keys.
 * reset != 0 zeroes hist_hi and hist_lo in place afterwards. */
int qb_finalize(int32_t* hist_hi, int32_t* hist_lo, const int32_t* sel, const int32_t* r_lo,
                int E, float* bias_out, uint16_t* qkey_out, int reset, void* stream);

/* ----------------------------------------------------------------- K3 ---- */

/* Route one microbatch and accumulate the K3 uniform histogram
 * ([QB-PR] "Quantile estimator" and "Implementation"):
 *   w = RN(hi - lo), scale = RN(nbins / w),
 *   idx = floor(RN(RN(r - lo) * scale)), clamped to [0, nbins-1],
 *   hist[j][idx] += 1, with r the fp32 margin.
 *   bounds    device fp32 [2] = {lo, hi}, lo < hi (read on the device).
 *   hist      device int32 [E, nbins]; 1 <= nbins <= 65536.
 *   alpha_out device fp32 [N]: receives alpha of every token.  The first of
 *             the call's two launches routes the tokens and writes alpha
 *             there; the second recomputes each expert slice's scores from
 *             the logits and counts the margins' bins (a 1000-bin histogram
 *             per expert is too large to count in one routing pass).
 * Two launches on `stream`. */
int k3_route_hist(const void* logits, int dtype, const float* bias, int64_t N, int E, int k,
                  const float* bounds, int nbins, int32_t* hist, float* alpha_out,
                  void* stream);

/* A further microbatch of the same global batch: the same operation and
 * arguments as k3_route_hist, for a call issued on `stream` directly after a
 * k3_route_hist or k3_route_hist_next call of the same batch (same bias,
 * bounds and hist).  At E = 256 its alpha pass may start on the SMs that the
 * previous call's counting leaves, so alpha_out must not be the previous
 * call's alpha_out (two buffers used in turn suffice: the call before that
 * has finished).  Ownership and ordering otherwise as qb_route_hist_hi_next.
 * Other E: the same as k3_route_hist. */
int k3_route_hist_next(const void* logits, int dtype, const float* bias, int64_t N, int E,
                       int k, const float* bounds, int nbins, int32_t* hist, float* alpha_out,
                       void* stream);

/* K3 quantile, centering and next bounds ([QB-PR] "Quantile estimator"):
 *   b*  = first bin with cumulative count >= r, before = count below it,
 *   q_j = (lo + b* * width) + width * ((r - before) / count[b*]) in fp64,
 *         width = (hi - lo) / nbins;
 *   bias_out[j] = RN32(q_j - mean_j q_j);
 *   bounds <- {min_j bias_out - 1, max_j bias_out + 1} (fp32, in place).
 * Device arithmetic differs from these formulas only in rounding, far
 * inside this mode's 1e-6 relative tolerance: width = (hi - lo) * RN(1/nbins)
 * and the in-bin fraction (r - before) / count is an fp32 quotient; the fp64
 * sum behind the mean is a fixed tree (8 groups of E/8 experts, then the 8
 * partial sums in order), not the ascending serial order.  E <= 512.
 * reset != 0 zeroes hist afterwards.  bounds and bias_out are device. */
int k3_finalize(int32_t* hist, int E, int nbins, int64_t r, float* bounds, float* bias_out,
                int reset, void* stream);

/* ---------------------------------------------------------------- LEI ---- */

/* Load-error injection on a run of local batches ([EQB] LEI paragraph).
 * The N tokens are split into consecutive local batches of `batch_tokens`
 * tokens (0 means one batch of N; the last batch may be shorter).  For each
 * batch with n tokens:
 *   load_e   = #{(i,t) : topk_idx[i,t] == e},   T = n * k / E
 *   rho_raw  = (load_e - T) / T,   rho_e = tanh(rho_raw_e) - mean_e tanh(rho_raw)
 *   grad[i,e] = RN32(grad[i,e] + RN32(eta * rho_e)) for every token i of it.
 * rho and eta*rho are evaluated in fp32 (loads and T are exact); eta*rho
 * agrees with the real-number formula to about 1e-11 at eta = 8e-5, well
 * inside the 1e-6 absolute tolerance on grad.
 *   grad      device fp32 [N, E], updated in place; 16-byte aligned.
 *   topk_idx  device int32 [N, k], entries in [0, E).
 *   workspace device fp32 [num_batches * E] scratch owned by the caller
 *             (num_batches = ceil(N / batch_tokens)); it receives eta*rho. */
int lei_inject(float* grad, const int32_t* topk_idx, int64_t N, int E, int k, float eta,
               int64_t batch_tokens, float* workspace, void* stream);

/* lei_inject in two calls, for schedules that run the two halves at
 * different times (e.g. the grad update beside the next layer's routing).
 * lei_rho(...) + lei_apply(...) on one stream with the same workspace give
 * exactly the result of lei_inject(...).
 * lei_rho: the per-batch loads and eta*rho of lei_inject written to
 *   `workspace` (fp32 [num_batches * E], 16-byte aligned, caller-owned);
 *   grad is not touched.  Arguments and errors as in lei_inject.
 * lei_apply: grad[i,e] = RN32(grad[i,e] + workspace[batch(i) * E + e]) for
 *   every token i, batch(i) = i / batch_tokens (0 means one batch of N);
 *   grad and workspace 16-byte aligned.  The grad update is one launch of
 *   small CTAs (128 threads), so that it fits beside other resident kernels. */
int lei_rho(const int32_t* topk_idx, int64_t N, int E, int k, float eta, int64_t batch_tokens,
            float* workspace, void* stream);
int lei_apply(float* grad, int64_t N, int E, int64_t batch_tokens, const float* workspace,
              void* stream);

/* lei_apply launched to run beside the kernel enqueued just before it on
 * `stream` (a programmatic dependent launch): it may start as soon as every
 * CTA of that kernel has started (qb_route_hist_hi, qb_route_hist_lo and
 * k3_route_hist signal this at their start; any other kernel at its exit)
 * and it completes only after that kernel has completed, so work enqueued
 * after it sees both.  Use it to overlap the grad stream of one layer with
 * the routing pass of the next.  Same arguments and result as lei_apply,
 * bit for bit.  The adds are done by the bulk-copy unit
 * (cp.reduce.async.bulk .add.f32 into L2, binary32 round-to-nearest-even),
 * one 32-thread CTA with 4 KB of shared memory per SM.  The caller must
 * make sure that the preceding kernel neither reads nor writes grad and
 * does not write workspace (it runs concurrently), and that workspace was
 * complete before that kernel was enqueued. */
int lei_apply_overlap(float* grad, int64_t N, int E, int64_t batch_tokens, const float* workspace,
                      void* stream);

/* --------------------------------------------------------- router GEMM ---- */

/* Router logits on the tensor cores: logits[M, E] = hidden[M, H] x W[H, E],
 * bf16 inputs, fp32 accumulation (tcgen05.mma, accumulator in tensor memory).
 * The router of [QB-PR] ("Implementation": the histogram is added to the
 * existing router kernel) produces these scores.
 *   hidden     device bf16 [M, H] row-major, 16-byte aligned.
 *   w_t        device bf16 [E, H]: W transposed (each expert's column of W
 *              contiguous), 16-byte aligned.
 *   logits_out device fp32 [M, E], 16-byte aligned.
 * Supported: E a multiple of 32 from 32 to 256 (the MMA's N), H a positive
 * multiple of 64.  The accumulation order
 * over H is the tensor core's; results agree with an fp64 product within
 * fp32 accumulation error. */
int qb_router_gemm(const void* hidden, const void* w_t, int64_t M, int H, int E, float* logits_out,
                   void* stream);

/* The router GEMM with the EQB hi pass in its epilogue ([QB-PR]
 * "Implementation": classification and histogram counts added to the router
 * kernel, no full score tensor kept): the logits stay in tensor memory and
 * sigmoid, top-(k+1), margins, keys and hi-byte counts are computed there.
 * Outputs equal qb_route_hist_hi run on this GEMM's fp32 logits (same
 * binary32 steps): hist_hi += counts; keys_out, topk_out, alpha_out as in
 * qb_route_hist_hi (each optional); logits_out optional (fp32 [M, E],
 * written only when given, e.g. to check the outputs).  Arguments as in
 * qb_router_gemm and qb_route_hist_hi; 1 <= k <= 15.  E = 256: one launch,
 * a persistent CTA per SM; tokens with more than 8 candidate groups of 8
 * experts (ties) or a tie at alpha take a slower exact path.  Other E (a
 * multiple of 32 up to 256) require logits_out (QB_EUNSUPPORTED without
 * it): qb_router_gemm into logits_out, then qb_route_hist_hi on it. */
int qb_router_gemm_hist_hi(const void* hidden, const void* w_t, int64_t M, int H, int E, int k,
                           const float* bias, float* logits_out, int32_t* hist_hi,
                           uint16_t* keys_out, int32_t* topk_out, float* alpha_out,
                           void* stream);

/* A further microbatch of the same global batch: the same operation and
 * arguments as qb_router_gemm_hist_hi, for a call issued on `stream`
 * directly after a qb_router_gemm_hist_hi or qb_router_gemm_hist_hi_next
 * call of the same batch (same bias and hist_hi).  At E = 256 the call's CTAs
 * may start on the SMs that the previous call's CTAs leave while its last
 * tiles are still in their epilogues; the ownership and ordering rules are
 * those of qb_route_hist_hi_next.  Other E: the same as
 * qb_router_gemm_hist_hi. */
int qb_router_gemm_hist_hi_next(const void* hidden, const void* w_t, int64_t M, int H, int E,
                                int k, const float* bias, float* logits_out, int32_t* hist_hi,
                                uint16_t* keys_out, int32_t* topk_out, float* alpha_out,
                                void* stream);

/* Load-error injection without a caller workspace.  The pages have no
 * counterpart to this entry point; it exists for callers that cannot allocate
 * device memory where LEI is applied -- code under a framework whose caching
 * allocator owns the memory pool, services with a device-memory budget fixed
 * at start-up, or call sites that hold no allocator.
 * Same arguments and results as lei_inject, minus `workspace`: the eta*rho
 * scratch lives in a fixed array inside the library's device memory
 * (65536 floats = 256 KiB per GPU, held until process exit).  Requires
 * ceil(N / batch_tokens) * E <= 65536, else returns QB_EINVAL before
 * launching anything.  Allocates nothing itself (no cudaMalloc or cudaFree).
 * The first successful call on a device looks up the array's device address
 * there (cudaGetSymbolAddress).  Under CUDA's default lazy module loading that
 * lookup is also when the driver loads the library's device code on that
 * device and reserves the 256 KiB (with CUDA_MODULE_LOADING=EAGER it happens
 * when the context is created), so a caller with a fixed memory budget should
 * make one call at start-up, and that first call must come before any stream
 * capture.  A failed lookup returns QB_ECUDA, clears the CUDA error it left
 * and is retried by the next call.  All calls share the one array, which
 * keeps the last call's contents (every value read is first written by the
 * same call, so nothing needs clearing); calls that overlap on the GPU -- on
 * different streams, or from different host threads -- race on it and must
 * be serialised by the caller. */
int lei_inject_noalloc(float* grad, const int32_t* topk_idx, int64_t N, int E, int k, float eta,
                       int64_t batch_tokens, void* stream);

/* ------------------------------------------------ comparison and diagnostics ---- */

/* Rank-averaged QB, the sharding-dependent scheme that [EQB]'s opening
 * paragraph attributes to the MARIN implementation (average of rank-local
 * quantiles).  Each of P ranks runs the EQB steps on its own tokens only
 * (qb_route_hist_hi ... qb_finalize with its own rank R_p = ceil(k*N_p/E)) and
 * hands over the selected keys (qb_finalize's qkey_out).  Then
 *   avg[j]      = (sum over p in rank order of q_p[j], fp64) / P,
 *                 q_p[j] the fp32 value of the bf16 number with key qkeys[p,j]
 *   bias_out[j] = RN32(avg[j] - mu),  mu = (sum_j avg[j] in fp64, ascending j)/E
 *   qkeys    device uint16 [P, E];  bias_out device fp32 [E].
 * One launch; the same arithmetic order as the plain definition (results
 * bit-equal to it). */
int qb_rank_average(const uint16_t* qkeys, int P, int E, float* bias_out, void* stream);

/* MaxVio load-imbalance diagnostic ([EQB] testbed paragraph: how far the
 * busiest expert exceeds uniform load).  The N tokens' top-k sets are split
 * into local batches of batch_tokens (0 = one batch; the last may be shorter):
 *   loads_out[b][e] = #{(i,t) in batch b : topk_idx[i,t] == e}
 *   maxvio_out[0]   = (max_e sum_b loads[b][e] - T) / T,  T = N*k/E   (global)
 *   maxvio_out[1]   = mean_b (max_e loads[b][e] - T_b) / T_b,  T_b = n_b*k/E (local)
 * in fp64, batches in order.  topk_idx device int32 [N, k] (16-byte
 * aligned), loads_out device int32 [num_batches, E], maxvio_out device
 * double [2].  Two launches. */
int qb_maxvio(const int32_t* topk_idx, int64_t N, int E, int k, int64_t batch_tokens,
              int32_t* loads_out, double* maxvio_out, void* stream);

/* Reads and clears the device status word that kernels set instead of
 * trapping (bit 0: a bounded wait timed out).  Synchronous; returns QB_OK
 * when clear, QB_EDEVICE when a flag was set, QB_ECUDA on a CUDA error. */
int qb_device_status(int* flags_out);

/* Diagnostic for the bounded-wait path of every kernel: launches one warp
 * that waits on a shared-memory mbarrier nothing will complete (no arrival,
 * no copy issued against it) with a limit of `polls` polls (1 <= polls <=
 * 2^24).  The wait gives up, sets bit 0 of the device status word and the
 * kernel returns, leaving no copy in flight; qb_device_status then reports
 * QB_EDEVICE once.  The pages have no counterpart: it exists so that the
 * status reporting can be tested without a GPU fault. */
int qb_selftest_wait_timeout(int64_t polls, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* QB_H */
