/*
 * qb_oracle.h -- plain CPU oracle for bias-based quantile balancing (QB).
 *
 * TEST INFRASTRUCTURE ONLY.  This library is the slow, obviously-correct
 * restatement of what the GPU path computes.  It exists so that tests, the
 * smoke check and the benchmark's CPU-baseline leg can compare against it.
 * Nothing in the product path may link, load or call it, and it shares no
 * code, header, table or constant with the CUDA library.
 *
 * Sources (web pages; cited by title and section):
 *   [QB-PR]  "[Dev] Add global-batch quantile balancing" (Megatron-LM pull
 *            request 6637), sections "Quantile estimator" and "Implementation".
 *   [EQB]    "Exact Quantile Balancing and Load-Error Injection for
 *            Mixture-of-Experts" (paper summary), the EQB paragraph and the
 *            LEI paragraph.
 *
 * Every floating-point step below is an IEEE-754 basic operation in round-to-
 * nearest-even, in program order; the file is compiled with
 * -ffp-contract=off so that no multiply-add is fused unless fmaf() is called.
 */
#ifndef QB_ORACLE_H
#define QB_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Pinned logistic function (the "raw sigmoid router score", [QB-PR]
 * "Quantile estimator").  See qb_oracle.c for the exact operation sequence. */
float orc_sigmoid(float x);
void orc_sigmoid_array(const float* x, float* s, int64_t n);
/* The exp(-x) stage of orc_sigmoid, exposed for accuracy tests. */
float orc_exp_neg(float x);
/* Taylor coefficients used by the exp stage, c[0..7] = RN((-1)^i / i!). */
void orc_exp_coeffs(float* c8);

/* fp32 -> bf16 bit pattern, round to nearest, ties to even. */
uint16_t orc_bf16_rne(float r);
/* Order-preserving 16-bit key of RN_bf16(r): -0 folds to +0, then
 * key = bits ^ (sign ? 0xFFFF : 0x8000) ([EQB] EQB paragraph). */
uint16_t orc_key(float r);
/* Inverse of the key map: the fp32 value of the bf16 number with that key. */
float orc_key_decode(uint16_t key);
void orc_keys_array(const float* r, uint16_t* keys, int64_t n);
void orc_bf16_array(const float* r, uint16_t* bits, int64_t n);

/* Routing of N tokens with E experts ([QB-PR] "Quantile estimator"):
 *   s = sigmoid(logit), v_j = RN(s_j + b_j),
 *   alpha = (k+1)-th largest v (full sort, ties kept with multiplicity),
 *   margins r_j = RN(alpha - s_j),
 *   topk = the k experts first in the order (v descending, j ascending).
 * logits are fp32 [N,E] row-major; the bf16 variant takes raw bf16 bits.
 * Any output pointer may be NULL. */
void orc_route(const float* logits, const float* bias, int64_t N, int E, int k,
               float* alpha, float* scores, float* margins, int32_t* topk);
void orc_route_bf16(const uint16_t* logits_bf16, const float* bias, int64_t N, int E, int k,
                    float* alpha, float* scores, float* margins, int32_t* topk);

/* Rank of the k/E quantile among n_pool samples: ceil(k*n_pool/E), 1-based. */
int64_t orc_rank(int64_t n_pool, int E, int k);

/* EQB histograms by direct counting ([EQB] EQB paragraph).  Both accumulate
 * (+=) into int32 [E,256] (expert-major). */
void orc_hist_hi(const uint16_t* keys, int64_t N, int E, int32_t* hist_hi);
void orc_hist_lo(const uint16_t* keys, int64_t N, int E, const int32_t* sel, int32_t* hist_lo);

/* Rank select on a 256-bin histogram row: sel = first bin whose cumulative
 * count reaches R, r_lo = R minus the count of the bins below sel. */
void orc_select_hi(const int32_t* hist_hi, int E, int64_t R, int32_t* sel, int32_t* r_lo);
void orc_select_lo(const int32_t* hist_lo, int E, const int32_t* r_lo, int32_t* lo);

/* The exact R-th smallest key of every expert column, by sorting all keys of
 * that column (keys [N_pool,E]). */
void orc_kth_key_sort(const uint16_t* keys, int64_t n_pool, int E, int64_t R, uint16_t* qkey);

/* Mean-centering ([QB-PR] "Quantile estimator", last line):
 * mu = (sum_j q_j in fp64, ascending j) / E;  b_j = RN32(q_j - mu). */
void orc_center(const double* q, int E, float* b_out);

/* K3 uniform histogram ([QB-PR] "Quantile estimator" and "Implementation"):
 * width w = RN(hi - lo), scale = RN(nbins / w),
 * idx = floor(RN(RN(r - lo) * scale)) clamped to [0, nbins-1]; += into
 * int32 [E,nbins]. */
void orc_k3_hist(const float* margins, int64_t N, int E, float lo, float hi, int nbins,
                 int32_t* hist);
/* K3 quantile by linear interpolation inside the bin where the cumulative
 * count reaches R, then centering, then the next bounds
 * [min b - 1, max b + 1] in fp32.  q_out (fp64 [E]) may be NULL. */
void orc_k3_finalize(const int32_t* hist, int E, int nbins, int64_t R, float lo, float hi,
                     float* b_out, float* bounds_out, double* q_out);

/* Load-error injection ([EQB] LEI paragraph) on one local batch:
 * load_e = #(i,t) with topk[i,t]==e, T = N*k/E, rho_raw = (load-T)/T,
 * rho = tanh(rho_raw) - mean(tanh(rho_raw)), grad[i,e] = RN32(grad[i,e] +
 * RN32(eta*rho_e)) for every token i.  load_out / rho_out may be NULL. */
void orc_lei(float* grad, const int32_t* topk, int64_t N, int E, int k, float eta,
             int64_t* load_out, double* rho_out);

/* Number of OpenMP threads the oracle uses (1 when built without OpenMP). */
int orc_num_threads(void);
void orc_set_num_threads(int n);

#ifdef __cplusplus
}
#endif
#endif
