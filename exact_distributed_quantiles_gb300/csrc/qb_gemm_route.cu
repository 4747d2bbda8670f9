// qb_gemm_route.cu -- the router GEMM with the routing pass in its epilogue:
// logits = hidden x W on the tensor cores, then, straight from the TMEM
// accumulator, sigmoid, top-(k+1), margins, BF16 keys and the hi-byte
// histogram, without the logits ever reaching global memory (unless asked).
//
// "[Dev] Add global-batch quantile balancing", "Implementation": the fused
// path adds bin classification and histogram atomics to the router kernel
// and keeps no full score tensor; "Quantile estimator": s = sigmoid(logit),
// alpha = (k+1)-th largest of s + b, r = alpha - s.  "Exact Quantile
// Balancing and Load-Error Injection for Mixture-of-Experts", EQB paragraph:
// the hi-byte histogram of the BF16 margins.  Every step computes the same
// binary32 values as the routing kernel, so the keys, top-k sets and counts
// equal those of the routing kernel run on this GEMM's fp32 logits.
//
// One persistent CTA per SM over tiles of 128 tokens x 256 experts:
//   warp 0      TMA producer (3-stage ring of hidden and W^T K-slices);
//   warp 1      allocates all 512 TMEM columns (two accumulators) and issues
//               tcgen05.mma into accumulator (local tile index & 1);
//   warps 2-9   two epilogue warpgroups, warpgroup b serving accumulator b,
//               one thread per token (TMEM lane), 32 columns at a time:
//     A  sigmoid of the row (packed path when |x| <= 86), v = s + b, the max
//        of every group of 8 experts; the scores go back into TMEM;
//     B  the (k+1)-th largest group max tau bounds alpha from below; the
//        groups whose max reaches tau (k+1 of them for nearly every token)
//        are staged in shared memory and merged by sorting networks into
//        alpha; the top-k set is read off the staged groups;
//     C  r = alpha - s, keys out, one shared increment per element into the
//        32-bin window: 16-bit counter pairs (two experts per word), rows of
//        129 words, so the 32 tokens of a warp that hit different bins of
//        one expert use different banks.  The launcher keeps every CTA under
//        2^16 tokens per launch.
//   A token with more candidate groups than the staging holds, or with a tie
//   at alpha in its top-k set, takes an exact one-thread path (insertion over
//   all 256 values) -- rare, and correct for any input.
// Every wait is bounded; a timeout sets the device status word and the CTA
// still frees its TMEM before returning.
#include "qb_device.cuh"
#include "qb_internal.h"
#include "qb_route.cuh"
#include "qb_tc.cuh"

namespace qb {
namespace {

using route::first_block8;
using route::merge_block8;

constexpr int kE = 256;        // experts: TMEM columns per accumulator
constexpr int kBM = 128;       // tokens per tile: TMEM lanes
constexpr int kBK = 64;        // K per stage (one 128-byte swizzle row of bf16)
constexpr int kStages = 3;
constexpr int kABytes = kBM * kBK * 2;
constexpr int kBBytes = kE * kBK * 2;
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kEpiWarps = 8;
constexpr int kThreads = (2 + kEpiWarps) * 32;
constexpr int kStageGroups = 8;          // candidate groups staged per token
constexpr int kWinRow = kE / 2 + 1;      // words per window slot row (16-bit counter pairs)
constexpr int kWinSlots = route::kWin + 1;
constexpr uint32_t kIdescGR = idesc_bf16_f32(kBM, kE);

constexpr int kOffWin = kStages * kStageBytes;
constexpr int kOffStage = kOffWin + ((kWinSlots * kWinRow * 4 + 15) & ~15);
constexpr int kOffBias = kOffStage + kEpiWarps * 32 * kStageGroups * 32;
constexpr int kOffLut = kOffBias + kE * 4;
constexpr int kOffBar = kOffLut + 256;
constexpr int kSmemUsed = kOffBar + 12 * 8 + 16;
constexpr int kSmemBytes = kSmemUsed + 1024;  // + alignment slack

struct FusedArgs {
  const float* bias;
  int64_t M;
  int K;
  int k;
  int32_t* hist;       // [256, 256] += hi-byte counts
  uint16_t* keys_out;  // [M, 256] or null
  int32_t* topk_out;   // [M, k] or null
  float* alpha_out;    // [M] or null
  float* logits_out;   // [M, 256] or null
  int* status;
  // a later microbatch of the same global batch, issued right after another
  // fused call on the stream (qb_router_gemm_hist_hi_next): skips the wait
  // for the previous kernel at its start and waits at its end instead
  int chained;
};

// The window slot of a hi byte computed in registers (the same map as the
// routing kernel's table: bytes 0x40-0x4F -> 0-15, 0xB0-0xBF -> 16-31, any
// other -> the dummy row 32).  The epilogue has issue slots to spare, and a
// table load would put shared-memory latency in front of every increment.
__device__ __forceinline__ uint32_t window_slot(uint32_t bin) {
  const uint32_t in_window = (0x0810u >> (bin >> 4)) & 1u;  // hi nibble 4 or 11
  const uint32_t slot = (bin & 15u) | ((bin >> 3) & 16u);
  return in_window ? slot : (uint32_t)route::kDummy;
}

// No "memory" clobber: the window is read only after the __syncthreads
// before the flush, and without the clobber the compiler can issue the
// loads of a chunk ahead of its increments.
template <uint32_t V>
__device__ __forceinline__ void red_shared_addc(uint32_t addr) {
  asm volatile("red.shared.add.u32 [%0], %1;" ::"r"(addr), "n"(V));
}

template <int KL, int K1>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_route_kernel(const __grid_constant__ CUtensorMap map_a,
                      const __grid_constant__ CUtensorMap map_b, const FusedArgs g) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* sb = smem_raw + (base - raw);
  uint32_t* win = reinterpret_cast<uint32_t*>(sb + kOffWin);
  float* stage_all = reinterpret_cast<float*>(sb + kOffStage);
  float* bias_s = reinterpret_cast<float*>(sb + kOffBias);
  uint8_t* lut = sb + kOffLut;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sb + kOffBar);
  uint64_t* full = bars;            // [kStages]
  uint64_t* empty = bars + 4;       // [kStages]
  uint64_t* tfull = bars + 8;       // [2]
  uint64_t* tempty = bars + 10;     // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 12);

  const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);
  const int lane = threadIdx.x & 31;
  const int ktiles = g.K / kBK;
  const int64_t n_tiles = (g.M + kBM - 1) / kBM;
  const int k = g.k;

  for (int i = threadIdx.x; i < kWinSlots * kWinRow; i += blockDim.x) win[i] = 0;
  for (int i = threadIdx.x; i < 256; i += blockDim.x) lut[i] = (uint8_t)route::window_slot_of(i);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull + b, 1);
      mbar_init(tempty + b, kEpiWarps / 2 * 32);
    }
    fence_mbar_init();
  }
  // Launched as a programmatic dependent of the kernel before it: wait for
  // its completion (and its memory) before the first global read and before
  // taking tensor memory.  A chained call follows another fused call of the
  // same global batch that has itself waited (its counts only add to the
  // same histogram, its outputs are other rows), so it goes on at once and
  // waits at its end instead, so that it completes after the call before it.
  // The next chained call may launch from here on; one CTA fills an SM
  // (shared memory), so its CTAs take SMs as this call's CTAs leave them.
  if (!g.chained) asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  for (int i = threadIdx.x; i < kE; i += blockDim.x) bias_s[i] = g.bias[i];
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), 2 * kE);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---- TMA producer
    if (lane == 0) {
      bool ok = true;
      uint32_t gk = 0;
      for (int64_t tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
        for (int kt = 0; kt < ktiles; ++kt, ++gk) {
          const int s = (int)(gk % kStages);
          const uint32_t round = gk / kStages;
          if (gk >= (uint32_t)kStages && !mbar_wait_bounded(empty + s, (round - 1) & 1u, g.status)) {
            ok = false;
            break;
          }
          const uint32_t sa = base + (uint32_t)(s * kStageBytes);
          mbar_arrive_expect_tx(full + s, (uint32_t)kStageBytes);
          tma_load_2d(sa, &map_a, kt * kBK, (int)(tile * kBM), smem_u32(full + s));
          tma_load_2d(sa + kABytes, &map_b, kt * kBK, 0, smem_u32(full + s));
        }
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer
    if (lane == 0) {
      bool ok = true;
      uint32_t gk = 0, lt = 0;
      for (int64_t tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x, ++lt) {
        const uint32_t b = lt & 1u, use = lt >> 1;
        if (use >= 1 && !mbar_wait_bounded(tempty + b, (use - 1) & 1u, g.status)) break;
        tc_fence_after();
        const uint32_t d = tmem + b * (uint32_t)kE;
        for (int kt = 0; kt < ktiles; ++kt, ++gk) {
          const int s = (int)(gk % kStages);
          if (!mbar_wait_bounded(full + s, (gk / kStages) & 1u, g.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = base + (uint32_t)(s * kStageBytes);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            tc_mma(d, smem_desc_sw128(sa + 32u * kk), smem_desc_sw128(sa + kABytes + 32u * kk),
                   kIdescGR, (kt > 0 || kk > 0) ? 1u : 0u);
          tc_commit(smem_u32(empty + s));
        }
        if (ok) tc_commit(smem_u32(tfull + b));
      }
    }
  } else {
    // ---- epilogue: warpgroup wg serves accumulator wg; thread = token
    const int wg = (warp - 2) >> 2;
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int et = (warp - 2) * 32 + lane;
    float* stage = stage_all + et * (kStageGroups * 8);
    const uint32_t win_b = smem_u32(win);
    uint32_t use = 0;
    for (int64_t tile = blockIdx.x + (int64_t)wg * gridDim.x; tile < n_tiles;
         tile += 2 * (int64_t)gridDim.x, ++use) {
      bool ok = mbar_wait_bounded(tfull + wg, use & 1u, g.status);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const uint32_t ta = tmem + (uint32_t)(wg * kE) + ((uint32_t)(32 * q) << 16);
      const int64_t row = tile * kBM + 32 * q + lane;
      const bool valid = row < g.M;

      // ---- A: scores, group maxima; scores back into TMEM.  Chunks alternate
      // between two register sets so that the next chunk's TMEM load is in
      // flight while this one is computed.
      float gmx[32];
      bool ext = false;
      auto chunk_a = [&](int c, uint32_t(&r)[32]) {
        float x[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(r[i]);
        if (g.logits_out && valid) {
          float4* dst = reinterpret_cast<float4*>(g.logits_out + row * kE + 32 * c);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[i] = make_float4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]);
        }
        float m = 0.0f;
#pragma unroll
        for (int i = 0; i < 32; ++i) m = fmaxf(m, fabsf(x[i]));
        ext |= m > kFoldAbsX;
        float s[32];
        if (m <= kFastAbsX) {
#pragma unroll
          for (int i = 0; i < 16; ++i)
            f2_unpack(sigmoid2_fast(f2_pack(x[2 * i], x[2 * i + 1])), s[2 * i], s[2 * i + 1]);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) s[i] = sigmoid_pinned(x[i]);
        }
        // group maxima collected by a shift (constant register indices):
        // after chunk 7, gmx[4c + gi] holds chunk c's group gi
#pragma unroll
        for (int i = 0; i < 28; ++i) gmx[i] = gmx[i + 4];
#pragma unroll
        for (int gi = 0; gi < 4; ++gi) {
          float v[8];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 b2 = *reinterpret_cast<const float2*>(bias_s + 32 * c + 8 * gi + 2 * i);
            f2_unpack(f2_add(f2_pack(s[8 * gi + 2 * i], s[8 * gi + 2 * i + 1]), f2_pack(b2.x, b2.y)),
                      v[2 * i], v[2 * i + 1]);
          }
          gmx[28 + gi] = fmaxf(fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3])),
                               fmaxf(fmaxf(v[4], v[5]), fmaxf(v[6], v[7])));
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(s[i]);
        tmem_st32(ta + 32u * c, r);
      };
      {
        uint32_t ra[32], rb[32];
        tmem_ld32_nowait(ta, ra);
#pragma unroll 1
        for (int c = 0; c < 8; c += 2) {
          tmem_wait_ld(ra);
          tmem_ld32_nowait(ta + 32u * (c + 1), rb);
          chunk_a(c, ra);
          tmem_wait_ld(rb);
          if (c + 2 < 8) tmem_ld32_nowait(ta + 32u * (c + 2), ra);
          chunk_a(c + 1, rb);
        }
      }
      tmem_wait_st();

      // ---- B: tau from the group maxima, stage the candidate groups, alpha
      float L[KL];
#pragma unroll
      for (int i = 0; i < KL; ++i) L[i] = -INFINITY;
#pragma unroll
      for (int b0 = 0; b0 < 32; b0 += 8) {
        float v8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v8[i] = gmx[b0 + i];
        if (b0 == 0)
          first_block8<KL>(L, v8);
        else
          merge_block8<KL>(L, v8);
      }
      const float tau = route::pick<KL, K1>(L, k);
      uint32_t cand = 0;
#pragma unroll
      for (int gi = 0; gi < 32; ++gi) cand |= (gmx[gi] >= tau ? 1u : 0u) << gi;
      const int ncand = __popc(cand);
      bool slow = valid && ncand > kStageGroups;
      int nst = 0;
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        if (!__any_sync(0xffffffffu, ((cand >> (4 * c)) & 0xFu) != 0u)) continue;
        uint32_t r[32];
        tmem_ld32(ta + 32u * c, r);
#pragma unroll
        for (int gi = 0; gi < 4; ++gi) {
          if (((cand >> (4 * c + gi)) & 1u) && nst < kStageGroups) {
            float v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
              v[i] = __fadd_rn(__uint_as_float(r[8 * gi + i]), bias_s[32 * c + 8 * gi + i]);
            float4* d4 = reinterpret_cast<float4*>(stage + 8 * nst);
            d4[0] = make_float4(v[0], v[1], v[2], v[3]);
            d4[1] = make_float4(v[4], v[5], v[6], v[7]);
            ++nst;
          }
        }
      }
#pragma unroll
      for (int i = 0; i < KL; ++i) L[i] = -INFINITY;
#pragma unroll 1
      for (int i = 0; i < nst; ++i) {
        const float4 a0 = reinterpret_cast<const float4*>(stage + 8 * i)[0];
        const float4 a1 = reinterpret_cast<const float4*>(stage + 8 * i)[1];
        float v8[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        if (i == 0)
          first_block8<KL>(L, v8);
        else
          merge_block8<KL>(L, v8);
      }
      float alpha = route::pick<KL, K1>(L, k);
      int c_gt = 0;
#pragma unroll
      for (int i = 0; i < KL; ++i) c_gt += (i < k && L[i] > alpha) ? 1 : 0;
      if (g.topk_out) slow = slow || (valid && c_gt < k);

      // exact path for the rare tokens above: insertion over all 256 values
      if (__any_sync(0xffffffffu, slow)) {
        float L3[KL];
#pragma unroll
        for (int i = 0; i < KL; ++i) L3[i] = -INFINITY;
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          uint32_t r[32];
          tmem_ld32(ta + 32u * c, r);
          if (slow) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              route::insert_desc<KL>(L3, __fadd_rn(__uint_as_float(r[i]), bias_s[32 * c + i]));
          }
        }
        if (slow) {
          alpha = route::pick<KL, K1>(L3, k);
          c_gt = 0;
#pragma unroll
          for (int i = 0; i < KL; ++i) c_gt += (i < k && L3[i] > alpha) ? 1 : 0;
        }
        if (g.topk_out) {
          int32_t* out = g.topk_out + row * k;
          int tl = k - c_gt, cnt = 0;
#pragma unroll 1
          for (int c = 0; c < 8; ++c) {
            uint32_t r[32];
            tmem_ld32(ta + 32u * c, r);
            if (slow) {
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                const float v = __fadd_rn(__uint_as_float(r[i]), bias_s[32 * c + i]);
                const bool gt = v > alpha;
                if ((gt || (v == alpha && tl > 0)) && cnt < k) {
                  if (!gt) --tl;
                  out[cnt++] = 32 * c + i;
                }
              }
            }
          }
        }
      }
      if (g.topk_out && valid && !slow) {
        // the k experts above alpha, ascending: the staged groups in order
        int32_t* out = g.topk_out + row * k;
        int cnt = 0;
        uint32_t m = cand;
#pragma unroll 1
        for (int i = 0; i < nst; ++i) {
          const int gi = __ffs((int)m) - 1;
          m &= m - 1;
          const float4 a0 = reinterpret_cast<const float4*>(stage + 8 * i)[0];
          const float4 a1 = reinterpret_cast<const float4*>(stage + 8 * i)[1];
          const float v8[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (v8[j] > alpha && cnt < k) out[cnt++] = 8 * gi + j;
        }
      }
      if (g.alpha_out && valid) g.alpha_out[row] = alpha;

      // ---- C: margins, keys, window counts (two register sets, as in A)
      const bool fold = __any_sync(0xffffffffu, ext);
      auto chunk_c = [&](int c, const uint32_t(&r)[32]) {
        uint32_t kw[16];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float s8[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) s8[i] = __uint_as_float(r[8 * j + i]);
          uint32_t w4[4];
          if (fold)
            route::keys8<true>(alpha, s8, w4);
          else
            route::keys8<false>(alpha, s8, w4);
#pragma unroll
          for (int i = 0; i < 4; ++i) kw[4 * j + i] = w4[i];
        }
        if (valid) {
          if (g.keys_out) {
            uint4* dst = reinterpret_cast<uint4*>(g.keys_out + row * kE + 32 * c);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              dst[i] = make_uint4(kw[4 * i], kw[4 * i + 1], kw[4 * i + 2], kw[4 * i + 3]);
          }
          // every element is counted in the window without branching; a bin
          // outside it lands in the dummy row (never flushed) and is counted
          // again below, in global memory, by the rare second loop
          uint32_t mslot = 0;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const uint32_t bin = prmt(kw[i >> 1], 0u, (i & 1) ? 0x4443u : 0x4441u);
            const uint32_t slot = window_slot(bin);
            mslot = slot > mslot ? slot : mslot;
            const uint32_t addr = win_b + 4u * (slot * (uint32_t)kWinRow + 16u * c + (i >> 1));
            if (i & 1)
              red_shared_addc<0x10000u>(addr);
            else
              red_shared_addc<1u>(addr);
          }
          if (mslot == (uint32_t)route::kDummy) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const uint32_t bin = prmt(kw[i >> 1], 0u, (i & 1) ? 0x4443u : 0x4441u);
              if (lut[bin] == (uint32_t)route::kDummy)
                atomicAdd(g.hist + (int64_t)(32 * c + i) * 256 + bin, 1);
            }
          }
        }
      };
      {
        uint32_t ra[32], rb[32];
        tmem_ld32_nowait(ta, ra);
#pragma unroll 1
        for (int c = 0; c < 8; c += 2) {
          tmem_wait_ld(ra);
          tmem_ld32_nowait(ta + 32u * (c + 1), rb);
          chunk_c(c, ra);
          tmem_wait_ld(rb);
          if (c + 2 < 8) tmem_ld32_nowait(ta + 32u * (c + 2), ra);
          chunk_c(c + 1, rb);
        }
      }
      tc_fence_before();
      mbar_arrive(tempty + wg);
    }
  }

  // ---- flush the window, free TMEM
  tc_fence_before();
  __syncthreads();
  for (int i = threadIdx.x; i < route::kWin * (kE / 2); i += blockDim.x) {
    const int slot = i / (kE / 2), p = i % (kE / 2);
    const uint32_t w = win[slot * kWinRow + p];
    const uint32_t bin = route::slot_bin(slot);
    if (w & 0xFFFFu) atomicAdd(g.hist + (int64_t)(2 * p) * 256 + bin, (int)(w & 0xFFFFu));
    if (w >> 16) atomicAdd(g.hist + (int64_t)(2 * p + 1) * 256 + bin, (int)(w >> 16));
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 2 * kE);
  }
  if (g.chained) asm volatile("griddepcontrol.wait;" ::: "memory");
}

int64_t grid_of(int64_t M) {
  const int64_t n_tiles = (M + kBM - 1) / kBM;
  const int64_t sms = sm_count();
  return n_tiles < sms ? n_tiles : sms;
}

template <int KL, int K1>
int launch_fused(const CUtensorMap& ma, const CUtensorMap& mb, const FusedArgs& g,
                 cudaStream_t stream) {
  auto kern = gemm_route_kernel<KL, K1>;
  static bool attr_set = false;  // per instantiation; benign race (idempotent)
  if (!attr_set) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
        cudaSuccess)
      return launch_status();
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid_of(g.M));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, ma, mb, g) != cudaSuccess) {
    (void)cudaGetLastError();
    return QB_ECUDA;
  }
  return launch_status();
}

}  // namespace

int launch_router_gemm_route(const void* hidden, const void* w_t, int64_t M, int K, int k,
                             const float* bias, int32_t* hist, uint16_t* keys_out,
                             int32_t* topk_out, float* alpha_out, float* logits_out,
                             cudaStream_t stream, bool chained) {
  if (K % kBK != 0 || K <= 0) return QB_EUNSUPPORTED;
  int* status = device_status_ptr();
  if (!status) return QB_ECUDA;
  // The window's 16-bit counters hold at most 2^16 - 1 tokens per CTA: one
  // launch covers at most 511 tiles per CTA; larger calls take several.
  const int64_t chunk = (int64_t)sm_count() * 511 * kBM;
  for (int64_t off = 0; off < M; off += chunk) {
    const int64_t m = M - off < chunk ? M - off : chunk;
    CUtensorMap ma, mb;
    if (!make_bf16_kmajor_map(&ma, static_cast<const __nv_bfloat16*>(hidden) + off * K,
                              (uint64_t)m, (uint64_t)K, kBM))
      return QB_EINVAL;
    if (!make_bf16_kmajor_map(&mb, w_t, (uint64_t)kE, (uint64_t)K, kE)) return QB_EINVAL;
    // every launch after the first of a call continues the same batch
    FusedArgs g{bias, m, K, k, hist,
                keys_out ? keys_out + off * kE : nullptr, topk_out ? topk_out + off * k : nullptr,
                alpha_out ? alpha_out + off : nullptr, logits_out ? logits_out + off * kE : nullptr,
                status, (chained || off > 0) ? 1 : 0};
    int st;
    if (k + 1 == 7)
      st = launch_fused<8, 7>(ma, mb, g, stream);
    else if (k + 1 == 9)
      st = launch_fused<16, 9>(ma, mb, g, stream);
    else if (k + 1 <= 8)
      st = launch_fused<8, 0>(ma, mb, g, stream);
    else
      st = launch_fused<16, 0>(ma, mb, g, stream);
    if (st != QB_OK) return st;
  }
  return QB_OK;
}

}  // namespace qb
