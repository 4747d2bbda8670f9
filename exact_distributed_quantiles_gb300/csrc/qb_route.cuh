// qb_route.cuh -- the fused router pass (sigmoid, top-(k+1), margins, keys,
// histograms) shared by the EQB hi pass, the recomputing EQB lo pass and the
// K3 pass.  Included by qb_route_hi.cu, qb_route_lo.cu and qb_route_k3.cu,
// each of which instantiates one mode.
//
// "[Dev] Add global-batch quantile balancing", "Quantile estimator":
//   s = sigmoid(logit), alpha[i] = (k+1)-th largest of s[i,:] + b,
//   r[i,j] = alpha[i] - s[i,j];  "Implementation": the fused path adds shared-
//   memory bin classification and histogram atomics to the router pass and
//   keeps no full score tensor.
// "Exact Quantile Balancing and Load-Error Injection for Mixture-of-Experts",
//   EQB paragraph: hi-byte histogram of the BF16 margins, then the lo byte
//   inside the selected bin.
//
// Work decomposition (one CTA per SM, NW warps, each warp independent):
//   a warp owns a tile of 32 consecutive tokens held in shared memory,
//   filled by cp.async.bulk (one mbarrier per warp);
//   phase A  element-wise over the tile: s = sigma(x) written back in place,
//            v = s + b, the max of every group of 8 experts;
//   phase B  one lane per token: the (k+1)-th largest group max is a lower
//            bound tau of alpha; only groups whose max reaches tau can hold
//            any of the k+1 largest v, so alpha is the (k+1)-th largest v of
//            those groups (a register insertion network);
//   phase C  element-wise: r = alpha - s, key of RN_bf16(r), keys out,
//            histogram increments; rows freed here are refilled at once with
//            the warp's next tile.
// EQB hi histograms are privatised per CTA for the 32 hi-byte bins that hold
// margins with 2^-30 <= |r| < 2 (key hi byte 0x40-0x4F and 0xB0-0xBF); other
// bins go straight to the global histogram.  The shared copy is flushed with
// one atomic add per non-zero counter when the CTA finishes.
#pragma once
#include <cuda_bf16.h>

#include "qb_device.cuh"
#include "qb_internal.h"

namespace qb {
namespace route {

constexpr int kTile = 32;  // tokens per warp tile
constexpr int kWin = 32;   // hi-byte bins privatised in shared memory
constexpr int kSmemLimit = 227 * 1024;

struct Args {
  const void* logits;
  const float* bias;
  int64_t N;
  int k;
  int32_t* hist;  // hi: [E,256]  lo: [E,256]  k3: [E,nbins]
  uint16_t* keys_out;
  int32_t* topk_out;
  float* alpha_out;
  const int32_t* sel;    // lo mode
  const float* bounds;   // k3 mode
  int nbins;             // k3 mode
  int* status;
};

template <int E>
struct Geo {
  static constexpr int G = E / 8;                                   // groups of 8 experts
  static constexpr int GP = ((G / 4 + 1) % 2 == 1) ? G + 4 : G + 8;  // padded gmax row (words)
  static constexpr int LPR = E >= 256 ? 32 : E / 8;                 // lanes per row in a step
  static constexpr int NCOPY = E >= 256 ? 1 : 256 / E;              // histogram copies
  static constexpr int CSTRIDE = kWin * E + (NCOPY > 1 ? LPR : 0);  // words per copy
  static constexpr int STEPS = kTile * E / 256;                     // 256-element steps per tile
  static constexpr int BREG = E == 512 ? 16 : 8;                    // per-lane bias registers
  // Position of expert e inside one histogram slot row: for a fixed element
  // index t the 32 lanes of a step land in 32 distinct banks.
  __device__ static __forceinline__ int pi(int e) {
    if (E == 512) return (e >> 8) * 256 + (e & 7) * 32 + ((e & 255) >> 3);
    return (e & 7) * LPR + (e >> 3);
  }
  __device__ static __forceinline__ int pi_inv(int p) {
    if (E == 512) {
      const int h = p >> 8, q = p & 255;
      return h * 256 + (q & 31) * 8 + (q >> 5);
    }
    return (p % LPR) * 8 + p / LPR;
  }
};

__host__ __device__ constexpr int round16(int b) { return (b + 15) & ~15; }

template <int E, typename T, int MODE>
struct Smem {
  using GE = Geo<E>;
  static constexpr int kHist = MODE == kModeHi ? GE::NCOPY * GE::CSTRIDE * 4 : 0;
  static constexpr int kBias = E * 4;
  static constexpr int kFixed = kHist + kBias;
  static constexpr int kTileBytes = kTile * E * 4;  // fp32 scores; bf16 input sits in the upper half
  static constexpr int kGmax = round16(kTile * GE::GP * 4);
  static constexpr int kAlpha = round16(kTile * 4);
  static constexpr int kWarp = kTileBytes + kGmax + kAlpha + 16;  // + mbarrier
  static constexpr int nw_fit() {
    int n = (kSmemLimit - kFixed) / kWarp;
    return n > 16 ? 16 : n;
  }
  static constexpr int NW = nw_fit();
  static constexpr int kTotal = kFixed + NW * kWarp;
};

// Insert v into the descending list L[0..KMAX) (drops the smallest).
template <int KMAX>
__device__ __forceinline__ void insert_desc(float (&L)[KMAX], float v) {
#pragma unroll
  for (int t = 0; t < KMAX; ++t) {
    const float hi = fmaxf(L[t], v);
    v = fminf(L[t], v);
    L[t] = hi;
  }
}

template <int KMAX>
__device__ __forceinline__ float pick(const float (&L)[KMAX], int k) {
  float a = L[0];
#pragma unroll
  for (int t = 1; t < KMAX; ++t) a = (t == k) ? L[t] : a;
  return a;
}

// Slot of a hi-byte bin in the shared window, or 255 when outside it.
__device__ __forceinline__ uint32_t window_slot(uint32_t bin) {
  const uint32_t m = bin ^ ((bin >> 7) * 0xF0u);  // 0xB0..0xBF -> 0x40..0x4F
  return ((m >> 4) == 4u) ? ((m & 15u) | ((bin >> 7) << 4)) : 255u;
}

__device__ __forceinline__ uint32_t slot_bin(int slot) {
  return slot < 16 ? 0x40u + slot : 0xB0u + (slot - 16);
}


// Shared-memory address of the x element f (flat index inside the tile) and
// of the score element f.  fp32: in place.  bf16: x lives in the upper half
// of the fp32 score area; writing score f only overwrites x elements below f.
template <int E, typename T>
__device__ __forceinline__ T* x_ptr(unsigned char* tile, int f) {
  if constexpr (sizeof(T) == 4) {
    return reinterpret_cast<T*>(tile) + f;
  } else {
    return reinterpret_cast<T*>(tile + kTile * E * 2) + f;
  }
}

// Rows of the next tile whose shared bytes are free once the scores of the
// first F flat elements of this tile have been consumed.
template <int E, typename T>
__device__ __forceinline__ int rows_free(int F) {
  if constexpr (sizeof(T) == 4) {
    return F / E;
  } else {
    const int r = (2 * F - kTile * E) / E;
    return r < 0 ? 0 : (r > kTile ? kTile : r);
  }
}

template <int E, typename T>
__device__ __forceinline__ void issue_rows(unsigned char* tile, const T* logits, int64_t tile_start,
                                           int r0, int r1, uint64_t* bar) {
  if (r1 <= r0) return;
  fence_proxy_async_smem();
  bulk_g2s(x_ptr<E, T>(tile, r0 * E), logits + (tile_start + r0) * (int64_t)E,
           (uint32_t)((r1 - r0) * E * sizeof(T)), bar);
}

__device__ __forceinline__ void load8(const float* p, float (&x)[8]) {
  const float4 a = reinterpret_cast<const float4*>(p)[0];
  const float4 b = reinterpret_cast<const float4*>(p)[1];
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
  x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&x)[8]) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ void store8(float* p, const float (&x)[8]) {
  reinterpret_cast<float4*>(p)[0] = make_float4(x[0], x[1], x[2], x[3]);
  reinterpret_cast<float4*>(p)[1] = make_float4(x[4], x[5], x[6], x[7]);
}

template <int E, int KMAX, typename T, int MODE>
__global__ void __launch_bounds__(Smem<E, T, MODE>::NW * 32, 1) route_kernel(const Args a) {
  using GE = Geo<E>;
  using SM = Smem<E, T, MODE>;
  constexpr int NW = SM::NW;
  extern __shared__ __align__(128) unsigned char smem[];
  int32_t* hist_s = reinterpret_cast<int32_t*>(smem);
  float* bias_s = reinterpret_cast<float*>(smem + SM::kHist);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  unsigned char* wbase = smem + SM::kFixed + warp * SM::kWarp;
  unsigned char* tile = wbase;
  float* sc = reinterpret_cast<float*>(tile);
  float* gmax = reinterpret_cast<float*>(wbase + SM::kTileBytes);
  float* alpha_s = reinterpret_cast<float*>(wbase + SM::kTileBytes + SM::kGmax);
  uint64_t* bar = reinterpret_cast<uint64_t*>(wbase + SM::kTileBytes + SM::kGmax + SM::kAlpha);
  const T* logits = static_cast<const T*>(a.logits);
  const int k = a.k;

  // ---- prologue: zero the shared histogram, stage the bias, init barrier
  if constexpr (MODE == kModeHi) {
    for (int i = threadIdx.x; i < GE::NCOPY * GE::CSTRIDE; i += blockDim.x) hist_s[i] = 0;
  }
  for (int i = threadIdx.x; i < E; i += blockDim.x) bias_s[i] = a.bias[i];
  if (lane == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncthreads();

  // Per-lane expert block of the element-wise phases and its constants.
  float breg[GE::BREG];
  int32_t selreg[GE::BREG];
#pragma unroll
  for (int i = 0; i < GE::BREG; ++i) {
    const int e = (E == 512 ? (i >> 3) * 256 + 8 * lane : (8 * lane) % E) + (i & 7);
    breg[i] = bias_s[e];
    selreg[i] = (MODE == kModeLo) ? a.sel[e] : 0;
  }
  float k3_lo = 0.f, k3_scale = 0.f, k3_nb = 0.f;
  if constexpr (MODE == kModeK3) {
    k3_lo = a.bounds[0];
    const float w = __fsub_rn(a.bounds[1], a.bounds[0]);
    k3_nb = (float)a.nbins;
    k3_scale = __fdiv_rn(k3_nb, w);
  }

  const int64_t n_tiles = (a.N + kTile - 1) / kTile;
  const int64_t wstride = (int64_t)gridDim.x * NW;
  int64_t tix = (int64_t)blockIdx.x * NW + warp;
  uint32_t parity = 0;
  bool ok = true;

  if (tix < n_tiles && lane == 0) {
    const int64_t t0 = tix * kTile;
    const int rows = (int)((a.N - t0) < kTile ? (a.N - t0) : kTile);
    mbar_arrive_expect_tx(bar, (uint32_t)(rows * E * sizeof(T)));
    issue_rows<E, T>(tile, logits, t0, 0, rows, bar);
  }

  for (; tix < n_tiles && ok; tix += wstride) {
    const int64_t t0 = tix * kTile;
    const int rows = (int)((a.N - t0) < kTile ? (a.N - t0) : kTile);
    const int64_t nt = tix + wstride;
    const int64_t n0 = nt * kTile;
    const int nrows = nt < n_tiles ? (int)((a.N - n0) < kTile ? (a.N - n0) : kTile) : 0;

    ok = mbar_wait_bounded(bar, parity, a.status);
    parity ^= 1u;
    if (!ok) break;

    // ---- phase A: scores in place, group maxima
#pragma unroll 1
    for (int st = 0; st < GE::STEPS; ++st) {
      const int f = st * 256 + 8 * lane;
      const int row = f / E;
      const int e0 = f % E;
      float x[8];
      if (row < rows) load8(x_ptr<E, T>(tile, f), x);
      if constexpr (sizeof(T) != 4) __syncwarp();
      if (row < rows) {
        float s[8];
        float g = -INFINITY;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          s[i] = sigmoid_pinned(x[i]);
          const float b = (E == 512 && (st & 1)) ? breg[(8 + i) % GE::BREG] : breg[i];
          g = fmaxf(g, __fadd_rn(s[i], b));
        }
        store8(sc + f, s);
        gmax[row * GE::GP + (e0 >> 3)] = g;
      }
    }
    __syncwarp();

    // ---- phase B: one lane per token, alpha and the top-k set
    if (lane < rows) {
      float gm[GE::G];
#pragma unroll
      for (int q = 0; q < GE::G / 4; ++q) {
        const float4 v4 = reinterpret_cast<const float4*>(gmax + lane * GE::GP)[q];
        gm[4 * q] = v4.x; gm[4 * q + 1] = v4.y; gm[4 * q + 2] = v4.z; gm[4 * q + 3] = v4.w;
      }
      float L[KMAX];
#pragma unroll
      for (int t = 0; t < KMAX; ++t) L[t] = -INFINITY;
#pragma unroll
      for (int g = 0; g < GE::G; ++g) insert_desc<KMAX>(L, gm[g]);
      const float tau = pick<KMAX>(L, k);
      uint64_t mask = 0;
#pragma unroll
      for (int g = 0; g < GE::G; ++g) mask |= (gm[g] >= tau ? 1ull : 0ull) << g;
#pragma unroll
      for (int t = 0; t < KMAX; ++t) L[t] = -INFINITY;
      for (uint64_t m = mask; m; m &= m - 1) {
        const int g = __ffsll((long long)m) - 1;
        float s8[8], b8[8];
        load8(sc + lane * E + 8 * g, s8);
        load8(bias_s + 8 * g, b8);
#pragma unroll
        for (int i = 0; i < 8; ++i) insert_desc<KMAX>(L, __fadd_rn(s8[i], b8[i]));
      }
      const float alpha = pick<KMAX>(L, k);
      alpha_s[lane] = alpha;
      const int64_t tok = t0 + lane;
      if (a.alpha_out) a.alpha_out[tok] = alpha;
      if (a.topk_out) {
        int c_gt = 0;
#pragma unroll
        for (int t = 0; t < KMAX; ++t) c_gt += (t < k && L[t] > alpha) ? 1 : 0;
        int ties = k - c_gt;
        int c = 0;
        int32_t* out = a.topk_out + tok * k;
        for (uint64_t m = mask; m; m &= m - 1) {
          const int g = __ffsll((long long)m) - 1;
          float s8[8], b8[8];
          load8(sc + lane * E + 8 * g, s8);
          load8(bias_s + 8 * g, b8);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float v = __fadd_rn(s8[i], b8[i]);
            const bool take = (v > alpha) || (v == alpha && ties > 0);
            if (take) {
              if (!(v > alpha)) --ties;
              out[c++] = 8 * g + i;
            }
          }
        }
      }
    }
    __syncwarp();

    // ---- phase C: margins, keys, histograms; refill freed rows
    if (lane == 0 && nrows > 0) mbar_arrive_expect_tx(bar, (uint32_t)(nrows * E * sizeof(T)));
    int copied = 0;
#pragma unroll 1
    for (int st = 0; st < GE::STEPS; ++st) {
      const int f = st * 256 + 8 * lane;
      const int row = f / E;
      const int e0 = f % E;
      if (row < rows) {
        float s[8];
        load8(sc + f, s);
        const float alpha = alpha_s[row];
        const int64_t tok = t0 + row;
        if constexpr (MODE == kModeK3) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float r = __fsub_rn(alpha, s[i]);
            const float tt = __fmul_rn(__fsub_rn(r, k3_lo), k3_scale);
            int idx;
            if (!(tt >= 0.0f))
              idx = 0;
            else if (tt >= k3_nb)
              idx = a.nbins - 1;
            else
              idx = __float2int_rz(tt);
            atomicAdd(a.hist + (int64_t)(e0 + i) * a.nbins + idx, 1);
          }
        } else {
          uint32_t kw[4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            kw[i] = keys_from_bf16x2(
                bf16x2_rn(__fsub_rn(alpha, s[2 * i]), __fsub_rn(alpha, s[2 * i + 1])));
          if (MODE == kModeHi && a.keys_out)
            *reinterpret_cast<uint4*>(a.keys_out + tok * E + e0) =
                make_uint4(kw[0], kw[1], kw[2], kw[3]);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint32_t key = (kw[i >> 1] >> ((i & 1) * 16)) & 0xFFFFu;
            const uint32_t bin = key >> 8;
            const int e = e0 + i;
            if constexpr (MODE == kModeHi) {
              const uint32_t slot = window_slot(bin);
              if (slot < (uint32_t)kWin) {
                const int copy = (E >= 256) ? 0 : (8 * lane) / E;
                atomicAdd(hist_s + copy * GE::CSTRIDE + slot * E + GE::pi(e), 1);
              } else {
                atomicAdd(a.hist + (int64_t)e * 256 + bin, 1);
              }
            } else {
              const int sl = (E == 512 && (st & 1)) ? selreg[(8 + i) % GE::BREG] : selreg[i];
              if ((int)bin == sl) atomicAdd(a.hist + (int64_t)e * 256 + (key & 0xFFu), 1);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0 && nrows > 0) {
        int nf = rows_free<E, T>((st + 1) * 256);
        nf = nf < nrows ? nf : nrows;
        issue_rows<E, T>(tile, logits, n0, copied, nf, bar);
        if (nf > copied) copied = nf;
      }
    }
  }

  // ---- epilogue: flush the shared hi histogram
  if constexpr (MODE == kModeHi) {
    __syncthreads();
    for (int i = threadIdx.x; i < kWin * E; i += blockDim.x) {
      int c = 0;
#pragma unroll
      for (int cp = 0; cp < GE::NCOPY; ++cp) c += hist_s[cp * GE::CSTRIDE + i];
      if (c) {
        const int slot = i / E;
        const int e = GE::pi_inv(i % E);
        atomicAdd(a.hist + (int64_t)e * 256 + slot_bin(slot), c);
      }
    }
  }
}

template <int E, int KMAX, typename T, int MODE>
int launch_one(const Args& a, cudaStream_t stream) {
  using SM = Smem<E, T, MODE>;
  static_assert(SM::NW >= 1, "tile does not fit shared memory");
  auto kern = route_kernel<E, KMAX, T, MODE>;
  static bool attr_set = false;  // per instantiation; benign race (idempotent)
  if (!attr_set) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SM::kTotal) !=
        cudaSuccess)
      return launch_status();
    attr_set = true;
  }
  const int64_t n_tiles = (a.N + kTile - 1) / kTile;
  int64_t grid = sm_count();
  const int64_t need = (n_tiles + SM::NW - 1) / SM::NW;
  if (need < grid) grid = need;
  if (grid < 1) grid = 1;
  kern<<<(unsigned)grid, SM::NW * 32, SM::kTotal, stream>>>(a);
  return launch_status();
}

template <int MODE, typename T>
int dispatch_E(int E, int kmax, const Args& a, cudaStream_t st) {
#define QB_CASE(EE)                                                      \
  case EE:                                                               \
    return kmax <= 8 ? launch_one<EE, 8, T, MODE>(a, st)                 \
                     : launch_one<EE, 16, T, MODE>(a, st);
  switch (E) {
    QB_CASE(32)
    QB_CASE(64)
    QB_CASE(128)
    QB_CASE(256)
    QB_CASE(512)
    default:
      return QB_EUNSUPPORTED;
  }
#undef QB_CASE
}

template <int MODE>
int launch_mode(const void* logits, int dtype, const float* bias, int64_t N, int E, int k,
                int32_t* hist, uint16_t* keys_out, int32_t* topk_out, float* alpha_out,
                const int32_t* sel, const float* bounds, int nbins, cudaStream_t stream) {
  Args a{logits, bias, N, k, hist, keys_out, topk_out, alpha_out, sel, bounds, nbins,
         device_status_ptr()};
  if (!a.status) return QB_ECUDA;
  if (dtype == QB_F32) return dispatch_E<MODE, float>(E, k + 1, a, stream);
  return dispatch_E<MODE, __nv_bfloat16>(E, k + 1, a, stream);
}

}  // namespace route
}  // namespace qb
