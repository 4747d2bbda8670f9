// qb_route.cuh -- the fused router pass (sigmoid, top-(k+1), margins, keys,
// histograms) shared by the EQB hi pass, the recomputing EQB lo pass and the
// K3 pass (which stops after alpha; qb_k3.cu counts).  Included by
// qb_route_hi.cu, qb_route_lo.cu and qb_route_k3.cu, each of which
// instantiates one mode; E = 256 routes through qb_route256.cuh instead.
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
//   a warp owns a tile of TILE consecutive tokens held in shared memory,
//   filled by cp.async.bulk in groups of rows, one mbarrier per row group, so
//   that phase A waits only for the rows it is about to read;
//   phase A  element-wise over the tile, 8 experts per lane: s = sigma(x)
//            (packed f32x2 arithmetic) written back in place, v = s + b, the
//            max of every group of 8 experts;
//   phase B  32/TILE lanes per token: the (k+1)-th largest group max is a
//            lower bound tau of alpha; only groups whose max reaches tau can
//            hold any of the k+1 largest v, so alpha is the (k+1)-th largest
//            v of those groups (register sorting networks and bitonic merges,
//            the token's lanes merging by shuffles);
//   phase C  element-wise: r = alpha - s, packed BF16 conversion, key map,
//            keys out, histogram increments; rows freed here are refilled at
//            once with the warp's next tile.
// EQB hi histograms are privatised per CTA for the 32 hi-byte bins that hold
// margins with 2^-30 <= |r| < 2 (key hi byte 0x40-0x4F and 0xB0-0xBF); a
// 256-entry table maps a hi byte to its slot, every other byte to a dummy
// slot that is never flushed, and a warp vote sends the rare steps that saw
// such a byte through a second loop of direct global atomics.  The shared
// copy is flushed with one atomic add per non-zero counter per CTA.
#pragma once
#include <cuda_bf16.h>

#include <type_traits>

#include "qb_device.cuh"
#include "qb_internal.h"

namespace qb {
namespace route {

#ifndef QB_ROUTE_MAXW
#define QB_ROUTE_MAXW 20  // warps per CTA (one CTA per SM), if shared memory allows
#endif
constexpr int kWin = 32;      // hi-byte bins privatised in shared memory
constexpr int kDummy = kWin;  // slot of every other bin (never flushed)
constexpr int kSmemLimit = 227 * 1024;

struct Args {
  const void* logits;
  const float* bias;
  int64_t N;
  int k;
  int32_t* hist;  // hi: [E,256]  lo: [E,256]  k3: unused
  uint16_t* keys_out;  // hi: EQB keys [N,E] (optional)
  int32_t* topk_out;
  float* alpha_out;
  const int32_t* sel;   // lo mode
  const float* bounds;  // k3 mode
  int nbins;            // k3 mode
  int* status;
  // Experts per row in memory (logits, bias, keys, sel, top-k indices).  The
  // kernel's tile geometry is for E (a power of two); a call with
  // e_real < E (any multiple of 32) pads each row in shared memory: the
  // padded experts get bias -inf and score 0, so v = -inf keeps them out of
  // the top-(k+1), and nothing of theirs is stored or counted.
  int e_real;
  // E = 256 pass only: the call continues a global batch right after another
  // such call on the same stream (qb_route_hist_hi_next): it skips the wait
  // for the previous kernel at its start and waits at its end instead.
  int chained = 0;
};

template <int E, int TILE>
struct Geo {
  static constexpr int G = E / 8;                                   // groups of 8 experts
  static constexpr int GP = ((G / 4 + 1) % 2 == 1) ? G + 4 : G + 8;  // padded gmax row (words)
  static constexpr int LPR = E >= 256 ? 32 : E / 8;                 // lanes per row in a step
  static constexpr int NCOPY = E >= 256 ? 1 : 256 / E;              // histogram copies
  static constexpr int NSLOT = kWin + 1;                            // + dummy slot
  static constexpr int CSTRIDE = NSLOT * E + (NCOPY > 1 ? LPR : 0);  // words per copy
  static constexpr int STEPS = TILE * E / 256;                      // 256-element steps per tile
  static constexpr int NQ = E >= 512 ? E / 256 : 1;                 // 256-expert quarters of a row
  static constexpr int BREG = 8 * NQ;                               // per-lane bias registers
  // Position of expert e inside one histogram slot row: for a fixed element
  // index the 32 lanes of a step land in 32 distinct banks.
  __host__ __device__ static constexpr int pi(int e) {
    return E >= 512 ? (e >> 8) * 256 + (e & 7) * 32 + ((e & 255) >> 3) : (e & 7) * LPR + (e >> 3);
  }
  __device__ static __forceinline__ int pi_inv(int p) {
    if (E >= 512) {
      const int h = p >> 8, q = p & 255;
      return h * 256 + (q & 31) * 8 + (q >> 5);
    }
    return (p % LPR) * 8 + p / LPR;
  }
};

__host__ __device__ constexpr int round16(int b) { return (b + 15) & ~15; }

// Bit mask over the groups of 8 experts of a token (32 bits up to E = 256).
template <int G>
using GroupMask = typename std::conditional<
    (G <= 32), uint32_t,
    typename std::conditional<(G <= 64), unsigned long long, unsigned __int128>::type>::type;
__device__ __forceinline__ int lowest_bit(uint32_t m) { return __ffs((int)m) - 1; }  // -1 if 0
__device__ __forceinline__ int lowest_bit(unsigned long long m) {
  return __ffsll((long long)m) - 1;
}
__device__ __forceinline__ int lowest_bit(unsigned __int128 m) {
  const unsigned long long lo = (unsigned long long)m, hi = (unsigned long long)(m >> 64);
  return lo ? __ffsll((long long)lo) - 1 : (hi ? 63 + __ffsll((long long)hi) : -1);
}
// OR of the group mask of lane ^ o
__device__ __forceinline__ uint32_t shfl_xor_mask(uint32_t m, int o) {
  return __shfl_xor_sync(0xffffffffu, m, o);
}
__device__ __forceinline__ unsigned long long shfl_xor_mask(unsigned long long m, int o) {
  return __shfl_xor_sync(0xffffffffu, m, o);
}
__device__ __forceinline__ unsigned __int128 shfl_xor_mask(unsigned __int128 m, int o) {
  const unsigned long long lo = __shfl_xor_sync(0xffffffffu, (unsigned long long)m, o);
  const unsigned long long hi = __shfl_xor_sync(0xffffffffu, (unsigned long long)(m >> 64), o);
  return ((unsigned __int128)hi << 64) | lo;
}

template <int E, typename T, int MODE, int TILE>
struct Smem {
  using GE = Geo<E, TILE>;
  static constexpr int kHist = MODE == kModeHi ? round16(GE::NCOPY * GE::CSTRIDE * 4) : 0;
  static constexpr int kStatic = 256 + E * 4 + 1024;  // static lut + bias, and a margin
  static constexpr int kFixed = kHist + kStatic;
  static constexpr int kTileBytes = TILE * E * 4;  // fp32 scores; bf16 input sits in the upper half
  static constexpr int kGmax = round16(TILE * GE::GP * 4);  // group maxima
  static constexpr int kAlpha = round16(TILE * 4);
  static constexpr int GR = (256 / E) > 4 ? 256 / E : 4;  // rows per load group
  static constexpr int NGRP = TILE / GR;                   // mbarriers per warp
  static constexpr int kWarp = kTileBytes + kGmax + kAlpha + round16(NGRP * 8);
  static constexpr int nw_fit() {
    int n = (kSmemLimit - kFixed) / kWarp;
    return n > QB_ROUTE_MAXW ? QB_ROUTE_MAXW : n;
  }
  static constexpr int NW = nw_fit();
  static constexpr int kTotal = kHist + NW * kWarp;  // dynamic shared memory
};

// ---- register selection networks (all descending) ----
__device__ __forceinline__ void cas_desc(float& a, float& b) {
  const float hi = fmaxf(a, b);
  b = fminf(a, b);
  a = hi;
}

// Insert v into the descending list L[0..KL) (drops the smallest).
template <int KL>
__device__ __forceinline__ void insert_desc(float (&L)[KL], float v) {
#pragma unroll
  for (int t = 0; t < KL; ++t) cas_desc(L[t], v);
}

// Sort 8 values descending: a 19-comparator network (checked on all 0/1
// inputs, which by the 0-1 principle covers every input).
__device__ __forceinline__ void sort8_desc(float (&v)[8]) {
  cas_desc(v[0], v[2]); cas_desc(v[1], v[3]); cas_desc(v[4], v[6]); cas_desc(v[5], v[7]);
  cas_desc(v[0], v[4]); cas_desc(v[1], v[5]); cas_desc(v[2], v[6]); cas_desc(v[3], v[7]);
  cas_desc(v[0], v[1]); cas_desc(v[2], v[3]); cas_desc(v[4], v[5]); cas_desc(v[6], v[7]);
  cas_desc(v[2], v[4]); cas_desc(v[3], v[5]);
  cas_desc(v[1], v[4]); cas_desc(v[3], v[6]);
  cas_desc(v[1], v[2]); cas_desc(v[3], v[4]); cas_desc(v[5], v[6]);
}

// L <- the KL largest of L and B, both descending: elementwise max against
// the reversed B is bitonic and holds them; a bitonic merger sorts it.
template <int KL>
__device__ __forceinline__ void merge_desc(float (&L)[KL], const float (&B)[KL]) {
#pragma unroll
  for (int i = 0; i < KL; ++i) L[i] = fmaxf(L[i], B[KL - 1 - i]);
#pragma unroll
  for (int d = KL / 2; d >= 1; d /= 2) {
#pragma unroll
    for (int i = 0; i < KL; ++i)
      if ((i & d) == 0) cas_desc(L[i], L[i + d]);
  }
}

// Merge a block of 8 values into the descending list L (KL >= 8).
template <int KL>
__device__ __forceinline__ void merge_block8(float (&L)[KL], float (&v)[8]) {
  sort8_desc(v);
  float B[KL];
#pragma unroll
  for (int i = 0; i < KL; ++i) B[i] = i < 8 ? v[i] : -INFINITY;
  merge_desc<KL>(L, B);
}

// L <- the block of 8 values sorted descending (L was empty).
template <int KL>
__device__ __forceinline__ void first_block8(float (&L)[KL], float (&v)[8]) {
  sort8_desc(v);
#pragma unroll
  for (int i = 0; i < KL; ++i) L[i] = i < 8 ? v[i] : -INFINITY;
}

// Merge the list of lane ^ o into L.
template <int KL>
__device__ __forceinline__ void merge_partner(float (&L)[KL], int o) {
  float P[KL];
#pragma unroll
  for (int i = 0; i < KL; ++i) P[i] = __shfl_xor_sync(0xffffffffu, L[i], o);
  merge_desc<KL>(L, P);
}

// L[k]: a compile-time index when K1 = k + 1 is known, else a select chain.
template <int KL, int K1>
__device__ __forceinline__ float pick(const float (&L)[KL], int k) {
  if constexpr (K1 > 0) {
    return L[K1 - 1];
  } else {
    float a = L[0];
#pragma unroll
    for (int t = 1; t < KL; ++t) a = (t == k) ? L[t] : a;
    return a;
  }
}

// Shared-window slot of a hi byte (kDummy outside the window).
__host__ __device__ constexpr uint32_t window_slot_of(uint32_t bin) {
  return (((bin ^ ((bin >> 7) * 0xF0u)) >> 4) == 4u)
             ? (((bin ^ ((bin >> 7) * 0xF0u)) & 15u) | ((bin >> 7) << 4))
             : (uint32_t)kDummy;
}

__device__ __forceinline__ uint32_t slot_bin(int slot) {
  return slot < 16 ? 0x40u + slot : 0xB0u + (slot - 16);
}

// Shared-memory address of the x element f (flat index inside the tile).
// fp32: in place.  bf16: x lives in the upper half of the fp32 score area;
// writing score f only overwrites x elements below f.
template <int E, typename T, int TILE>
__device__ __forceinline__ T* x_ptr(unsigned char* tile, int f) {
  if constexpr (sizeof(T) == 4) {
    return reinterpret_cast<T*>(tile) + f;
  } else {
    return reinterpret_cast<T*>(tile + TILE * E * 2) + f;
  }
}

// Rows of the next tile whose shared bytes are free once the scores of the
// first F flat elements of this tile have been consumed.
template <int E, typename T, int TILE>
__device__ __forceinline__ int rows_free(int F) {
  if constexpr (sizeof(T) == 4) {
    return F / E;
  } else {
    const int r = (2 * F - TILE * E) / E;
    return r < 0 ? 0 : (r > TILE ? TILE : r);
  }
}

template <int E, typename T, int TILE>
__device__ __forceinline__ void issue_rows(unsigned char* tile, const T* logits, int64_t tile_start,
                                           int r0, int r1, int er, uint64_t* bar) {
  if (r1 <= r0) return;
  fence_proxy_async_smem();
  if (er == E) {
    bulk_g2s(x_ptr<E, T, TILE>(tile, r0 * E), logits + (tile_start + r0) * (int64_t)E,
             (uint32_t)((r1 - r0) * E * sizeof(T)), bar);
  } else {
    // padded rows: one copy of the er experts of each row
    for (int r = r0; r < r1; ++r)
      bulk_g2s(x_ptr<E, T, TILE>(tile, r * E), logits + (tile_start + r) * (int64_t)er,
               (uint32_t)(er * sizeof(T)), bar);
  }
}

// Issue the load of every row group of the next tile that is complete inside
// [0, nf) and not issued yet (groups below `issued`); one mbarrier per group.
template <int E, typename T, int TILE, int GR>
// Called by every lane with the same arguments (the bookkeeping stays warp-
// uniform); only the leader lane issues the barrier arrival and the copy.
__device__ __forceinline__ void issue_groups(unsigned char* tile, const T* logits, int64_t start,
                                             int nrows, int nf, int& issued, uint64_t* bars,
                                             bool leader, int er) {
  while (issued * GR < nrows) {
    const int r0 = issued * GR;
    const int r1 = (r0 + GR < nrows) ? r0 + GR : nrows;
    if (nf < r1) break;
    if (leader) {
      mbar_arrive_expect_tx(bars + issued, (uint32_t)((r1 - r0) * er * sizeof(T)));
      issue_rows<E, T, TILE>(tile, logits, start, r0, r1, er, bars + issued);
    }
    ++issued;
  }
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

// Eight margins alpha - s -> four packed key pairs.  `fold` maps margins that
// round to bf16 -0 onto the +0 key; they only occur when some score is below
// 2^-100 (a logit below -75), which phase A flags per tile.
template <bool FOLD>
__device__ __forceinline__ void keys8(float alpha, const float (&s)[8], uint32_t (&kw)[4]) {
  const f2_t A = f2_splat(alpha);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float r0, r1;
    f2_unpack(f2_sub(A, f2_pack(s[2 * i], s[2 * i + 1])), r0, r1);
    uint32_t w = bf16x2_rn(r0, r1);
    if constexpr (FOLD) {
      const uint32_t nz = (w & 0x7FFF7FFFu) + 0x7FFF7FFFu;
      w &= (nz | 0x7FFF7FFFu);
    }
    kw[i] = w ^ (prmt(w, 0u, 0xBB99u) | 0x80008000u);
  }
}


// No "memory" clobber: the window is read only after the __syncthreads
// before the flush, and without the clobber the compiler can issue a step's
// table loads ahead of its increments.
__device__ __forceinline__ void red_shared_add1(uint32_t addr) {
  asm volatile("red.shared.add.u32 [%0], 1;" ::"r"(addr));
}

__device__ __forceinline__ uint32_t lut_load(const uint8_t* lut, uint32_t bin) {
  return lut[bin];
}

template <int E, int KL, int K1, typename T, int MODE, int TILE>
__global__ void __launch_bounds__(Smem<E, T, MODE, TILE>::NW * 32, 1) route_kernel(const Args a) {
  static_assert(TILE == 8 || TILE == 16 || TILE == 32, "lanes per token must divide 32");
  using GE = Geo<E, TILE>;
  using SM = Smem<E, T, MODE, TILE>;
  constexpr int NW = SM::NW;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ uint8_t lut[256];
  __shared__ __align__(16) float bias_s[E];
  int32_t* hist_s = reinterpret_cast<int32_t*>(smem);
  // warp index as a value the compiler knows to be warp-uniform, so that the
  // per-tile branches below need no divergence handling
  const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);
  const int lane = threadIdx.x & 31;
  // A kernel launched as this one's programmatic dependent (lei_apply_overlap)
  // may be scheduled into the room left beside this CTA from now on.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  unsigned char* wbase = smem + SM::kHist + warp * SM::kWarp;
  unsigned char* tile = wbase;
  float* sc = reinterpret_cast<float*>(tile);
  float* gmax = reinterpret_cast<float*>(wbase + SM::kTileBytes);
  float* alpha_s = reinterpret_cast<float*>(wbase + SM::kTileBytes + SM::kGmax);
  constexpr int GR = SM::GR;
  uint64_t* bars = reinterpret_cast<uint64_t*>(wbase + SM::kTileBytes + SM::kGmax + SM::kAlpha);
  const T* logits = static_cast<const T*>(a.logits);
  const int k = a.k;
  const int er = a.e_real;  // experts per row in memory (<= E)

  // ---- prologue: zero the shared histogram, slot table, bias, barrier
  if constexpr (MODE == kModeHi) {
    for (int i = threadIdx.x; i < GE::NCOPY * GE::CSTRIDE; i += blockDim.x) hist_s[i] = 0;
    for (int i = threadIdx.x; i < 256; i += blockDim.x) lut[i] = (uint8_t)window_slot_of(i);
  }
  for (int i = threadIdx.x; i < E; i += blockDim.x) bias_s[i] = i < er ? a.bias[i] : -INFINITY;
  if (lane == 0) {
    for (int q = 0; q < SM::NGRP; ++q) mbar_init(bars + q, 1);
    fence_mbar_init();
  }
  __syncthreads();

  // Per-lane expert block of the element-wise phases and its constants.
  const int e0l = (E >= 512) ? 8 * lane : (8 * lane) % E;
  float breg[GE::BREG];
  int32_t selreg[GE::BREG];
#pragma unroll
  for (int i = 0; i < GE::BREG; ++i) {
    const int e = e0l + (i >> 3) * 256 + (i & 7);
    breg[i] = bias_s[e];
    selreg[i] = (MODE == kModeLo && e < er) ? a.sel[e] : -1;
  }
  // shared byte address of this lane's counter for element i, slot 0
  const int copy = (E >= 256) ? 0 : (8 * lane) / E;
  const uint32_t hbase = smem_u32(hist_s) + 4u * (uint32_t)(copy * GE::CSTRIDE + (lane % GE::LPR));

  const int64_t n_tiles = (a.N + TILE - 1) / TILE;
  const int64_t wstride = (int64_t)gridDim.x * NW;
  int64_t tix = (int64_t)blockIdx.x * NW + warp;
  uint32_t parity = 0;
  bool ok = true;

  if (tix < n_tiles && lane == 0) {
    const int64_t t0 = tix * TILE;
    const int rows = (int)((a.N - t0) < TILE ? (a.N - t0) : TILE);
    int issued = 0;
    issue_groups<E, T, TILE, GR>(tile, logits, t0, rows, rows, issued, bars, true, er);
  }

  for (; tix < n_tiles && ok; tix += wstride) {
    const int64_t t0 = tix * TILE;
    const int rows = (int)((a.N - t0) < TILE ? (a.N - t0) : TILE);
    const int64_t nt = tix + wstride;
    const int64_t n0 = nt * TILE;
    const int nrows = nt < n_tiles ? (int)((a.N - n0) < TILE ? (a.N - n0) : TILE) : 0;


    // ---- phase A: scores in place, group maxima.  Two 8-element chunks per
    // lane per iteration (all loads first, one fast/slow decision for both,
    // then straight-line packed arithmetic) for instruction-level parallelism.
    bool ext = false;
    constexpr int NS = (GE::STEPS % 2 == 0) ? 2 : 1;
#pragma unroll 1
    for (int st0 = 0; st0 < GE::STEPS; st0 += NS) {
      float x[NS][8];
      bool act[NS];
#pragma unroll
      for (int u = 0; u < NS; ++u) {
        const int st = st0 + u;
        act[u] = (st * 256 + 8 * lane) / E < rows;
        if ((st * 256) % (GR * E) == 0) {
          const int q = (st * 256) / (GR * E);
          if (q * GR < rows && !mbar_wait_bounded(bars + q, parity, a.status)) ok = false;
        }
      }
#pragma unroll
      for (int u = 0; u < NS; ++u)
        if (act[u] && ok) load8(x_ptr<E, T, TILE>(tile, (st0 + u) * 256 + 8 * lane), x[u]);
      if constexpr (sizeof(T) != 4) __syncwarp();
      float m = 0.0f;
#pragma unroll
      for (int u = 0; u < NS; ++u)
        if (act[u]) m = fmaxf(m, max_abs8(x[u]));
      ext |= m > kFoldAbsX;
      float s[NS][8];
      // one decision per warp: the packed path unless some lane holds a large x
      if (__all_sync(0xffffffffu, m <= kFastAbsX)) {
#pragma unroll
        for (int u = 0; u < NS; ++u)
#pragma unroll
          for (int i = 0; i < 4; ++i)
            f2_unpack(sigmoid2_fast(f2_pack(x[u][2 * i], x[u][2 * i + 1])), s[u][2 * i],
                      s[u][2 * i + 1]);
      } else {
#pragma unroll
        for (int u = 0; u < NS; ++u)
#pragma unroll
          for (int i = 0; i < 8; ++i) s[u][i] = sigmoid_pinned(x[u][i]);
      }
#pragma unroll
      for (int u = 0; u < NS; ++u) {
        if (!act[u]) continue;
        const int st = st0 + u;
        const int f = st * 256 + 8 * lane;
        if (er < E && (f % E) >= er) {
          // a padded expert: score 0 (its logit slot holds stale bytes), v = -inf
#pragma unroll
          for (int i = 0; i < 8; ++i) s[u][i] = 0.0f;
        }
        const int qtr = st % GE::NQ;  // which 256-expert quarter of the row
        float v[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float b0 = breg[2 * i], b1 = breg[2 * i + 1];
#pragma unroll
          for (int qq = 1; qq < GE::NQ; ++qq) {
            b0 = qtr == qq ? breg[8 * qq + 2 * i] : b0;
            b1 = qtr == qq ? breg[8 * qq + 2 * i + 1] : b1;
          }
          const f2_t B = f2_pack(b0, b1);
          f2_unpack(f2_add(f2_pack(s[u][2 * i], s[u][2 * i + 1]), B), v[2 * i], v[2 * i + 1]);
        }
        const float g = fmaxf(fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3])),
                              fmaxf(fmaxf(v[4], v[5]), fmaxf(v[6], v[7])));
        store8(sc + f, s[u]);
        gmax[(f / E) * GE::GP + ((f % E) >> 3)] = g;
      }
    }
    parity ^= 1u;
    if (!__all_sync(0xffffffffu, ok)) break;
    const bool tile_ext = __any_sync(0xffffffffu, ext);

    // ---- phase B: LPT = 32 / TILE lanes per token (lane % TILE = token,
    // lane / TILE = part).  tau: each lane takes the top KL of its part of the
    // group maxima, the lanes of a token merge theirs by shuffles.  alpha: the
    // candidate groups (max >= tau) are dealt out by rank modulo LPT; each
    // lane merges its groups' sorted values, then the token's lanes merge.
    {
      constexpr int LPT = 32 / TILE;
      constexpr int GH = GE::G / LPT;
      const int t = lane & (TILE - 1);
      const int h = lane / TILE;
      const bool actB = t < rows;
      float gm[GH];
      if constexpr (GH % 4 == 0) {
#pragma unroll
        for (int q = 0; q < GH / 4; ++q) {
          const float4 v4 = actB ? reinterpret_cast<const float4*>(gmax + t * GE::GP + h * GH)[q]
                                 : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
          gm[4 * q] = v4.x; gm[4 * q + 1] = v4.y; gm[4 * q + 2] = v4.z; gm[4 * q + 3] = v4.w;
        }
      } else {
#pragma unroll
        for (int g = 0; g < GH; ++g) gm[g] = actB ? gmax[t * GE::GP + h * GH + g] : -INFINITY;
      }
      float L[KL];
#pragma unroll
      for (int i = 0; i < KL; ++i) L[i] = -INFINITY;
      if constexpr (GH % 8 == 0) {
        // the first block sorted is the list (merging it into -inf would
        // only copy it); later blocks merge
#pragma unroll
        for (int b0 = 0; b0 < GH; b0 += 8) {
          float v8[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) v8[i] = gm[b0 + i];
          if (b0 == 0)
            first_block8<KL>(L, v8);
          else
            merge_block8<KL>(L, v8);
        }
      } else {
#pragma unroll
        for (int g = 0; g < GH; ++g) insert_desc<KL>(L, gm[g]);
      }
#pragma unroll
      for (int o = TILE; o < 32; o <<= 1) merge_partner<KL>(L, o);
      const float tau = pick<KL, K1>(L, k);
      using MaskT = GroupMask<GE::G>;
      MaskT cand = 0;
#pragma unroll
      for (int g = 0; g < GH; ++g) cand |= (MaskT)(gm[g] >= tau ? 1u : 0u) << (h * GH + g);
      cand = actB ? cand : (MaskT)0;
#pragma unroll
      for (int o = TILE; o < 32; o <<= 1) cand |= shfl_xor_mask(cand, o);
#pragma unroll
      for (int i = 0; i < KL; ++i) L[i] = -INFINITY;
      const float* srow = sc + t * E;
      bool fresh = true;  // L still empty: the first group is sorted into it directly
      for (MaskT m = cand; m;) {
        int g = -1;
#pragma unroll
        for (int p = 0; p < LPT; ++p) {
          const int gp = lowest_bit(m);
          m &= m - 1;
          g = (p == h) ? gp : g;
        }
        if (g >= 0) {
          float s8[8], b8[8];
          load8(srow + 8 * g, s8);
          load8(bias_s + 8 * g, b8);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            f2_unpack(f2_add(f2_pack(s8[2 * i], s8[2 * i + 1]), f2_pack(b8[2 * i], b8[2 * i + 1])),
                      s8[2 * i], s8[2 * i + 1]);
          if (fresh)
            first_block8<KL>(L, s8);
          else
            merge_block8<KL>(L, s8);
          fresh = false;
        }
      }
#pragma unroll
      for (int o = TILE; o < 32; o <<= 1) merge_partner<KL>(L, o);
      const float alpha = pick<KL, K1>(L, k);
      const int64_t tok = t0 + t;
      if (actB && h == 0) {
        alpha_s[t] = alpha;
        if (a.alpha_out) a.alpha_out[tok] = alpha;
      }
      if (a.topk_out) {
        // experts with v > alpha, then ties at alpha by ascending index
        int c_gt = 0;
#pragma unroll
        for (int i = 0; i < KL; ++i) c_gt += (i < k && L[i] > alpha) ? 1 : 0;
        const int ties = k - c_gt;
        int32_t* out = a.topk_out + tok * k;
        if (__any_sync(0xffffffffu, actB && ties > 0)) {
          // rare: a tie at alpha; one lane per token scans in index order
          if (actB && h == 0) {
            int tl = ties, c = 0;
            for (MaskT m = cand; m; m &= m - 1) {
              const int g = lowest_bit(m);
              float s8[8], b8[8];
              load8(srow + 8 * g, s8);
              load8(bias_s + 8 * g, b8);
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const float v = __fadd_rn(s8[i], b8[i]);
                if (v > alpha || (v == alpha && tl > 0)) {
                  if (!(v > alpha)) --tl;
                  out[c++] = 8 * g + i;
                }
              }
            }
          }
        } else if constexpr (GH <= 8) {
          // The k experts above alpha in ascending order.  Lane h owns the
          // token's groups [h*GH, (h+1)*GH): it tests the elements of each
          // of its groups whose max exceeds alpha into a bit mask, the
          // token's lanes scan their counts (lane h's experts all precede
          // lane h+1's), and each lane writes its own indices in order.
          uint32_t own = 0;
#pragma unroll
          for (int g = 0; g < GH; ++g) own |= (gm[g] > alpha ? 1u : 0u) << g;
          own = actB ? own : 0u;
          unsigned long long bits = 0;
          for (uint32_t m = own; m; m &= m - 1) {
            const int gl = __ffs((int)m) - 1;
            float s8[8], b8[8];
            load8(srow + 8 * (h * GH + gl), s8);
            load8(bias_s + 8 * (h * GH + gl), b8);
            uint32_t m8 = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              float v0, v1;
              f2_unpack(f2_add(f2_pack(s8[2 * i], s8[2 * i + 1]), f2_pack(b8[2 * i], b8[2 * i + 1])),
                        v0, v1);
              m8 |= (v0 > alpha ? 1u : 0u) << (2 * i);
              m8 |= (v1 > alpha ? 2u : 0u) << (2 * i);
            }
            bits |= (unsigned long long)m8 << (8 * gl);
          }
          const int cnt = __popcll(bits);
          int incl = cnt;
#pragma unroll
          for (int o = TILE; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
          }
          int pos = incl - cnt;
          const int ebase = h * GH * 8;
          for (unsigned long long m = bits; m; m &= m - 1) {
            if (pos < k) out[pos] = ebase + (__ffsll((long long)m) - 1);
            ++pos;
          }
        } else {
          // The k experts above alpha in ascending order.  Only groups whose
          // max exceeds alpha hold any; the token's lanes take each of them
          // in turn, lane h testing EPL consecutive elements, and EPL warp
          // ballots tell every lane how many of the group's elements below
          // its own are set, so each index goes straight to its slot.
          constexpr int EPL = 8 / LPT;
          constexpr uint32_t PAT = TILE == 8 ? 0x01010101u : (TILE == 16 ? 0x00010001u : 1u);
          MaskT gsel = 0;
#pragma unroll
          for (int g = 0; g < GH; ++g) gsel |= (MaskT)(gm[g] > alpha ? 1u : 0u) << (h * GH + g);
          gsel = actB ? gsel : (MaskT)0;
#pragma unroll
          for (int o = TILE; o < 32; o <<= 1) gsel |= shfl_xor_mask(gsel, o);
          const uint32_t below = (1u << (TILE * h)) - 1u;  // bits of the token's lower lanes
          const float* sp = srow + EPL * h;
          const float* bp = bias_s + EPL * h;
          int base = 0;
          while (__any_sync(0xffffffffu, gsel != 0)) {
            const bool has = gsel != 0;
            const int g = has ? lowest_bit(gsel) : 0;
            gsel &= gsel - 1;
            float sv[EPL];
            if constexpr (EPL == 2) {
              const float2 s2 = *reinterpret_cast<const float2*>(sp + 8 * g);
              const float2 b2 = *reinterpret_cast<const float2*>(bp + 8 * g);
              f2_unpack(f2_add(f2_pack(s2.x, s2.y), f2_pack(b2.x, b2.y)), sv[0], sv[1]);
            } else {
#pragma unroll
              for (int i = 0; i < EPL; ++i) sv[i] = __fadd_rn(sp[8 * g + i], bp[8 * g + i]);
            }
            int pre = 0, tot = 0;
            bool pr[EPL];
#pragma unroll
            for (int i = 0; i < EPL; ++i) {
              pr[i] = has && sv[i] > alpha;
              const uint32_t x = (__ballot_sync(0xffffffffu, pr[i]) >> t) & PAT;
              pre += __popc(x & below);
              tot += __popc(x);
            }
#pragma unroll
            for (int i = 0; i < EPL; ++i) {
              if (pr[i]) {
                if (base + pre < k) out[base + pre] = 8 * g + EPL * h + i;
                ++pre;
              }
            }
            base += tot;
          }
        }
      }
    }
    __syncwarp();

    // ---- phase C: margins, keys, histograms; refill freed rows
    int issued = 0;
#pragma unroll 1
    for (int st = 0; st < GE::STEPS; ++st) {
      const int f = st * 256 + 8 * lane;
      const int row = f / E;
      const int e0 = f % E;
      const bool act = row < rows;
      const int64_t tok = t0 + row;
      const bool real = e0 < er;  // not a padded expert
      if constexpr (MODE == kModeK3) {
        // alpha only (phase B wrote it): the K3 counts are taken by the
        // counting kernel from the logits and alpha
        (void)tok;
        (void)e0;
        (void)act;
        (void)real;
      } else {
        uint32_t kw[4] = {0u, 0u, 0u, 0u};
        bool out_of_window = false;
        if (act && real) {
          float s[8];
          load8(sc + f, s);
          if (tile_ext)
            keys8<true>(alpha_s[row], s, kw);
          else
            keys8<false>(alpha_s[row], s, kw);
          if (MODE == kModeHi && a.keys_out)
            *reinterpret_cast<uint4*>(a.keys_out + tok * er + e0) =
                make_uint4(kw[0], kw[1], kw[2], kw[3]);
          if constexpr (MODE == kModeHi) {
            const uint32_t hoff = 1024u * (uint32_t)(st % GE::NQ);  // +256 experts per quarter
            uint32_t mslot = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const uint32_t bin = prmt(kw[i >> 1], 0u, (i & 1) ? 0x4443u : 0x4441u);
              const uint32_t slot = lut_load(lut, bin);
              mslot = slot > mslot ? slot : mslot;
              red_shared_add1(hbase + hoff + 4u * (uint32_t)(i * GE::LPR) + slot * (4u * E));
            }
            out_of_window = mslot == (uint32_t)kDummy;
          } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const uint32_t key = (kw[i >> 1] >> ((i & 1) * 16)) & 0xFFFFu;
              int sl = selreg[i];
#pragma unroll
              for (int qq = 1; qq < GE::NQ; ++qq) sl = (st % GE::NQ) == qq ? selreg[8 * qq + i] : sl;
              if ((int)(key >> 8) == sl)
                atomicAdd(a.hist + (int64_t)(e0 + i) * 256 + (key & 0xFFu), 1);
            }
          }
        }
        if constexpr (MODE == kModeHi) {
          // rare: hi bytes outside the shared window go to the global histogram
          if (__any_sync(0xffffffffu, out_of_window) && out_of_window) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const uint32_t bin = prmt(kw[i >> 1], 0u, (i & 1) ? 0x4443u : 0x4441u);
              if (lut_load(lut, bin) == (uint32_t)kDummy)
                atomicAdd(a.hist + (int64_t)(e0 + i) * 256 + bin, 1);
            }
          }
        }
      }
      __syncwarp();
      if (nrows > 0)
        issue_groups<E, T, TILE, GR>(tile, logits, n0, nrows, rows_free<E, T, TILE>((st + 1) * 256),
                                     issued, bars, lane == 0, er);
    }
  }

  // ---- epilogue: flush the shared hi histogram (window slots only)
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

template <int E, int KL, int K1, typename T, int MODE, int TILE>
int launch_one(const Args& a, cudaStream_t stream) {
  using SM = Smem<E, T, MODE, TILE>;
  static_assert(SM::NW >= 1, "tile does not fit shared memory");
  auto kern = route_kernel<E, KL, K1, T, MODE, TILE>;
  static bool attr_set = false;  // per instantiation; benign race (idempotent)
  if (!attr_set) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SM::kTotal) !=
        cudaSuccess)
      return launch_status();
    attr_set = true;
  }
  const int64_t n_tiles = (a.N + TILE - 1) / TILE;
  int64_t grid = sm_count();
  const int64_t need = (n_tiles + SM::NW - 1) / SM::NW;
  if (need < grid) grid = need;
  if (grid < 1) grid = 1;
  kern<<<(unsigned)grid, SM::NW * 32, SM::kTotal, stream>>>(a);
  return launch_status();
}

template <int MODE, typename T, int TILE>
int dispatch_E(int E, int k, const Args& a, cudaStream_t st) {
#define QB_CASE(EE)                                                       \
  case EE:                                                                \
    if (k + 1 == 7) return launch_one<EE, 8, 7, T, MODE, TILE>(a, st);   \
    if (k + 1 == 9) return launch_one<EE, 16, 9, T, MODE, TILE>(a, st);  \
    if (k + 1 <= 8) return launch_one<EE, 8, 0, T, MODE, TILE>(a, st);   \
    return launch_one<EE, 16, 0, T, MODE, TILE>(a, st);
  switch (E) {
    QB_CASE(32)
    QB_CASE(64)
    QB_CASE(128)
    QB_CASE(256)
    QB_CASE(512)
    QB_CASE(1024)
    default:
      return QB_EUNSUPPORTED;
  }
#undef QB_CASE
}

#ifndef QB_ROUTE_TILE
#define QB_ROUTE_TILE 8
#endif

template <int MODE>
int launch_mode(const void* logits, int dtype, const float* bias, int64_t N, int E, int k,
                int32_t* hist, uint16_t* keys_out, int32_t* topk_out, float* alpha_out,
                const int32_t* sel, const float* bounds, int nbins, cudaStream_t stream) {
  Args a{logits, bias, N, k, hist, keys_out, topk_out, alpha_out, sel, bounds, nbins,
         device_status_ptr(), E};
  if (!a.status) return QB_ECUDA;
  // the tile geometry of the next power of two (a row of E = 96 sits in a
  // 128-expert slot)
  int ep = 32;
  while (ep < E) ep <<= 1;
  if (dtype == QB_F32) return dispatch_E<MODE, float, QB_ROUTE_TILE>(ep, k, a, stream);
  return dispatch_E<MODE, __nv_bfloat16, QB_ROUTE_TILE>(ep, k, a, stream);
}

}  // namespace route
}  // namespace qb
