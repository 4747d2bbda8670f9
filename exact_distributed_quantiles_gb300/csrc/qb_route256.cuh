// qb_route256.cuh -- the fused router pass specialised to E = 256 experts
// (the pages' testbed width): sigmoid, top-(k+1), margins, BF16 keys and the
// EQB hi-byte histogram in one streaming pass.
//
// "[Dev] Add global-batch quantile balancing", "Quantile estimator":
//   s = sigmoid(logit), alpha[i] = (k+1)-th largest of s[i,:] + b,
//   r[i,j] = alpha[i] - s[i,j]; "Implementation": shared-memory bin
//   classification and histogram atomics inside the router pass.
// "Exact Quantile Balancing and Load-Error Injection for Mixture-of-Experts",
//   EQB paragraph: 256-bin histogram of the high byte of the BF16 margins.
//
// Same results as the generic routing kernel (qb_route.cuh), bit for bit; the
// layout is chosen for sm_103a's shared memory and issue rate:
//   * a warp owns a tile of 8 tokens; each token row sits in its own 1040-byte
//     slot (1024 bytes of fp32 scores + 16 bytes of padding), filled by one
//     cp.async.bulk per row and one mbarrier per pair of rows;
//   * lane L's 8 experts are {4L..4L+3} and {128+4L..128+4L+3}: its two
//     16-byte loads of a row are conflict-free across the warp, and this set
//     is "group L" of the top-(k+1) search (any partition into groups of 8
//     works; this one needs no transposition);
//   * the padding staggers rows over the banks, so the four lanes of each of
//     the 8 tokens in the top-(k+1) phase read their groups with few conflicts;
//   * scores are kept negated (sn = -s): the logistic's last Newton step then
//     needs no separate negation, and v = b - sn, r = alpha + sn are the same
//     IEEE operations as s + b and alpha - s;
//   * per-tile bookkeeping is static (which rows to wait for and refill), and
//     only the last, ragged tile of a launch runs the masked variant.
#pragma once
#include <cuda_bf16.h>

#include "qb_device.cuh"
#include "qb_internal.h"
#include "qb_route.cuh"

namespace qb {
namespace r256 {

using route::Args;

constexpr int kE = 256;
constexpr int kTile = 8;         // tokens per warp tile
constexpr int kPitch = 1040;     // bytes per row slot in shared memory
constexpr int kGP = 36;          // words per group-maximum row (36 = 4 mod 32)
constexpr int kPairs = kTile / 2;  // row pairs per tile, one mbarrier each
constexpr int kWin = route::kWin;
constexpr int kDummy = route::kDummy;
constexpr int kHistBytes = (kWin + 1) * kE * 4;  // [slot][i * 32 + lane] int32
constexpr int kStg = 36;  // words per staged window row at the flush (144 bytes)

// Modes of the pass: the EQB hi pass (phases A-C), or alpha only (phases A
// and B: alpha per token, the input of the K3 counting kernel).
enum Mode256 { kHi256 = 0, kAlpha256 = 1 };
constexpr int kWarpBytes = kTile * kPitch + kTile * kGP * 4 + 32 + 8 * kPairs;
constexpr int kStaticBytes = kE * 4 + 1024;  // bias, and a margin
__host__ __device__ constexpr int hist_bytes(int mode) { return mode == kHi256 ? kHistBytes : 0; }
__host__ __device__ constexpr int warps_max(int mode) {
  return (227 * 1024 - hist_bytes(mode) - kStaticBytes) / kWarpBytes > 20
             ? 20
             : (227 * 1024 - hist_bytes(mode) - kStaticBytes) / kWarpBytes;
}
constexpr int kNW = warps_max(kHi256);
static_assert(kNW >= 16, "route256 tile does not fit shared memory");

template <typename T>
struct In;
template <>
struct In<float> {
  static constexpr int kRowBytes = 1024, kOff = 0;
};
template <>
struct In<__nv_bfloat16> {
  // bf16 rows sit in the upper half of the slot; a lane's fp32 score stores
  // of a row only overwrite logits of that row, which the step read first
  static constexpr int kRowBytes = 512, kOff = 528;
};

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// max |x| of 16 values.
__device__ __forceinline__ float max_abs16(const float (&x)[16]) {
  const float m1 = fmax3(fabsf(x[0]), fabsf(x[1]), fabsf(x[2]));
  const float m2 = fmax3(fabsf(x[3]), fabsf(x[4]), fabsf(x[5]));
  const float m3 = fmax3(fabsf(x[6]), fabsf(x[7]), fabsf(x[8]));
  const float m4 = fmax3(fabsf(x[9]), fabsf(x[10]), fabsf(x[11]));
  const float m5 = fmax3(fabsf(x[12]), fabsf(x[13]), fabsf(x[14]));
  return fmaxf(fmax3(m1, m2, fabsf(x[15])), fmax3(m3, m4, m5));
}

__device__ __forceinline__ float max8(const float* v) {
  return fmaxf(fmax3(v[0], v[1], v[2]), fmax3(v[3], v[4], fmax3(v[5], v[6], v[7])));
}

// Row r of the tile -> lane's 8 logits as fp32 (experts 4L..4L+3, 128+4L..).
__device__ __forceinline__ void load_x(const unsigned char* row, int lane, const float*,
                                       float* x) {
  const float4 a = *reinterpret_cast<const float4*>(row + 16 * lane);
  const float4 b = *reinterpret_cast<const float4*>(row + 512 + 16 * lane);
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
  x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}
__device__ __forceinline__ void load_x(const unsigned char* row, int lane, const __nv_bfloat16*,
                                       float* x) {
  const uint2 a = *reinterpret_cast<const uint2*>(row + 528 + 8 * lane);
  const uint2 b = *reinterpret_cast<const uint2*>(row + 528 + 256 + 8 * lane);
  x[0] = __uint_as_float(a.x << 16); x[1] = __uint_as_float(a.x & 0xFFFF0000u);
  x[2] = __uint_as_float(a.y << 16); x[3] = __uint_as_float(a.y & 0xFFFF0000u);
  x[4] = __uint_as_float(b.x << 16); x[5] = __uint_as_float(b.x & 0xFFFF0000u);
  x[6] = __uint_as_float(b.y << 16); x[7] = __uint_as_float(b.y & 0xFFFF0000u);
}

// Group g of a row (8 negated scores) -> v = b - sn in element order.
__device__ __forceinline__ void group_v(const unsigned char* row, const float* bias_s, int g,
                                        float (&v)[8]) {
  const float4 s0 = *reinterpret_cast<const float4*>(row + 16 * g);
  const float4 s1 = *reinterpret_cast<const float4*>(row + 512 + 16 * g);
  const float4 b0 = *reinterpret_cast<const float4*>(bias_s + 4 * g);
  const float4 b1 = *reinterpret_cast<const float4*>(bias_s + 128 + 4 * g);
  f2_unpack(f2_sub(f2_pack(b0.x, b0.y), f2_pack(s0.x, s0.y)), v[0], v[1]);
  f2_unpack(f2_sub(f2_pack(b0.z, b0.w), f2_pack(s0.z, s0.w)), v[2], v[3]);
  f2_unpack(f2_sub(f2_pack(b1.x, b1.y), f2_pack(s1.x, s1.y)), v[4], v[5]);
  f2_unpack(f2_sub(f2_pack(b1.z, b1.w), f2_pack(s1.z, s1.w)), v[6], v[7]);
}

// Half `half` of group g of a row (4 negated scores) -> v = b - sn.
__device__ __forceinline__ void half_v(const unsigned char* row, const float* bias_s, int g,
                                       int half, float (&v)[4]) {
  const float4 s0 = *reinterpret_cast<const float4*>(row + 512 * half + 16 * g);
  const float4 b0 = *reinterpret_cast<const float4*>(bias_s + 128 * half + 4 * g);
  f2_unpack(f2_sub(f2_pack(b0.x, b0.y), f2_pack(s0.x, s0.y)), v[0], v[1]);
  f2_unpack(f2_sub(f2_pack(b0.z, b0.w), f2_pack(s0.z, s0.w)), v[2], v[3]);
}

// Merge 4 values into the descending list L (KL >= 8): sort them (5
// comparators), then L[i] = max(L[i], B[KL-1-i]) against the 4 sorted values
// padded with -inf (only the last 4 positions change) and a bitonic merger.
template <int KL>
__device__ __forceinline__ void merge_block4(float (&L)[KL], float (&v)[4]) {
  route::cas_desc(v[0], v[1]); route::cas_desc(v[2], v[3]);
  route::cas_desc(v[0], v[2]); route::cas_desc(v[1], v[3]);
  route::cas_desc(v[1], v[2]);
#pragma unroll
  for (int j = 0; j < 4; ++j) L[KL - 4 + j] = fmaxf(L[KL - 4 + j], v[3 - j]);
#pragma unroll
  for (int d = KL / 2; d >= 1; d /= 2) {
#pragma unroll
    for (int i = 0; i < KL; ++i)
      if ((i & d) == 0) route::cas_desc(L[i], L[i + d]);
  }
}

// The M-th largest (1-based) of the union of this lane's descending list L
// and the list of lane ^ o, without merging them: for two descending lists A
// and B it is max over i in [0, M] of min(A[i-1], B[M-1-i]), out-of-range
// entries being +inf.  Only the partner's first M entries travel.
template <int KL, int M>
__device__ __forceinline__ float select_with_partner(const float (&L)[KL], const float (&P)[KL]) {
  static_assert(M >= 1 && M <= KL, "rank out of range");
  float best = fmaxf(P[M - 1], L[M - 1]);  // i = 0 and i = M
#pragma unroll
  for (int i = 1; i < M; ++i) best = fmaxf(best, fminf(L[i - 1], P[M - 1 - i]));
  return best;
}

// Lists of KL = 16 entries whose last 8 are -inf (a block of 8 sorted into
// an empty list): the general merges would take element-wise maxima against
// -inf; these give the same lists with half the shuffles and no maxima.
// Lane ^ o's 8 values, reversed after this lane's 8, form a bitonic sequence
// that the bitonic merger sorts.
__device__ __forceinline__ void bitonic_clean16(float (&L)[16]) {
#pragma unroll
  for (int d = 8; d >= 1; d /= 2) {
#pragma unroll
    for (int i = 0; i < 16; ++i)
      if ((i & d) == 0) route::cas_desc(L[i], L[i + d]);
  }
}
__device__ __forceinline__ void merge_partner_8of16(float (&L)[16], int o) {
  float P[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) P[i] = __shfl_xor_sync(0xffffffffu, L[i], o);
#pragma unroll
  for (int j = 0; j < 8; ++j) L[8 + j] = P[7 - j];
  bitonic_clean16(L);
}
// a block of 8 values into such a list
__device__ __forceinline__ void append_block8_16(float (&L)[16], float (&v)[8]) {
  route::sort8_desc(v);
#pragma unroll
  for (int j = 0; j < 8; ++j) L[8 + j] = v[7 - j];
  bitonic_clean16(L);
}
template <int KL>
__device__ __forceinline__ void merge_partner_first(float (&L)[KL], int o) {
  if constexpr (KL == 16)
    merge_partner_8of16(L, o);
  else
    route::merge_partner<KL>(L, o);
}

template <int KL, int M>
__device__ __forceinline__ void partner_head(const float (&L)[KL], float (&P)[KL], int o) {
#pragma unroll
  for (int i = 0; i < KL; ++i) P[i] = i < M ? __shfl_xor_sync(0xffffffffu, L[i], o) : -INFINITY;
}

// Expert of element i (0..7) of lane L.
__device__ __forceinline__ int expert_of(int lane, int i) {
  return (i < 4) ? 4 * lane + i : 128 + 4 * lane + (i - 4);
}

// Shared-window slot of the hi byte of one key of a packed pair (half 0 or 1).
// The window holds the hi bytes 0xB0-0xBF (margins 2^-30 <= r < 2, slots
// 0-15) and 0x40-0x4F (-2 < r <= -2^-30, slots 16-31); every other byte maps
// to kDummy (32), a row that is never flushed.  Computed in registers: with
// the pair xor 0x40004000, the in-window hi bytes become 0xF0-0xFF and
// 0x00-0x0F, i.e. the signed bytes -16..15; sign-extended (one prmt) and
// offset by 16 they are the slots 0..31, and an unsigned min sends the rest
// to 32.
__device__ __forceinline__ uint32_t window_slot(uint32_t kw, int half) {
  const uint32_t sx = prmt(kw ^ 0x40004000u, 0u, half ? 0xBBB3u : 0x9991u);
  return min(sx + 16u, (uint32_t)kDummy);
}

// Hi byte counted by window slot s (the inverse of window_slot on the window).
__device__ __forceinline__ int slot_bin(int s) { return s < 16 ? 0xB0 + s : 0x40 + (s - 16); }

struct Ctx {
  const Args* a;
  unsigned char* tile;
  float* gmax;
  float* alpha_s;
  uint64_t* bars;
  const float* bias_s;
  uint32_t hb;  // shared byte address of this lane's slot-0 counter of element 0
  int lane;
  int k;
};

// Issue the loads of row pair q of the tile at token `start` (nrows rows):
// every lane copies its 16-byte chunks of the pair with cp.async (global to
// shared, no registers) and then makes the pair's mbarrier track their
// completion (cp.async.mbarrier.arrive.noinc; the barrier expects one such
// arrival per lane).  The copies go through the load/store path, not the
// bulk-copy unit: that unit stays free for the bulk reductions of a kernel
// running beside this one (lei_apply_overlap), which stalled badly behind
// one bulk copy per row.
template <typename T>
__device__ __forceinline__ void issue_pair(const Ctx& c, int64_t start, int nrows, int q) {
  constexpr int kChunks = In<T>::kRowBytes / 16;  // 16-byte chunks per row
  const int r0 = 2 * q;
  if (nrows <= r0) return;  // warp-uniform
  const int nr = nrows - r0 >= 2 ? 2 : 1;
  const char* src = reinterpret_cast<const char*>(static_cast<const T*>(c.a->logits) +
                                                  (start + r0) * (int64_t)kE);
  const uint32_t dst = smem_u32(c.tile + r0 * kPitch + In<T>::kOff);
#pragma unroll
  for (int j = 0; j < 2 * kChunks / 32; ++j) {
    const int ch = c.lane + 32 * j;  // chunk of the pair
    const int row = ch / kChunks;
    if (row < nr)
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                       dst + (uint32_t)(row * kPitch + (ch % kChunks) * 16)),
                   "l"(src + row * In<T>::kRowBytes + (ch % kChunks) * 16)
                   : "memory");
  }
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(c.bars + q))
               : "memory");
}

// Bounded wait on an mbarrier phase, decided by the whole warp at once (a
// vote per poll keeps the loop warp-uniform); gives up after ~2^24 polls,
// records kDevTimeout and returns false.
__device__ __forceinline__ bool warp_wait_bounded(uint64_t* bar, uint32_t parity, int* status) {
  for (uint32_t it = 0; it < (1u << 24); ++it) {
    if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
    if (it > 64) __nanosleep(64);
  }
  if (lane_id() == 0) atomicOr(status, kDevTimeout);
  return false;
}

// Phase C of a tile: r = alpha + sn (= alpha - s), BF16 keys, key stores and
// the hi-byte counts, two rows at a time; after each pair its rows are
// refilled with the next tile's.  FOLD: the tile held a logit beyond the range
// where no margin can round to bf16 -0, so -0 is folded to +0 first.
template <typename T, bool FULL, bool FOLD>
__device__ __forceinline__ void phase_c(const Ctx& c, int64_t t0, int rows, int64_t n0,
                                        int nrows) {
  const Args& a = *c.a;
  const int lane = c.lane;
  uint16_t* kp = a.keys_out ? a.keys_out + t0 * kE + 4 * lane : nullptr;
#pragma unroll 1
  for (int q = 0; q < kPairs; ++q) {
    uint32_t kw[2][4];
    uint32_t mslot = 0;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int st = 2 * q + u;
      if (FULL || st < rows) {
        const unsigned char* row = c.tile + st * kPitch;
        const float4 s0 = *reinterpret_cast<const float4*>(row + 16 * lane);
        const float4 s1 = *reinterpret_cast<const float4*>(row + 512 + 16 * lane);
        const f2_t A = f2_splat(c.alpha_s[st]);
        const f2_t SN[4] = {f2_pack(s0.x, s0.y), f2_pack(s0.z, s0.w), f2_pack(s1.x, s1.y),
                            f2_pack(s1.z, s1.w)};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float r0, r1;
          f2_unpack(f2_add(A, SN[i]), r0, r1);
          uint32_t w = bf16x2_rn(r0, r1);
          if constexpr (FOLD) {
            const uint32_t nz = (w & 0x7FFF7FFFu) + 0x7FFF7FFFu;
            w &= (nz | 0x7FFF7FFFu);  // -0 -> +0
          }
          kw[u][i] = w ^ (prmt(w, 0u, 0xBB99u) | 0x80008000u);
        }
        if (kp) {
          *reinterpret_cast<uint2*>(kp + st * kE) = make_uint2(kw[u][0], kw[u][1]);
          *reinterpret_cast<uint2*>(kp + st * kE + 128) = make_uint2(kw[u][2], kw[u][3]);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint32_t slot = window_slot(kw[u][i >> 1], i & 1);
          mslot = slot > mslot ? slot : mslot;
          route::red_shared_add1(c.hb + 128u * (uint32_t)i + (slot << 10));
        }
      }
    }
    if (__any_sync(0xffffffffu, mslot == (uint32_t)kDummy)) {
      // rare: hi bytes outside the shared window go to the global histogram
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        if (FULL || 2 * q + u < rows) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            if (window_slot(kw[u][i >> 1], i & 1) == (uint32_t)kDummy) {
              const uint32_t bin = prmt(kw[u][i >> 1], 0u, (i & 1) ? 0x4443u : 0x4441u);
              atomicAdd(a.hist + (int64_t)expert_of(lane, i) * 256 + bin, 1);
            }
          }
        }
      }
    }
    __syncwarp();
    issue_pair<T>(c, n0, nrows, q);
  }
}

// One tile: phase A (scores, group maxima), B (alpha, top-k), C (keys and
// counts; refills).  FULL: all 8 rows are tokens.  Returns false if a wait
// on a row pair timed out (the warp then stops).
template <typename T, int KL, int K1, int MODE, bool FULL>
__device__ __forceinline__ bool tile_pass(const Ctx& c, const float (&breg)[8], int64_t t0,
                                          int rows, int64_t n0, int nrows, uint32_t parity) {
  const Args& a = *c.a;
  const int lane = c.lane;
  const int k = c.k;
  unsigned char* tile = c.tile;

  if constexpr (!FULL) {
    // the rows past the end hold no token: give them zeros
    uint4* z = reinterpret_cast<uint4*>(tile + rows * kPitch);
    for (int i = lane; i < (kTile - rows) * (kPitch / 16); i += 32) z[i] = make_uint4(0, 0, 0, 0);
    __syncwarp();
  }

  // ---- phase A: two rows per iteration
  bool ext = false;
  bool ok = true;
#pragma unroll 1
  for (int q = 0; q < kPairs; ++q) {
    if (FULL || 2 * q < rows) ok = warp_wait_bounded(c.bars + q, parity, a.status);
    if (!ok) return false;
    unsigned char* r0 = tile + 2 * q * kPitch;
    float x[16];
    load_x(r0, lane, static_cast<const T*>(nullptr), x);
    load_x(r0 + kPitch, lane, static_cast<const T*>(nullptr), x + 8);
    if constexpr (sizeof(T) != 4) __syncwarp();  // all logits read before scores overwrite them
    const float m = max_abs16(x);
    ext |= m > kFoldAbsX;
    float sn[16];
    if (__all_sync(0xffffffffu, m <= kFastAbsX)) {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        f2_unpack(neg_sigmoid2_fast(f2_pack(x[2 * i], x[2 * i + 1])), sn[2 * i], sn[2 * i + 1]);
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) sn[i] = -sigmoid_pinned(x[i]);
    }
    float v[16];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      f2_unpack(f2_sub(f2_pack(breg[(2 * i) & 7], breg[(2 * i + 1) & 7]),
                       f2_pack(sn[2 * i], sn[2 * i + 1])),
                v[2 * i], v[2 * i + 1]);
    *reinterpret_cast<float4*>(r0 + 16 * lane) = make_float4(sn[0], sn[1], sn[2], sn[3]);
    *reinterpret_cast<float4*>(r0 + 512 + 16 * lane) = make_float4(sn[4], sn[5], sn[6], sn[7]);
    *reinterpret_cast<float4*>(r0 + kPitch + 16 * lane) = make_float4(sn[8], sn[9], sn[10], sn[11]);
    *reinterpret_cast<float4*>(r0 + kPitch + 512 + 16 * lane) =
        make_float4(sn[12], sn[13], sn[14], sn[15]);
    c.gmax[(2 * q) * kGP + lane] = max8(v);
    c.gmax[(2 * q + 1) * kGP + lane] = max8(v + 8);
  }
  __syncwarp();
  const bool tile_ext = __any_sync(0xffffffffu, ext);

  // ---- phase B: 4 lanes per token (lane = t + 8h), lane h holds groups
  // 8h..8h+7.  tau = the (k+1)-th largest group maximum is a lower bound of
  // alpha, and every v > tau lies in a group whose maximum exceeds tau (at
  // most k such groups).  Those groups are dealt to the token's lanes in
  // ascending order (round r, lane h: the (4r+h)-th lowest); each lane sorts
  // and merges its groups, the lanes merge, and alpha = max(tau, L[k]).
  {
    constexpr int R = KL == 8 ? 2 : 4;  // rounds: at most k <= KL-1 groups
    const int t = lane & 7;
    const int h = lane >> 3;
    const bool actB = FULL || t < rows;
    const unsigned char* trow = tile + t * kPitch;
    float gm[8];
    {
      const float4 g0 = *reinterpret_cast<const float4*>(c.gmax + t * kGP + 8 * h);
      const float4 g1 = *reinterpret_cast<const float4*>(c.gmax + t * kGP + 8 * h + 4);
      gm[0] = g0.x; gm[1] = g0.y; gm[2] = g0.z; gm[3] = g0.w;
      gm[4] = g1.x; gm[5] = g1.y; gm[6] = g1.z; gm[7] = g1.w;
    }
    float L[KL];
    {
      float w8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) w8[i] = gm[i];
      route::first_block8<KL>(L, w8);
    }
    merge_partner_first<KL>(L, 8);
    float tau;
    if constexpr (K1 > 0) {
      float P[KL];
      partner_head<KL, K1>(L, P, 16);
      tau = select_with_partner<KL, K1>(L, P);
    } else {
      route::merge_partner<KL>(L, 16);
      tau = route::pick<KL, K1>(L, k);
    }
    uint32_t gt = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) gt |= (gm[i] > tau ? 1u : 0u) << (8 * h + i);
    gt |= __shfl_xor_sync(0xffffffffu, gt, 8);
    gt |= __shfl_xor_sync(0xffffffffu, gt, 16);
    int gr[R];
    {
      uint32_t m = gt;
#pragma unroll
      for (int r = 0; r < R; ++r) {
        int g = -1;
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const int gp = route::lowest_bit(m);
          m &= m - 1;
          g = (p == h) ? gp : g;
        }
        gr[r] = g;
      }
    }
    {
      float w8[8];
      group_v(trow, c.bias_s, gr[0] < 0 ? 0 : gr[0], w8);
#pragma unroll
      for (int i = 0; i < 8; ++i) w8[i] = gr[0] < 0 ? -INFINITY : w8[i];
      route::first_block8<KL>(L, w8);
    }
    // k = 6 (at most 6 groups): the second round deals the halves of the
    // groups of rank 4 and 5 (lane h: rank 4 + h/2, half h%2), so that every
    // lane sorts 4 values instead of two lanes sorting 8 each.
    int g1 = -1, half1 = 0;
    if constexpr (K1 == 7) {
      uint32_t m = gt;
#pragma unroll
      for (int p = 0; p < 4; ++p) m &= m - 1;
      const int g4 = route::lowest_bit(m);
      m &= m - 1;
      const int g5 = route::lowest_bit(m);
      g1 = (h >> 1) ? g5 : g4;
      half1 = h & 1;
      if (__any_sync(0xffffffffu, g1 >= 0)) {
        float w4[4];
        half_v(trow, c.bias_s, g1 < 0 ? 0 : g1, half1, w4);
#pragma unroll
        for (int i = 0; i < 4; ++i) w4[i] = g1 < 0 ? -INFINITY : w4[i];
        merge_block4<KL>(L, w4);
      }
    } else {
#pragma unroll
      for (int r = 1; r < R; ++r) {
        if (__any_sync(0xffffffffu, gr[r] >= 0)) {
          float w8[8];
          group_v(trow, c.bias_s, gr[r] < 0 ? 0 : gr[r], w8);
#pragma unroll
          for (int i = 0; i < 8; ++i) w8[i] = gr[r] < 0 ? -INFINITY : w8[i];
          if constexpr (KL == 16) {
            if (r == 1)
              append_block8_16(L, w8);  // round 0 left 8 values and 8 -inf
            else
              route::merge_block8<KL>(L, w8);
          } else {
            route::merge_block8<KL>(L, w8);
          }
        }
      }
    }
    route::merge_partner<KL>(L, 8);
    // alpha = max(tau, the (k+1)-th largest v of the dealt groups); ties at
    // alpha exist exactly when the k-th largest of those is not above it
    float alpha;
    bool tie;
    if constexpr (K1 > 0) {
      float P[KL];
      partner_head<KL, K1>(L, P, 16);
      alpha = fmaxf(tau, select_with_partner<KL, K1>(L, P));
      tie = !(select_with_partner<KL, K1 - 1>(L, P) > alpha);
    } else {
      route::merge_partner<KL>(L, 16);
      alpha = fmaxf(tau, route::pick<KL, K1>(L, k));
      int c_gt = 0;
#pragma unroll
      for (int i = 0; i < KL; ++i) c_gt += (i < k && L[i] > alpha) ? 1 : 0;
      tie = c_gt < k;
    }
    const int64_t tok = t0 + t;
    if (actB && h == 0) {
      c.alpha_s[t] = alpha;
      if (a.alpha_out) a.alpha_out[tok] = alpha;
    }
    if (MODE == kHi256 && a.topk_out) {
      int32_t* out = a.topk_out + tok * k;
      if (__any_sync(0xffffffffu, actB && tie)) {
        // rare: ties at alpha.  One lane per token scans the groups whose
        // maximum reaches alpha in expert order (low halves, then high).
        uint32_t ge = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) ge |= (gm[i] >= alpha ? 1u : 0u) << (8 * h + i);
        ge |= __shfl_xor_sync(0xffffffffu, ge, 8);
        ge |= __shfl_xor_sync(0xffffffffu, ge, 16);
        if (actB && h == 0) {
          // k minus the number of v > alpha: the ties to take, in index order
          int tl = k;
          for (uint32_t m = ge; m; m &= m - 1) {
            const int g = route::lowest_bit(m);
            for (int half = 0; half < 2; ++half)
              for (int i = 0; i < 4; ++i) {
                const int e = half * 128 + 4 * g + i;
                const float sv = *reinterpret_cast<const float*>(trow + 4 * e);
                tl -= __fsub_rn(c.bias_s[e], sv) > alpha ? 1 : 0;
              }
          }
          int n = 0;
          for (int half = 0; half < 2; ++half) {
            for (uint32_t m = ge; m; m &= m - 1) {
              const int g = route::lowest_bit(m);
              for (int i = 0; i < 4; ++i) {
                const int e = half * 128 + 4 * g + i;
                const float sv = *reinterpret_cast<const float*>(trow + 4 * e);
                const float vv = __fsub_rn(c.bias_s[e], sv);
                if (vv > alpha || (vv == alpha && tl > 0)) {
                  if (!(vv > alpha)) --tl;
                  out[n++] = e;
                }
              }
            }
          }
        }
      } else if constexpr (K1 == 7) {
        // the 6 experts with v > alpha, ascending.  Pieces in expert order:
        // the low halves of ranks 0-3 (round 0, lanes 0-3), of rank 4 (lane 0)
        // and 5 (lane 2), then the high halves of ranks 0-3, 4 (lane 1), 5
        // (lane 3).  Packed 8-bit counts per lane: A = round-0 low half,
        // B = round-0 high half, Ce / Co = the round-1 half on even / odd lanes.
        uint32_t b0lo = 0, b0hi = 0, b1 = 0;
        {
          float w8[8];
          group_v(trow, c.bias_s, gr[0] < 0 ? 0 : gr[0], w8);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            b0lo |= (w8[i] > alpha ? 1u : 0u) << i;
            b0hi |= (w8[4 + i] > alpha ? 1u : 0u) << i;
          }
          if (gr[0] < 0 || !actB) b0lo = b0hi = 0u;
        }
        if (__any_sync(0xffffffffu, g1 >= 0)) {
          float w4[4];
          half_v(trow, c.bias_s, g1 < 0 ? 0 : g1, half1, w4);
#pragma unroll
          for (int i = 0; i < 4; ++i) b1 |= (w4[i] > alpha ? 1u : 0u) << i;
          if (g1 < 0 || !actB) b1 = 0u;
        }
        const uint32_t c1 = (uint32_t)__popc(b1);
        const uint32_t cnt = (uint32_t)__popc(b0lo) | ((uint32_t)__popc(b0hi) << 8) |
                             ((half1 ? 0u : c1) << 16) | ((half1 ? c1 : 0u) << 24);
        uint32_t incl = cnt;
        {
          uint32_t y = __shfl_up_sync(0xffffffffu, incl, 8);
          if (h >= 1) incl += y;
          y = __shfl_up_sync(0xffffffffu, incl, 16);
          if (h >= 2) incl += y;
        }
        const uint32_t tot = __shfl_sync(0xffffffffu, incl, t + 24);
        const uint32_t excl = incl - cnt;
        const int totA = (int)(tot & 0xFFu), totB = (int)((tot >> 8) & 0xFFu);
        const int base_hi = totA + (int)((tot >> 16) & 0xFFu);
        int pos = (int)(excl & 0xFFu);
        for (uint32_t b = b0lo; b; b &= b - 1) out[pos++] = 4 * gr[0] + __ffs((int)b) - 1;
        pos = base_hi + (int)((excl >> 8) & 0xFFu);
        for (uint32_t b = b0hi; b; b &= b - 1) out[pos++] = 128 + 4 * gr[0] + __ffs((int)b) - 1;
        pos = half1 ? base_hi + totB + (int)(excl >> 24) : totA + (int)((excl >> 16) & 0xFFu);
        for (uint32_t b = b1; b; b &= b - 1) out[pos++] = 128 * half1 + 4 * g1 + __ffs((int)b) - 1;
      } else {
        // the k experts with v > alpha, ascending: every lane's dealt groups
        // in dealing order (ascending group index), low halves first
        uint32_t blo[R], bhi[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
          blo[r] = bhi[r] = 0u;
          if (r == 0 || __any_sync(0xffffffffu, gr[r] >= 0)) {
            float w8[8];
            group_v(trow, c.bias_s, gr[r] < 0 ? 0 : gr[r], w8);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              blo[r] |= (w8[i] > alpha ? 1u : 0u) << i;
              bhi[r] |= (w8[4 + i] > alpha ? 1u : 0u) << i;
            }
            if (gr[r] < 0 || !actB) blo[r] = bhi[r] = 0u;
          }
        }
        // packed 8-bit counts: lo of round r at field r, hi at field R + r
        using PK = typename std::conditional<(R <= 2), uint32_t, unsigned long long>::type;
        PK cnt = 0;
#pragma unroll
        for (int r = 0; r < R; ++r)
          cnt |= ((PK)__popc(blo[r]) << (8 * r)) | ((PK)__popc(bhi[r]) << (8 * (R + r)));
        PK incl = cnt;
        {
          PK y = __shfl_up_sync(0xffffffffu, incl, 8);
          if (h >= 1) incl += y;
          y = __shfl_up_sync(0xffffffffu, incl, 16);
          if (h >= 2) incl += y;
        }
        const PK tot = __shfl_sync(0xffffffffu, incl, t + 24);
        const PK excl = incl - cnt;
        int base = 0;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const int f = 8 * (half * R + r);
            int pos = base + (int)((excl >> f) & 0xFFu);
            base += (int)((tot >> f) & 0xFFu);
            const int e0 = half * 128 + 4 * gr[r];
            for (uint32_t b = half ? bhi[r] : blo[r]; b; b &= b - 1) {
              out[pos] = e0 + __ffs((int)b) - 1;
              ++pos;
            }
          }
        }
      }
    }
  }
  __syncwarp();

  // ---- phase C: margins, keys, counts; refill each freed row pair
  if constexpr (MODE == kHi256) {
    if (tile_ext)
      phase_c<T, FULL, true>(c, t0, rows, n0, nrows);
    else
      phase_c<T, FULL, false>(c, t0, rows, n0, nrows);
  } else {
    // alpha only: every row is free once phase B is done
#pragma unroll
    for (int q = 0; q < kPairs; ++q) issue_pair<T>(c, n0, nrows, q);
  }
  return true;
}

template <typename T, int KL, int K1, int MODE>
__global__ void __launch_bounds__(warps_max(MODE) * 32, 1) route256_kernel(const Args a) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ __align__(16) float bias_s[kE];
  const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);
  const int lane = threadIdx.x & 31;
  int32_t* hist_s = reinterpret_cast<int32_t*>(smem);
  unsigned char* wb = smem + hist_bytes(MODE) + warp * kWarpBytes;
  Ctx c;
  c.a = &a;
  c.tile = wb;
  c.gmax = reinterpret_cast<float*>(wb + kTile * kPitch);
  c.alpha_s = c.gmax + kTile * kGP;
  c.bars = reinterpret_cast<uint64_t*>(c.alpha_s + 8);
  c.bias_s = bias_s;
  c.hb = smem_u32(hist_s) + 4u * (uint32_t)lane;
  c.lane = lane;
  c.k = a.k;

  if constexpr (MODE == kHi256)
    for (int i = threadIdx.x; i < (kWin + 1) * kE; i += blockDim.x) hist_s[i] = 0;
  // Launched as a programmatic dependent of the kernel before it: this CTA
  // may have started while that kernel still runs, so wait for its
  // completion (and its memory) before the first global access.  A chained
  // call follows another hi pass of the same global batch, which has itself
  // waited before it let this one launch: nothing this call reads is still
  // being written, and its counts only add to the same histogram, so it
  // starts at once (and waits at its end, so that it completes after the
  // call before it).
  if (!a.chained) asm volatile("griddepcontrol.wait;" ::: "memory");
  // From here on, a kernel launched as this one's programmatic dependent (the
  // next chained call, or lei_apply_overlap) may take the room this CTA
  // leaves: everything before this kernel has completed, except the earlier
  // hi passes of a chain, which only add to the histogram.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  for (int i = threadIdx.x; i < kE; i += blockDim.x) bias_s[i] = a.bias[i];
  if (lane == 0) {
    // one arrival per lane per phase: each lane's cp.async completions
    for (int q = 0; q < kPairs; ++q) mbar_init(c.bars + q, 32);
    fence_mbar_init();
  }
  __syncthreads();
  float breg[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) breg[i] = bias_s[expert_of(lane, i)];

  // warps per CTA of this launch (<= kNW; the launcher balances the tiles)
  const int nw = (int)(blockDim.x >> 5);
  const int64_t n_tiles = (a.N + kTile - 1) / kTile;
  const int64_t wstride = (int64_t)gridDim.x * nw;
  int64_t tix = (int64_t)blockIdx.x * nw + warp;
  if (tix < n_tiles) {
    const int64_t s0 = tix * kTile;
    const int rows0 = (int)((a.N - s0) < kTile ? (a.N - s0) : kTile);
#pragma unroll
    for (int q = 0; q < kPairs; ++q) issue_pair<T>(c, s0, rows0, q);
  }
  uint32_t parity = 0;
  bool clean = true;  // no wait of this warp gave up
  for (; tix < n_tiles; tix += wstride) {
    const int64_t t0 = tix * kTile;
    const int rows = (int)((a.N - t0) < kTile ? (a.N - t0) : kTile);
    const int64_t nt = tix + wstride;
    const int64_t n0 = nt * kTile;
    const int nrows = nt < n_tiles ? (int)((a.N - n0) < kTile ? (a.N - n0) : kTile) : 0;
    const bool ok = rows == kTile
                        ? tile_pass<T, KL, K1, MODE, true>(c, breg, t0, rows, n0, nrows, parity)
                        : tile_pass<T, KL, K1, MODE, false>(c, breg, t0, rows, n0, nrows, parity);
    if (!ok) {
      clean = false;
      break;
    }
    parity ^= 1u;
  }

  // ---- flush the shared window (after every warp's increments)
  if constexpr (MODE == kHi256) {
    const int nw = (int)(blockDim.x >> 5);
    const bool all_clean = __syncthreads_and(clean ? 1 : 0) != 0;
    if (all_clean && (reinterpret_cast<uintptr_t>(a.hist) & 15) == 0 &&
        nw * kWarpBytes >= kE * kStg * 4) {
      // Through the (now idle) tile buffers: the window is copied into rows
      // r = 32 i + L (expert expert_of(L, i)) of kStg words, whose slots 0-15
      // and 16-31 are two runs of 16 consecutive counters of the expert's
      // histogram row (hi bytes 0xB0-0xBF and 0x40-0x4F); each run is then
      // added by one 64-byte bulk reduction in L2 (512 per CTA instead of
      // one atomic per counter).  Both copies are conflict-free: the reads
      // take 32 consecutive words, and the 16-byte writes of a quarter-warp
      // land on 8 different 16-byte bank groups ((9 r + q) % 8 differs).
      // Taken only when no wait of the CTA gave up, so no row copy or its
      // barrier arrival is outstanding; every lane still waits for its own
      // copies, and the row-pair barriers living in the buffers are
      // invalidated before the buffers are reused.
      asm volatile("cp.async.wait_all;" ::: "memory");
      if (lane == 0)
        for (int q = 0; q < kPairs; ++q)
          asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(c.bars + q))
                       : "memory");
      __syncthreads();
      int32_t* stg = reinterpret_cast<int32_t*>(smem + hist_bytes(MODE));
      for (int p = warp; p < 8 * (kWin / 4); p += nw) {
        const int i = p & 7, q = p >> 3;  // rows 32 i + lane, slots 4q .. 4q+3
        const int32_t* src = hist_s + lane + 32 * i + 256 * (4 * q);
        *reinterpret_cast<int4*>(stg + (32 * i + lane) * kStg + 4 * q) =
            make_int4(src[0], src[256], src[512], src[768]);
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncthreads();
      for (int j = threadIdx.x; j < 2 * kE; j += blockDim.x) {
        const int r = j >> 1, run = j & 1;
        int32_t* dst = a.hist + (int64_t)expert_of(r & 31, r >> 5) * 256 + (run ? 0x40 : 0xB0);
        asm volatile(
            "cp.reduce.async.bulk.global.shared::cta.bulk_group.add.u32 [%0], [%1], 64;" ::"l"(dst),
            "r"(smem_u32(stg + r * kStg + 16 * run))
            : "memory");
      }
      asm volatile("cp.async.bulk.commit_group;" ::: "memory");
      asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    } else {
      // a histogram that is not 16-byte aligned, or a wait that gave up (its
      // copies may still land in the tile buffers): one atomic per non-zero
      // counter, straight from the window
      for (int w = threadIdx.x; w < kWin * kE; w += blockDim.x) {
        const int cnt = hist_s[w];
        if (cnt) {
          const int slot = w >> 8, p = w & 255;
          atomicAdd(a.hist + (int64_t)expert_of(p & 31, p >> 5) * 256 + slot_bin(slot), cnt);
        }
      }
    }
  }
  if (a.chained) asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <typename T, int KL, int K1, int MODE>
int launch_one(const Args& a, cudaStream_t stream) {
  constexpr int kNWm = warps_max(MODE);
  auto kern = route256_kernel<T, KL, K1, MODE>;
  static bool attr_set = false;  // per instantiation; benign race (idempotent)
  if (!attr_set) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             hist_bytes(MODE) + kNWm * kWarpBytes) != cudaSuccess)
      return launch_status();
    attr_set = true;
  }
  // Tiles are dealt round-robin to every warp of the grid, so the launch
  // takes as many tile-times as its busiest warp has tiles.  Use every SM,
  // the fewest rounds that kNW warps per CTA allow, and then only as many
  // warps per CTA as those rounds need (a 32768-token call: 4096 tiles = 2
  // rounds of 14 warps on 152 SMs, not 20 warps of which a third idle in the
  // second round).
  const int64_t n_tiles = (a.N + kTile - 1) / kTile;
  int64_t grid = sm_count();
  if (n_tiles < grid) grid = n_tiles;
  if (grid < 1) grid = 1;
  const int64_t rounds = (n_tiles + grid * kNWm - 1) / (grid * kNWm);
  int64_t nw = rounds > 0 ? (n_tiles + grid * rounds - 1) / (grid * rounds) : 1;
  if (nw < 1) nw = 1;
  if (nw > kNWm) nw = kNWm;
  // A programmatic dependent launch: the CTAs of this call may take the SMs
  // that the previous kernel on the stream frees and run their shared-memory
  // set-up while it finishes (the kernel waits for it before touching global
  // memory); back-to-back microbatch calls lose less time between launches.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)(nw * 32));
  cfg.dynamicSmemBytes = (size_t)(hist_bytes(MODE) + (int)nw * kWarpBytes);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, a) != cudaSuccess) {
    (void)cudaGetLastError();
    return QB_ECUDA;
  }
  return launch_status();
}

template <typename T, int MODE>
int dispatch_k(int k, const Args& a, cudaStream_t st) {
  if (k + 1 == 7) return launch_one<T, 8, 7, MODE>(a, st);
  if (k + 1 == 9) return launch_one<T, 16, 9, MODE>(a, st);
  if (k + 1 <= 8) return launch_one<T, 8, 0, MODE>(a, st);
  return launch_one<T, 16, 0, MODE>(a, st);
}

// EQB hi pass at E = 256 for one input type (same contract as
// route::launch_mode<kModeHi>); instantiated by qb_route256_f32.cu and
// qb_route256_bf16.cu.
template <typename T>
int launch_hi_t(const void* logits, const float* bias, int64_t N, int k, int32_t* hist,
                uint16_t* keys_out, int32_t* topk_out, float* alpha_out, cudaStream_t stream,
                bool chained = false) {
  Args a{logits, bias, N, k, hist, keys_out, topk_out, alpha_out, nullptr, nullptr, 0,
         device_status_ptr(), kE};
  a.chained = chained ? 1 : 0;
  if (!a.status) return QB_ECUDA;
  return dispatch_k<T, kHi256>(k, a, stream);
}

// alpha per token only (phases A and B), for the K3 counting kernel.
template <typename T>
int launch_alpha_t(const void* logits, const float* bias, int64_t N, int k, float* alpha_out,
                   cudaStream_t stream, bool chained = false) {
  Args a{logits, bias, N, k, nullptr, nullptr, nullptr, alpha_out, nullptr, nullptr, 0,
         device_status_ptr(), kE};
  a.chained = chained ? 1 : 0;
  if (!a.status) return QB_ECUDA;
  return dispatch_k<T, kAlpha256>(k, a, stream);
}

}  // namespace r256
}  // namespace qb
