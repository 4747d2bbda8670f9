// qb_gemm.cu -- router GEMM front end: logits = hidden (bf16) x W (bf16),
// fp32 accumulation on the 5th-generation tensor cores (tcgen05, TMEM).
//
// The router of "[Dev] Add global-batch quantile balancing" computes its
// scores from hidden states; the histogram passes then run on those scores
// ("Implementation": the fused path extends the existing router kernel).
//
// One persistent CTA per SM walks tiles of 128 x E logits (all experts of
// 128 tokens; E a multiple of 32 up to 256), tile = blockIdx.x + i * gridDim.x:
//   warp 0      TMA producer: hidden tile 128 x 64 and W^T tile E x 64 per
//               stage (bf16, 128-byte swizzle) into a 4-deep ring;
//   warp 1      allocates 512 TMEM columns (two accumulators of up to 256
//               columns); one lane issues tcgen05.mma (M=128, N=E, K=16)
//               four times per stage into
//               accumulator (local tile index & 1), commits each stage back to
//               the producer and each finished tile to its epilogue;
//   warps 2-9   two epilogue warpgroups, warpgroup b draining accumulator b
//               (tcgen05.ld 32 lanes x 32 columns at a time, fp32 stores), so
//               that one tile's stores overlap the next tile's MMAs.
// At full MMA rate the hidden-state slices (16 KB per 0.33 us per SM) would
// need more than the HBM bandwidth: the kernel is bound by HBM, not by the
// tensor cores (W^T comes from L2).  Every mbarrier wait is bounded; a
// timeout sets the device status flag and the CTA still frees its TMEM
// before returning.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "qb_device.cuh"
#include "qb_internal.h"
#include "qb_tc.cuh"

namespace qb {
namespace {

constexpr int kBM = 128;        // tokens per tile (TMEM lanes)
constexpr int kBN = 256;        // TMEM columns per accumulator (the largest expert count)
constexpr int kBK = 64;         // K per stage: one 128-byte swizzle row of bf16
constexpr int kStages = 4;
constexpr int kABytes = kBM * kBK * 2;  // 16 KB
constexpr int kBBytes = kBN * kBK * 2;  // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kEpiWarps = 8;
constexpr int kThreads = (2 + kEpiWarps) * 32;
constexpr int kSmemBytes = kStages * kStageBytes + 1024 /*align*/ + 256 /*barriers*/;


struct GemmArgs {
  float* logits;  // [M, E] fp32
  int64_t M;
  int K;
  int* status;
  int E;  // experts: the MMA's N (a multiple of 32, at most 256)
  uint32_t idesc;  // instruction descriptor for M = 128, N = E
};

__global__ void __launch_bounds__(kThreads, 1)
    router_gemm_kernel(const __grid_constant__ CUtensorMap map_a,
                       const __grid_constant__ CUtensorMap map_b, const GemmArgs g) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // 1024-byte alignment for the swizzled tiles
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* sbase = smem_raw + (base - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sbase + kStages * kStageBytes);
  uint64_t* full = bars;                  // [kStages]
  uint64_t* empty = bars + kStages;       // [kStages]
  uint64_t* tfull = bars + 2 * kStages;   // [2]
  uint64_t* tempty = tfull + 2;           // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);

  const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);
  const int lane = threadIdx.x & 31;
  const int ktiles = g.K / kBK;
  const int64_t n_tiles = (g.M + kBM - 1) / kBM;

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
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), 2 * kBN);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      uint32_t gk = 0;
      bool ok = true;
      for (int64_t tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
        for (int kt = 0; kt < ktiles; ++kt, ++gk) {
          const int s = (int)(gk % kStages);
          const uint32_t round = gk / kStages;
          if (gk >= (uint32_t)kStages && !mbar_wait_bounded(empty + s, (round - 1) & 1u, g.status)) {
            ok = false;
            break;
          }
          const uint32_t sa = base + (uint32_t)(s * kStageBytes);
          mbar_arrive_expect_tx(full + s, (uint32_t)(kABytes + g.E * kBK * 2));
          tma_load_2d(sa, &map_a, kt * kBK, (int)(tile * kBM), smem_u32(full + s));
          tma_load_2d(sa + kABytes, &map_b, kt * kBK, 0, smem_u32(full + s));
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = g.idesc;
      uint32_t gk = 0, lt = 0;
      bool ok = true;
      for (int64_t tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x, ++lt) {
        const uint32_t b = lt & 1u, use = lt >> 1;
        if (use >= 1 && !mbar_wait_bounded(tempty + b, (use - 1) & 1u, g.status)) break;
        tc_fence_after();
        const uint32_t d = tmem + b * (uint32_t)kBN;
        for (int kt = 0; kt < ktiles; ++kt, ++gk) {
          const int s = (int)(gk % kStages);
          if (!mbar_wait_bounded(full + s, (gk / kStages) & 1u, g.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = base + (uint32_t)(s * kStageBytes);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            // the 16-element K slice starts 32 bytes further along the row
            const uint64_t ad = smem_desc_sw128(sa + 32u * kk);
            const uint64_t bd = smem_desc_sw128(sa + kABytes + 32u * kk);
            tc_mma(d, ad, bd, idesc, (kt > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(smem_u32(empty + s));  // frees the stage once these MMAs are done
        }
        if (ok) tc_commit(smem_u32(tfull + b));  // all MMAs of the tile
      }
    }
  } else {
    // epilogue: warpgroup wg drains accumulator wg; warp w reads TMEM lanes
    // 32*(w%4) .. +31 (one token each)
    const int wg = (warp - 2) >> 2;
    const int q = warp & 3;
    uint32_t use = 0;
    for (int64_t tile = blockIdx.x + (int64_t)wg * gridDim.x; tile < n_tiles;
         tile += 2 * (int64_t)gridDim.x, ++use) {
      bool ok = mbar_wait_bounded(tfull + wg, use & 1u, g.status);
      ok = __all_sync(0xffffffffu, ok);  // tcgen05.ld is warp-collective
      if (!ok) break;
      tc_fence_after();
      const int64_t row = tile * kBM + 32 * q + lane;
      const uint32_t lane_base = tmem + (uint32_t)(wg * kBN) + ((uint32_t)(32 * q) << 16);
#pragma unroll 1
      for (int c0 = 0; c0 < g.E; c0 += 32) {
        uint32_t r[32];
        tmem_ld32(lane_base + (uint32_t)c0, r);
        if (row < g.M) {
          float4* dst = reinterpret_cast<float4*>(g.logits + row * g.E + c0);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[i] = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                 __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
        }
      }
      tc_fence_before();
      mbar_arrive(tempty + wg);  // the accumulator may be overwritten
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 2 * kBN);
  }
}

// ---- host side: tensor maps -------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool encode_fn() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

// 2-D bf16 tensor [rows, cols] row-major, box [box_rows, 64], 128-byte swizzle.
bool make_map(CUtensorMap* map, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kBK, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool make_bf16_kmajor_map(CUtensorMap* map, const void* ptr, uint64_t rows, uint64_t cols,
                          uint32_t box_rows) {
  return encode_fn() && make_map(map, ptr, rows, cols, box_rows);
}

int launch_router_gemm(const void* hidden, const void* w_t, int64_t M, int K, int E,
                       float* logits, cudaStream_t stream) {
  if (E < 32 || E > kBN || E % 32 != 0) return QB_EUNSUPPORTED;
  if (K % kBK != 0 || K <= 0) return QB_EUNSUPPORTED;
  if (!encode_fn()) return QB_ECUDA;
  CUtensorMap ma, mb;
  if (!make_map(&ma, hidden, (uint64_t)M, (uint64_t)K, kBM)) return QB_EINVAL;
  if (!make_map(&mb, w_t, (uint64_t)E, (uint64_t)K, (uint32_t)E)) return QB_EINVAL;
  GemmArgs g{logits, M, K, device_status_ptr(), E, idesc_bf16_f32(kBM, E)};
  if (!g.status) return QB_ECUDA;
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(router_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes) != cudaSuccess)
      return launch_status();
    attr = true;
  }
  const int64_t tiles = (M + kBM - 1) / kBM;
  int64_t grid = sm_count();
  if (grid > tiles) grid = tiles;
  router_gemm_kernel<<<(unsigned)grid, kThreads, kSmemBytes, stream>>>(ma, mb, g);
  return launch_status();
}

}  // namespace qb
