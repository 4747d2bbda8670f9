// qb_gemm.cu -- router GEMM front end: logits = hidden (bf16) x W (bf16),
// fp32 accumulation on the 5th-generation tensor cores (tcgen05, TMEM).
//
// The router of "[Dev] Add global-batch quantile balancing" computes its
// scores from hidden states; the histogram passes then run on those scores
// ("Implementation": the fused path extends the existing router kernel).
//
// One CTA computes a 128 x 256 tile of logits (all experts of 128 tokens):
//   warp 0      TMA producer: hidden tile 128 x 64 and W^T tile 256 x 64 per
//               stage (bf16, 128-byte swizzle) into a 4-deep ring;
//   warp 1      allocates 256 TMEM columns; one lane issues tcgen05.mma
//               (M=128, N=256, K=16) four times per stage and commits each
//               stage back to the producer, and the last one to the epilogue;
//   warps 2-5   epilogue: tcgen05.ld 32 lanes x 32 columns at a time, fp32
//               stores of the logits.
// Every mbarrier wait is bounded; a timeout sets the device status flag and
// the CTA still frees its TMEM before returning.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "qb_device.cuh"
#include "qb_internal.h"
#include "qb_tc.cuh"

namespace qb {
namespace {

constexpr int kBM = 128;        // tokens per tile (TMEM lanes)
constexpr int kBN = 256;        // experts per tile (TMEM columns)
constexpr int kBK = 64;         // K per stage: one 128-byte swizzle row of bf16
constexpr int kStages = 4;
constexpr int kABytes = kBM * kBK * 2;  // 16 KB
constexpr int kBBytes = kBN * kBK * 2;  // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kThreads = 192;
constexpr int kSmemBytes = kStages * kStageBytes + 1024 /*align*/ + 256 /*barriers*/;

constexpr uint32_t kIdesc = idesc_bf16_f32(kBM, kBN);

struct GemmArgs {
  float* logits;  // [M, 256] fp32
  int64_t M;
  int K;
  int* status;
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
  uint64_t* full = bars;                 // [kStages]
  uint64_t* empty = bars + kStages;      // [kStages]
  uint64_t* accum = bars + 2 * kStages;  // [1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t m0 = (int64_t)blockIdx.x * kBM;
  const int ktiles = g.K / kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    mbar_init(accum, 1);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), kBN);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;

  if (warp == 0) {
    if (lane == 0) {
      for (int kt = 0; kt < ktiles && ok; ++kt) {
        const int s = kt % kStages;
        const uint32_t round = (uint32_t)(kt / kStages);
        if (kt >= kStages) ok = mbar_wait_bounded(empty + s, (round - 1) & 1u, g.status);
        if (!ok) break;
        const uint32_t sa = base + (uint32_t)(s * kStageBytes);
        mbar_arrive_expect_tx(full + s, (uint32_t)kStageBytes);
        tma_load_2d(sa, &map_a, kt * kBK, (int)m0, smem_u32(full + s));
        tma_load_2d(sa + kABytes, &map_b, kt * kBK, 0, smem_u32(full + s));
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      for (int kt = 0; kt < ktiles && ok; ++kt) {
        const int s = kt % kStages;
        ok = mbar_wait_bounded(full + s, (uint32_t)(kt / kStages) & 1u, g.status);
        if (!ok) break;
        tc_fence_after();
        const uint32_t sa = base + (uint32_t)(s * kStageBytes);
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk) {
          // the 16-element K slice starts 32 bytes further along the row
          const uint64_t ad = smem_desc_sw128(sa + 32u * kk);
          const uint64_t bd = smem_desc_sw128(sa + kABytes + 32u * kk);
          tc_mma(tmem, ad, bd, kIdesc, (kt > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(smem_u32(empty + s));  // frees the stage once these MMAs are done
      }
      tc_commit(smem_u32(accum));  // all MMAs of the tile
    }
  } else {
    // epilogue warps 2..5: warp w reads TMEM lanes 32*(w%4) .. +31
    const int q = warp & 3;
    ok = mbar_wait_bounded(accum, 0u, g.status);
    ok = __all_sync(0xffffffffu, ok);  // tcgen05.ld is warp-collective
    tc_fence_after();
    if (ok) {
      const int64_t row = m0 + 32 * q + lane;
      const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
#pragma unroll 1
      for (int c0 = 0; c0 < kBN; c0 += 32) {
        uint32_t r[32];
        tmem_ld32(lane_base + (uint32_t)c0, r);
        if (row < g.M) {
          float4* dst = reinterpret_cast<float4*>(g.logits + row * kBN + c0);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[i] = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                 __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kBN);
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
  if (E != kBN) return QB_EUNSUPPORTED;
  if (K % kBK != 0 || K <= 0) return QB_EUNSUPPORTED;
  if (!encode_fn()) return QB_ECUDA;
  CUtensorMap ma, mb;
  if (!make_map(&ma, hidden, (uint64_t)M, (uint64_t)K, kBM)) return QB_EINVAL;
  if (!make_map(&mb, w_t, (uint64_t)E, (uint64_t)K, kBN)) return QB_EINVAL;
  GemmArgs g{logits, M, K, device_status_ptr()};
  if (!g.status) return QB_ECUDA;
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(router_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes) != cudaSuccess)
      return launch_status();
    attr = true;
  }
  const int64_t tiles = (M + kBM - 1) / kBM;
  router_gemm_kernel<<<(unsigned)tiles, kThreads, kSmemBytes, stream>>>(ma, mb, g);
  return launch_status();
}

}  // namespace qb
