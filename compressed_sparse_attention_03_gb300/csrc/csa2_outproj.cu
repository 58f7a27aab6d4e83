// Grouped output projection.  "Inside DeepSeek V4.1", section "Attention that looks at 640
// places": the 64 head outputs go back through 8 groups of a 1,024-wide bottleneck; page
// "DeepSeek V4.1 - Pooled group / Source layer, pairs pooled": o^g_{t,r} = [O-bar_{h,t}]_{h in r}
// W_OA,r.  Group r holds heads 8r .. 8r+7, concatenated head after head, so its 4096 inputs are
// one contiguous slice of the attention output row.
//
// Per group a bf16 GEMM C_r[M, 1024] = A_r[M, 4096] W_r^T with W_r stored [1024 outputs][4096
// inputs] (K contiguous), fp32 accumulation in tensor memory, bf16 output.  One persistent block
// per SM walks output tiles of 128 rows x 256 outputs; the four 256-output tiles of one
// (group, row tile) are adjacent in the walk, so blocks that run at the same time share each A
// tile through L2 and it is read from HBM about once.
//   warp 0      TMA producer: A [128 x 64] and W [256 x 64] bf16 boxes, 128-byte swizzle, into a
//               ring of kStages stages (48 KB each)
//   warp 1      TMEM allocation and the MMA-issuing thread: per stage four M=128, N=256, K=16
//               MMAs into one of two accumulators (256 columns each)
//   warps 2-5   epilogue (TMEM lane quarter = warp % 4): accumulator -> bf16 -> global
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "csa2_common.cuh"
#include "csa2_internal.h"
#include "csa2_sm100.cuh"

namespace csa2 {
namespace {

using namespace sm100;

constexpr int kBM = 128, kBN = 256, kBK = 64, kStages = 4;
constexpr int kGroups = 8, kGroupIn = 8 * 512, kGroupOut = 1024;
constexpr int kNTiles = kGroupOut / kBN;  // 4
constexpr uint32_t kABytes = kBM * kBK * 2, kBBytes = kBN * kBK * 2, kStageBytes = kABytes + kBBytes;
constexpr uint32_t kOutDyn = kStages * kStageBytes + 1024;
constexpr int kOutThreads = 6 * 32;

__device__ int g_outproj_error;

struct OutBars {
  uint64_t full[kStages], empty[kStages], acc_full[2], acc_empty[2];
};

__global__ void __launch_bounds__(kOutThreads, 1) outproj_kernel(const __grid_constant__ CUtensorMap ta,
                                                                 const __grid_constant__ CUtensorMap tw, int64_t M,
                                                                 uint16_t* out) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ OutBars bars;
  __shared__ uint32_t tmem_base_sh;
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  unsigned char* sm = smem_raw + (sbase - smem_u32(smem_raw));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int* err = &g_outproj_error;
  const int n_mt = (int)((M + kBM - 1) / kBM);
  const int n_tiles = kGroups * n_mt * kNTiles;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars.full[s], 1);
      mbar_init(&bars.empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&bars.acc_full[a], 1);
      mbar_init(&bars.acc_empty[a], 4);
    }
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  if (warp == 0) {
    // ============================================================ TMA producer
    if (lane == 0) {
      int it = 0;  // stage uses so far
      for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
        const int nt = tile % kNTiles, mt = (tile / kNTiles) % n_mt, r = tile / (kNTiles * n_mt);
        for (int kb = 0; kb < kGroupIn / kBK; ++kb, ++it) {
          const int s = it % kStages;
          if (it >= kStages) mbar_wait(&bars.empty[s], ((it / kStages) - 1) & 1, err, 1);
          unsigned char* st = sm + s * kStageBytes;
          mbar_arrive_expect_tx(&bars.full[s], kStageBytes);
          tma_load_2d(st, &ta, r * kGroupIn + kb * kBK, mt * kBM, &bars.full[s]);
          tma_load_2d(st + kABytes, &tw, kb * kBK, r * kGroupOut + nt * kBN, &bars.full[s]);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ============================================================ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(false, false, kBM, kBN, true);
      int it = 0, lt = 0;  // stage uses, local tiles
      for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++lt) {
        const int a = lt & 1;
        if (lt >= 2) mbar_wait(&bars.acc_empty[a], ((lt >> 1) - 1) & 1, err, 2);
        const uint32_t d = tmem + 256u * a;
        for (int kb = 0; kb < kGroupIn / kBK; ++kb, ++it) {
          const int s = it % kStages;
          mbar_wait(&bars.full[s], (it / kStages) & 1, err, 3);
          tc_fence_after();
          const uint32_t sa = sbase + s * kStageBytes, sw = sa + kABytes;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            mma_f16_ss(d, sw128_desc(sa + kk * 32, 16, 1024), sw128_desc(sw + kk * 32, 16, 1024), idesc,
                       (kb | kk) != 0);
          mma_commit(&bars.empty[s]);  // the stage is free once these MMAs have read it
        }
        mma_commit(&bars.acc_full[a]);
      }
    }
    __syncwarp();
  } else {
    // ============================================================ epilogue
    const int q4 = warp & 3;
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * q4) << 16);
    int lt = 0;
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++lt) {
      const int nt = tile % kNTiles, mt = (tile / kNTiles) % n_mt, r = tile / (kNTiles * n_mt);
      const int a = lt & 1;
      mbar_wait(&bars.acc_full[a], (lt >> 1) & 1, err, 4);
      tc_fence_after();
      const int64_t row = (int64_t)mt * kBM + 32 * q4 + lane;
      uint16_t* dst = out + row * (kGroups * kGroupOut) + r * kGroupOut + nt * kBN;
#pragma unroll 1
      for (int c = 0; c < kBN / 32; ++c) {
        uint32_t u[32];
        tmem_ld32(lane_addr + 256u * a + 32 * c, u);
        tmem_wait_ld();
        if (row < M) {
          uint4* o4 = reinterpret_cast<uint4*>(dst + 32 * c);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint32_t w[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(u[8 * v + 2 * k]), __uint_as_float(u[8 * v + 2 * k + 1]));
              w[k] = *reinterpret_cast<const uint32_t*>(&h2);
            }
            o4[v] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.acc_empty[a]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool encode_tiled_2d(CUtensorMap* map, CUtensorMapDataType dtype, int elem_bytes, const void* base, uint64_t cols,
                     uint64_t rows, uint64_t pitch_bytes, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle swizzle) {
  auto fn = encode_fn();
  if (!fn || (reinterpret_cast<uintptr_t>(base) & 15u) || (pitch_bytes & 15u) || (box_cols * elem_bytes) % 16u)
    return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {pitch_bytes};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tiled_1d(CUtensorMap* map, CUtensorMapDataType dtype, int elem_bytes, const void* base, uint64_t n,
                     uint32_t box) {
  auto fn = encode_fn();
  if (!fn || (reinterpret_cast<uintptr_t>(base) & 15u) || (box * elem_bytes) % 16u) return false;
  const cuuint64_t dims[1] = {n};
  const cuuint64_t strides[1] = {(cuuint64_t)n * elem_bytes};  // unused for one dimension
  const cuuint32_t boxd[1] = {box};
  const cuuint32_t estr[1] = {1};
  return fn(map, dtype, 1, const_cast<void*>(base), dims, strides, boxd, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {
// bf16 [rows][cols] row-major (row pitch `pitch` elements), box [box_rows][64], 128-byte swizzle
bool encode_2d(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows, uint64_t pitch, uint32_t box_rows) {
  return encode_tiled_2d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, cols, rows, pitch * 2, kBK, box_rows,
                         CU_TENSOR_MAP_SWIZZLE_128B);
}
}  // namespace

cudaError_t launch_out_group_proj(const uint16_t* o, const uint16_t* w, int64_t M, uint16_t* out, int num_sms,
                                  cudaStream_t st) {
  CUtensorMap ta, tw;
  if (!encode_2d(&ta, o, 64 * 512, (uint64_t)M, 64 * 512, kBM)) return cudaErrorInvalidValue;
  if (!encode_2d(&tw, w, kGroupIn, (uint64_t)kGroups * kGroupOut, kGroupIn, kBN)) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(outproj_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kOutDyn);
  if (e != cudaSuccess) return e;
  const int64_t tiles = (int64_t)kGroups * ((M + kBM - 1) / kBM) * kNTiles;
  const int grid = (int)std::min<int64_t>(tiles, num_sms);
  outproj_kernel<<<grid, kOutThreads, kOutDyn, st>>>(ta, tw, M, out);
  note_launch();
  return cudaGetLastError();
}

cudaError_t take_outproj_error(int* code) {
  const int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(code, g_outproj_error, sizeof(int));
  if (e == cudaSuccess && *code != 0) e = cudaMemcpyToSymbol(g_outproj_error, &zero, sizeof(int));
  return e;
}

}  // namespace csa2
