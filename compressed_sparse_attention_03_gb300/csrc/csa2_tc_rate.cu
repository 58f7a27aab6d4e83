// Tensor-core rate probe: the peak against which the tensor-bound kernels of this library are
// quoted, measured on the device at hand for each operand kind they use.  One block per SM;
// its elected thread issues MMAs of M = 128, N = 256 back to back on fixed shared-memory
// operands into one TMEM accumulator (no memory traffic, no epilogue), so the time is the
// tensor pipe's:
//   kind 0  kind::f16, fp16 operands, K = 16 per MMA (128-byte swizzle)
//   kind 1  kind::f8f6f4, E5M2 operands, K = 32
//   kind 2  kind::mxf4, packed E2M1 operands with UE8M0 scales per 32 values, K = 64 (64-byte
//           swizzle; scale words 2^0 in TMEM)
// Operand values are small finite numbers of each type (no NaN or Inf).
#include <cuda_runtime.h>

#include <algorithm>

#include "csa2_common.cuh"
#include "csa2_internal.h"
#include "csa2_sm100.cuh"

namespace csa2 {
namespace {

using namespace sm100;

constexpr int kRateThreads = 128;
constexpr uint32_t kRateSmem = 48 * 1024 + 1024;  // A 128 x 128 B, B 256 x 128 B, alignment slack
constexpr uint32_t kSfaCol = 256, kSfbCol = 288;  // TMEM: D at 0 (256 columns), scale words

__device__ int g_rate_error;

__global__ void __launch_bounds__(kRateThreads, 1) tc_rate_kernel(int kind, int iters) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_base_sh;
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  unsigned char* sm = smem_raw + (sbase - smem_u32(smem_raw));
  const int tid = threadIdx.x, warp = tid >> 5;
  // fp16 in [0.5, 1), E5M2 codes in [0.5, 1) (exponent field 14), E2M1 codes of magnitude <= 4
  for (int i = tid; i < 48 * 1024 / 4; i += kRateThreads) {
    const uint32_t h = (uint32_t)i * 2654435761u;
    const uint32_t v = kind == 0 ? (0x38003800u | (h & 0x03ff03ffu))
                       : kind == 1 ? (0x38383838u | (h & 0x03030303u))
                                   : (h & 0x66666666u);
    reinterpret_cast<uint32_t*>(sm)[i] = v;
  }
  fence_proxy_async();
  if (tid == 0) {
    mbar_init(&bar, 1);
    mbar_fence_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base_sh, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  const uint32_t lane_addr = tmem + ((uint32_t)(32 * warp) << 16);
  for (int c = 0; c < 4; ++c) tmem_st1(lane_addr + kSfaCol + c, 0x7F7F7F7Fu);
  for (int c = 0; c < 8; ++c) tmem_st1(lane_addr + kSfbCol + c, 0x7F7F7F7Fu);
  tmem_wait_st();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0) {
    const uint32_t sa = sbase, sb = sbase + 16384;
    if (kind == 0) {
      const uint32_t id = idesc_f16(false, false, 128, 256);
      for (int it = 0; it < iters; ++it)
        mma_f16_ss(tmem, sw128_desc(sa + 32 * (it & 3), 16, 1024), sw128_desc(sb + 32 * (it & 3), 16, 1024), id,
                   it > 0 ? 1u : 0u);
    } else if (kind == 1) {
      const uint32_t id = idesc_e5m2(128, 256);
      for (int it = 0; it < iters; ++it)
        mma_f8_ss(tmem, sw128_desc(sa + 32 * (it & 3), 16, 1024), sw128_desc(sb + 32 * (it & 3), 16, 1024), id,
                  it > 0 ? 1u : 0u);
    } else {
      for (int it = 0; it < iters; ++it)
        mma_mxf4(tmem, sw64_desc(sa + 32 * (it & 1)), sw64_desc(sb + 32 * (it & 1)),
                 idesc_mxf4(128, 256, 2 * (it & 1), 2 * (it & 1)), tmem + kSfaCol, tmem + kSfbCol, it > 0 ? 1u : 0u);
    }
    mma_commit(&bar);
  }
  __syncwarp();
  mbar_wait(&bar, 0, &g_rate_error, 1);
  tc_fence_after();
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t measure_tc_rate(int kind, int iters, int num_sms, cudaStream_t st, double* tflops, int* timed_out) {
  cudaError_t e = cudaFuncSetAttribute(tc_rate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kRateSmem);
  if (e != cudaSuccess) return e;
  cudaEvent_t a = nullptr, b = nullptr;
  if ((e = cudaEventCreate(&a)) != cudaSuccess) return e;
  if ((e = cudaEventCreate(&b)) != cudaSuccess) {
    cudaEventDestroy(a);
    return e;
  }
  float best = 0.f;
  for (int r = 0; r < 3 && e == cudaSuccess; ++r) {  // the best of three launches
    cudaEventRecord(a, st);
    tc_rate_kernel<<<num_sms, kRateThreads, kRateSmem, st>>>(kind, iters);
    note_launch();
    e = cudaGetLastError();
    cudaEventRecord(b, st);
    if (e == cudaSuccess) e = cudaEventSynchronize(b);
    float ms = 0.f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, a, b);
    if (e == cudaSuccess && ms > 0.f) {
      const double k = kind == 0 ? 16.0 : kind == 1 ? 32.0 : 64.0;
      const double tf = 2.0 * 128 * 256 * k * iters * num_sms / (ms * 1e-3) / 1e12;
      best = (float)std::max((double)best, tf);
    }
  }
  cudaEventDestroy(a);
  cudaEventDestroy(b);
  if (e != cudaSuccess) return e;
  int code = 0;
  const int zero = 0;
  if ((e = cudaMemcpyFromSymbol(&code, g_rate_error, sizeof(int))) != cudaSuccess) return e;
  if (code && (e = cudaMemcpyToSymbol(g_rate_error, &zero, sizeof(int))) != cudaSuccess) return e;
  *timed_out = code != 0;
  *tflops = best;
  return cudaSuccess;
}

}  // namespace csa2
