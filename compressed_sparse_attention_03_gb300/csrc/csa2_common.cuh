// Device helpers shared by the CSA2 kernels: FP4 (E2M1 + UE8M0/32) and FP8 (E4M3fn)
// codecs, RoPE angles, bf16 loads and block reductions.  Formats follow "Inside DeepSeek
// V4.1", section "890 bytes" (FP4 entries with 8-bit scales, FP8 window) with the scale
// rule fixed by this library (one UE8M0 per 32 values, OCP MX choice of exponent).
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "csa2_internal.h"

namespace csa2 {

// Programmatic dependent launch.  A kernel launched with launch_dependent may be scheduled
// while the kernel before it on the stream is still running; it calls grid_dep_wait() before
// its first access to global memory, which returns once that kernel has completed and its
// writes are visible (at once after a normal launch).  grid_dep_trigger() lets the next
// kernel's blocks be scheduled from then on.  Only the launch and block scheduling overlap:
// no memory access moves ahead of the previous kernel's end.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void grid_dep_trigger() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                             Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

__host__ __device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
__host__ __device__ __forceinline__ int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// E2M1 code (4 bits) -> value.  1 sign, 2 exponent (bias 1), 1 mantissa; exponent 0 is
// subnormal.  Written as arithmetic on the fields.
__device__ __forceinline__ float e2m1_to_f32(uint32_t c) {
  uint32_t e = (c >> 1) & 3, m = c & 1;
  float mag = e == 0 ? 0.5f * (float)m : __uint_as_float((e + 126u) << 23) * (1.0f + 0.5f * (float)m);
  return (c & 8) ? -mag : mag;
}

// Scaled value x (already divided by the block scale) -> E2M1 code, round to nearest with
// ties to the even code (mantissa bit 0), saturating at 6.  The decision points are the
// midpoints 0.25 0.75 1.25 1.75 2.5 3.5 5; at a midpoint the even neighbour wins, which is
// the lower one at 0.25 1.25 2.5 5 (codes 0 2 4 6) and the upper one at 0.75 1.75 3.5.
__device__ __forceinline__ uint32_t f32_to_e2m1(float x) {
  uint32_t s = (__float_as_uint(x) >> 28) & 8u;
  float a = fabsf(x);
  uint32_t m = (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) + (a > 2.5f) + (a >= 3.5f) + (a > 5.0f);
  return s | m;
}

// Order-preserving map of a float score to uint32 (larger score -> larger key, -0 == +0).
__device__ __forceinline__ uint32_t score_key(float x) {
  uint32_t u = __float_as_uint(x);
  if ((u << 1) == 0) u = 0;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_score(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Score histograms for the top-k: a bin is the top kHistBits bits of a score key (sign, the 8
// exponent bits and 2 mantissa bits), so a bin spans at most a factor 1.25 of |score|.
constexpr int kHistBits = 11, kHistBins = 1 << kHistBits, kHistShift = 32 - kHistBits;

// 2^k as a float built from its bits: exact for -149 <= k <= 127 (subnormal below -126).
__device__ __forceinline__ float pow2f(int k) {
  if (k > 127) return __uint_as_float(0x7f800000u);
  if (k >= -126) return __uint_as_float((uint32_t)(k + 127) << 23);
  if (k >= -149) return __uint_as_float(1u << (k + 149));
  return 0.f;
}

// UE8M0 exponent for a block with absolute maximum amax: floor(log2 amax) - 2, clamped to
// [-127, 127]; amax == 0 (or subnormal) gives -127.
__device__ __forceinline__ int mx_scale_exp(float amax) {
  int E = (int)((__float_as_uint(amax) >> 23) & 255u);
  if (E == 0) return -127;
  return max(-127, E - 127 - 2);
}

// E4M3fn: value = (E + 6) * 8 + q form.  Round to nearest even within the binade of `a`
// (subnormals share the step of the lowest binade), saturate to 448 (code 0x7E).
__device__ __forceinline__ uint32_t f32_to_e4m3(float v) {
  uint32_t s = (__float_as_uint(v) >> 24) & 0x80u;
  float a = fabsf(v);
  if (a != a) return 0x7Fu;
  if (!(a < 448.0f)) return s | 0x7Eu;
  int E = (int)((__float_as_uint(a) >> 23) & 255u) - 127;  // floor(log2 a) for normal a
  E = max(E, -6);
  float q = rintf(ldexpf(a, 3 - E));  // exact scaling, then round half to even
  return s | (uint32_t)((E + 6) * 8 + (int)q);
}

__device__ __forceinline__ float e4m3_to_f32(uint32_t c) {
  uint32_t e = (c >> 3) & 15, m = c & 7;
  float mag = e == 0 ? ldexpf((float)m, -9) : ldexpf(1.0f + 0.125f * (float)m, (int)e - 7);
  return (c & 0x80) ? -mag : mag;
}

// cos/sin of pos * inv_freq: the angle is formed and reduced modulo 2*pi in fp64 (positions
// reach ~2^21, where an fp32 product would be off by ~0.1 rad) and evaluated in fp32 at the
// rounded angle rf, then corrected to first order for d = r - rf (|d| <= 2e-7):
// cos(r) ~ cos(rf) - d sin(rf), sin(r) ~ sin(rf) + d cos(rf).
__device__ __forceinline__ void rope_cs(int64_t pos, double inv_freq, float sign, float& c, float& s) {
  const double two_pi_hi = 6.283185307179586;          // nearest double to 2*pi
  const double two_pi_lo = 2.4492935982947064e-16;     // 2*pi - two_pi_hi
  double ang = (double)pos * inv_freq;
  double k = rint(ang * 0.15915494309189535);
  double r = fma(-k, two_pi_hi, ang);
  r = fma(-k, two_pi_lo, r);
  r *= (double)sign;
  const float rf = (float)r;
  const float d = (float)(r - (double)rf);
  float s0, c0;
  sincosf(rf, &s0, &c0);
  c = fmaf(-d, s0, c0);
  s = fmaf(d, c0, s0);
}

// Double-float (s + c) accumulation in fp32: error-free two-sum of each addend, so that a
// sum of squares keeps ~2^-44 relative accuracy without fp64 arithmetic (slow on this GPU).
struct DFSum {
  float s = 0.f, c = 0.f;
  __device__ __forceinline__ void add(float x) {
    const float t = s + x;
    const float bb = t - s;
    c += (s - (t - bb)) + (x - bb);
    s = t;
  }
  __device__ __forceinline__ void add_sq(float x) {  // x * x exactly (product + fma error)
    const float p = x * x;
    add(p);
    c += fmaf(x, x, -p);
  }
  __device__ __forceinline__ void add(const DFSum& o) {
    add(o.s);
    c += o.c;
  }
  __device__ __forceinline__ float value() const { return s + c; }
};

__device__ __forceinline__ DFSum warp_sum_df(DFSum v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    DFSum p;
    p.s = __shfl_xor_sync(0xffffffffu, v.s, o);
    p.c = __shfl_xor_sync(0xffffffffu, v.c, o);
    v.add(p);
  }
  return v;
}

// 1 / sqrt(ss / n + eps) in fp32 with correctly rounded division and square root.
__device__ __forceinline__ float rms_inv(float ss, float n, double eps) {
  return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, n), (float)eps)));
}

// Two independent fp32 FMAs (a.x * b.x + c.x, a.y * b.y + c.y), each rounded to nearest, as one
// packed instruction: the same results as two fmaf calls.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;\n"
      : "=l"(r)
      : "l"(*reinterpret_cast<const uint64_t*>(&a)), "l"(*reinterpret_cast<const uint64_t*>(&b)),
        "l"(*reinterpret_cast<const uint64_t*>(&c)));
  return *reinterpret_cast<const float2*>(&r);
}

template <typename T>
__device__ __forceinline__ T warp_sum(T v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Sum over a block of NT threads (NT multiple of 32, <= 1024).  `red` holds NT/32 values.
template <int NT, typename T>
__device__ __forceinline__ T block_sum(T v, T* red) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  T t = 0;
#pragma unroll
  for (int i = 0; i < NT / 32; ++i) t += red[i];
  return t;
}

}  // namespace csa2
