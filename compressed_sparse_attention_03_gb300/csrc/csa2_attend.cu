// Sink-softmax MQA over the gathered rows.  Page "DeepSeek V4.1 - Pooled group / Source
// layer, pairs pooled", block "Compressed sparse attention": J^w_t = {max(0,t-127)..t},
// Y = [W; Z], J = [J^w; I + |W|], G_t = Y[J_t], S = Q.G/sqrt(512),
// A = exp S / (exp s_h + sum exp S), O = sum A G, O-bar_{448:} = R_t^{-1} O_{448:}.
// "Inside DeepSeek V4.1", section "Attention that looks at 640 places": 64 heads x 512, one
// shared key/value row per place, a learned sink per head, 640 = 128 + 512 places.
//
// Kernel shape: one block per (query, row split).  Rows are gathered 32 at a time, decoded
// exactly to bf16 in shared memory (E2M1 x 2^k and E4M3 are exact in bf16), and multiplied
// with bf16 tensor-core MMAs (fp32 accumulation); the softmax is online over the chunks.
// Decode (few queries) splits the rows across blocks and merges in a combine kernel.
#include "csa2_common.cuh"

namespace csa2 {
namespace {

constexpr int kAttThreads = 256;       // 8 warps
constexpr int kChunk = 32;             // rows per gathered chunk
constexpr int kQStride = kD + 8;       // padded smem row (bf16 elements)
constexpr int kPStride = kChunk + 8;
constexpr int kMaxRows = kWin + kTopK; // 640
constexpr float kLog2e = 1.4426950408889634f;

struct AttSmem {
  __nv_bfloat16 q[kH][kQStride];
  __nv_bfloat16 g[kChunk][kQStride];
  __nv_bfloat16 p[kH][kPStride];
  float s[kH][kChunk + 1];
  float m[kH], l[kH], alpha[kH];
  int32_t rows[kMaxRows];
  uint16_t lut8[256];  // e4m3 code -> bf16 bits
  int nrows, nwin;
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
               : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float x) {
  __nv_bfloat16 v = __float2bfloat16_rn(x);
  return *reinterpret_cast<uint16_t*>(&v);
}

// grid (T, nb, nsplit).  nsplit == 1: writes out.  Otherwise writes the split's unnormalised
// O, running max m (log2 units) and sum l to the workspace for attend_combine_kernel.
__global__ void __launch_bounds__(kAttThreads, 1) attend_kernel(AttendArgs a, SeqPos pos, int b0, RopeFreq rf, int nsplit,
                                                                int rows_per_split, float* part_o, float* part_ml) {
  extern __shared__ __align__(16) unsigned char smraw[];
  AttSmem& sm = *reinterpret_cast<AttSmem*>(smraw);
  const int t = blockIdx.x, bl = blockIdx.y, split = blockIdx.z;
  const int b = b0 + bl;
  const int T = a.T;
  const int64_t p0 = pos.p0[bl];
  const int64_t p = p0 + t;
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const int64_t qrow = (int64_t)b * T + t;

  // ---- row list: window rows (view row index) then the selected Z entries
  for (int i = tid; i < 256; i += kAttThreads) sm.lut8[i] = f32_to_bf16_bits(e4m3_to_f32((uint32_t)i));
  if (tid < 32) {
    const int nw = (int)min64(kWin, p + 1);
    const int32_t* ip = a.idx + qrow * kTopK;
    int base = nw;
    for (int r0 = 0; r0 < kTopK; r0 += 32) {
      const int32_t j = ip[r0 + lane];
      const bool ok = j >= 0 && j < a.cap;  // out-of-range indices are skipped
      const uint32_t bal = __ballot_sync(0xffffffffu, ok);
      if (ok) sm.rows[base + __popc(bal & ((1u << lane) - 1u))] = j;
      base += __popc(bal);
    }
    for (int i = lane; i < nw; i += 32) sm.rows[i] = t + 128 - nw + i;
    if (lane == 0) {
      sm.nrows = base;
      sm.nwin = nw;
    }
  }
  for (int i = tid; i < kH; i += kAttThreads) {
    sm.m[i] = -INFINITY;
    sm.l[i] = 0.f;
  }
  // ---- Q [64][512] bf16 -> smem
  {
    const uint4* qs = reinterpret_cast<const uint4*>(a.q + qrow * kH * kD);
    for (int i = tid; i < kH * kD / 8; i += kAttThreads) {
      const int h = i / (kD / 8), c = i % (kD / 8);
      *reinterpret_cast<uint4*>(&sm.q[h][c * 8]) = qs[i];
    }
  }
  __syncthreads();
  const int n = sm.nrows, nw = sm.nwin;
  const int r_begin = split * rows_per_split;
  const int r_end = min(n, r_begin + rows_per_split);

  const int hg = w & 3;       // head group of 16
  const int half = w >> 2;    // S: row half of the chunk; O: dim half
  const int g = lane >> 2, c4 = lane & 3;
  float o[32][4];
#pragma unroll
  for (int i = 0; i < 32; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  const float scale_log2 = rsqrtf((float)kD) * kLog2e;

  for (int r0 = r_begin; r0 < r_end; r0 += kChunk) {
    const int nchunk = min(kChunk, r_end - r0);
    // ---- gather + decode: thread -> (row tid/8, 64 dims)
    {
      const int rr = tid >> 3, seg = tid & 7;
      uint32_t outw[32];
      if (rr < nchunk) {
        const int ri = r0 + rr;
        if (ri < nw) {
          const uint4* src = reinterpret_cast<const uint4*>(a.window + ((int64_t)b * (127 + T) + sm.rows[ri]) * kD + 64 * seg);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4 x = src[v];
            const uint32_t wd[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              outw[8 * v + 2 * k] = (uint32_t)sm.lut8[wd[k] & 255] | ((uint32_t)sm.lut8[(wd[k] >> 8) & 255] << 16);
              outw[8 * v + 2 * k + 1] = (uint32_t)sm.lut8[(wd[k] >> 16) & 255] | ((uint32_t)sm.lut8[wd[k] >> 24] << 16);
            }
          }
        } else {
          const int64_t j = sm.rows[ri];
          const uint4* src = reinterpret_cast<const uint4*>(a.z_codes + ((int64_t)b * a.cap + j) * 256 + 32 * seg);
          const uint8_t* scp = a.z_scales + ((int64_t)b * a.cap + j) * 16 + 2 * seg;
#pragma unroll
          for (int v = 0; v < 2; ++v) {
            uint4 x = src[v];
            const float s = ldexpf(1.0f, (int)scp[v] - 127);
            const uint32_t wd[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int k = 0; k < 4; ++k)
#pragma unroll
              for (int q = 0; q < 4; ++q)
                outw[16 * v + 4 * k + q] = pack_bf16(e2m1_to_f32((wd[k] >> (8 * q)) & 15) * s,
                                                     e2m1_to_f32((wd[k] >> (8 * q + 4)) & 15) * s);
          }
        }
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) outw[i] = 0u;
      }
      uint4* dst = reinterpret_cast<uint4*>(&sm.g[rr][64 * seg]);
#pragma unroll
      for (int v = 0; v < 8; ++v) dst[v] = make_uint4(outw[4 * v], outw[4 * v + 1], outw[4 * v + 2], outw[4 * v + 3]);
    }
    __syncthreads();
    // ---- S = Q G^T for heads 16hg.., rows 16half..
    {
      float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      const int arow = 16 * hg + (lane & 7) + 8 * ((lane >> 3) & 1), acol = 8 * (lane >> 4);
      const int brow = 16 * half + (lane & 7) + 8 * (lane >> 4), bcol = 8 * ((lane >> 3) & 1);
#pragma unroll 4
      for (int kk = 0; kk < kD / 16; ++kk) {
        uint32_t a0, a1, a2, a3, b0r, b1r, b2r, b3r;
        ldsm_x4(smem_u32(&sm.q[arow][16 * kk + acol]), a0, a1, a2, a3);
        ldsm_x4(smem_u32(&sm.g[brow][16 * kk + bcol]), b0r, b1r, b2r, b3r);
        mma_bf16(s[0], a0, a1, a2, a3, b0r, b1r);
        mma_bf16(s[1], a0, a1, a2, a3, b2r, b3r);
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int h = 16 * hg + g + 8 * (q >> 1);
          const int r = 16 * half + 8 * nt + 2 * c4 + (q & 1);
          sm.s[h][r] = r < nchunk ? s[nt][q] * scale_log2 : -INFINITY;
        }
    }
    __syncthreads();
    // ---- online softmax statistics: 4 threads per head, 8 rows each
    {
      const int h = tid >> 2, qd = tid & 3;
      const float m_old = sm.m[h], l_old = sm.l[h];
      float v[8], cmax = -INFINITY;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        v[i] = sm.s[h][8 * qd + i];
        cmax = fmaxf(cmax, v[i]);
      }
      cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, 1));
      cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, 2));
      const float m_new = fmaxf(m_old, cmax);
      const float alpha = exp2f(m_old - m_new);
      float sum = 0.f;
      uint32_t pk[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 pb = __floats2bfloat162_rn(exp2f(v[2 * i] - m_new), exp2f(v[2 * i + 1] - m_new));
        const float2 pf = __bfloat1622float2(pb);
        sum += pf.x + pf.y;
        pk[i] = *reinterpret_cast<const uint32_t*>(&pb);
      }
      *reinterpret_cast<uint4*>(&sm.p[h][8 * qd]) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      sum += __shfl_xor_sync(0xffffffffu, sum, 1);
      sum += __shfl_xor_sync(0xffffffffu, sum, 2);
      __syncwarp();
      if (qd == 0) {
        sm.m[h] = m_new;
        sm.l[h] = l_old * alpha + sum;
        sm.alpha[h] = alpha;
      }
    }
    __syncthreads();
    // ---- O = alpha O + P G for heads 16hg.., dims 256half..
    {
      const float al0 = sm.alpha[16 * hg + g], al1 = sm.alpha[16 * hg + g + 8];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        o[i][0] *= al0; o[i][1] *= al0;
        o[i][2] *= al1; o[i][3] *= al1;
      }
      const int arow = 16 * hg + (lane & 7) + 8 * ((lane >> 3) & 1), acol = 8 * (lane >> 4);
      const int brow = (lane & 7) + 8 * ((lane >> 3) & 1), bcol = 8 * (lane >> 4);
#pragma unroll
      for (int kk = 0; kk < kChunk / 16; ++kk) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(smem_u32(&sm.p[arow][16 * kk + acol]), a0, a1, a2, a3);
#pragma unroll
        for (int np = 0; np < 16; ++np) {
          uint32_t b0r, b1r, b2r, b3r;
          ldsm_x4_t(smem_u32(&sm.g[16 * kk + brow][256 * half + 16 * np + bcol]), b0r, b1r, b2r, b3r);
          mma_bf16(o[2 * np], a0, a1, a2, a3, b0r, b1r);
          mma_bf16(o[2 * np + 1], a0, a1, a2, a3, b2r, b3r);
        }
      }
    }
    __syncthreads();
  }

  const int h0 = 16 * hg + g, h1 = h0 + 8;
  if (nsplit == 1) {
    const float den0 = sm.l[h0] + exp2f(a.sinks[h0] * kLog2e - sm.m[h0]);
    const float den1 = sm.l[h1] + exp2f(a.sinks[h1] * kLog2e - sm.m[h1]);
    const float inv0 = 1.f / den0, inv1 = 1.f / den1;
    uint16_t* out0 = a.out + (qrow * kH + h0) * kD;
    uint16_t* out1 = a.out + (qrow * kH + h1) * kD;
#pragma unroll
    for (int nt = 0; nt < 32; ++nt) {
      const int d = 256 * half + 8 * nt + 2 * c4;
      float x0 = o[nt][0] * inv0, x1 = o[nt][1] * inv0, y0 = o[nt][2] * inv1, y1 = o[nt][3] * inv1;
      if (d >= kD - kDR) {
        float cs, sn;
        rope_cs(p, rf.inv_freq[(d - (kD - kDR)) / 2], -1.0f, cs, sn);
        const float rx0 = x0 * cs - x1 * sn, rx1 = x0 * sn + x1 * cs;
        const float ry0 = y0 * cs - y1 * sn, ry1 = y0 * sn + y1 * cs;
        x0 = rx0; x1 = rx1; y0 = ry0; y1 = ry1;
      }
      *reinterpret_cast<uint32_t*>(out0 + d) = pack_bf16(x0, x1);
      *reinterpret_cast<uint32_t*>(out1 + d) = pack_bf16(y0, y1);
    }
  } else {
    const int64_t pr = ((int64_t)bl * T + t) * nsplit + split;
    float* po0 = part_o + (pr * kH + h0) * kD;
    float* po1 = part_o + (pr * kH + h1) * kD;
#pragma unroll
    for (int nt = 0; nt < 32; ++nt) {
      const int d = 256 * half + 8 * nt + 2 * c4;
      *reinterpret_cast<float2*>(po0 + d) = make_float2(o[nt][0], o[nt][1]);
      *reinterpret_cast<float2*>(po1 + d) = make_float2(o[nt][2], o[nt][3]);
    }
    if (tid < kH) {
      part_ml[(pr * kH + tid) * 2] = sm.m[tid];
      part_ml[(pr * kH + tid) * 2 + 1] = sm.l[tid];
    }
  }
}

// grid (T, nb, 64 heads), 128 threads x 4 dims.  Merges the split partials with the sink.
__global__ void __launch_bounds__(128) attend_combine_kernel(AttendArgs a, SeqPos pos, int b0, RopeFreq rf, int nsplit,
                                                             const float* part_o, const float* part_ml) {
  const int t = blockIdx.x, bl = blockIdx.y, h = blockIdx.z;
  const int b = b0 + bl;
  const int64_t qrow = (int64_t)b * a.T + t;
  const int64_t lrow = (int64_t)bl * a.T + t;  // row within this launch's partials
  const int64_t p = pos.p0[bl] + t;
  float mstar = a.sinks[h] * kLog2e;
  for (int s = 0; s < nsplit; ++s) mstar = fmaxf(mstar, part_ml[((lrow * nsplit + s) * kH + h) * 2]);
  float den = exp2f(a.sinks[h] * kLog2e - mstar);
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  const int d = 4 * threadIdx.x;
  for (int s = 0; s < nsplit; ++s) {
    const int64_t pr = lrow * nsplit + s;
    const float ms = part_ml[(pr * kH + h) * 2], ls = part_ml[(pr * kH + h) * 2 + 1];
    if (ls == 0.f) continue;  // split without rows
    const float wgt = exp2f(ms - mstar);
    den += wgt * ls;
    const float4 v = *reinterpret_cast<const float4*>(part_o + (pr * kH + h) * kD + d);
    acc[0] += wgt * v.x; acc[1] += wgt * v.y; acc[2] += wgt * v.z; acc[3] += wgt * v.w;
  }
  const float inv = 1.f / den;
#pragma unroll
  for (int i = 0; i < 4; ++i) acc[i] *= inv;
  if (d >= kD - kDR) {
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      float cs, sn;
      rope_cs(p, rf.inv_freq[(d - (kD - kDR)) / 2 + q], -1.0f, cs, sn);
      const float x0 = acc[2 * q], x1 = acc[2 * q + 1];
      acc[2 * q] = x0 * cs - x1 * sn;
      acc[2 * q + 1] = x0 * sn + x1 * cs;
    }
  }
  uint2 packed = make_uint2(pack_bf16(acc[0], acc[1]), pack_bf16(acc[2], acc[3]));
  *reinterpret_cast<uint2*>(a.out + (qrow * kH + h) * kD + d) = packed;
}

int choose_splits(int nq, int num_sms) {
  if (nq >= num_sms) return 1;
  int s = (2 * num_sms + nq - 1) / nq;
  return max(1, min(s, kMaxRows / kChunk));
}

}  // namespace

size_t attend_workspace_bytes(int B, int T, int num_sms) {
  const int nb = min(B, kMaxSeqPerLaunch);
  const int s = choose_splits(nb * T, num_sms);
  if (s == 1) return 0;
  const size_t rows = (size_t)nb * T * s;
  return rows * kH * kD * 4 + rows * kH * 2 * 4;
}

cudaError_t launch_attend(const AttendArgs& a, const SeqPos& pos, int b0, int nb, const RopeFreq& rf, void* ws,
                          size_t ws_bytes, int num_sms, cudaStream_t st) {
  const int s = choose_splits(nb * a.T, num_sms);
  const size_t smem = sizeof(AttSmem);
  cudaError_t e = cudaFuncSetAttribute(attend_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int rps = kMaxRows;
  float *po = nullptr, *pml = nullptr;
  if (s > 1) {
    rps = ((kMaxRows / s + kChunk - 1) / kChunk) * kChunk;
    const size_t rows = (size_t)nb * a.T * s;
    if (ws_bytes < rows * kH * kD * 4 + rows * kH * 2 * 4) return cudaErrorInvalidValue;
    po = static_cast<float*>(ws);
    pml = po + rows * kH * kD;
  }
  attend_kernel<<<dim3((unsigned)a.T, (unsigned)nb, (unsigned)s), kAttThreads, smem, st>>>(a, pos, b0, rf, s, rps, po, pml);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (s > 1) {
    attend_combine_kernel<<<dim3((unsigned)a.T, (unsigned)nb, kH), 128, 0, st>>>(a, pos, b0, rf, s, po, pml);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace csa2
