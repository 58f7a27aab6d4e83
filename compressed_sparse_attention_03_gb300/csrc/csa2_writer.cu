// Compressed-KV writer.  Page "DeepSeek V4.1 - Pooled group / Source layer, pairs pooled",
// block "Compressed sparse attention": k^p_j (pair softmax pooling), c (RMSNorm, gain
// gamma_C), Z (RoPE by 2j on dims 448..511, FP4), k^i = c W_IK, k^n (RMSNorm, gamma_IK),
// K^I (RoPE by 2j on dims 64..127, FP4) and the window W (RMSNorm of w^a, RoPE by t, FP8).
// RMSNorm as on "DeepSeek V4.1 - Window layer / Attention RMSNorm" (eps 1e-20).
//
// Precision: fp32 elementwise work, compensated (double-float fp32) sums of squares and a
// compensated dot product for c W_IK (fp32 FMA chains of kChain terms, each folded into a
// double-float sum), so that the values reaching the FP4/FP8 rounding differ from an fp64
// evaluation by about 1e-7 of the row's rms and the codes match except at rounding midpoints.
#include "csa2_common.cuh"
#include "csa2_sm100.cuh"

namespace csa2 {
namespace {

constexpr int kWriterThreads = 128;       // window kernel: one token per block
constexpr int kEntryThreads = 512;        // entries kernel: four groups of 128
constexpr int kEntriesPerBlock = 4;       // one per group
// Products of c W_IK summed in plain fp32 before joining the double-float sum: a chain of 16
// terms of size ~|c||w| carries a rounding error of a few 1e-8 of the result's rms.
constexpr int kChain = 16;

// Pack the four 4-bit codes of one thread (4 consecutive values) into two bytes.
__device__ __forceinline__ uint16_t pack4(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3) {
  return (uint16_t)(c0 | (c1 << 4) | (c2 << 8) | (c3 << 12));
}

// Blocks of 32 values held 4 per thread by 8 consecutive lanes: returns the 4 codes packed
// and writes the block's scale byte from the first of the 8 lanes.
__device__ __forceinline__ uint16_t fp4_quant4(const float v[4], uint8_t* scale_out) {
  float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
  int e = mx_scale_exp(amax);
  if ((threadIdx.x & 7) == 0) *scale_out = (uint8_t)(e + 127);
  const float s = pow2f(-e);  // exact: -e is in [-125, 127]
  return pack4(f32_to_e2m1(v[0] * s), f32_to_e2m1(v[1] * s), f32_to_e2m1(v[2] * s), f32_to_e2m1(v[3] * s));
}

// Double-float accumulation of sum(x*w): error-free product (fma) and two-sum.
struct DF {
  float s, c;
  __device__ __forceinline__ void add(float p) {  // two-sum
    float t = s + p;
    float bb = t - s;
    c += (s - (t - bb)) + (p - bb);
    s = t;
  }
  __device__ __forceinline__ void add_prod(float x, float w) {
    float p = x * w;
    float pe = fmaf(x, w, -p);
    float t = s + p;
    float bb = t - s;
    float te = (s - (t - bb)) + (p - bb);
    s = t;
    c += te + pe;
  }
};

// Double-float sum over the 128 threads of group g (four whole warps), on named barrier 1 + g.
__device__ __forceinline__ float group_sum(DFSum v, float2* red, int g) {
  v = warp_sum_df(v);
  const int wg = (threadIdx.x >> 5) & 3;
  sm100::named_bar_sync(1 + g, 128);  // earlier readers of red[] are done
  if ((threadIdx.x & 31) == 0) red[wg] = make_float2(v.s, v.c);
  sm100::named_bar_sync(1 + g, 128);
  DFSum t;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    t.add(red[i].x);
    t.c += red[i].y;
  }
  return t.value();
}

// grid (entry groups of 4, sequences), 512 threads.  Group g = tid / 128 pools, normalises and
// quantises entry g (thread = 4 channels); the k^i = c W_IK products are split over the
// groups by K quarter (thread = output column), each a double-float partial, combined in
// phase 3 where group g again owns entry g (thread = output column).  NE = 1: launches where
// no sequence gains more than one entry (decode); the thread's weights then load in two
// batches of 64, so that their latency is paid twice rather than eight times.
template <int NE>
__global__ void __launch_bounds__(kEntryThreads) writer_entries_kernel(WriterArgs a, SeqPos pos, int b0, RopeFreq rf) {
  __shared__ float sc[kEntriesPerBlock][kD];
  __shared__ float2 part[4][kEntriesPerBlock][kDI];  // (s, c) of each K quarter
  __shared__ float2 red[kEntriesPerBlock][4];

  grid_dep_trigger();  // the window kernel may be scheduled now (it waits for this one's end)
  const int bl = blockIdx.y;
  const int b = b0 + bl;
  const int64_t p0 = seq_p0(pos, bl);
  const int T = a.T;
  const int rs = a.rshift;
  const int64_t n_new = ((p0 + T) >> rs) - (p0 >> rs);
  const int64_t e_base = (int64_t)blockIdx.x * kEntriesPerBlock;
  if (e_base >= n_new) return;
  const int ne = (int)min64(kEntriesPerBlock, n_new - e_base);
  const int tid = threadIdx.x, g = tid >> 7, gt = tid & 127;
  const int ch = 4 * gt;
  const int64_t j = (p0 >> rs) + e_base + g;  // this group's entry (valid when g < ne)
  const int64_t jpos = j << rs;                // the position the entry is rotated by

  // ---- phase 1: pooled key, RMSNorm, Z (the branch is uniform over a group)
  if (g < ne) {
    const int64_t t1 = jpos + (1 << rs) - 1 - p0;  // local index of the entry's last token
    const uint16_t* k1p = a.kc + ((int64_t)b * T + t1) * kD + ch;
    const uint16_t* g1p = a.gc + ((int64_t)b * T + t1) * kD + ch;
    float k0[4], g0[4], k1[4], g1[4];
    uint2 kk1 = *reinterpret_cast<const uint2*>(k1p), gg1 = *reinterpret_cast<const uint2*>(g1p);
    k1[0] = bf16_to_f32(kk1.x & 0xffff); k1[1] = bf16_to_f32(kk1.x >> 16);
    k1[2] = bf16_to_f32(kk1.y & 0xffff); k1[3] = bf16_to_f32(kk1.y >> 16);
    g1[0] = bf16_to_f32(gg1.x & 0xffff); g1[1] = bf16_to_f32(gg1.x >> 16);
    g1[2] = bf16_to_f32(gg1.y & 0xffff); g1[3] = bf16_to_f32(gg1.y >> 16);
    if (rs == 0) {  // ratio 1: the entry is the token itself (a softmax over one token is 1)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        k0[i] = 0.f;
        g0[i] = -INFINITY;
      }
    } else if (t1 >= 1) {
      uint2 kk0 = *reinterpret_cast<const uint2*>(k1p - kD), gg0 = *reinterpret_cast<const uint2*>(g1p - kD);
      k0[0] = bf16_to_f32(kk0.x & 0xffff); k0[1] = bf16_to_f32(kk0.x >> 16);
      k0[2] = bf16_to_f32(kk0.y & 0xffff); k0[3] = bf16_to_f32(kk0.y >> 16);
      g0[0] = bf16_to_f32(gg0.x & 0xffff); g0[1] = bf16_to_f32(gg0.x >> 16);
      g0[2] = bf16_to_f32(gg0.y & 0xffff); g0[3] = bf16_to_f32(gg0.y >> 16);
    } else {  // token 2j is the one the pair buffer kept from the previous call
      float4 kb = *reinterpret_cast<const float4*>(a.pair_kc + (int64_t)b * kD + ch);
      float4 gb = *reinterpret_cast<const float4*>(a.pair_gc + (int64_t)b * kD + ch);
      k0[0] = kb.x; k0[1] = kb.y; k0[2] = kb.z; k0[3] = kb.w;
      g0[0] = gb.x; g0[1] = gb.y; g0[2] = gb.z; g0[3] = gb.w;
    }
    float kp[4];
    DFSum ssq;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (rs == 0) {
        kp[i] = k1[i];
      } else {
        float m = fmaxf(g0[i], g1[i]);
        float e0 = expf(g0[i] - m), e1 = expf(g1[i] - m);
        float den = e0 + e1;
        kp[i] = (e0 / den) * k0[i] + (e1 / den) * k1[i];
      }
      ssq.add_sq(kp[i]);
    }
    const float r = rms_inv(group_sum(ssq, red[g], g), (float)kD, a.eps);
    float c[4], z[4];
    float4 gm = *reinterpret_cast<const float4*>(a.gamma_c + ch);
    c[0] = gm.x * (kp[0] * r); c[1] = gm.y * (kp[1] * r);
    c[2] = gm.z * (kp[2] * r); c[3] = gm.w * (kp[3] * r);
    *reinterpret_cast<float4*>(&sc[g][ch]) = make_float4(c[0], c[1], c[2], c[3]);
#pragma unroll
    for (int i = 0; i < 4; ++i) z[i] = c[i];
    if (ch >= kD - kDR) {
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int pi = (ch - (kD - kDR)) / 2 + q;
        float cs, sn;
        rope_cs(jpos, rf.inv_freq[pi], 1.0f, cs, sn);
        float x0 = c[2 * q], x1 = c[2 * q + 1];
        z[2 * q] = x0 * cs - x1 * sn;
        z[2 * q + 1] = x0 * sn + x1 * cs;
      }
    }
    uint16_t packed = fp4_quant4(z, a.z_scales + ((int64_t)b * a.cap + j) * 16 + gt / 8);
    *reinterpret_cast<uint16_t*>(a.z_codes + ((int64_t)b * a.cap + j) * 256 + 2 * gt) = packed;
  } else {
    *reinterpret_cast<float4*>(&sc[g][ch]) = make_float4(0.f, 0.f, 0.f, 0.f);  // no entry: zero row
  }
  __syncthreads();

  // ---- phase 2: quarter g of k^i = c W_IK for the block's entries (thread = output column)
  if constexpr (NE == 1) {
    const int o = gt;
    DF acc{0.f, 0.f};
#pragma unroll
    for (int hb = 0; hb < 2; ++hb) {
      const int d0 = 128 * g + 64 * hb;
      float w[64];
#pragma unroll
      for (int u = 0; u < 64; ++u) w[u] = bf16_to_f32(__ldg(a.w_ik + (d0 + u) * kDI + o));
#pragma unroll
      for (int c = 0; c < 64; c += kChain) {  // the same chains, in the same order, as below
        float s = 0.f;
#pragma unroll
        for (int u = 0; u < kChain; u += 4) {
          const float4 x = *reinterpret_cast<const float4*>(&sc[0][d0 + c + u]);
          s = fmaf(x.x, w[c + u], s);
          s = fmaf(x.y, w[c + u + 1], s);
          s = fmaf(x.z, w[c + u + 2], s);
          s = fmaf(x.w, w[c + u + 3], s);
        }
        acc.add(s);
      }
    }
    part[g][0][o] = make_float2(acc.s, acc.c);
  } else {
    const int o = gt;
    const int nacc = ne == 1 ? 1 : kEntriesPerBlock;  // one entry skips the empty rows
    DF acc[kEntriesPerBlock];
#pragma unroll
    for (int e = 0; e < kEntriesPerBlock; ++e) acc[e] = DF{0.f, 0.f};
    for (int d0 = 128 * g; d0 < 128 * g + 128; d0 += kChain) {
      float w[kChain];
#pragma unroll
      for (int u = 0; u < kChain; ++u) w[u] = bf16_to_f32(__ldg(a.w_ik + (d0 + u) * kDI + o));
#pragma unroll
      for (int e = 0; e < kEntriesPerBlock; ++e) {
        if (e < nacc) {
          float s = 0.f;
#pragma unroll
          for (int u = 0; u < kChain; u += 4) {
            const float4 x = *reinterpret_cast<const float4*>(&sc[e][d0 + u]);
            s = fmaf(x.x, w[u], s);
            s = fmaf(x.y, w[u + 1], s);
            s = fmaf(x.z, w[u + 2], s);
            s = fmaf(x.w, w[u + 3], s);
          }
          acc[e].add(s);
        }
      }
    }
#pragma unroll
    for (int e = 0; e < kEntriesPerBlock; ++e)
      if (e < nacc) part[g][e][o] = make_float2(acc[e].s, acc[e].c);
  }
  __syncthreads();

  // ---- phase 3: RMSNorm, RoPE by 2j on dims 64..127, FP4 for entry g (thread = output column)
  if (g < ne) {
    const int o = gt;
    DF t{0.f, 0.f};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      t.add_prod(part[q][g][o].x, 1.f);
      t.add_prod(part[q][g][o].y, 1.f);
    }
    const float ki = t.s + t.c;
    DFSum ssq;
    ssq.add_sq(ki);
    const float r = rms_inv(group_sum(ssq, red[g], g), (float)kDI, a.eps);
    float kn = a.gamma_ik[o] * (ki * r);
    const float partner = __shfl_xor_sync(0xffffffffu, kn, 1);
    if (o >= 64) {
      float cs, sn;
      rope_cs(jpos, rf.inv_freq[(o - 64) / 2], 1.0f, cs, sn);
      kn = (o & 1) ? (partner * sn + kn * cs) : (kn * cs - partner * sn);
    }
    const float amax = warp_max(fabsf(kn));
    const int ex = mx_scale_exp(amax);
    const uint32_t code = f32_to_e2m1(kn * pow2f(-ex));
    const uint32_t hi = __shfl_xor_sync(0xffffffffu, code, 1);
    if ((o & 1) == 0) a.ki_codes[((int64_t)b * a.cap + j) * 64 + o / 2] = (uint8_t)(code | (hi << 4));
    if ((o & 31) == 0) a.ki_scales[((int64_t)b * a.cap + j) * 4 + o / 32] = (uint8_t)(ex + 127);
  }
}

__global__ void __launch_bounds__(kWriterThreads) writer_window_kernel(WriterArgs a, SeqPos pos, int b0, RopeFreq rf) {
  __shared__ float2 red[kWriterThreads / 32];
  __shared__ float r_sh;
  grid_dep_wait();  // launched dependent on the entry kernel (which reads the pair buffer)
  const int t = blockIdx.x;
  const int bl = blockIdx.y;
  const int b = b0 + bl;
  const int64_t p0 = seq_p0(pos, bl);
  const int T = a.T;
  const int tid = threadIdx.x;
  const int ch = 4 * tid;
  const int64_t row = (int64_t)b * T + t;
  uint2 ww = *reinterpret_cast<const uint2*>(a.wa + row * kD + ch);
  float x[4] = {bf16_to_f32(ww.x & 0xffff), bf16_to_f32(ww.x >> 16), bf16_to_f32(ww.y & 0xffff),
                bf16_to_f32(ww.y >> 16)};
  DFSum ssq;
#pragma unroll
  for (int i = 0; i < 4; ++i) ssq.add_sq(x[i]);
  ssq = warp_sum_df(ssq);
  if ((tid & 31) == 0) red[tid >> 5] = make_float2(ssq.s, ssq.c);
  __syncthreads();
  if (tid == 0) {
    DFSum tot;
#pragma unroll
    for (int i = 0; i < kWriterThreads / 32; ++i) {
      tot.add(red[i].x);
      tot.c += red[i].y;
    }
    r_sh = rms_inv(tot.value(), (float)kD, a.eps);
  }
  __syncthreads();
  const float r = r_sh;
  float4 gm = *reinterpret_cast<const float4*>(a.gamma_w + ch);
  float y[4] = {gm.x * (x[0] * r), gm.y * (x[1] * r), gm.z * (x[2] * r), gm.w * (x[3] * r)};
  if (ch >= kD - kDR) {
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      float cs, sn;
      rope_cs(p0 + t, rf.inv_freq[(ch - (kD - kDR)) / 2 + q], 1.0f, cs, sn);
      float x0 = y[2 * q], x1 = y[2 * q + 1];
      y[2 * q] = x0 * cs - x1 * sn;
      y[2 * q + 1] = x0 * sn + x1 * cs;
    }
  }
  uint32_t packed = f32_to_e4m3(y[0]) | (f32_to_e4m3(y[1]) << 8) | (f32_to_e4m3(y[2]) << 16) | (f32_to_e4m3(y[3]) << 24);
  *reinterpret_cast<uint32_t*>(a.window + ((int64_t)b * (127 + T) + 127 + t) * kD + ch) = packed;
  // the last token of an unfinished pair waits in the pair buffer for its partner (ratio 2)
  if (a.rshift == 1 && t == T - 1 && ((p0 + T) & 1)) {
    uint2 kk = *reinterpret_cast<const uint2*>(a.kc + row * kD + ch);
    uint2 gg = *reinterpret_cast<const uint2*>(a.gc + row * kD + ch);
    *reinterpret_cast<float4*>(a.pair_kc + (int64_t)b * kD + ch) =
        make_float4(bf16_to_f32(kk.x & 0xffff), bf16_to_f32(kk.x >> 16), bf16_to_f32(kk.y & 0xffff), bf16_to_f32(kk.y >> 16));
    *reinterpret_cast<float4*>(a.pair_gc + (int64_t)b * kD + ch) =
        make_float4(bf16_to_f32(gg.x & 0xffff), bf16_to_f32(gg.x >> 16), bf16_to_f32(gg.y & 0xffff), bf16_to_f32(gg.y >> 16));
  }
}

// Window roll between calls ([PG] paragraph "Between forward calls": the window keeps the last
// 128 positions).  Row r of the next call's view holds position p0 + T - 127 + r, which is row
// T + r of this call's view: rows T .. T+126 move to rows 0 .. 126.  One block per sequence
// loads all of its 127 rows (65,024 bytes, 16 per thread and load) before storing any, so a
// sequence's rows may move within one buffer.
constexpr int kRollThreads = 512;
constexpr int kRollVec = 127 * kD / 16;
constexpr int kRollPer = (kRollVec + kRollThreads - 1) / kRollThreads;

__global__ void __launch_bounds__(kRollThreads) roll_window_kernel(const uint8_t* window, int T, uint8_t* next,
                                                                   int T_next) {
  const int b = blockIdx.x;
  const uint4* src = reinterpret_cast<const uint4*>(window + ((int64_t)b * (127 + T) + T) * kD);
  uint4* dst = reinterpret_cast<uint4*>(next + (int64_t)b * (127 + T_next) * kD);
  uint4 v[kRollPer];
#pragma unroll
  for (int k = 0; k < kRollPer; ++k) {
    const int i = threadIdx.x + k * kRollThreads;
    if (i < kRollVec) v[k] = src[i];
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < kRollPer; ++k) {
    const int i = threadIdx.x + k * kRollThreads;
    if (i < kRollVec) dst[i] = v[k];
  }
}

}  // namespace

cudaError_t launch_roll_window(const uint8_t* window, int B, int T, uint8_t* next, int T_next, cudaStream_t st) {
  roll_window_kernel<<<(unsigned)B, kRollThreads, 0, st>>>(window, T, next, T_next);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_writer(const WriterArgs& a, const SeqPos& pos, int b0, int nb, const RopeFreq& rf, cudaStream_t st) {
  // new entries per sequence: from the positions, or (positions read on the device) the most any
  // position can give, T at ratio 1 and ceil(T / 2) at ratio 2; each block checks its own count
  int64_t max_new = 0;
  if (pos.dev)
    max_new = a.rshift ? (a.T + 1) >> 1 : a.T;
  else
    for (int i = 0; i < nb; ++i) max_new = max(max_new, ((pos.p0[i] + a.T) >> a.rshift) - (pos.p0[i] >> a.rshift));
  if (max_new > 0) {
    dim3 grid((unsigned)((max_new + kEntriesPerBlock - 1) / kEntriesPerBlock), (unsigned)nb);
    if (max_new == 1)
      writer_entries_kernel<1><<<grid, kEntryThreads, 0, st>>>(a, pos, b0, rf);
    else
      writer_entries_kernel<kEntriesPerBlock><<<grid, kEntryThreads, 0, st>>>(a, pos, b0, rf);
    note_launch();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = launch_dependent(writer_window_kernel, dim3((unsigned)a.T, (unsigned)nb), dim3(kWriterThreads), 0, st, a,
                                   pos, b0, rf);
  note_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace csa2
