// Sink-softmax MQA over the gathered rows, on the 5th-generation tensor cores (tcgen05).
// Page "DeepSeek V4.1 - Pooled group / Source layer, pairs pooled", block "Compressed sparse
// attention": J^w_t = {max(0,t-127)..t}, Y = [W; Z], J = [J^w; I + |W|], G_t = Y[J_t],
// S = Q.G/sqrt(512), A = exp S / (exp s_h + sum exp S), O = sum A G, O-bar_{448:} =
// R_t^{-1} O_{448:}.  "Inside DeepSeek V4.1", section "Attention that looks at 640 places":
// 64 heads x 512, one shared key/value row per place, a learned sink per head, 640 places.
//
// One block per (query, row split).  The gathered rows form chunks of 128 (at most 5), and
// G is decoded twice into a 4-slot ring of "atoms" (128 rows x 64 dims, fp16, 128B-swizzled):
//   pass 1  S^T_c[rows, heads] = G_c Q^T    M=128 rows, N=64 heads, K=512 (8 atoms, K-major)
//           into its own TMEM tile per chunk; the softmax turns each S tile into
//           P_c = exp2(S - m) (fp16, kept in smem for all chunks) while the next chunk's MMAs run
//   pass 2  O^T[dims, heads] += G_c^T P_c^T  M=128 dims, N=64, K=128 rows (atom pairs, MN-major)
//           for dims 0..255 over all chunks, then dims 256..511, plus l_h = sum_rows P
//           from a ones x P^T MMA (one 1 KB swizzle atom of ones, zero row-group stride).
// Operands are fp16: E2M1 x 2^e (scale exponents -22..12) and E4M3 values are exact in fp16
// and convert with one hardware instruction per pair; accumulation is fp32 in TMEM.
// Measured on GB300: a 128 x 64 x 16 fp16 MMA takes ~50 cycles and alternating accumulators
// costs more, so every accumulator receives its MMAs consecutively.
//
// Warp roles (416 threads):
//   warps 0-3   softmax + epilogue; thread = TMEM lane = row of S^T / dim of O^T
//   warps 4-11  producers: Q -> smem, then the atom sequence (pass 1: chunk-major, 8 atoms per
//               chunk; pass 2: dims 0..255 then 256..511), two threads per row and atom, raw
//               rows fetched 4 atoms ahead into registers
//   warp 12     TMEM allocation and the single MMA-issuing thread
// Online softmax with a lazy reference: a head's reference m only moves when a chunk's
// maximum exceeds it by more than kTau (log2 units), so P <= 2^kTau; when it moves, the
// earlier chunks' P (still in smem, before any O MMA) are rescaled.
#include <cuda_fp16.h>

#include "csa2_common.cuh"
#include "csa2_sm100.cuh"

namespace csa2 {
namespace {

using namespace sm100;

constexpr int kThreads = 416;
constexpr int kRows = 128;                  // rows per chunk
constexpr int kMaxRows = kWin + kTopK;      // 640
constexpr int kMaxChunks = kMaxRows / kRows;
constexpr int kSlots = 4;                   // G atom ring
constexpr int kAhead = 4;                   // raw atoms prefetched per producer thread
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kTau = 8.0f;                // lazy-rescale threshold (log2 units)
// dynamic shared memory (1024-aligned): Q 8 atoms x [64 heads x 128 B] (later: epilogue
// staging), P 5 chunks x [128 rows x 128 B], G ring 4 atoms x [128 rows x 128 B], ones 1 KB
constexpr uint32_t kQOff = 0, kPOff = 65536, kGOff = 147456, kOnesOff = 212992, kDynBytes = 214016 + 1024;
// TMEM columns: O^T dims 0..127 at 0, 128..255 at 64, row sums at 128, S^T chunk c at 192+64c;
// pass 2b puts O^T dims 256..383 / 384..511 into the S columns of chunks 0 / 1
constexpr uint32_t kTmemCols = 512, kLCol = 128, kSCol = 192;
constexpr int kStage = 68;                  // epilogue staging row (floats) in the Q region

__device__ int g_attend_error;

struct Bars {
  uint64_t q_full, p_all, o_lo, o_hi;
  uint64_t s_full[kMaxChunks];
  uint64_t atom_full[kSlots], atom_free[kSlots];
};

__device__ __forceinline__ uint32_t cvt_e2m1x2_f16x2(uint32_t byte) {
  uint32_t r;
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %1;\n cvt.rn.f16x2.e2m1x2 %0, b0;\n}\n" : "=r"(r) : "r"(byte));
  return r;
}
__device__ __forceinline__ uint32_t cvt_e4m3x2_f16x2(uint32_t two) {
  uint32_t r;
  asm("{\n .reg .b16 h0, h1;\n mov.b32 {h0, h1}, %1;\n cvt.rn.f16x2.e4m3x2 %0, h0;\n}\n" : "=r"(r) : "r"(two));
  return r;
}
__device__ __forceinline__ uint32_t hmul2(uint32_t x, uint32_t y) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;\n" : "=r"(r) : "r"(x), "r"(y));
  return r;
}
__device__ __forceinline__ uint32_t f2_to_h2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Reduce v[32] over the 32 lanes of the warp; lane l receives the result for entry l.
// Each round a lane keeps half of its entries and exchanges the other half.
template <bool kMax>
__device__ __forceinline__ float transpose_reduce32(const float (&v)[32], int lane) {
  auto op = [](float x, float y) { return kMax ? fmaxf(x, y) : x + y; };
  float a[16], b[8], c[4], d[2];
  bool up = lane & 16;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float send = up ? v[i] : v[16 + i], keep = up ? v[16 + i] : v[i];
    a[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 16));
  }
  up = lane & 8;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float send = up ? a[i] : a[8 + i], keep = up ? a[8 + i] : a[i];
    b[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 8));
  }
  up = lane & 4;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float send = up ? b[i] : b[4 + i], keep = up ? b[4 + i] : b[i];
    c[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 4));
  }
  up = lane & 2;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float send = up ? c[i] : c[2 + i], keep = up ? c[2 + i] : c[i];
    d[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 2));
  }
  up = lane & 1;
  const float send = up ? d[0] : d[1], keep = up ? d[1] : d[0];
  return op(keep, __shfl_xor_sync(0xffffffffu, send, 1));
}

// Atom `seq` of the sequence, in the order the MMAs consume them: pass 1 (seq < 8n) chunk
// seq/8, dims block seq%8; pass 2, for each 128-dim tile (blocks 2u, 2u+1, u = 0..3), the
// block pair of every chunk in turn.
struct AtomId {
  int chunk, blk;
};
__device__ __forceinline__ AtomId atom_of(int seq, int nloc) {
  if (seq < 8 * nloc) return {seq >> 3, seq & 7};
  const int s2 = seq - 8 * nloc, tile = s2 / (2 * nloc), w = s2 % (2 * nloc);
  return {w >> 1, 2 * tile + (w & 1)};
}

// grid (T, nb, nsplit).  nsplit == 1 writes `out`; otherwise the split's unnormalised O, its
// reference m (log2 units) and sum l go to the partial buffers for attend_combine_kernel.
__global__ void __launch_bounds__(kThreads, 1) attend_tc_kernel(AttendArgs a, SeqPos pos, int b0, RopeFreq rf,
                                                                int nsplit, int chunks_per_split, float* part_o,
                                                                float* part_ml) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ Bars bars;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int32_t rows[kMaxRows];
  __shared__ float red_max[4][64];
  __shared__ float m_ref[64], alpha_s[64], den_s[64], l_s[64];  // den_s: 1 / denominator
  __shared__ float2 rope_s[kDR / 2];                            // cos, sin of -t per rotated pair
  __shared__ int nrows_sh, nwin_sh;

  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  unsigned char* sm = smem_raw + (sbase - smem_u32(smem_raw));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t = blockIdx.x, bl = blockIdx.y, split = blockIdx.z;
  const int b = b0 + bl;
  const int T = a.T;
  const int64_t p = pos.p0[bl] + t;
  const int64_t qrow = (int64_t)b * T + t;
  int* err = &g_attend_error;

  // ---------------------------------------------------------------- setup
  if (warp == 0) {
    // all 512 indices in one round trip (16 per lane); the order of the gathered rows does not
    // matter to the result, so each lane appends its valid entries after a warp prefix sum
    const int nw = (int)min64(kWin, p + 1);
    const int4* ip = reinterpret_cast<const int4*>(a.idx + qrow * kTopK);
    int32_t jv[16];
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const int4 x = ip[v * 32 + lane];
      jv[4 * v] = x.x; jv[4 * v + 1] = x.y; jv[4 * v + 2] = x.z; jv[4 * v + 3] = x.w;
    }
    int cnt = 0;
#pragma unroll
    for (int k = 0; k < 16; ++k) cnt += (jv[k] >= 0 && jv[k] < a.cap) ? 1 : 0;  // out-of-range entries are skipped
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    int wpos = nw + incl - cnt;
#pragma unroll
    for (int k = 0; k < 16; ++k)
      if (jv[k] >= 0 && jv[k] < a.cap) rows[wpos++] = jv[k];
    const int base = nw + __shfl_sync(0xffffffffu, incl, 31);
    for (int i = lane; i < nw; i += 32) rows[i] = t + 128 - nw + i;  // window-view row of position p-nw+1+i
    if (lane == 0) {
      nrows_sh = base;
      nwin_sh = nw;
    }
  }
  if (warp == 1) {
    float cs, sn;
    rope_cs(p, rf.inv_freq[lane], -1.0f, cs, sn);
    rope_s[lane] = make_float2(cs, sn);
  }
  if (tid == 64) {
    mbar_init(&bars.q_full, 8);
    mbar_init(&bars.p_all, 4);
    mbar_init(&bars.o_lo, 1);
    mbar_init(&bars.o_hi, 1);
    for (int i = 0; i < kMaxChunks; ++i) mbar_init(&bars.s_full[i], 1);
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(&bars.atom_full[i], 8);
      mbar_init(&bars.atom_free[i], 1);
    }
    mbar_fence_init();
  }
  if (warp == 12) {
    tmem_alloc(&tmem_base_sh, kTmemCols);
    tmem_relinquish();
  }
  if (tid < 64) m_ref[tid] = -INFINITY;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  const int n = nrows_sh, nw = nwin_sh;
  const int nch = (n + kRows - 1) / kRows;
  const int c_begin = split * chunks_per_split;
  const int nloc = max(0, min(nch, c_begin + chunks_per_split) - c_begin);
  const int n_atoms = 16 * nloc;

  if (warp >= 4 && warp < 12) {
    // ============================================================ producers
    const int pidx = tid - 128;
    const int row = pidx >> 1, sub = pidx & 1;  // row of the chunk, 32-dim half of the atom
    uint4 raw[kAhead][2];
    uint32_t sc[kAhead];
    int kind[kAhead];  // 0: no row (zeros), 1: window (FP8), 2: Z (FP4)
    auto fetch = [&](int seq, int s) {  // s == seq % kAhead, a compile-time constant at every call
      kind[s] = 0;
      if (seq >= n_atoms) return;
      const AtomId id = atom_of(seq, nloc);
      const int ri = (c_begin + id.chunk) * kRows + row;
      if (ri >= n) return;
      const int d0 = 64 * id.blk + 32 * sub;
      if (ri < nw) {
        kind[s] = 1;
        const uint4* src = reinterpret_cast<const uint4*>(a.window + ((int64_t)b * (127 + T) + rows[ri]) * kD + d0);
        raw[s][0] = src[0];
        raw[s][1] = src[1];
      } else {
        kind[s] = 2;
        const int64_t j = rows[ri];
        raw[s][0] = *reinterpret_cast<const uint4*>(a.z_codes + ((int64_t)b * a.cap + j) * 256 + d0 / 2);
        sc[s] = a.z_scales[((int64_t)b * a.cap + j) * 16 + d0 / 32];
      }
    };
    if (nloc > 0) {
      // Q (bf16 [64][512]) -> fp16, 8 K-major atoms of [64 heads x 64 dims]; the first raw atoms
      // are requested between the two halves so that the latencies overlap
      const uint4* qs = reinterpret_cast<const uint4*>(a.q + qrow * kH * kD);
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        uint4 qv[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) qv[k] = qs[pidx + 256 * (8 * part + k)];
        if (part == 0)
#pragma unroll
          for (int s = 0; s < kAhead; ++s) fetch(s, s);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int i = pidx + 256 * (8 * part + k);
          const int h = i >> 6, d0 = (i & 63) * 8;
          const uint32_t w[4] = {qv[k].x, qv[k].y, qv[k].z, qv[k].w};
          uint32_t o[4];
#pragma unroll
          for (int m = 0; m < 4; ++m) o[m] = f2_to_h2(bf16_to_f32(w[m] & 0xffffu), bf16_to_f32(w[m] >> 16));
          *reinterpret_cast<uint4*>(sm + kQOff + (d0 >> 6) * 8192 + sw128_off(h, (d0 & 63) >> 3)) =
              make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
      if (pidx < 64) *reinterpret_cast<uint4*>(sm + kOnesOff + 16 * pidx) = make_uint4(0x3C003C00u, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u);
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.q_full);
    }
    static_assert(kAhead == kSlots, "the producer loop is unrolled by the ring depth");
    for (int seq0 = 0; seq0 < n_atoms; seq0 += kSlots) {  // n_atoms is a multiple of 4
#pragma unroll
      for (int s = 0; s < kSlots; ++s) {
        const int seq = seq0 + s, slot = s;
        if (seq >= kSlots) mbar_wait(&bars.atom_free[slot], ((seq / kSlots) - 1) & 1, err, 1);
        uint32_t o[16];
        if (kind[s] == 1) {
          const uint32_t w[8] = {raw[s][0].x, raw[s][0].y, raw[s][0].z, raw[s][0].w,
                                 raw[s][1].x, raw[s][1].y, raw[s][1].z, raw[s][1].w};
#pragma unroll
          for (int m = 0; m < 8; ++m) {
            o[2 * m] = cvt_e4m3x2_f16x2(w[m] & 0xffffu);
            o[2 * m + 1] = cvt_e4m3x2_f16x2(w[m] >> 16);
          }
        } else if (kind[s] == 2) {
          const float sf = ldexpf(1.0f, (int)sc[s] - 127);
          const uint32_t s2 = f2_to_h2(sf, sf);
          const uint32_t w[4] = {raw[s][0].x, raw[s][0].y, raw[s][0].z, raw[s][0].w};
#pragma unroll
          for (int m = 0; m < 4; ++m)
#pragma unroll
            for (int by = 0; by < 4; ++by) o[4 * m + by] = hmul2(cvt_e2m1x2_f16x2((w[m] >> (8 * by)) & 255u), s2);
        } else {
#pragma unroll
          for (int q = 0; q < 16; ++q) o[q] = 0u;
        }
        unsigned char* dst = sm + kGOff + slot * 16384;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          *reinterpret_cast<uint4*>(dst + sw128_off(row, 4 * sub + q)) = make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.atom_full[slot]);
        fetch(seq + kAhead, s);
      }
    }
  } else if (warp == 12) {
    // ============================================================ MMA issuer
    if (lane == 0 && nloc > 0) {
      const uint32_t idS = idesc_f16(false, false, 128, 64);
      const uint32_t idO = idesc_f16(true, true, 128, 64);
      const uint32_t idL = idesc_f16(false, true, 128, 64);  // ones (any layout) x P^T (MN-major)
      const uint32_t gq = sbase + kQOff, gg = sbase + kGOff, gp = sbase + kPOff;
      const uint64_t ones_desc = sw128_desc(sbase + kOnesOff, 16, 0);  // every row group reads the same atom
      mbar_wait(&bars.q_full, 0, err, 2);
      int seq = 0;
      // pass 1: S^T of every chunk
      for (int c = 0; c < nloc; ++c) {
        for (int k = 0; k < 8; ++k, ++seq) {
          const int slot = seq % kSlots;
          mbar_wait(&bars.atom_full[slot], (seq / kSlots) & 1, err, 3);
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_f16_ss(tmem + kSCol + 64 * c, sw128_desc(gg + slot * 16384 + kk * 32, 16, 1024),
                       sw128_desc(gq + k * 8192 + kk * 32, 16, 1024), idS, (k | kk) != 0);
          mma_commit(&bars.atom_free[slot]);
        }
        mma_commit(&bars.s_full[c]);
      }
      mbar_wait(&bars.p_all, 0, err, 4);
      tc_fence_after();
      // pass 2: O^T 128-dim tiles over all chunks; atoms come in (even, odd) slot pairs
      for (int half = 0; half < 2; ++half) {
        for (int tile = 0; tile < 2; ++tile) {
          // dims 128*(2*half+tile) ..: accumulator column
          const uint32_t ocol = half == 0 ? 64u * tile : kSCol + 64u * tile;
          for (int c = 0; c < nloc; ++c) {
            const int s0 = 8 * nloc + 2 * nloc * (2 * half + tile) + 2 * c;  // first atom of the pair (even)
            const int slot = s0 % kSlots;
            mbar_wait(&bars.atom_full[slot], (s0 / kSlots) & 1, err, 3);
            mbar_wait(&bars.atom_full[slot + 1], ((s0 + 1) / kSlots) & 1, err, 3);
            tc_fence_after();
            const uint32_t pc = gp + c * 16384;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_f16_ss(tmem + ocol, sw128_desc(gg + slot * 16384 + kk * 2048, 16384, 1024),
                         sw128_desc(pc + kk * 2048, 8192, 1024), idO, (c > 0 || kk > 0) ? 1u : 0u);
            mma_commit(&bars.atom_free[slot]);
            mma_commit(&bars.atom_free[slot + 1]);
          }
        }
        if (half == 0) {
          // row sums l_h = sum over all rows of P[row, h]
          for (int c = 0; c < nloc; ++c)
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_f16_ss(tmem + kLCol, ones_desc, sw128_desc(gp + c * 16384 + kk * 2048, 8192, 1024), idL,
                         (c > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&bars.o_lo);
        } else {
          mma_commit(&bars.o_hi);
        }
      }
    }
    __syncwarp();
  } else {
    // ============================================================ softmax (warps 0-3)
    const int r = 32 * warp + lane;  // row of the chunk = TMEM lane
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * warp) << 16);
    const float scale_log2 = rsqrtf((float)kD) * kLog2e;
    auto load_x = [&](int c, int hh, bool valid, float (&x)[32]) {
      uint32_t u[32];
      tmem_ld32(lane_addr + kSCol + 64 * c + 32 * hh, u);
      tmem_wait_ld();
#pragma unroll
      for (int h = 0; h < 32; ++h) x[h] = valid ? __uint_as_float(u[h]) * scale_log2 : -INFINITY;
    };
    // P_c = exp2(x - m) as fp16, MN-major [rows][heads]; true if some score exceeds its head's
    // reference by more than kTau
    auto write_p = [&](int c, bool valid) {
      bool over = false;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float x[32];
        load_x(c, hh, valid, x);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t w[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int h0 = 8 * q + 2 * k;
            const float m0 = m_ref[32 * hh + h0], m1 = m_ref[32 * hh + h0 + 1];
            over |= (x[h0] > m0 + kTau) | (x[h0 + 1] > m1 + kTau);
            w[k] = f2_to_h2(exp2f(x[h0] - m0), exp2f(x[h0 + 1] - m1));
          }
          *reinterpret_cast<uint4*>(sm + kPOff + c * 16384 + sw128_off(r, 4 * hh + q)) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      return over;
    };
    for (int c = 0; c < nloc; ++c) {
      mbar_wait(&bars.s_full[c], 0, err, 5);
      tc_fence_after();
      const bool valid = (c_begin + c) * kRows + r < n;
      // optimistic pass with the current references (-inf before the first chunk, so the check
      // always fails there); one barrier ORs whether any head needs a new reference
      if (bar_red_or(1, 128, write_p(c, valid))) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          float x[32];
          load_x(c, hh, valid, x);
          red_max[warp][32 * hh + lane] = transpose_reduce32<true>(x, lane);
        }
        named_bar_sync(1, 128);
        if (tid < 64) {
          const float mc = fmaxf(fmaxf(red_max[0][tid], red_max[1][tid]), fmaxf(red_max[2][tid], red_max[3][tid]));
          const float mo = m_ref[tid];
          float al = 1.f;
          if (mc > mo + kTau) {
            al = exp2f(mo - mc);
            m_ref[tid] = mc;
          }
          alpha_s[tid] = al;
        }
        named_bar_sync(1, 128);
        // earlier chunks' P (this thread's rows) *= alpha[head]; no O MMA has read them yet
        for (int c2 = 0; c2 < c; ++c2)
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            uint4* pp = reinterpret_cast<uint4*>(sm + kPOff + c2 * 16384 + sw128_off(r, q));
            uint4 v = *pp;
            uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[k]));
              w[k] = f2_to_h2(f.x * alpha_s[8 * q + 2 * k], f.y * alpha_s[8 * q + 2 * k + 1]);
            }
            *pp = make_uint4(w[0], w[1], w[2], w[3]);
          }
        write_p(c, valid);
      }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncwarp();
    if (lane == 0 && nloc > 0) mbar_arrive(&bars.p_all);
    // ------------------------------------------------------------ epilogue
    // row sums: every lane of the sum tile holds sum_rows P[row, h]
    if (nloc > 0) {
      mbar_wait(&bars.o_lo, 0, err, 7);
      tc_fence_after();
    }
    if (tid < 64) {
      float l = 0.f;
      if (nloc > 0) {
        uint32_t u[32];
        tmem_ld32(lane_addr + kLCol + 32 * (tid >> 5), u);
        tmem_wait_ld();
#pragma unroll
        for (int h = 0; h < 32; ++h)
          if (h == lane) l = __uint_as_float(u[h]);
      }
      l_s[tid] = l;
      den_s[tid] = nsplit == 1 ? 1.f / (l + exp2f(a.sinks[tid] * kLog2e - m_ref[tid])) : 1.f;
    }
    named_bar_sync(1, 128);
    // O^T tile by tile through smem (the Q region): thread = dim writes its 64 heads as a row,
    // then tasks (head, 8 dims) read columns and store 16 bytes (bf16 out) or 32 (fp32 partials)
    float* stage = reinterpret_cast<float*>(sm + kQOff);
    const int64_t pr_row = ((int64_t)bl * T + t) * nsplit + split;
    for (int m = 0; m < 4; ++m) {
      if (m == 2 && nloc > 0) {
        mbar_wait(&bars.o_hi, 0, err, 8);
        tc_fence_after();
      }
      const uint32_t ocol = m < 2 ? 64u * m : kSCol + 64u * (m - 2);
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t u[32];
        if (nloc > 0) {
          tmem_ld32(lane_addr + ocol + 32 * hh, u);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int h = 0; h < 32; ++h) u[h] = 0u;
        }
#pragma unroll
        for (int q = 0; q < 8; ++q)
          *reinterpret_cast<float4*>(stage + r * kStage + 32 * hh + 4 * q) =
              make_float4(__uint_as_float(u[4 * q]) * den_s[32 * hh + 4 * q], __uint_as_float(u[4 * q + 1]) * den_s[32 * hh + 4 * q + 1],
                          __uint_as_float(u[4 * q + 2]) * den_s[32 * hh + 4 * q + 2], __uint_as_float(u[4 * q + 3]) * den_s[32 * hh + 4 * q + 3]);
      }
      named_bar_sync(1, 128);
#pragma unroll 2
      for (int task = tid; task < 64 * 16; task += 128) {
        const int h = task & 63, g = task >> 6;  // head, group of 8 dims
        float o[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) o[k] = stage[(8 * g + k) * kStage + h];
        const int d0 = 128 * m + 8 * g;
        if (nsplit == 1) {
          if (d0 >= kD - kDR) {  // rotate each (even, odd) pair back by -t
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float2 cs = rope_s[(d0 - (kD - kDR)) / 2 + k];
              const float x0 = o[2 * k], x1 = o[2 * k + 1];
              o[2 * k] = x0 * cs.x - x1 * cs.y;
              o[2 * k + 1] = x0 * cs.y + x1 * cs.x;
            }
          }
          uint32_t w[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const __nv_bfloat162 v = __floats2bfloat162_rn(o[2 * k], o[2 * k + 1]);
            w[k] = *reinterpret_cast<const uint32_t*>(&v);
          }
          *reinterpret_cast<uint4*>(a.out + (qrow * kH + h) * kD + d0) = make_uint4(w[0], w[1], w[2], w[3]);
        } else {
          float4* po = reinterpret_cast<float4*>(part_o + (pr_row * kH + h) * kD + d0);
          po[0] = make_float4(o[0], o[1], o[2], o[3]);
          po[1] = make_float4(o[4], o[5], o[6], o[7]);
        }
      }
      named_bar_sync(1, 128);
    }
    if (nsplit > 1 && tid < 64) {
      part_ml[(pr_row * kH + tid) * 2] = m_ref[tid];
      part_ml[(pr_row * kH + tid) * 2 + 1] = l_s[tid];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 12) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
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
  for (int s = 0; s < nsplit; ++s) {
    const int64_t pr = lrow * nsplit + s;
    if (part_ml[(pr * kH + h) * 2 + 1] > 0.f) mstar = fmaxf(mstar, part_ml[(pr * kH + h) * 2]);
  }
  float den = exp2f(a.sinks[h] * kLog2e - mstar);
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  const int d = 4 * threadIdx.x;
  for (int s = 0; s < nsplit; ++s) {
    const int64_t pr = lrow * nsplit + s;
    const float ms = part_ml[(pr * kH + h) * 2], ls = part_ml[(pr * kH + h) * 2 + 1];
    if (!(ls > 0.f)) continue;  // split without rows
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
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc[0], acc[1]), hi = __floats2bfloat162_rn(acc[2], acc[3]);
  *reinterpret_cast<uint2*>(a.out + (qrow * kH + h) * kD + d) =
      make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
}

int choose_splits(int nq, int num_sms) {
  if (nq >= num_sms) return 1;
  return max(1, min(kMaxChunks, num_sms / nq));
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
  cudaError_t e = cudaFuncSetAttribute(attend_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDynBytes);
  if (e != cudaSuccess) return e;
  const int cps = (kMaxChunks + s - 1) / s;
  float *po = nullptr, *pml = nullptr;
  if (s > 1) {
    const size_t rows = (size_t)nb * a.T * s;
    if (ws_bytes < rows * kH * kD * 4 + rows * kH * 2 * 4) return cudaErrorInvalidValue;
    po = static_cast<float*>(ws);
    pml = po + rows * kH * kD;
  }
  attend_tc_kernel<<<dim3((unsigned)a.T, (unsigned)nb, (unsigned)s), kThreads, kDynBytes, st>>>(a, pos, b0, rf, s, cps,
                                                                                                 po, pml);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (s > 1) {
    attend_combine_kernel<<<dim3((unsigned)a.T, (unsigned)nb, kH), 128, 0, st>>>(a, pos, b0, rf, s, po, pml);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace csa2
