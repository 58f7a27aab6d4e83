// Sink-softmax MQA over the gathered rows, on the 5th-generation tensor cores (tcgen05).
// Page "DeepSeek V4.1 - Pooled group / Source layer, pairs pooled", block "Compressed sparse
// attention": J^w_t = {max(0,t-127)..t}, Y = [W; Z], J = [J^w; I + |W|], G_t = Y[J_t],
// S = Q.G/sqrt(512), A = exp S / (exp s_h + sum exp S), O = sum A G, O-bar_{448:} =
// R_t^{-1} O_{448:}.  "Inside DeepSeek V4.1", section "Attention that looks at 640 places":
// 64 heads x 512, one shared key/value row per place, a learned sink per head, 640 places.
//
// One block per (query, row split).  The gathered rows form chunks of 128 (at most 5):
//   S^T_c[rows, heads] = G_c Q^T     M=128 rows, N=64 heads, K=512 (8 K-major atoms)
//   O^T[dims, heads] += G_c^T P_c^T  M=128 dims x 4 tiles, N=64, K=128 rows (MN-major)
//   l_h += sum_rows P_c[row, h]      a ones x P^T MMA (one 1 KB swizzle atom of ones read
//                                    for every row group through a zero row-group stride)
// An "atom" is 128 rows x 64 dims of G in fp16, 128B-swizzled; the same atom serves as the
// K-major A operand of S and, in (even, odd) pairs, the MN-major A operand of one O tile.
// The MMA stream is software-pipelined: S(0), then S(c) and O(c-1) for c = 1..n-1, then
// O(n-1), so the softmax of chunk c (S -> P_c in smem) overlaps the MMAs of S(c+1).  G is
// decoded twice (for S and for O) from FP4 / FP8 rows: E2M1 x 2^e (scale exponents -22..12)
// and E4M3 are exact in fp16 and convert with one hardware instruction per pair.
//
// Measured on GB300: a 128x64x16 fp16 MMA takes ~50 cycles and alternating accumulators
// costs more, so each accumulator receives its MMAs consecutively; and a barrier arrive with
// release semantics waits for the arriving thread's outstanding loads, so raw rows are staged
// with cp.async (not ordered by the arrive) several atoms ahead.
//
// Warp roles (416 threads):
//   warps 0-3   softmax + epilogue; thread = TMEM lane = row of S^T / dim of O^T
//   warps 4-11  producers: Q -> smem, then every atom: raw 32 dims per thread (cp.async into a
//               5-deep staging ring) -> decode -> 4-slot atom ring; two threads per row
//   warp 12     TMEM allocation and the single MMA-issuing thread
// Online softmax with a lazy reference: a head's reference m only moves when a chunk's
// maximum exceeds it by more than kTau (log2 units), so P <= 2^kTau; when it moves, O and l
// are rescaled in TMEM after the previous chunk's MMAs complete.
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
constexpr int kSlots = 4;                   // decoded atom ring
constexpr int kStg = 5;                     // raw staging ring (cp.async depth)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kTau = 8.0f;                // lazy-rescale threshold (log2 units)
// dynamic shared memory (1024-aligned)
constexpr uint32_t kQOff = 0;                        // Q: 8 atoms x [64 heads x 128 B]
constexpr uint32_t kPOff = 65536;                    // P: 2 x [128 rows x 128 B]
constexpr uint32_t kGOff = 98304;                    // atoms: 4 x [128 rows x 128 B] (epilogue staging later)
constexpr uint32_t kStgOff = 163840;                 // raw: 5 x [128 rows x 64 B]
constexpr uint32_t kScOff = 204800;                  // Z scale rows: 3 chunks x [128 x 16 B]
constexpr uint32_t kOnesOff = 210944;                // 1 KB of fp16 ones
constexpr uint32_t kDynBytes = 211968 + 1024;
// TMEM columns: O^T dims tiles at 0, 64, 128, 192; row sums at 256; S^T buffers at 320, 384
constexpr uint32_t kTmemCols = 512, kLCol = 256, kSCol = 320;
constexpr int kStage = 68;                           // epilogue staging row (floats)

__device__ int g_attend_error;

struct Bars {
  uint64_t q_full;
  uint64_t s_full[kMaxChunks];
  uint64_t p_full[2], o_done[2];
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

// Atom `pos` of the stream S(0); S(1), O(0); ...; S(n-1), O(n-2); O(n-1): chunk, dims block
// (0..7), and whether it belongs to an S pass.  O atoms come in tile order (pairs 0-1, ..., 6-7).
struct AtomId {
  int chunk, blk;
  bool s;
};
__device__ __forceinline__ AtomId atom_of(int pos, int n) {
  if (pos < 8) return {0, pos, true};
  if (pos >= 16 * n - 8) return {n - 1, pos - (16 * n - 8), false};
  const int q = (pos - 8) >> 4, r = (pos - 8) & 15;
  return r < 8 ? AtomId{q + 1, r, true} : AtomId{q, r - 8, false};
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
  __shared__ int nrows_sh, nwin_sh, moved_sh;

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
      moved_sh = 0;
    }
  }
  if (warp == 1) {
    float cs, sn;
    rope_cs(p, rf.inv_freq[lane], -1.0f, cs, sn);
    rope_s[lane] = make_float2(cs, sn);
  }
  if (tid == 64) {
    mbar_init(&bars.q_full, 8);
    for (int i = 0; i < kMaxChunks; ++i) mbar_init(&bars.s_full[i], 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.p_full[i], 4);
      mbar_init(&bars.o_done[i], 1);
    }
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
    const int row = pidx >> 1, sub = pidx & 1;  // row of the chunk, 32-dim half of each atom
    // raw bytes of atom `at` (this thread's 32 dims) -> staging slot at % kStg, asynchronously
    auto issue = [&](int at) {
      if (at < n_atoms) {
        const AtomId id = atom_of(at, nloc);
        const int ri = (c_begin + id.chunk) * kRows + row;
        unsigned char* st = sm + kStgOff + (at % kStg) * 8192 + row * 64 + 32 * sub;
        if (ri < n) {
          const int d0 = 64 * id.blk + 32 * sub;
          if (ri < nw) {
            const unsigned char* src = a.window + ((int64_t)b * (127 + T) + rows[ri]) * kD + d0;
            cp_async16(st, src);
            cp_async16(st + 16, src + 16);
          } else {
            const int64_t j = rows[ri];
            cp_async16(st, a.z_codes + ((int64_t)b * a.cap + j) * 256 + d0 / 2);
            // the chunk's scale row, with its first atom; both threads of the row copy the same 16
            // bytes so that each only depends on its own copies
            if (id.s && id.blk == 0)
              cp_async16(sm + kScOff + (id.chunk % 3) * 2048 + row * 16, a.z_scales + ((int64_t)b * a.cap + j) * 16);
          }
        }
      }
      cp_async_commit();  // one group per atom, possibly empty
    };
    if (nloc > 0) {
      // Q (bf16 [64][512]) -> fp16, 8 K-major atoms of [64 heads x 64 dims]; the first raw atoms
      // are requested first so that the latencies overlap
#pragma unroll 1
      for (int at = 0; at < kStg; ++at) issue(at);
      const uint4* qs = reinterpret_cast<const uint4*>(a.q + qrow * kH * kD);
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        uint4 qv[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) qv[k] = qs[pidx + 256 * (8 * part + k)];
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
#pragma unroll 1
    for (int at = 0; at < n_atoms; ++at) {
      cp_async_wait<kStg - 1>();  // this thread's copies for atom `at` have landed
      const AtomId id = atom_of(at, nloc);
      const int ri = (c_begin + id.chunk) * kRows + row;
      const unsigned char* st = sm + kStgOff + (at % kStg) * 8192 + row * 64 + 32 * sub;
      uint32_t o[16];
      if (ri < n && ri < nw) {
        const uint4 v0 = *reinterpret_cast<const uint4*>(st), v1 = *reinterpret_cast<const uint4*>(st + 16);
        const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          o[2 * m] = cvt_e4m3x2_f16x2(w[m] & 0xffffu);
          o[2 * m + 1] = cvt_e4m3x2_f16x2(w[m] >> 16);
        }
      } else if (ri < n) {
        const uint4 v = *reinterpret_cast<const uint4*>(st);
        const int e = (int)sm[kScOff + (id.chunk % 3) * 2048 + row * 16 + 2 * id.blk + sub] - 127;
        const float sf = ldexpf(1.0f, e);
        const uint32_t s2 = f2_to_h2(sf, sf);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int m = 0; m < 4; ++m)
#pragma unroll
          for (int by = 0; by < 4; ++by) o[4 * m + by] = hmul2(cvt_e2m1x2_f16x2((w[m] >> (8 * by)) & 255u), s2);
      } else {
#pragma unroll
        for (int q = 0; q < 16; ++q) o[q] = 0u;
      }
      const int slot = at % kSlots;
      if (at >= kSlots) mbar_wait(&bars.atom_free[slot], ((at / kSlots) - 1) & 1, err, 1);
      unsigned char* dst = sm + kGOff + slot * 16384;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        *reinterpret_cast<uint4*>(dst + sw128_off(row, 4 * sub + q)) = make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.atom_full[slot]);
      issue(at + kStg);
    }
    cp_async_wait<0>();
  } else if (warp == 12) {
    // ============================================================ MMA issuer
    if (lane == 0 && nloc > 0) {
      const uint32_t idS = idesc_f16(false, false, 128, 64);
      const uint32_t idO = idesc_f16(true, true, 128, 64);
      const uint32_t idL = idesc_f16(false, true, 128, 64);  // ones (any layout) x P^T (MN-major)
      const uint32_t gq = sbase + kQOff, gg = sbase + kGOff, gp = sbase + kPOff;
      const uint64_t ones_desc = sw128_desc(sbase + kOnesOff, 16, 0);  // every row group reads the same atom
      mbar_wait(&bars.q_full, 0, err, 2);
      int at = 0;
      auto s_pass = [&](int c) {
        for (int k = 0; k < 8; ++k, ++at) {
          const int slot = at % kSlots;
          mbar_wait(&bars.atom_full[slot], (at / kSlots) & 1, err, 3);
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_f16_ss(tmem + kSCol + 64 * (c & 1), sw128_desc(gg + slot * 16384 + kk * 32, 16, 1024),
                       sw128_desc(gq + k * 8192 + kk * 32, 16, 1024), idS, (k | kk) != 0);
          mma_commit(&bars.atom_free[slot]);
        }
        mma_commit(&bars.s_full[c]);
      };
      auto o_pass = [&](int c) {
        mbar_wait(&bars.p_full[c & 1], (c >> 1) & 1, err, 4);
        tc_fence_after();
        const uint32_t pc = gp + (c & 1) * 16384;
        for (int tile = 0; tile < 4; ++tile, at += 2) {
          const int slot = at % kSlots;  // even: the pair is (slot, slot + 1)
          mbar_wait(&bars.atom_full[slot], (at / kSlots) & 1, err, 3);
          mbar_wait(&bars.atom_full[slot + 1], ((at + 1) / kSlots) & 1, err, 3);
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_f16_ss(tmem + 64 * tile, sw128_desc(gg + slot * 16384 + kk * 2048, 16384, 1024),
                       sw128_desc(pc + kk * 2048, 8192, 1024), idO, (c > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&bars.atom_free[slot]);
          mma_commit(&bars.atom_free[slot + 1]);
        }
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_f16_ss(tmem + kLCol, ones_desc, sw128_desc(pc + kk * 2048, 8192, 1024), idL, (c > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bars.o_done[c & 1]);
      };
      s_pass(0);
      for (int c = 1; c < nloc; ++c) {
        s_pass(c);
        o_pass(c - 1);
      }
      o_pass(nloc - 1);
    }
    __syncwarp();
  } else {
    // ============================================================ softmax (warps 0-3)
    const int r = 32 * warp + lane;  // row of the chunk = TMEM lane
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * warp) << 16);
    const float scale_log2 = rsqrtf((float)kD) * kLog2e;
    auto load_x = [&](int c, int hh, bool valid, float (&x)[32]) {
      uint32_t u[32];
      tmem_ld32(lane_addr + kSCol + 64 * (c & 1) + 32 * hh, u);
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
          *reinterpret_cast<uint4*>(sm + kPOff + (c & 1) * 16384 + sw128_off(r, 4 * hh + q)) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      return over;
    };
    for (int c = 0; c < nloc; ++c) {
      mbar_wait(&bars.s_full[c], 0, err, 5);
      if (c >= 2) mbar_wait(&bars.o_done[c & 1], ((c - 2) >> 1) & 1, err, 6);  // O(c-2) has read P buffer
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
            if (c > 0) moved_sh = 1;
          }
          alpha_s[tid] = al;
        }
        named_bar_sync(1, 128);
        if (moved_sh) {
          // O^T tiles and row sums (lane = dim, column = head) *= alpha[head] once O(c-1) is done
          mbar_wait(&bars.o_done[(c - 1) & 1], ((c - 1) >> 1) & 1, err, 7);
          tc_fence_after();
          for (int m = 0; m < 5; ++m)
            for (int hh = 0; hh < 2; ++hh) {
              uint32_t u[32];
              tmem_ld32(lane_addr + 64 * m + 32 * hh, u);
              tmem_wait_ld();
#pragma unroll
              for (int h = 0; h < 32; ++h) u[h] = __float_as_uint(__uint_as_float(u[h]) * alpha_s[32 * hh + h]);
              tmem_st32(lane_addr + 64 * m + 32 * hh, u);
            }
          tmem_wait_st();
        }
        write_p(c, valid);
        named_bar_sync(1, 128);
        if (tid == 0) moved_sh = 0;
      }
      fence_proxy_async();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.p_full[c & 1]);
    }
    // ------------------------------------------------------------ epilogue
    if (nloc > 0) {
      mbar_wait(&bars.o_done[(nloc - 1) & 1], ((nloc - 1) >> 1) & 1, err, 8);
      tc_fence_after();
    }
    // row sums: every lane of the sum tile holds sum_rows P[row, h]
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
    // O^T tile by tile through smem (the atom ring, idle now): thread = dim writes its 64 heads
    // as a row, then tasks (head, 8 dims) read columns and store 16 bytes (bf16) or 32 (fp32)
    float* stage = reinterpret_cast<float*>(sm + kGOff);
    const int64_t pr_row = ((int64_t)bl * T + t) * nsplit + split;
    for (int m = 0; m < 4; ++m) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t u[32];
        if (nloc > 0) {
          tmem_ld32(lane_addr + 64 * m + 32 * hh, u);
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
