// Sink-softmax MQA over the gathered rows, on the 5th-generation tensor cores (tcgen05).
// Page "DeepSeek V4.1 - Pooled group / Source layer, pairs pooled", block "Compressed sparse
// attention": J^w_t = {max(0,t-127)..t}, Y = [W; Z], J = [J^w; I + |W|], G_t = Y[J_t],
// S = Q.G/sqrt(512), A = exp S / (exp s_h + sum exp S), O = sum A G, O-bar_{448:} =
// R_t^{-1} O_{448:}.  "Inside DeepSeek V4.1", section "Attention that looks at 640 places":
// 64 heads x 512, one shared key/value row per place, a learned sink per head, 640 places.
//
// One block per (query, row split).  The gathered rows are processed in chunks of 128:
//   S^T[rows, heads] = G_c Q^T    (M = 128 rows, N = 64 heads, K = 512; A, B K-major)
//   O^T[dims, heads] += G_c^T P^T (M = 128 dims x 4 tiles, N = 64, K = 128 rows; A, B MN-major)
// so that both MMAs have M = 128 and the same shared-memory copy of G_c serves as the
// K-major A operand of the first and the MN-major A operand of the second.  Operands are
// fp16: E2M1 x 2^e (for scale exponents -22..12) and E4M3 values are exact in fp16 and
// convert with one hardware instruction per pair; accumulation is fp32 in tensor memory.
//
// The per-head row sums l_h = sum_rows P[row, h] come from the tensor core too: a fifth O-phase
// accumulator multiplies P^T by an all-ones A operand held in tensor memory (so those MMAs read
// only P from shared memory), and the softmax never reduces across lanes after the first chunk.
// Measured on GB300: a 128x64x16 fp16 MMA takes ~50 cycles and alternating between
// accumulators costs more, so each accumulator receives its MMAs consecutively.
//
// Warp roles (448 threads):
//   warps 0-3   softmax (thread = TMEM lane = row of S^T), then the row sums and 1/denominator;
//               with the producers, the output epilogue (thread = TMEM lane = dim of O^T)
//   warps 4-11  producers: Q -> smem once, then gather + decode 128 rows per chunk, two
//               threads per row (atoms 2a and 2a+1 of tile a); the raw rows of chunk c+1
//               wait in registers while chunk c is consumed and are written as soon as the
//               O MMAs free each 128-dim tile.  Both threads of a row sit in one warp and
//               work on the same tile at each step, so no lane waits for a later tile.
//   warp 12     TMEM allocation and the thread issuing the S MMAs
//   warp 13     the thread issuing the O and row-sum MMAs: while one issuer waits (and its MMAs
//               drain) the other keeps the tensor pipe busy, so the next chunk's S MMAs overlap
//               this chunk's O MMAs
// Online softmax with a lazy reference: a head's reference m only moves when a chunk's
// maximum exceeds it by more than kTau (log2 units), so P <= 2^kTau and O is rescaled in
// TMEM rarely (in practice only at the first chunk, where there is nothing to rescale).
#include <cuda_fp16.h>

#include <algorithm>

#include "csa2_common.cuh"
#include "csa2_fp16.cuh"
#include "csa2_sm100.cuh"

namespace csa2 {
namespace {

using namespace sm100;

constexpr int kThreads = 448;
constexpr int kRows = 128;                  // rows per chunk
constexpr int kMaxRows = kWin + kTopK;      // 640
constexpr int kMaxChunks = kMaxRows / kRows;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kTau = 8.0f;                // lazy-rescale threshold (log2 units)
// dynamic shared memory (1024-aligned): Q 8 atoms x [64 x 128 B], G 8 atoms x [128 x 128 B],
// P [128 rows x 128 B], one 1 KB swizzle atom of fp16 ones
constexpr uint32_t kQOff = 0, kGOff = 65536, kPOff = 196608, kDynBytes = 212992 + 1024;
static_assert(kPOff - kGOff == kH * kD * 4, "the G area holds one fp32 output row (split partials)");
// TMEM columns: O^T tiles at 0, 64, 128, 192; row sums at 256; S^T at 320; at 384 the all-ones
// A operand of the row-sum MMAs (128 lanes x 16 fp16 ones = 8 columns, written once per block)
constexpr uint32_t kTmemCols = 512, kLCol = 256, kSCol = 320, kOnesCol = 384;

__device__ int g_attend_error;
// Set when a producer read a Z scale above 2^13 (scale byte > 140), where E2M1 x 2^e overflows
// the fp16 operand, or a query value that overflows fp16.  csa2_check reports it.
__device__ unsigned g_attend_domain;

struct Bars {
  uint64_t q_raw, q_full, s_full, p_full, l_done;
  uint64_t atom_full[8];
  uint64_t tile_free[4];
};

// 2^x by the hardware approximation (relative error ~2^-22, results below 2^-126 flushed to 0,
// 2^-inf = 0): P is stored as fp16, whose rounding (2^-11) and smallest subnormal (2^-24)
// are far coarser.
__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
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

// grid (T, nb, nsplit).  nsplit == 1 writes `out`; otherwise the split's unnormalised O, its
// reference m (log2 units) and sum l go to the partial buffers for attend_combine_kernel.
// wst: per-sequence replay starts s (0 = none); the window rows are positions max(s, t-127)..t.
__global__ void __launch_bounds__(kThreads, 1) attend_tc_kernel(AttendArgs a, SeqPos pos, SeqPos wst, int b0,
                                                                RopeFreq rf, int nsplit, int chunks_per_split,
                                                                float* part_o, float* part_ml) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ Bars bars;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int32_t rows[kMaxRows];
  __shared__ float red_max[4][64];
  __shared__ float m_ref[64], alpha_s[64], l_run[64], den_s[64];  // den_s: 1 / denominator
  __shared__ int nrows_sh, nwin_sh;
  grid_dep_wait();  // launched dependent: nothing is read before the previous kernel has ended
  grid_dep_trigger();

  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  unsigned char* sm = smem_raw + (sbase - smem_u32(smem_raw));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t = blockIdx.x, bl = blockIdx.y, split = blockIdx.z;
  const int b = b0 + bl;
  const int T = a.T;
  const int64_t p = seq_p0(pos, bl) + t;
  const int64_t qrow = (int64_t)b * T + t;
  int* err = &g_attend_error;

  // ---------------------------------------------------------------- setup
  if (warp == 0) {
    // all 512 indices in one round trip (16 per lane); the order of the gathered rows does not
    // matter to the result, so each lane appends its valid entries after a warp prefix sum
    const int nw = (int)min64(kWin, p + 1 - wst.p0[bl]);  // window rows: max(s, p-127) .. p
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
  if (tid == 32) {
    mbar_init(&bars.q_raw, 1);
    mbar_init(&bars.q_full, 8);
    mbar_init(&bars.s_full, 1);
    mbar_init(&bars.p_full, 8);  // softmax warps 0-3 and producer warps 4-7
    mbar_init(&bars.l_done, 1);
    for (int i = 0; i < 8; ++i) mbar_init(&bars.atom_full[i], 8);
    for (int i = 0; i < 4; ++i) mbar_init(&bars.tile_free[i], 1);
    mbar_fence_init();
    // Q (bf16 [64][512], 64 KB) into the G area with one bulk copy, while warp 0 reads the
    // indices; the producers convert it after the setup barrier
    mbar_arrive_expect_tx(&bars.q_raw, kH * kD * 2);
    bulk_g2s(sm + kGOff, a.q + qrow * kH * kD, kH * kD * 2, &bars.q_raw);
    // the query one wave of blocks ahead (it will most likely run on some SM when this block
    // ends): its Q and index row into L2, so that its prologue starts from L2
    uint32_t nsm;
    asm("mov.u32 %0, %%nsmid;" : "=r"(nsm));  // SMs of the device: one block each at a time
    const int ahead = (int)nsm;
    if (split == 0 && t + ahead < T) {
      bulk_prefetch_l2(a.q + (qrow + ahead) * kH * kD, kH * kD * 2);
      bulk_prefetch_l2(a.idx + (qrow + ahead) * kTopK, kTopK * 4);
    }
  }
  if (warp == 12) {
    tmem_alloc(&tmem_base_sh, kTmemCols);
    tmem_relinquish();
  }
  if (tid < 64) {
    m_ref[tid] = -INFINITY;
    l_run[tid] = 0.f;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  const int n = nrows_sh, nw = nwin_sh;
  const int nch = (n + kRows - 1) / kRows;
  const int c_begin = split * chunks_per_split;
  const int nloc = max(0, min(nch, c_begin + chunks_per_split) - c_begin);

  const float scale_log2 = rsqrtf((float)kD) * kLog2e;
  // P[r, 32hh .. 32hh+31] = exp2(x - m) as fp16 into the MN-major [rows][heads] operand, for the
  // chunk row r = this thread's TMEM lane (lane quarter warp % 4); true if some score exceeds
  // its head's reference by more than kTau
  auto p_half = [&](int hh, int r, uint32_t lane_addr, bool valid) -> bool {
    uint32_t u[32];
    tmem_ld32(lane_addr + kSCol + 32 * hh, u);
    tmem_wait_ld();
    bool over = false;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t w[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int h0 = 8 * q + 2 * k;
        const float x0 = valid ? __uint_as_float(u[h0]) * scale_log2 : -INFINITY;
        const float x1 = valid ? __uint_as_float(u[h0 + 1]) * scale_log2 : -INFINITY;
        const float m0 = m_ref[32 * hh + h0], m1 = m_ref[32 * hh + h0 + 1];
        over |= (x0 > m0 + kTau) | (x1 > m1 + kTau);
        w[k] = f2_to_h2(ex2_ftz(x0 - m0), ex2_ftz(x1 - m1));
      }
      *reinterpret_cast<uint4*>(sm + kPOff + sw128_off(r, 4 * hh + q)) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    return over;
  };
  // red_max[warp % 4][32hh + lane] = max over the warp's 32 rows of head 32hh + lane
  auto warp_max_half = [&](int hh, uint32_t lane_addr, bool valid) {
    uint32_t u[32];
    tmem_ld32(lane_addr + kSCol + 32 * hh, u);
    tmem_wait_ld();
    float x[32];
#pragma unroll
    for (int h = 0; h < 32; ++h) x[h] = valid ? __uint_as_float(u[h]) * scale_log2 : -INFINITY;
    red_max[warp & 3][32 * hh + lane] = transpose_reduce32<true>(x, lane);
  };

  if (warp >= 4 && warp < 12) {
    // ============================================================ producers
    const int pidx = tid - 128;
    const int row = pidx >> 1, half = pidx & 1;
    uint4 raw[16];
    int kind = 0;  // 0: no row (zeros), 1: window (FP8), 2: Z (FP4)
    auto load = [&](int i) {
      const int ri = (c_begin + i) * kRows + row;
      kind = 0;
      if (ri < n) {
        // atom k = 2 * at + half covers dims 64k .. 64k+63
        if (ri < nw) {
          kind = 1;
          const uint4* src = reinterpret_cast<const uint4*>(a.window + ((int64_t)b * (127 + T) + rows[ri]) * kD);
#pragma unroll
          for (int at = 0; at < 4; ++at)
#pragma unroll
            for (int q = 0; q < 4; ++q) raw[4 * at + q] = src[4 * (2 * at + half) + q];  // 64 FP8 bytes
        } else {
          kind = 2;
          const int64_t j = rows[ri];
          const uint4* src = reinterpret_cast<const uint4*>(a.z_codes + ((int64_t)b * a.cap + j) * 256);
#pragma unroll
          for (int at = 0; at < 4; ++at)
#pragma unroll
            for (int q = 0; q < 2; ++q) raw[2 * at + q] = src[2 * (2 * at + half) + q];  // 32 FP4 code bytes
          raw[8] = *reinterpret_cast<const uint4*>(a.z_scales + ((int64_t)b * a.cap + j) * 16);  // all 16 scales
          if (__vcmpgtu4(raw[8].x, 0x8C8C8C8Cu) | __vcmpgtu4(raw[8].y, 0x8C8C8C8Cu) | __vcmpgtu4(raw[8].z, 0x8C8C8C8Cu) |
              __vcmpgtu4(raw[8].w, 0x8C8C8C8Cu))
            atomicOr(&g_attend_domain, 1u);
        }
      }
    };
    // the first chunk's rows are requested before waiting for the staged Q, so that the two
    // latencies overlap (the row list is complete at the setup barrier)
    if (nloc > 0) load(0);
    mbar_wait(&bars.q_raw, 0, err, 8);  // the staged Q has landed (waited for even without chunks)
    if (nloc > 0) {
      // Q (bf16, staged in the G area) -> fp16, 8 K-major atoms of [64 heads x 64 dims]
      const uint4* qs = reinterpret_cast<const uint4*>(sm + kGOff);
#pragma unroll 4
      for (int k = 0; k < 16; ++k) {
        const int i = pidx + 256 * k;
        const uint4 qv = qs[i];
        const int h = i >> 6, d0 = (i & 63) * 8;
        const uint32_t w[4] = {qv.x, qv.y, qv.z, qv.w};
        uint32_t o[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) o[m] = f2_to_h2(bf16_to_f32(w[m] & 0xffffu), bf16_to_f32(w[m] >> 16));
        // |q| >= 65520 (bf16 exponent field >= 143) becomes inf in fp16
        const uint32_t big = __vcmpgeu2(qv.x & 0x7f807f80u, 0x47804780u) | __vcmpgeu2(qv.y & 0x7f807f80u, 0x47804780u) |
                             __vcmpgeu2(qv.z & 0x7f807f80u, 0x47804780u) | __vcmpgeu2(qv.w & 0x7f807f80u, 0x47804780u);
        if (big) atomicOr(&g_attend_domain, 1u);
        *reinterpret_cast<uint4*>(sm + kQOff + (d0 >> 6) * 8192 + sw128_off(h, (d0 & 63) >> 3)) =
            make_uint4(o[0], o[1], o[2], o[3]);
      }
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.q_full);
      named_bar_sync(2, 256);  // every producer has read its staged Q before G is written
    }
    for (int i = 0; i < nloc; ++i) {
#pragma unroll
      for (int at = 0; at < 4; ++at) {
        const int k = 2 * at + half;  // atom: 64 dims, in tile at
        if (i > 0) mbar_wait(&bars.tile_free[at], (i - 1) & 1, err, 1);
        uint32_t o[32];
        if (kind == 1) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint4 v = raw[4 * at + q];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              o[8 * q + 2 * m] = cvt_e4m3x2_f16x2(w[m] & 0xffffu);
              o[8 * q + 2 * m + 1] = cvt_e4m3x2_f16x2(w[m] >> 16);
            }
          }
        } else if (kind == 2) {
          const uint32_t sw = k < 2 ? raw[8].x : k < 4 ? raw[8].y : k < 6 ? raw[8].z : raw[8].w;  // bytes 2k, 2k+1
#pragma unroll
          for (int blk = 0; blk < 2; ++blk) {  // 32 dims per scale byte
            const uint32_t s2 = pow2_h2((int)((sw >> (16 * (k & 1) + 8 * blk)) & 255u) - 127);
            const uint4 v = raw[2 * at + blk];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              cvt_e2m1x8_f16x8(w[m], o + 16 * blk + 4 * m);
#pragma unroll
              for (int by = 0; by < 4; ++by) o[16 * blk + 4 * m + by] = hmul2(o[16 * blk + 4 * m + by], s2);
            }
          }
        } else {
#pragma unroll
          for (int q = 0; q < 32; ++q) o[q] = 0u;
        }
        unsigned char* dst = sm + kGOff + k * 16384;
#pragma unroll
        for (int q = 0; q < 8; ++q)
          *reinterpret_cast<uint4*>(dst + sw128_off(row, q)) = make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
        fence_proxy_async();
        __syncwarp();
        if (lane < 2) mbar_arrive(&bars.atom_full[2 * at + lane]);
      }
      if (warp < 8) {
        // warps 4-7 (lane quarters 0-3): heads 32..63 of this chunk's softmax (the barriers as
        // in the softmax warps), then their share of p_full.  The tiles of the chunk are
        // written, so the raw registers are free until load(i + 1).
        mbar_wait(&bars.s_full, i & 1, err, 10);
        if (i > 0) mbar_wait(&bars.l_done, (i - 1) & 1, err, 12);  // P of the last chunk has been read
        tc_fence_after();
        const int r = 32 * (warp & 3) + lane;
        const uint32_t lane_addr = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
        const bool valid = (c_begin + i) * kRows + r < n;
        if (i == 0) {
          warp_max_half(1, lane_addr, valid);
          named_bar_sync(5, 256);  // the chunk maximum of every head is in red_max
          named_bar_sync(4, 256);  // the references are set
          p_half(1, r, lane_addr, valid);
        } else {
          named_bar_sync(5, 256);
          bar_red_or(4, 256, p_half(1, r, lane_addr, valid));
        }
        fence_proxy_async();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.p_full);
      }
      if (i + 1 < nloc) load(i + 1);
    }
  } else if (warp == 12) {
    // ============================================================ S issuer
    if (lane == 0 && nloc > 0) {
      const uint32_t idS = idesc_f16(false, false, 128, 64);
      const uint32_t gq = sbase + kQOff, gg = sbase + kGOff;
      mbar_wait(&bars.q_full, 0, err, 2);
      for (int i = 0; i < nloc; ++i) {
        // S^T = G_c Q^T into one accumulator.  The softmax has read the last chunk's S^T by then:
        // the atoms of chunk c are refilled only after the O MMAs of chunk c-1, which the other
        // thread issues after p_full.  Every wait of this thread stalls until its MMAs in flight
        // drain, so it waits for atoms 2 k2 and 2 k2 + 1 together (the two producer halves write
        // them at the same time); the O issuer's MMAs keep the tensor pipe busy meanwhile.
        for (int k2 = 0; k2 < 4; ++k2) {
          mbar_wait(&bars.atom_full[2 * k2], i & 1, err, 3);
          mbar_wait(&bars.atom_full[2 * k2 + 1], i & 1, err, 3);
          tc_fence_after();
#pragma unroll
          for (int hk = 0; hk < 2; ++hk) {
            const int k = 2 * k2 + hk;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_f16_ss(tmem + kSCol, sw128_desc(gg + k * 16384 + kk * 32, 16, 1024),
                         sw128_desc(gq + k * 8192 + kk * 32, 16, 1024), idS, (k2 | hk | kk) != 0);
          }
        }
        mma_commit(&bars.s_full);
      }
    }
    __syncwarp();
  } else if (warp == 13) {
    // ============================================================ O issuer
    if (lane == 0 && nloc > 0) {
      const uint32_t idO = idesc_f16(true, true, 128, 64);
      const uint32_t idL = idesc_f16(false, true, 128, 64);  // ones (TMEM) x P^T (MN-major)
      const uint32_t gg = sbase + kGOff, gp = sbase + kPOff;
      for (int i = 0; i < nloc; ++i) {
        mbar_wait(&bars.p_full, i & 1, err, 4);
        tc_fence_after();
        // O^T tiles one after the other in the order the producers refill them (each frees its
        // two atoms for the next chunk), then the row sums.
        for (int m = 0; m < 4; ++m) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_f16_ss(tmem + 64 * m, sw128_desc(gg + 2 * m * 16384 + kk * 2048, 16384, 1024),
                       sw128_desc(gp + kk * 2048, 8192, 1024), idO, (i > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&bars.tile_free[m]);
        }
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_f16_ts(tmem + kLCol, tmem + kOnesCol, sw128_desc(gp + kk * 2048, 8192, 1024), idL, (i > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bars.l_done);
      }
    }
    __syncwarp();
  } else {
    // ============================================================ softmax (warps 0-3)
    const int r = 32 * warp + lane;  // row of the chunk = TMEM lane
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * warp) << 16);
    // x[32] = scaled scores of heads 32hh..32hh+31 for this thread's row (sum of the S halves)
    auto load_x = [&](int hh, bool valid, float (&x)[32]) {
      uint32_t u[32];
      tmem_ld32(lane_addr + kSCol + 32 * hh, u);
      tmem_wait_ld();
#pragma unroll
      for (int h = 0; h < 32; ++h) x[h] = valid ? __uint_as_float(u[h]) * scale_log2 : -INFINITY;
    };
    if (nloc > 0) {  // the row-sum MMAs' all-ones A operand; the first p_full arrive publishes it
      uint32_t ones[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) ones[k] = 0x3C003C00u;
      tmem_st16(lane_addr + kOnesCol, ones);
      tmem_wait_st();
    }
    for (int i = 0; i < nloc; ++i) {
      mbar_wait(&bars.s_full, i & 1, err, 5);
      // P is rewritten below: the last chunk's O and row-sum MMAs (the other issuer) must have read it
      if (i > 0) mbar_wait(&bars.l_done, (i - 1) & 1, err, 11);
      tc_fence_after();
      const bool valid = (c_begin + i) * kRows + r < n;
      // Heads 0..31 here, 32..63 in producer warps 4-7 (same rows: lane quarter warp % 4); barriers
      // 5 and 4 are taken by warps 0-7 (256 threads) at every chunk.
      // First chunk: the references are -inf, so they are set to the chunk maxima (each group
      // reduces its heads; barrier 5: all maxima in red_max; barrier 4: references set).
      // Later chunks: an optimistic pass with the current references; barrier 5 makes this
      // group's reference updates of the last chunk visible to warps 4-7, barrier 4 ORs whether
      // any head needs a new reference.
      bool redo = false;
      if (i == 0) {
        warp_max_half(0, lane_addr, valid);
        named_bar_sync(5, 256);
        if (tid < 64)
          m_ref[tid] = fmaxf(fmaxf(red_max[0][tid], red_max[1][tid]), fmaxf(red_max[2][tid], red_max[3][tid]));
        named_bar_sync(4, 256);
        p_half(0, r, lane_addr, valid);
      } else {
        named_bar_sync(5, 256);
        redo = bar_red_or(4, 256, p_half(0, r, lane_addr, valid));
      }
      if (redo) {  // new references where needed, O rescaled, then P for all 64 heads
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          float x[32];
          load_x(hh, valid, x);
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
        if (i > 0) {
          // O^T tiles and row sums (lane = dim, column = head) *= alpha[head], once the previous
          // chunk's MMAs are done
          mbar_wait(&bars.l_done, (i - 1) & 1, err, 6);
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
        p_half(0, r, lane_addr, valid);
        p_half(1, r, lane_addr, valid);
      }
      fence_proxy_async();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.p_full);
    }
    // ------------------------------------------------------------ epilogue
    if (nloc > 0) {
      mbar_wait(&bars.l_done, (nloc - 1) & 1, err, 7);
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
      l_run[tid] = l;
      den_s[tid] = nsplit == 1 ? 1.f / (l + exp2f(a.sinks[tid] * kLog2e - m_ref[tid])) : 1.f;
    }
    if (nsplit != 1) {
      named_bar_sync(1, 128);
      const int64_t pr_row = ((int64_t)bl * T + t) * nsplit + split;
      float* po = part_o + pr_row * kH * kD;
      // the split's O [64 heads][512 dims] fp32 (128 KB, the whole G area) in shared memory,
      // then one bulk copy; a split without chunks first lets the staged Q copy land
      float* ost = reinterpret_cast<float*>(sm + kGOff);
      if (nloc == 0) mbar_wait(&bars.q_raw, 0, err, 9);
      for (int m = 0; m < 4; ++m) {
        const int d = 128 * m + r;
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
          for (int h = 0; h < 32; ++h) ost[(32 * hh + h) * kD + d] = __uint_as_float(u[h]);
        }
      }
      fence_proxy_async();
      named_bar_sync(1, 128);
      if (tid == 0) {
        bulk_s2g(po, ost, kH * kD * 4);
        bulk_commit();
        bulk_wait_read();
      }
      if (tid < 64) {
        part_ml[(pr_row * kH + tid) * 2] = m_ref[tid];
        part_ml[(pr_row * kH + tid) * 2 + 1] = l_run[tid];
      }
    }
  }
  if (nsplit == 1 && warp < 12) {
    // ------------------------------------------------------------ output (warps 0-11)
    // O^T tile m, heads 32hh..32hh+31 -> bf16, straight to global: lane = dim, so a warp writes
    // 64 contiguous bytes per head.  The producers are idle by now and reach the same TMEM lane
    // quarters (warp % 4), so each quarter's eight (tile, head half) units go to three warps.
    named_bar_sync(3, 384);  // warps 0-3 have seen the last MMAs complete and written den_s
    tc_fence_after();
    const int q4 = warp & 3, slot = warp >> 2;
    const int r = 32 * q4 + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * q4) << 16);
    uint16_t* orow = a.out + qrow * kH * kD;
    for (int u = slot; u < 8; u += 3) {
      const int m = u >> 1, hh = u & 1, d = 128 * m + r;
      float o[32];
      if (nloc > 0) {
        uint32_t v[32];
        tmem_ld32(lane_addr + 64 * m + 32 * hh, v);
        tmem_wait_ld();
#pragma unroll
        for (int h = 0; h < 32; ++h) o[h] = __uint_as_float(v[h]) * den_s[32 * hh + h];
      } else {
#pragma unroll
        for (int h = 0; h < 32; ++h) o[h] = 0.f;
      }
      if (m == 3 && q4 >= 2) {  // dims 448..511: rotate each (even, odd) pair back by -t
        float cs, sn;
        rope_cs(p, rf.inv_freq[(d - (kD - kDR)) >> 1], -1.0f, cs, sn);
        const bool odd = d & 1;
#pragma unroll
        for (int h = 0; h < 32; ++h) {
          const float partner = __shfl_xor_sync(0xffffffffu, o[h], 1);
          o[h] = odd ? fmaf(partner, sn, o[h] * cs) : fmaf(-partner, sn, o[h] * cs);
        }
      }
#pragma unroll
      for (int h = 0; h < 32; ++h) {
        const __nv_bfloat16 bv = __float2bfloat16_rn(o[h]);
        orow[(32 * hh + h) * kD + d] = *reinterpret_cast<const uint16_t*>(&bv);
      }
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
  grid_dep_wait();  // launched dependent on the split blocks
  const int t = blockIdx.x, bl = blockIdx.y, h = blockIdx.z;
  const int b = b0 + bl;
  const int64_t qrow = (int64_t)b * a.T + t;
  const int64_t lrow = (int64_t)bl * a.T + t;  // row within this launch's partials
  const int64_t p = seq_p0(pos, bl) + t;
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

namespace {
size_t attend_group_bytes(int nb, int T, int num_sms) {
  const int s = choose_splits(nb * T, num_sms);
  if (s == 1) return 0;
  const size_t rows = (size_t)nb * T * s;
  return rows * kH * kD * 4 + rows * kH * 2 * 4;
}
}  // namespace

// Launches take groups of kMaxSeqPerLaunch sequences; a smaller tail group may split more, so the
// need is the larger of the two group sizes.
size_t attend_workspace_bytes(int B, int T, int num_sms) {
  size_t need = attend_group_bytes(min(B, kMaxSeqPerLaunch), T, num_sms);
  if (B > kMaxSeqPerLaunch && B % kMaxSeqPerLaunch)
    need = std::max(need, attend_group_bytes(B % kMaxSeqPerLaunch, T, num_sms));
  return need;
}

cudaError_t launch_attend(const AttendArgs& a, const SeqPos& pos, const SeqPos& wst, int b0, int nb, const RopeFreq& rf, void* ws,
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
  // dependent launches: the kernel before each may still be ending when it is scheduled
  e = launch_dependent(attend_tc_kernel, dim3((unsigned)a.T, (unsigned)nb, (unsigned)s), dim3(kThreads), kDynBytes, st, a,
                       pos, wst, b0, rf, s, cps, po, pml);
  note_launch();
  if (e != cudaSuccess || (e = cudaGetLastError()) != cudaSuccess) return e;
  if (s > 1) {
    e = launch_dependent(attend_combine_kernel, dim3((unsigned)a.T, (unsigned)nb, kH), dim3(128), 0, st, a, pos, b0, rf,
                         s, po, pml);
    note_launch();
    if (e == cudaSuccess) e = cudaGetLastError();
  }
  return e;
}

// Reads and clears the attention kernels' device error word (0 = no bounded wait gave up).
// Reads and clears the domain flag of the attention kernel (0: every scale and query fitted fp16).
cudaError_t take_attend_domain(unsigned* flag) {
  const unsigned zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(flag, g_attend_domain, sizeof(unsigned));
  if (e == cudaSuccess && *flag != 0) e = cudaMemcpyToSymbol(g_attend_domain, &zero, sizeof(unsigned));
  return e;
}

cudaError_t take_attend_error(int* code) {
  const int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(code, g_attend_error, sizeof(int));
  if (e == cudaSuccess && *code != 0) e = cudaMemcpyToSymbol(g_attend_error, &zero, sizeof(int));
  return e;
}

}  // namespace csa2
