// Lightning-indexer scores for prefill on the tcgen05 tensor cores.
// Page "DeepSeek V4.1 - Pooled group / Source layer, pairs pooled", block "Compressed sparse
// attention": S^I_{t,j} = sum_h w^I_{t,h} ReLU(Q^I_{h,t} . K^I_j).
//
// As a GEMM: D[j, (t,h)] = K^I_j . Q^I_{t,h} with M = 128 keys, N = 256 = 8 queries x 32 heads,
// K = 128; the epilogue thread that owns key j (one TMEM lane) forms the 8 scores
// sum_h w_{t,h} ReLU(D[j, (t,h)]) in registers.  Both operands are the FP4 values re-encoded
// one per byte as E5M2 (E2M1 x 2^e is exact in E5M2 for scale exponents -15..13): Q^I is
// quantised to FP4 here exactly as in the CUDA-core path, then written as 32 KB "images" per
// query tile, K^I as 16 KB images per key tile, each image already in the 128B-swizzled
// K-major layout the MMA reads, so that one bulk copy (cp.async.bulk) stages it.  The score
// GEMM is four kind::f8f6f4 MMAs of K = 32 per key tile, one per 32-value scale block: within
// one MMA all key values share a scale and so do a head's query values, so each MMA's sum of
// 32 exact products is exact, and the fp32 accumulation across the four blocks is as for the
// CUDA-core path.
//
// Persistent kernel, 640 threads: warp 0 issues the bulk copies, warps 1 and 2 issue the MMAs
// of the even / odd key tiles (warp 1 allocates TMEM), warps 4-19 run the epilogue (four warps
// per TMEM lane quarter, each taking two of the tile's eight queries).  A query tile's image
// stays resident (double-buffered) while its causal key tiles stream through a kAStages ring;
// accumulators are double-buffered in TMEM (2 x 256 columns) so the epilogue of one tile
// overlaps the MMAs of the next.  Key tile i keeps ring stage i % kAStages and accumulator i % 2
// with the MMA thread of its parity (a commit tracks only its own thread's MMAs).  A thread's
// wait does not end before its own MMAs in flight have finished: with one MMA thread the tensor
// pipe idled during every wait, and with eight epilogue warps each waited out its own TMEM
// loads; both ran the kernel at well under its MMA time.
#include <cuda_fp16.h>

#include "csa2_common.cuh"
#include "csa2_fp16.cuh"
#include "csa2_sm100.cuh"

namespace csa2 {
namespace {

using namespace sm100;

constexpr int kQPerTile = 8;                       // queries per query tile (N = 256)
static_assert(kQPerTile % 2 == 0, "the epilogue reads two queries per TMEM wait");
constexpr uint32_t kQImg = 32768, kKImg = 16384;   // bytes per image: [256 | 128 rows][128 B] E5M2
constexpr int kEpiWarps = 16;                      // four per TMEM lane quarter, two queries each
constexpr int kThreadsTC = 128 + 32 * kEpiWarps;
constexpr int kAStages = 4;                        // key images in flight
static_assert(kAStages % 2 == 0 && kEpiWarps == 2 * kQPerTile, "stages keep their MMA thread; two queries per warp");
// dynamic smem: B (query images) 2 x 32 KB, A (key images) kAStages x 16 KB, w^I 2 x [8][32] floats,
// score-key histograms [8 queries][kHistBins] of the current query tile
constexpr uint32_t kBOff = 0, kAOff = 2 * kQImg, kWOff = kAOff + kAStages * kKImg, kHOff = kWOff + 2048,
                   kDynTC = kHOff + kQPerTile * kHistBins * 4 + 1024;

__device__ int g_index_error;
// Set when a kernel here read an FP4 scale above 2^13 (scale byte > 140): E2M1 x 2^e no longer
// fits fp16 (6 x 2^14 > 65504), so the tensor-core operands would overflow.  csa2_check reports it.
__device__ unsigned g_index_domain;
constexpr uint32_t kMaxScaleBytes = 0x8C8C8C8Cu;  // 140 in every byte: 2^13, the largest exact fp16 scale


// Q^I (bf16) -> FP4 (E2M1, UE8M0 per 32) -> E5M2 image.  grid (Tq, nb), 128 threads: warp w
// handles heads 8w..8w+7, lane l values 4l..4l+3.  Query t of the chunk lives in tile t/8,
// rows (t%8)*32 + h of the tile's [256 x 128] K-major image (one 128-byte swizzle atom per row).
__global__ void __launch_bounds__(128) qimage_kernel(IndexArgs a, int b0, int t0, int Tq, int nqt, uint8_t* qimg,
                                                     float* wq) {
  const int tl = blockIdx.x, bl = blockIdx.y;
  const int t = t0 + tl;
  const int b = b0 + bl;
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  const int64_t src = (int64_t)b * a.T + t;
  uint8_t* tile = qimg + ((int64_t)bl * nqt + tl / kQPerTile) * kQImg;
  uint2 rawv[8];  // the warp's eight head rows, all loads in flight before any store
#pragma unroll
  for (int k = 0; k < 8; ++k) rawv[k] = __ldg(reinterpret_cast<const uint2*>(a.qi + (src * kHI + 8 * w + k) * kDI + 4 * l));
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int h = 8 * w + k;
    const uint2 raw = rawv[k];
    float v[4] = {bf16_to_f32(raw.x & 0xffff), bf16_to_f32(raw.x >> 16), bf16_to_f32(raw.y & 0xffff), bf16_to_f32(raw.y >> 16)};
    float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
    const int e = mx_scale_exp(amax);
    if (e > 13 && l == 0) atomicOr(&g_index_domain, 1u);
    const float down = pow2f(-e), up = pow2f(e);  // exact powers of two
    float q[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) q[i] = e2m1_to_f32(f32_to_e2m1(v[i] * down)) * up;
    const uint32_t img = cvt_f32x2_e5m2x2(q[0], q[1]) | (cvt_f32x2_e5m2x2(q[2], q[3]) << 16);
    const int n = (tl % kQPerTile) * kHI + h, d = 4 * l;
    *reinterpret_cast<uint32_t*>(tile + sw128_off(n, d >> 4) + (d & 15)) = img;
  }
  if (threadIdx.x < kHI) wq[((int64_t)bl * Tq + tl) * kHI + threadIdx.x] = bf16_to_f32(a.wI[src * kHI + threadIdx.x]);
}

// K^I (FP4) -> E5M2 image.  grid (key tiles, nb), 128 threads: thread = key of the tile, its 128
// values one byte each in row r of the tile's [128 x 128] 128B-swizzled image.
__global__ void __launch_bounds__(128) kimage_kernel(IndexArgs a, int b0, int64_t n_keys, int nkt, uint8_t* kimg) {
  const int kt = blockIdx.x, bl = blockIdx.y;
  const int b = b0 + bl;
  const int r = threadIdx.x;
  const int64_t j = (int64_t)kt * 128 + r;
  uint8_t* tile = kimg + ((int64_t)bl * nkt + kt) * kKImg;
  uint4 c[4];
  uint32_t sc = 0;
  if (j < n_keys) {
    const uint4* src = reinterpret_cast<const uint4*>(a.ki_codes + ((int64_t)b * a.cap + j) * 64);
#pragma unroll
    for (int i = 0; i < 4; ++i) c[i] = src[i];
    sc = *reinterpret_cast<const uint32_t*>(a.ki_scales + ((int64_t)b * a.cap + j) * 4);
    if (__vcmpgtu4(sc, kMaxScaleBytes)) atomicOr(&g_index_domain, 1u);
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) c[i] = make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int blk = 0; blk < 4; ++blk) {  // 32 values: 16 bytes of codes, one scale byte
    const float s = pow2f((int)((sc >> (8 * blk)) & 255u) - 127);
    const uint32_t wd[4] = {c[blk].x, c[blk].y, c[blk].z, c[blk].w};
#pragma unroll
    for (int q = 0; q < 2; ++q) {  // 16 values = one 16-byte chunk of E5M2
      uint32_t o[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t word = wd[2 * q + (k >> 1)] >> (16 * (k & 1));  // four values: two code bytes
        const float v0 = e2m1_to_f32(word & 15u) * s, v1 = e2m1_to_f32((word >> 4) & 15u) * s;
        const float v2 = e2m1_to_f32((word >> 8) & 15u) * s, v3 = e2m1_to_f32((word >> 12) & 15u) * s;
        o[k] = cvt_f32x2_e5m2x2(v0, v1) | (cvt_f32x2_e5m2x2(v2, v3) << 16);
      }
      *reinterpret_cast<uint4*>(tile + sw128_off(r, 2 * blk + q)) = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

struct TcBars {
  uint64_t b_full[2], b_free[2], a_full[kAStages], a_free[kAStages], d_full[2], d_free[2];
};

// The static schedule: in round r CTA c takes query tile r*G + c (even rounds) or
// r*G + G-1-c (odd rounds), a zig-zag that balances the causal work (key tiles grow with the
// query index) across CTAs.  -1 past the last tile.
__device__ __forceinline__ int tile_of(int round, int G, int ntiles) {
  const int idx = round * G + ((round & 1) ? (G - 1 - (int)blockIdx.x) : (int)blockIdx.x);
  return idx < ntiles ? idx : -1;
}

// Lower edge (a score key) of the histogram bin that holds the K-th largest counted key, found
// by one warp: every key among the K largest is >= it.  0 when fewer than K keys were counted.
// Steps of 32 consecutive bins from the top (lane l: bin base - l, so the loads are free of bank
// conflicts), a running count (one warp reduction per step), and a prefix scan only in the first
// step that reaches K.
__device__ uint32_t warp_hist_lower(const uint32_t* hist, int K, int lane) {
  uint32_t carry = 0;
  for (int base = kHistBins - 1; base >= 0; base -= 32) {
    const uint32_t c = hist[base - lane];
    const uint32_t tot = __reduce_add_sync(0xffffffffu, c);
    if (carry + tot < (uint32_t)K) {
      carry += tot;
      continue;
    }
    uint32_t incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const uint32_t hit = __ballot_sync(0xffffffffu, carry + incl >= (uint32_t)K);
    if (hit) return (uint32_t)(base - (__ffs(hit) - 1)) << kHistShift;
    carry += __shfl_sync(0xffffffffu, incl, 31);
  }
  return 0u;
}

// lower_out (optional) [nb * Tq]: per query row, the histogram lower edge of its top-512 (keys
// below it cannot be selected), for the select that follows.
// cand (optional, with lower_out): instead of the dense score rows, each query row gets the list of
// its candidates, (score key, position) pairs in cand_key / cand_j: four segments of ld / 4 slots
// from row * ld, segment s for the keys of TMEM lane quarter s (key rows 32s .. 32s+31 of each
// tile), filled by the one warp that owns that (query, quarter), its count in cand_n[row * 4 + s].
// A key is a candidate unless it lies below the lower edge of the histogram bin of the K-th
// largest key counted so far for its query (thr_run, refreshed after 8, 16, 32, ... key tiles, so
// that each stretch between refreshes adds about K candidates at most, for a few refreshes): that
// edge only rises, and never above the row's final lower edge, so every key of the row's top-K is
// listed, and the lists hold all keys at or above the row's final edge.  ld is a multiple of 128.
__global__ void __launch_bounds__(kThreadsTC, 1) index_prefill_tc_kernel(IndexArgs a, SeqPos pos, int t0, int tq, int nqt,
                                                                         int nkt, const uint8_t* qimg, const uint8_t* kimg,
                                                                         const float* wq, float* scores, int64_t ld,
                                                                         int nb, int Tq, uint32_t* lower_out,
                                                                         int32_t* cand_j, int* cand_n) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ TcBars bars;
  __shared__ uint32_t tmem_base_sh;
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  unsigned char* sm = smem_raw + (sbase - smem_u32(smem_raw));
  float* sw = reinterpret_cast<float*>(sm + kWOff);  // [2][8][32]
  uint32_t* shist = reinterpret_cast<uint32_t*>(sm + kHOff);  // [8][kHistBins]
  __shared__ uint32_t thr_run[kQPerTile];                     // candidate bound per query of the tile
  uint32_t* cand_key = reinterpret_cast<uint32_t*>(scores);   // the score rows' space holds the keys
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nqt_act = (tq + kQPerTile - 1) / kQPerTile;  // query tiles of this pass (image stride: nqt)
  const int G = gridDim.x, ntiles = nb * nqt_act;
  int* err = &g_index_error;

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.b_full[i], 1);
      mbar_init(&bars.b_free[i], 2);  // both MMA threads
      mbar_init(&bars.d_full[i], 1);
      mbar_init(&bars.d_free[i], kEpiWarps);
    }
    for (int i = 0; i < kAStages; ++i) {
      mbar_init(&bars.a_full[i], 1);
      mbar_init(&bars.a_free[i], 1);
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

  // key tiles needed by query tile qt of sequence bl: entries visible to its last query
  auto n_key_tiles = [&](int bl, int qt) {
    const int tlast = min(tq, (qt + 1) * kQPerTile) - 1;
    const int64_t E = (seq_p0(pos, bl) + t0 + tlast + 1) >> a.rshift;
    return (int)((E + 127) / 128);
  };

  if (warp == 0) {
    // ============================================================ bulk-copy producer
    if (lane == 0) {
      int it = 0, qi = 0;
      for (int k = 0; k * G < ntiles; ++k) {
        const int tile = tile_of(k, G, ntiles);
        if (tile < 0) continue;
        const int bl = tile / nqt_act, qt = tile % nqt_act;
        const int nk = n_key_tiles(bl, qt);
        if (nk == 0) continue;
        const int sB = qi & 1;
        if (qi >= 2) mbar_wait(&bars.b_free[sB], ((qi >> 1) - 1) & 1, err, 11);
        mbar_arrive_expect_tx(&bars.b_full[sB], kQImg);
        const uint8_t* qsrc = qimg + ((int64_t)bl * nqt + qt) * kQImg;
        for (int c = 0; c < 2; ++c) bulk_g2s(sm + kBOff + sB * kQImg + c * 16384, qsrc + c * 16384, 16384, &bars.b_full[sB]);
        for (int kt = 0; kt < nk; ++kt, ++it) {
          const int sA = it % kAStages;
          if (it >= kAStages) mbar_wait(&bars.a_free[sA], ((it / kAStages) - 1) & 1, err, 12);
          mbar_arrive_expect_tx(&bars.a_full[sA], kKImg);
          bulk_g2s(sm + kAOff + sA * kKImg, kimg + ((int64_t)bl * nkt + kt) * kKImg, kKImg, &bars.a_full[sA]);
        }
        ++qi;
      }
    }
  } else if (warp == 1 || warp == 2) {
    // ============================================================ MMA threads (key tiles of parity warp - 1)
    if (lane == 0) {
      const uint32_t idesc = idesc_e5m2(128, 256);
      const int par = warp - 1;
      int it = 0, qi = 0, dc = 0;
      for (int k = 0; k * G < ntiles; ++k) {
        const int tile = tile_of(k, G, ntiles);
        if (tile < 0) continue;
        const int bl = tile / nqt_act, qt = tile % nqt_act;
        const int nk = n_key_tiles(bl, qt);
        if (nk == 0) continue;
        const int sB = qi & 1;
        mbar_wait(&bars.b_full[sB], (qi >> 1) & 1, err, 13);
        for (int kt = 0; kt < nk; ++kt, ++it, ++dc) {
          if ((it & 1) != par) continue;
          const int sA = it % kAStages, sD = dc & 1;
          mbar_wait(&bars.a_full[sA], (it / kAStages) & 1, err, 14);
          if (dc >= 2) mbar_wait(&bars.d_free[sD], ((dc >> 1) - 1) & 1, err, 15);
          tc_fence_after();
          const uint32_t abase = sbase + kAOff + sA * kKImg, bbase = sbase + kBOff + sB * kQImg;
#pragma unroll
          for (int k32 = 0; k32 < 4; ++k32)  // one MMA per 32-value scale block (32 bytes of each row)
            mma_f8_ss(tmem + 256 * sD, sw128_desc(abase + k32 * 32, 16, 1024), sw128_desc(bbase + k32 * 32, 16, 1024),
                      idesc, k32 > 0);
          mma_commit(&bars.a_free[sA]);
          mma_commit(&bars.d_full[sD]);
        }
        mma_commit(&bars.b_free[sB]);
        ++qi;
      }
    }
  } else if (warp >= 4) {
    // ============================================================ epilogue
    // warp 4 + 4*pair + quarter: keys 32*quarter .. (its TMEM lane quarter), queries 2*pair, +1
    const int ew = warp - 4, quarter = ew & 3, pair = ew >> 2, r = 32 * quarter + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * quarter) << 16);
    constexpr int kEpiThreads = 32 * kEpiWarps;
    int dc = 0, qi = 0;
    for (int k = 0; k * G < ntiles; ++k) {
      const int tile = tile_of(k, G, ntiles);
      if (tile < 0) continue;
      const int bl = tile / nqt_act, qt = tile % nqt_act;
      const int nk = n_key_tiles(bl, qt);
      if (nk == 0) continue;
      float* wsm = sw + (qi & 1) * 256;
      named_bar_sync(2, kEpiThreads);  // the previous use of this w buffer and of the histograms is finished
      for (int i = tid - 128; i < 256; i += kEpiThreads) {
        const int tl = qt * kQPerTile + i / kHI;
        wsm[i] = tl < tq ? wq[((int64_t)bl * Tq + tl) * kHI + (i % kHI)] : 0.f;
      }
      if (lower_out)
        for (int i = tid - 128; i < kQPerTile * kHistBins; i += kEpiThreads) shist[i] = 0u;
      if (tid - 128 < kQPerTile) thr_run[tid - 128] = 0u;
      named_bar_sync(2, kEpiThreads);
      const int64_t p0 = seq_p0(pos, bl) + t0;
      // key tiles below this bound are visible to all eight queries (the first has the fewest)
      const int64_t e_first = (p0 + qt * kQPerTile + 1) >> a.rshift;
      const bool all_queries = qt * kQPerTile + kQPerTile <= tq;
      int ncand[2] = {0, 0};  // this warp's candidates of its two queries (its lane quarter's segment)
      for (int kt = 0; kt < nk; ++kt, ++dc) {
        const int sD = dc & 1;
        mbar_wait(&bars.d_full[sD], (dc >> 1) & 1, err, 16);
        tc_fence_after();
        const int64_t j = (int64_t)kt * 128 + r;
        const bool full = all_queries && (int64_t)(kt + 1) * 128 <= e_first;
        // two queries per TMEM wait, four independent partial sums per query (heads h mod 4, two
        // packed pairs); four warps per sub-partition hide each other's load waits
        {
          const int q = 2 * pair;
          uint32_t u[2][32];
          tmem_ld32(lane_addr + 256 * sD + 32 * q, u[0]);
          tmem_ld32(lane_addr + 256 * sD + 32 * (q + 1), u[1]);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int tl = qt * kQPerTile + q + e;
            const float4* w4 = reinterpret_cast<const float4*>(wsm + 32 * (q + e));
            float2 s01 = make_float2(0.f, 0.f), s23 = make_float2(0.f, 0.f);
#pragma unroll
            for (int h4 = 0; h4 < 8; ++h4) {
              const float4 w = w4[h4];
              s01 = fma2(make_float2(w.x, w.y),
                         make_float2(fmaxf(__uint_as_float(u[e][4 * h4]), 0.f), fmaxf(__uint_as_float(u[e][4 * h4 + 1]), 0.f)),
                         s01);
              s23 = fma2(make_float2(w.z, w.w),
                         make_float2(fmaxf(__uint_as_float(u[e][4 * h4 + 2]), 0.f), fmaxf(__uint_as_float(u[e][4 * h4 + 3]), 0.f)),
                         s23);
            }
            const bool ok = full || (tl < tq && j < ((p0 + tl + 1) >> a.rshift));
            const float sc = (s01.x + s01.y) + (s23.x + s23.y);
            const int64_t rq = (int64_t)bl * Tq + tl;
            if (!cand_j) {
              if (ok) {
                scores[rq * ld + j] = sc;
                if (lower_out) atomicAdd(&shist[(q + e) * kHistBins + (score_key(sc) >> kHistShift)], 1u);
              }
            } else {
              // candidates: keys at or above the query's running bound, appended in warp batches
              const uint32_t key = score_key(sc);
              if (ok) atomicAdd(&shist[(q + e) * kHistBins + (key >> kHistShift)], 1u);
              const bool app = ok && key >= *reinterpret_cast<volatile uint32_t*>(&thr_run[q + e]);
              const uint32_t bal = __ballot_sync(0xffffffffu, app);
              if (app) {
                const int64_t at = rq * ld + quarter * (ld >> 2) + ncand[e] + __popc(bal & ((1u << lane) - 1u));
                cand_key[at] = key;
                cand_j[at] = (int32_t)j;
              }
              ncand[e] += __popc(bal);
            }
          }
        }
        // released after the scores are formed: releasing it right after the TMEM loads let the
        // MMAs two tiles on run beside these loads and made the kernel slower
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.d_free[sD]);
        if (cand_j && ew < kQPerTile && kt >= 7 && ((kt + 1) & kt) == 0) {
          // warp ew: a new bound for query ew from its histogram so far (other warps may still be
          // adding to it: a histogram with fewer keys only gives a lower bound)
          const int tl = qt * kQPerTile + ew;
          if (tl < tq) {
            const int64_t E = (p0 + tl + 1) >> a.rshift;
            const uint32_t lo = warp_hist_lower(shist + ew * kHistBins, (int)min64(kTopK, E), lane);
            if (lane == 0) thr_run[ew] = lo;
          }
        }
      }
      if (cand_j && lane == 0)
        for (int e = 0; e < 2; ++e) {
          const int tl = qt * kQPerTile + 2 * pair + e;
          if (tl < tq) cand_n[((int64_t)bl * Tq + tl) * 4 + quarter] = ncand[e];
        }
      if (lower_out) {  // warp ew < 8: the lower edge of query ew's top-512 from its histogram
        named_bar_sync(2, kEpiThreads);  // every count of this query tile is in
        const int tl = qt * kQPerTile + ew;
        if (ew < kQPerTile && tl < tq) {
          const int64_t E = (p0 + tl + 1) >> a.rshift;
          const uint32_t lo = warp_hist_lower(shist + ew * kHistBins, (int)min64(kTopK, E), lane);
          if (lane == 0) lower_out[(int64_t)bl * Tq + tl] = lo;
        }
      }
      ++qi;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------ decode (one query)
// Scores of one query per sequence against all its visible keys on the block-scaled FP4
// tensor-core path (tcgen05.mma kind::mxf4): the cached K^I codes and UE8M0 scales are the MMA
// operands as they are stored, with no decode.  D[key, head] = K^I_key . Q^I_head, M = 128 keys,
// N = 32 heads, K = 128 per tile as two MMAs of K = 64 (scale bytes 0-1, then 2-3).  Q^I is
// quantised to FP4 (E2M1, UE8M0 per 32) in the kernel exactly as in the oracle.  Each MMA's
// products are exact and the fp32 accumulation is the tensor core's.
// A unit is two tiles (256 positions); units cycle through kMSlots shared-memory stages and
// TMEM slots (accumulators 2 x 32 columns, A scale words 2 x 4 columns):
//  - warps 0 and 1 (one thread each): the even / odd units; per unit, one wait (sf_full), four
//    MMAs and one commit (done).  A thread's wait does not end before its own MMAs in flight
//    have finished, so one thread alone left the tensor pipe idle for half of each unit; with
//    two, one issues while the other waits.  A slot (s = u mod kMSlots, kMSlots even) stays with
//    one thread: a commit tracks only the MMAs of the thread that issues it.
//  - warp 2 (producer): TMA copies of the unit's code rows (64 bytes each) into a stage with the
//    64-byte swizzle the MMA reads (one 256-row box, or one 8-row box per pool block), and of its
//    scale words (4 bytes per key; boxes of 256 + 4 words, or 12 words per pool block, that start
//    at a multiple of 4 words: a tensor copy must start on a 16-byte boundary, and a sequence's
//    words start at word cap * b).  Every box lands at a multiple of 128 bytes in shared memory,
//    as tensor copies require (pool blocks' scale boxes 128 bytes apart).  A stage is refilled once the MMAs that read it have completed
//    (done of the unit kMSlots before).  Scale words read by each thread with plain loads arrived
//    too late: with the copies keeping ~100 KB per SM in flight, a load waited behind them for
//    several units' time.
//  - warps 3-6 (scale warps, TMEM lane quarter = warp % 4): once the epilogue has read the slot's
//    accumulators (d_free) and the unit's copies have landed (s_full), the unit's A scale words
//    from the stage into TMEM, the same words in every quarter (column c, lane i: row 32c + i);
//    then they release the unit to the MMA thread (sf_full).  They also write Q^I's codes and
//    scale words.
//  - warps 7-14 (epilogue, TMEM lane quarter = warp % 4; group (warp - 7) / 4 takes tile 0 or 1
//    of each unit): ReLU, the w^I weighting and the fp32 score stores.
// Earlier designs decoded the FP4 keys to fp16 in the kernel (sixteen decoder warps, eight
// kind::f16 MMAs per tile): every stage ran far below the copy bandwidth, and the chain of
// handshakes per tile set the pace.  Here a tile costs two MMAs and a unit one wait per role.
// Rows: one query (sequence bl, query t0 + tl) each; a row's key tiles are split evenly (an even
// count per block) over gridDim.x / rows persistent blocks.  With hist, each row also gets the
// histogram of its score keys (kHistBins bins, added up over its blocks) that lets the top-k skip
// most keys.  With a pool (hierarchical indexer, reindex scan) the row's positions p are its
// pool's entries 8 * pool[p / 8] + p % 8 instead of 0 .. E-1.  Positions past the row's end are
// computed from whatever rows the copies brought (or zeros) and never stored.
constexpr int kMSlots = 6;                          // units in flight: stages = TMEM slots
constexpr int kMThreads = 32 * 15;
constexpr int kMMma = 0, kMProd = 2, kMSf0 = 3, kMEpi0 = 7;  // MMA threads: warps 0 (even units) and 1 (odd)
constexpr uint32_t kMStage = 16384;                 // smem per stage: 256 rows x 64 B of codes
constexpr uint32_t kMQOff = 0;                      // smem: Q^I codes, 32 rows x 64 B (SW64)
constexpr uint32_t kMStageOff = 2048;               // smem: stages (1024-aligned)
constexpr uint32_t kMScw = 4096;                    // smem per stage: scale words (260, or 32 x 12 at 128 B)
constexpr uint32_t kMScOff = kMStageOff + kMSlots * kMStage;
constexpr uint32_t kDynMx = kMScOff + kMSlots * kMScw + 1024;
constexpr uint32_t kMAccCol = 0;                    // TMEM: slot s accumulators at 64 s (tile t: + 32 t)
constexpr uint32_t kMSfaCol = 64 * kMSlots;         // TMEM: slot s A scale words at kMSfaCol + 8 s (+ 4 t)
constexpr uint32_t kMSfbCol = kMSfaCol + 8 * kMSlots;  // TMEM: Q^I scale words (one column)
static_assert(kMSfbCol % 4 == 0 && kMSfbCol + 1 <= 512, "TMEM columns");
static_assert(kMStageOff % 1024 == 0 && kMStage % 1024 == 0 && kMScOff % 128 == 0 && kMScw % 128 == 0,
              "tensor-copy destinations: 128-byte aligned (1024 for the swizzled code rows)");
static_assert(kMEpi0 + 8 == kMThreads / 32 && kMSlots % 2 == 0, "warp roles; a slot keeps its MMA thread");

// s_full[s]: the unit's code rows and scale words landed (transaction count).  sf_full[s]: its scale words are
// in TMEM and its codes landed (4 scale warps).  done[s]: its MMAs completed (one commit): the
// stage is free and the accumulators hold its scores.  d_free[s]: the epilogue read them (8 warps).
struct MxBars {
  uint64_t s_full[kMSlots], sf_full[kMSlots], done[kMSlots], d_free[kMSlots];
};

__global__ void __launch_bounds__(kMThreads, 1) index_decode_mx_kernel(const __grid_constant__ CUtensorMap map_unit,
                                                                       const __grid_constant__ CUtensorMap map_block,
                                                                       const __grid_constant__ CUtensorMap map_sw256,
                                                                       const __grid_constant__ CUtensorMap map_sw4,
                                                                       const __grid_constant__ CUtensorMap map_sw12,
                                                                       IndexArgs a, SeqPos pos, int b0, int nb,
                                                                       int t0, int tq, int Tq, float* scores,
                                                                       int64_t ld, int* rowlen, uint32_t* hist) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ MxBars bars;
  __shared__ uint32_t shist[kHistBins];
  __shared__ uint32_t tmem_base_sh;
  __shared__ float wsh[kHI];
  grid_dep_trigger();  // the select that follows may be scheduled as this kernel's blocks end
  __shared__ uint32_t qsf[kHI];  // Q^I scale word per head (byte k: block k)
  __shared__ int32_t spool[kHsiBlocks];
  __shared__ int64_t n_sh;
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  unsigned char* sm = smem_raw + (sbase - smem_u32(smem_raw));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int* err = &g_index_error;
  // this block's query row and key-tile range
  const int nrows = nb * tq;
  const int per_row = max(1, (int)gridDim.x / nrows);
  const int rr = blockIdx.x / per_row, part = blockIdx.x % per_row;
  const bool active = rr < nrows;
  const int bl = active ? rr / tq : 0, tl = active ? rr % tq : 0;
  const int b = b0 + bl;
  const int64_t qrow = (int64_t)b * a.T + t0 + tl;
  const int64_t E = active ? (seq_p0(pos, bl) + t0 + tl + 1) >> a.rshift : 0;  // visible entries of the query
  const int32_t* prow = a.pool_in ? a.pool_in + qrow * kHsiBlocks : nullptr;
  if (active && prow)
    for (int i = tid; i < kHsiBlocks; i += kMThreads) spool[i] = prow[i];
  if (hist)
    for (int i = tid; i < kHistBins; i += kMThreads) shist[i] = 0u;
  __syncthreads();
  if (tid == 0) {
    int64_t n = E;
    if (prow) {  // ascending blocks, -1 padded; only the last (newest) block can be partial
      int lo = 0, hi = kHsiBlocks;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (spool[mid] >= 0) lo = mid + 1;
        else hi = mid;
      }
      n = lo == 0 ? 0 : (int64_t)kHsiBlock * (lo - 1) + min64(kHsiBlock, E - (int64_t)kHsiBlock * spool[lo - 1]);
      n = max64(n, 0);
    }
    n_sh = active ? n : 0;
    if (rowlen && active && part == 0) rowlen[bl * Tq + tl] = (int)n_sh;
  }
  __syncthreads();
  const int64_t n_pos = n_sh;  // positions of the row
  const int ntile = (int)((n_pos + 127) / 128);
  const int tpb = 2 * ((ntile + 2 * per_row - 1) / (2 * per_row));  // even: whole units
  const int t_begin = min(ntile, part * tpb), t_end = min(ntile, t_begin + tpb);
  const int nt = active ? t_end - t_begin : 0;
  const int nu = (nt + 1) / 2;

  if (tid == 0) {
    for (int i = 0; i < kMSlots; ++i) {
      mbar_init(&bars.s_full[i], 1);
      mbar_init(&bars.sf_full[i], 4);  // the four scale warps
      mbar_init(&bars.done[i], 1);
      mbar_init(&bars.d_free[i], 8);   // the eight epilogue warps
    }
    mbar_fence_init();
  }
  if (warp == kMMma) {
    tmem_alloc(&tmem_base_sh, 512);
    tmem_relinquish();
  }
  // Q^I -> FP4 codes (scale warps: warp heads 8(w - kMSf0)..+7, lane l values 4l..4l+3), w^I
  if (warp >= kMSf0 && warp < kMSf0 + 4 && active) {
    const int hw = warp - kMSf0;
    for (int h = 8 * hw; h < 8 * hw + 8; ++h) {
      const uint2 raw = *reinterpret_cast<const uint2*>(a.qi + (qrow * kHI + h) * kDI + 4 * lane);
      float v[4] = {bf16_to_f32(raw.x & 0xffff), bf16_to_f32(raw.x >> 16), bf16_to_f32(raw.y & 0xffff), bf16_to_f32(raw.y >> 16)};
      float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
      const int e = mx_scale_exp(amax);
      if (e > 13 && lane == 0) atomicOr(&g_index_domain, 1u);
      const float down = pow2f(-e);  // exact power of two
      const uint32_t c0 = f32_to_e2m1(v[0] * down), c1 = f32_to_e2m1(v[1] * down);
      const uint32_t c2 = f32_to_e2m1(v[2] * down), c3 = f32_to_e2m1(v[3] * down);
      *reinterpret_cast<uint16_t*>(sm + kMQOff + sw64_off(h, lane >> 3) + ((2 * lane) & 15)) =
          (uint16_t)(c0 | (c1 << 4) | (c2 << 8) | (c3 << 12));
      // scale byte of block lane / 8 (values 32k .. 32k+31) into byte k of the head's word
      const uint32_t sb = (uint32_t)(e + 127);
      const uint32_t w0 = __shfl_sync(0xffffffffu, sb, 0), w1 = __shfl_sync(0xffffffffu, sb, 8);
      const uint32_t w2 = __shfl_sync(0xffffffffu, sb, 16), w3 = __shfl_sync(0xffffffffu, sb, 24);
      if (lane == 0) qsf[h] = w0 | (w1 << 8) | (w2 << 16) | (w3 << 24);
    }
    if (hw == 0) wsh[lane] = bf16_to_f32(a.wI[qrow * kHI + lane]);
    fence_proxy_async();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  if (warp < kMProd) {
    // ============================================================ MMA threads
    if (lane == 0) {
      const uint32_t id0 = idesc_mxf4(128, 32, 0, 0), id1 = idesc_mxf4(128, 32, 2, 2);
      const uint64_t bq0 = sw64_desc(sbase + kMQOff), bq1 = sw64_desc(sbase + kMQOff + 32);
      for (int u = warp - kMMma; u < nu; u += 2) {
        const int s = u % kMSlots;
        mbar_wait(&bars.sf_full[s], (u / kMSlots) & 1, err, 22);
        tc_fence_after();
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const uint32_t d = tmem + kMAccCol + 64 * s + 32 * t, sfa = tmem + kMSfaCol + 8 * s + 4 * t;
          const uint32_t abase = sbase + kMStageOff + s * kMStage + t * 8192;
          mma_mxf4(d, sw64_desc(abase), bq0, id0, sfa, tmem + kMSfbCol, 0u);
          mma_mxf4(d, sw64_desc(abase + 32), bq1, id1, sfa, tmem + kMSfbCol, 1u);
        }
        mma_commit(&bars.done[s]);
      }
    }
    __syncwarp();
  } else if (warp == kMProd) {
    // ============================================================ producer: code rows
    const int64_t row0 = (int64_t)bl * a.cap;  // the sequence's first row (and scale word) in the tensor maps
    const int k0 = (int)(row0 & 3);            // scale boxes start k0 words early, on a 16-byte boundary
    const int64_t p_end = min64(n_pos, (int64_t)t_end * 128);
#pragma unroll 1
    for (int u = 0; u < nu; ++u) {
      const int s = u % kMSlots;
      if (u >= kMSlots) mbar_wait(&bars.done[s], ((u / kMSlots) - 1) & 1, err, 36);
      unsigned char* dst = sm + kMStageOff + s * kMStage;
      unsigned char* scd = sm + kMScOff + s * kMScw;
      const int64_t pu = (int64_t)(t_begin + 2 * u) * 128;  // first position of the unit
      if (!prow) {
        if (lane == 0) {
          const int x0 = (int)(row0 + pu - k0);  // words x0 .. x0 + 259 hold the unit's 256 at k0 ..
          mbar_arrive_expect_tx(&bars.s_full[s], kMStage + 1024 + 16);
          tma_load_2d(dst, &map_unit, 0, (int)(row0 + pu), &bars.s_full[s]);
          tma_load_1d(scd, &map_sw256, x0, &bars.s_full[s]);
          tma_load_1d(scd + 1024, &map_sw4, x0 + 256, &bars.s_full[s]);
        }
      } else {
        // lane k: pool block k of the unit (positions pu + 8k .. + 7, stage rows 8k .. + 7, scale
        // words 32k + k0 .. + 7)
        const int64_t pp = pu + 8 * lane;
        const int32_t blk = pp < p_end ? spool[pp >> 3] : -1;
        const uint32_t total = __reduce_add_sync(0xffffffffu, blk >= 0 ? 512u + 48u : 0u);
        if (lane == 0) mbar_arrive_expect_tx(&bars.s_full[s], total);
        __syncwarp();
        if (blk >= 0) {
          const int64_t j0 = row0 + (int64_t)kHsiBlock * blk;
          tma_load_2d(dst + lane * 512, &map_block, 0, (int)j0, &bars.s_full[s]);
          tma_load_1d(scd + lane * 128, &map_sw12, (int)(j0 - k0), &bars.s_full[s]);
        }
      }
    }
  } else if (warp < kMEpi0) {
    // ============================================================ scale warps: thread = row of column c
    const int q4 = warp & 3;
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * q4) << 16);
    const int k0 = (int)(((int64_t)bl * a.cap) & 3);  // offset of the stage's first scale word
    tmem_st1(lane_addr + kMSfbCol, qsf[lane]);         // Q^I row (head) lane, every quarter
#pragma unroll 1
    for (int u = 0; u < nu; ++u) {
      const int s = u % kMSlots;
      const int64_t pu = (int64_t)(t_begin + 2 * u) * 128;
      if (u >= kMSlots) mbar_wait(&bars.d_free[s], ((u / kMSlots) - 1) & 1, err, 34);
      mbar_wait(&bars.s_full[s], (u / kMSlots) & 1, err, 35);
      tc_fence_after();
      // tile t, column c -> unit row i = 128t + 32c + lane (1.0 in every byte past the row's end)
      const uint32_t* wsc = reinterpret_cast<const uint32_t*>(sm + kMScOff + s * kMScw) + k0;
      uint32_t v[8], big = 0;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int i = 128 * (k >> 2) + 32 * (k & 3) + lane;
        v[k] = pu + i < n_pos ? wsc[prow ? 32 * (i >> 3) + (i & 7) : i] : 0x7F7F7F7Fu;
        big |= __vcmpgtu4(v[k], kMaxScaleBytes);
      }
      if (big) atomicOr(&g_index_domain, 1u);
      tmem_st4(lane_addr + kMSfaCol + 8 * s, v[0], v[1], v[2], v[3]);
      tmem_st4(lane_addr + kMSfaCol + 8 * s + 4, v[4], v[5], v[6], v[7]);
      tmem_wait_st();
      fence_proxy_async();  // these reads of the stage, before the copy that next overwrites it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.sf_full[s]);
    }
  } else {
    // ============================================================ epilogue: thread = key lane
    const int q4 = warp & 3;            // TMEM lane quarter
    const int t = (warp - kMEpi0) >> 2;  // tile of the unit
    const int r = 32 * q4 + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * q4) << 16) + kMAccCol + 32 * t;
    float* out = scores + ((int64_t)bl * Tq + tl) * ld;  // indexed by position
    float wr[kHI];
#pragma unroll
    for (int h = 0; h < kHI; ++h) wr[h] = wsh[h];
    for (int u = 0; u < nu; ++u) {
      const int s = u % kMSlots;
      mbar_wait(&bars.done[s], (u / kMSlots) & 1, err, 24);
      tc_fence_after();
      uint32_t acc[32];
      tmem_ld32(lane_addr + 64 * s, acc);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.d_free[s]);
      float s4[4] = {0.f, 0.f, 0.f, 0.f};  // four independent chains of 8
#pragma unroll
      for (int h = 0; h < 32; ++h) s4[h & 3] = fmaf(wr[h], fmaxf(__uint_as_float(acc[h]), 0.f), s4[h & 3]);
      const int i = 2 * u + t;
      const int64_t pp = (int64_t)(t_begin + i) * 128 + r;
      if (i < nt && pp < n_pos) {
        const float sc = (s4[0] + s4[1]) + (s4[2] + s4[3]);
        out[pp] = sc;
        if (hist) atomicAdd(&shist[score_key(sc) >> kHistShift], 1u);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMMma) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (hist && nt > 0) {  // this block's counts into the row's histogram
    uint32_t* hrow = hist + ((int64_t)bl * Tq + tl) * kHistBins;
    for (int i = tid; i < kHistBins; i += kMThreads)
      if (shist[i]) atomicAdd(hrow + i, shist[i]);
  }
}

}  // namespace

cudaError_t launch_index_scores_decode_tc(const IndexArgs& a, const SeqPos& pos, int b0, int nb, int t0, int tq,
                                          int Tq, float* scores, int64_t ld, int* rowlen, uint32_t* hist,
                                          int num_sms, cudaStream_t st) {
  // the nb sequences' code rows [nb * cap][64 B]: 256-row boxes (a unit) and 8-row boxes (a pool
  // block); their scale words [nb * cap] (u32): boxes of 256 + 4 words and of 12 words
  CUtensorMap map_unit, map_block, map_sw256, map_sw4, map_sw12;
  const uint8_t* codes = a.ki_codes + (int64_t)b0 * a.cap * 64;
  const uint8_t* words = a.ki_scales + (int64_t)b0 * a.cap * 4;
  const uint64_t rows = (uint64_t)nb * a.cap;
  if (rows + 512 > (uint64_t)INT32_MAX) return cudaErrorInvalidValue;  // coordinates are 32-bit
  if (!encode_tiled_2d(&map_unit, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, codes, 64, rows, 64, 64, 256,
                       CU_TENSOR_MAP_SWIZZLE_64B) ||
      !encode_tiled_2d(&map_block, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, codes, 64, rows, 64, 64, 8,
                       CU_TENSOR_MAP_SWIZZLE_64B) ||
      !encode_tiled_1d(&map_sw256, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, words, rows, 256) ||
      !encode_tiled_1d(&map_sw4, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, words, rows, 4) ||
      !encode_tiled_1d(&map_sw12, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, words, rows, 12))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(index_decode_mx_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDynMx);
  if (e != cudaSuccess) return e;
  const int nrows = nb * tq;
  const int grid = nrows >= num_sms ? nrows : (num_sms / nrows) * nrows;
  if (hist) {  // the blocks add their counts
    e = cudaMemsetAsync(hist, 0, (size_t)nb * Tq * kHistBins * sizeof(uint32_t), st);
    if (e != cudaSuccess) return e;
  }
  index_decode_mx_kernel<<<grid, kMThreads, kDynMx, st>>>(map_unit, map_block, map_sw256, map_sw4, map_sw12, a, pos, b0, nb, t0, tq, Tq, scores, ld,
                                                          rowlen, hist);
  note_launch();
  return cudaGetLastError();
}

size_t index_tc_image_bytes(int nb, int Tq, int64_t max_entries) {
  const size_t nqt = (size_t)(Tq + kQPerTile - 1) / kQPerTile;
  const size_t nkt = (size_t)((max_entries + 127) / 128);
  return (size_t)nb * (nqt * kQImg + nkt * kKImg);
}

cudaError_t launch_index_scores_tc(const IndexArgs& a, const SeqPos& pos, int b0, int nb, int t0, int tq, int Tq,
                                   int64_t emax, int64_t emax_all, bool build_keys, uint8_t* img, float* wq,
                                   float* scores, int64_t ld, uint32_t* lower, int32_t* cand_j, int* cand_n,
                                   int num_sms, cudaStream_t st) {
  const int nqt = (Tq + kQPerTile - 1) / kQPerTile;
  const int nkt = (int)((emax_all + 127) / 128);  // key images of every pass of the call: one stride
  uint8_t* qimg = img;
  uint8_t* kimg = img + (size_t)nb * nqt * kQImg;
  qimage_kernel<<<dim3((unsigned)tq, (unsigned)nb), 128, 0, st>>>(a, b0, t0, Tq, nqt, qimg, wq);
  note_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (build_keys && nkt > 0) {  // once per call, for the entries visible to its last query
    kimage_kernel<<<dim3((unsigned)nkt, (unsigned)nb), 128, 0, st>>>(a, b0, emax_all, nkt, kimg);
    note_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  (void)emax;
  e = cudaFuncSetAttribute(index_prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDynTC);
  if (e != cudaSuccess) return e;
  const int ntiles = nb * ((tq + kQPerTile - 1) / kQPerTile);
  const int grid = max(1, min(num_sms, ntiles));
  index_prefill_tc_kernel<<<grid, kThreadsTC, kDynTC, st>>>(a, pos, t0, tq, nqt, nkt, qimg, kimg, wq, scores, ld, nb, Tq,
                                                             lower, cand_j, cand_n);
  note_launch();
  return cudaGetLastError();
}

// Reads and clears the indexer kernels' device error word (0 = no bounded wait gave up).
cudaError_t take_index_error(int* code) {
  const int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(code, g_index_error, sizeof(int));
  if (e == cudaSuccess && *code != 0) e = cudaMemcpyToSymbol(g_index_error, &zero, sizeof(int));
  return e;
}

// Reads and clears the FP4-scale domain flag of the indexer kernels (0: every scale read fitted).
cudaError_t take_index_domain(unsigned* flag) {
  const unsigned zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(flag, g_index_domain, sizeof(unsigned));
  if (e == cudaSuccess && *flag != 0) e = cudaMemcpyToSymbol(g_index_domain, &zero, sizeof(unsigned));
  return e;
}

namespace {
// One thread waits on a barrier that nothing arrives at: the bounded wait gives up after its
// spin limit (about 80 ms), records code 99 in the error word and the kernel returns.
__global__ void wait_probe_kernel() {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_fence_init();
    mbar_wait(&bar, 0, &g_index_error, 99);
  }
}
}  // namespace

cudaError_t launch_wait_probe(cudaStream_t st) {
  wait_probe_kernel<<<1, 32, 0, st>>>();
  note_launch();
  return cudaGetLastError();
}

}  // namespace csa2
