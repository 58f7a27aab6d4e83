// Lightning indexer and top-512.  Page "DeepSeek V4.1 - Pooled group / Source layer, pairs
// pooled", block "Compressed sparse attention": S^I_{t,j} = sum_h w^I_{t,h} ReLU(Q^I_{h,t} .
// K^I_j) over j < floor((t+1)/2), and I_t = top_512 of those scores.  "Inside DeepSeek
// V4.1", section "Attention that looks at 640 places": 32 heads of 128 numbers in FP4, one
// key per entry, the top 512 are kept.
//
// Q^I is quantised to FP4 (E2M1, UE8M0 per 32) like the keys; every per-head dot product
// is then a sum of exact products of E2M1 values times powers of two and is exact in fp32.
// Scores are fp32.  Top-k: larger score first, equal scores -> lower j first, output
// ascending in j, -1 padded.
#include <algorithm>

#include "csa2_common.cuh"

namespace csa2 {
namespace {

constexpr int kQprepThreads = 128;
constexpr int kScoreThreads = 256;  // one key per thread
constexpr int kQT = 4;              // queries per score block
constexpr int kTopkThreads = 512;  // select blocks that read a score histogram, merges, pools
constexpr int kTopkSmall = 128;    // select blocks of rows without a histogram (several per SM)
constexpr int kMaxChunks = 32;
constexpr int kMinChunk = 4096;
constexpr int kMaxChunk = 32768;
constexpr size_t kScoreBudget = size_t(1) << 30;  // bytes of fp32 scores per query chunk

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct IndexPlan {
  int Tq;           // queries (per sequence) per pass
  int64_t ld;       // score row stride (floats)
  int chunk;        // top-k stage-1 chunk
  int nchunks;
  bool tc;          // prefill: tensor-core score GEMM (queries per pass >= kMinTcQueries)
  int pnch;         // hierarchical pool: chunks of kPoolChunk blocks (pool mode)
  bool dec;         // scores from the per-query scan (one query, or a pool), with histograms
  bool cand;        // long prefill rows may take candidate lists instead of dense score rows
  size_t off_q, off_w, off_s, off_ck, off_cj, off_cn, off_img, off_rl, off_pk, off_pj, off_pn, off_h, off_lo,
      off_candj, off_candn, total;
};

constexpr int kPoolChunk = 16384;             // blocks per chunk of the pool select
constexpr int kPoolSel = kHsiBlocks - 1;      // best other blocks; the newest is always added

constexpr int kMinTcQueries = 8;
constexpr int64_t kMinHistRow = 16384;  // prefill rows this long get the scorer's histogram filter

IndexPlan make_plan(int nb, int T, int64_t max_entries, int mode = kIndexTopk) {
  IndexPlan p;
  // a reindex row holds the pool's positions (at most 2048 blocks of 8), not all entries
  if (mode == kIndexReindex) max_entries = min64(max_entries, (int64_t)kHsiBlock * kHsiBlocks);
  p.ld = ((max(max_entries, (int64_t)1) + 127) / 128) * 128;
  int64_t per_q = (int64_t)nb * p.ld * 4;
  int64_t tq = (int64_t)(kScoreBudget / (size_t)per_q);
  // scores to the caller's array (csa2_index_scores): one pass over all queries, no select
  const bool so = mode == kIndexScores;
  p.Tq = so ? T : (int)max64(1, min64(T, tq));
  int64_t c = kMinChunk;
  while (c * kMaxChunks < p.ld && c < kMaxChunk) c *= 2;
  p.chunk = (int)c;
  p.nchunks = (int)((p.ld + c - 1) / c);
  size_t rows = (size_t)nb * p.Tq;
  p.tc = T >= kMinTcQueries && mode != kIndexReindex;  // a pool scan gathers rows per query
  p.dec = T == 1 || mode == kIndexReindex;
  const int64_t nblk = (max_entries + kHsiBlock - 1) / kHsiBlock;
  p.pnch = mode == kIndexPool && nblk > kHsiBlocks ? (int)((nblk + kPoolChunk - 1) / kPoolChunk) : 0;
  size_t off = 0;
  p.off_q = off; off += p.tc ? 0 : align256(rows * kHI * kDI * 4);
  p.off_w = off; off += align256(rows * kHI * 4);
  p.off_s = off; off += so ? 0 : align256(rows * (size_t)p.ld * 4);
  p.off_ck = off; off += so ? 0 : align256(rows * p.nchunks * kTopK * 4);
  p.off_cj = off; off += so ? 0 : align256(rows * p.nchunks * kTopK * 4);
  p.off_cn = off; off += so ? 0 : align256(rows * p.nchunks * 4);
  p.off_img = off; off += p.tc ? align256(index_tc_image_bytes(nb, p.Tq, p.ld)) : 0;
  p.off_rl = off; off += mode == kIndexReindex ? align256(rows * 4) : 0;
  p.off_pk = off; off += align256(rows * p.pnch * kPoolSel * 4);
  p.off_pj = off; off += align256(rows * p.pnch * kPoolSel * 4);
  p.off_pn = off; off += align256(rows * p.pnch * 4);
  p.off_h = off; off += p.dec && !so ? align256(rows * kHistBins * 4) : 0;
  p.off_lo = off; off += p.tc && !so ? align256(rows * 4) : 0;  // per-row lower edges from the prefill scorer
  // candidate lists (csa2_index_topk on rows of kMinHistRow entries or more): positions beside the
  // keys, which take the score rows' space, and a count per row
  p.cand = p.tc && mode == kIndexTopk && max_entries >= kMinHistRow;
  p.off_candj = off; off += p.cand ? align256(rows * (size_t)p.ld * 4) : 0;
  p.off_candn = off; off += p.cand ? align256(rows * 4 * 4) : 0;
  p.total = off;
  return p;
}

// ------------------------------------------------------------------ Q^I -> FP4 -> fp32
// grid (Tq, nb): one block per query, warp w handles heads 8w..8w+7, lane l values 4l..4l+3.
__global__ void __launch_bounds__(kQprepThreads) qprep_kernel(IndexArgs a, int b0, int t0, int Tq, float* qdq, float* wq) {
  const int tl = blockIdx.x, bl = blockIdx.y;
  const int t = t0 + tl;
  if (t >= a.T) return;
  const int b = b0 + bl;
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  const int64_t src = ((int64_t)b * a.T + t);
  const int64_t dst = ((int64_t)bl * Tq + tl);
  for (int h = 8 * w; h < 8 * w + 8; ++h) {
    uint2 raw = *reinterpret_cast<const uint2*>(a.qi + (src * kHI + h) * kDI + 4 * l);
    float v[4] = {bf16_to_f32(raw.x & 0xffff), bf16_to_f32(raw.x >> 16), bf16_to_f32(raw.y & 0xffff), bf16_to_f32(raw.y >> 16)};
    float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
    const int e = mx_scale_exp(amax);
    float4 o;
    o.x = ldexpf(e2m1_to_f32(f32_to_e2m1(ldexpf(v[0], -e))), e);
    o.y = ldexpf(e2m1_to_f32(f32_to_e2m1(ldexpf(v[1], -e))), e);
    o.z = ldexpf(e2m1_to_f32(f32_to_e2m1(ldexpf(v[2], -e))), e);
    o.w = ldexpf(e2m1_to_f32(f32_to_e2m1(ldexpf(v[3], -e))), e);
    *reinterpret_cast<float4*>(qdq + (dst * kHI + h) * kDI + 4 * l) = o;
  }
  if (threadIdx.x < kHI) wq[dst * kHI + threadIdx.x] = bf16_to_f32(a.wI[src * kHI + threadIdx.x]);
}

// ------------------------------------------------------------------ score scan (CUDA cores)
// grid (key tiles of 256, query tiles of kQT, nb).  Thread = key j; the key's 128 FP4 values
// are decoded one 32-block at a time and dotted with the 32 heads of each query in smem.
__global__ void __launch_bounds__(kScoreThreads) score_kernel(IndexArgs a, SeqPos pos, int b0, int t0, int Tq,
                                                              const float* qdq, const float* wq, float* scores, int64_t ld) {
  extern __shared__ float4 smem4[];
  float* sq = reinterpret_cast<float*>(smem4);  // [kQT][32][128]
  __shared__ float sw[kQT][kHI];
  const int bl = blockIdx.z;
  const int b = b0 + bl;
  const int64_t p0 = seq_p0(pos, bl);
  const int tq0 = blockIdx.y * kQT;
  const int64_t j = (int64_t)blockIdx.x * kScoreThreads + threadIdx.x;
  // visible entries of the last query of the tile bound the whole tile
  const int tlast = min(tq0 + kQT, Tq) - 1;
  if (t0 + tq0 >= a.T) return;
  const int64_t Elast = (p0 + t0 + min(tlast, a.T - 1 - t0) + 1) >> a.rshift;
  if ((int64_t)blockIdx.x * kScoreThreads >= Elast) return;
  const int nq = min(kQT, min(Tq, a.T - t0) - tq0);
  for (int i = threadIdx.x; i < nq * kHI * kDI / 4; i += kScoreThreads)
    smem4[i] = reinterpret_cast<const float4*>(qdq + ((int64_t)bl * Tq + tq0) * kHI * kDI)[i];
  for (int i = threadIdx.x; i < nq * kHI; i += kScoreThreads)
    sw[i / kHI][i % kHI] = wq[((int64_t)bl * Tq + tq0) * kHI + i];
  __syncthreads();
  if (j >= Elast) return;
  uint4 cw[4];
  const uint4* kp = reinterpret_cast<const uint4*>(a.ki_codes + ((int64_t)b * a.cap + j) * 64);
#pragma unroll
  for (int i = 0; i < 4; ++i) cw[i] = kp[i];
  const uint32_t sc = *reinterpret_cast<const uint32_t*>(a.ki_scales + ((int64_t)b * a.cap + j) * 4);
  for (int qq = 0; qq < nq; ++qq) {
    const int t = t0 + tq0 + qq;
    const int64_t E = (p0 + t + 1) >> a.rshift;
    if (j >= E) continue;
    float acc[kHI];
#pragma unroll
    for (int h = 0; h < kHI; ++h) acc[h] = 0.f;
#pragma unroll
    for (int blk = 0; blk < 4; ++blk) {
      const float s = ldexpf(1.0f, (int)((sc >> (8 * blk)) & 255) - 127);
      float k[32];
      const uint32_t words[4] = {cw[blk].x, cw[blk].y, cw[blk].z, cw[blk].w};
#pragma unroll
      for (int wd = 0; wd < 4; ++wd)
#pragma unroll
        for (int nb = 0; nb < 8; ++nb) k[8 * wd + nb] = e2m1_to_f32((words[wd] >> (4 * nb)) & 15) * s;
      const float* qb = sq + (qq * kHI) * kDI + blk * 32;
#pragma unroll
      for (int h = 0; h < kHI; ++h) {
        const float4* q4 = reinterpret_cast<const float4*>(qb + h * kDI);
        float d = acc[h];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float4 qv = q4[i];
          d = fmaf(k[4 * i], qv.x, d);
          d = fmaf(k[4 * i + 1], qv.y, d);
          d = fmaf(k[4 * i + 2], qv.z, d);
          d = fmaf(k[4 * i + 3], qv.w, d);
        }
        acc[h] = d;
      }
    }
    float s = 0.f;
#pragma unroll
    for (int h = 0; h < kHI; ++h) s = fmaf(sw[qq][h], fmaxf(acc[h], 0.f), s);
    scores[((int64_t)bl * Tq + tq0 + qq) * ld + j] = s;
  }
}

// ------------------------------------------------------------------ top-k

template <int NT>
struct SelectShared {
  static constexpr int kWarps = NT / 32;
  uint32_t hist[kWarps][256];  // one histogram per warp: fewer same-address atomics
  uint32_t red[2][kWarps];
  int warp_tot[2][kWarps];
  uint32_t bucket;
  int krem;
  int exact;  // radix_select_pairs: the chosen bucket is taken whole
};

// Radix select over keys[0..n): on return *thr is the K-th largest key and *need_eq the
// number of keys equal to *thr that belong to the top K (the lowest-index ones).  The digits
// start at the highest bit in which the smallest and largest key differ (the bits above are
// common to every key and would put all keys into one bin).  Up to kSmallSelect keys share one
// histogram (clearing and folding one per warp would cost more than the few collisions);
// longer rows count into one histogram per warp.
constexpr int kSmallSelect = 4096;

template <int NT>
__device__ void radix_select(const uint32_t* keys, int n, int K, SelectShared<NT>& sh, uint32_t* thr, int* need_eq) {
  constexpr int kWarps = NT / 32;
  const int tid = threadIdx.x, w = tid >> 5, l = tid & 31;
  const bool one_hist = n <= kSmallSelect;
  const int hw = one_hist ? 0 : w;                   // this thread's histogram
  const int nclear = (one_hist ? 1 : kWarps) * 256;  // words to clear per pass
  uint32_t mn = 0xffffffffu, mx = 0u;
  for (int i = tid; i < n; i += NT) {
    const uint32_t k = keys[i];
    mn = min(mn, k);
    mx = max(mx, k);
  }
  mn = __reduce_min_sync(0xffffffffu, mn);
  mx = __reduce_max_sync(0xffffffffu, mx);
  if (l == 0) {
    sh.red[0][w] = mn;
    sh.red[1][w] = mx;
  }
  __syncthreads();
  mn = 0xffffffffu;
  mx = 0u;
  for (int x = 0; x < kWarps; ++x) {
    mn = min(mn, sh.red[0][x]);
    mx = max(mx, sh.red[1][x]);
  }
  __syncthreads();
  if (mn == mx) {  // every key equal: the K lowest positions
    *thr = mx;
    *need_eq = K;
    return;
  }
  const int top = 31 - __clz(mn ^ mx);
  uint32_t mask = top == 31 ? 0u : ~((2u << top) - 1u);
  uint32_t prefix = mx & mask;
  int krem = K;
  for (int hi = top; hi >= 0; hi -= 8) {
    const int lo = max(hi - 7, 0);
    const uint32_t dmask = (2u << (hi - lo)) - 1u;
    for (int i = tid; i < nclear; i += NT) (&sh.hist[0][0])[i] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += NT) {
      const uint32_t k = keys[i];
      if ((k & mask) == prefix) atomicAdd(&sh.hist[hw][(k >> lo) & dmask], 1u);
    }
    __syncthreads();
    if (!one_hist) {
      for (int b = tid; b < 256; b += NT) {  // fold the per-warp histograms into warp 0's
        uint32_t c = 0;
#pragma unroll
        for (int x = 0; x < kWarps; ++x) c += sh.hist[x][b];
        sh.hist[0][b] = c;
      }
      __syncthreads();
    }
    if (tid < 32) {
      // lane l owns bins 255-8l .. 248-8l (descending)
      uint32_t c[8], tot = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) { c[i] = sh.hist[0][255 - 8 * tid - i]; tot += c[i]; }
      uint32_t incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (tid >= o) incl += v;
      }
      const uint32_t excl = incl - tot;
      const bool mine = excl < (uint32_t)krem && incl >= (uint32_t)krem;
      if (mine) {
        uint32_t run = excl;
        for (int i = 0; i < 8; ++i) {
          if (run + c[i] >= (uint32_t)krem) {
            sh.bucket = 255 - 8 * tid - i;
            sh.krem = krem - (int)run;
            break;
          }
          run += c[i];
        }
      }
    }
    __syncthreads();
    prefix |= sh.bucket << lo;
    mask |= dmask << lo;
    krem = sh.krem;
    __syncthreads();
  }
  *thr = prefix;
  *need_eq = krem;
}

// Writes the K selected (key, j) pairs in ascending position order.  Keys > thr are all
// taken; of the keys == thr only the first need_eq (in position order).  js == nullptr
// means j = j0 + position.  Each warp owns one contiguous segment: a counting pass, one scan
// of the per-warp counts, then an ordered writing pass.
template <int NT>
__device__ void compact_selected(const uint32_t* keys, const int32_t* js, int64_t j0, int n, uint32_t thr, int need_eq,
                                 SelectShared<NT>& sh, uint32_t* out_key, int32_t* out_j) {
  constexpr int kWarps = NT / 32;
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  const uint32_t lt = (1u << l) - 1u;
  const int seg = (((n + kWarps - 1) / kWarps) + 31) & ~31;
  const int s0 = min(n, w * seg), s1 = min(n, s0 + seg);
  int gt = 0, eq = 0;
  for (int i0 = s0; i0 < s1; i0 += 32) {
    const int i = i0 + l;
    const bool v = i < s1;
    const uint32_t k = v ? keys[i] : 0u;
    gt += __popc(__ballot_sync(0xffffffffu, v && k > thr));
    eq += __popc(__ballot_sync(0xffffffffu, v && k == thr));
  }
  if (l == 0) {
    sh.warp_tot[0][w] = gt;
    sh.warp_tot[1][w] = eq;
  }
  __syncthreads();
  // lane x holds warp x's counts; exclusive scans give this warp's equal-key rank and output base
  const int g = l < kWarps ? sh.warp_tot[0][l] : 0, e = l < kWarps ? sh.warp_tot[1][l] : 0;
  int e_inc = e;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, e_inc, o);
    if (l >= o) e_inc += y;
  }
  const int e_exc = e_inc - e;
  const int taken = g + min(max(need_eq - e_exc, 0), e);
  int t_inc = taken;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, t_inc, o);
    if (l >= o) t_inc += y;
  }
  int run_eq = __shfl_sync(0xffffffffu, e_exc, w);
  int pos = __shfl_sync(0xffffffffu, t_inc - taken, w);
  for (int i0 = s0; i0 < s1; i0 += 32) {
    const int i = i0 + l;
    const bool v = i < s1;
    const uint32_t k = v ? keys[i] : 0u;
    const bool is_eq = v && k == thr;
    const uint32_t beq = __ballot_sync(0xffffffffu, is_eq);
    const bool take = (v && k > thr) || (is_eq && run_eq + __popc(beq & lt) < need_eq);
    const uint32_t bt = __ballot_sync(0xffffffffu, take);
    if (take) {
      const int p = pos + __popc(bt & lt);
      out_key[p] = k;
      out_j[p] = js ? js[i] : (int32_t)(j0 + i);
    }
    run_eq += __popc(beq);
    pos += __popc(bt);
  }
  __syncthreads();
}

// Stage 1: grid (nchunks, rows, nb).  Local top-512 of one chunk of one query's scores.
// With a single chunk the result is final and goes straight to idx / top_scores.
// With a pool (reindex), a row's positions map to entries 8 * pool[p / 8] + p % 8 and rowlen
// holds the number of visible positions.
__device__ __forceinline__ int32_t pool_entry(const int32_t* prow, int32_t p) {
  return prow ? kHsiBlock * prow[p >> 3] + (p & (kHsiBlock - 1)) : p;
}

// Lower edge (a key) of the histogram bin holding the K-th largest key of a row, so that all
// of the row's K largest keys are >= it (0 if the histogram holds fewer than K keys).
__device__ uint32_t hist_lower(const uint32_t* hist, int K, SelectShared<kTopkThreads>& sh) {
  static_assert(kTopkThreads * 4 == kHistBins, "four bins per thread");
  const int tid = threadIdx.x, w = tid >> 5, l = tid & 31;
  const int top = kHistBins - 1 - 4 * tid;  // this thread's bins top .. top-3, from the largest keys down
  const uint4 v4 = __ldg(reinterpret_cast<const uint4*>(hist + top - 3));
  const uint32_t v[4] = {v4.w, v4.z, v4.y, v4.x};
  const uint32_t s = v[0] + v[1] + v[2] + v[3];
  uint32_t x = s;  // inclusive scan over the threads (bins in descending order)
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (l >= o) x += y;
  }
  if (l == 31) sh.red[0][w] = x;
  if (tid == 0) sh.bucket = 0u;
  __syncthreads();
  if (w == 0) {
    uint32_t y = l < SelectShared<kTopkThreads>::kWarps ? sh.red[0][l] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t z = __shfl_up_sync(0xffffffffu, y, o);
      if (l >= o) y += z;
    }
    if (l < SelectShared<kTopkThreads>::kWarps) sh.red[1][l] = y;
  }
  __syncthreads();
  const uint32_t excl = x - s + (w ? sh.red[1][w - 1] : 0u);
  if (excl < (uint32_t)K && excl + s >= (uint32_t)K) {
    uint32_t c = excl;
    int b = top;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      c += v[u];
      if (c >= (uint32_t)K) {
        b = top - u;
        break;
      }
    }
    sh.bucket = (uint32_t)b << kHistShift;
  }
  __syncthreads();
  return sh.bucket;
}

// With hist (the row's score histogram) or lower_in (the lower edge of that bin, from the prefill
// scorer), a chunk whose keys at or above the K-th largest key's bin number at most 512 passes
// exactly those on (a superset of its part of the row's top-512, in position order) and skips
// the radix select.  NT threads per block: rows with a
// histogram take kTopkThreads (hist_lower reads four bins per thread); the others take
// kTopkSmall, so that several rows share an SM and hide one another's barrier latency.
template <int NT>
__global__ void __launch_bounds__(NT) topk_chunk_kernel(IndexArgs a, SeqPos pos, int b0, int t0, int Tq,
                                                        const float* scores, int64_t ld, int chunk, int nchunks,
                                                        uint32_t* ck, int32_t* cj, int* cn, const int* rowlen,
                                                        const uint32_t* hist, const uint32_t* lower_in) {
  extern __shared__ uint32_t skeys[];
  __shared__ SelectShared<NT> sh;
  __shared__ uint32_t okey[kTopK];
  __shared__ int32_t oj[kTopK];
  __shared__ int cnt_sh;
  grid_dep_wait();  // launched dependent on the scorer (histogram rows)
  grid_dep_trigger();
  const int c = blockIdx.x, tl = blockIdx.y, bl = blockIdx.z;
  const int t = t0 + tl;
  if (t >= a.T || tl >= Tq) return;
  const int b = b0 + bl;
  const int64_t row = (int64_t)bl * Tq + tl;
  const int64_t E = rowlen ? rowlen[row] : (seq_p0(pos, bl) + t + 1) >> a.rshift;
  const int64_t cs = (int64_t)c * chunk;
  const int n = (int)max64(0, min64(chunk, E - cs));
  // the candidates' lower bound, before the loads: from the row's score histogram, or as the
  // prefill scorer computed it from its own (lower_in)
  uint32_t lower = 0u;
  if constexpr (NT == kTopkThreads)
    if (hist && n > kTopK) lower = hist_lower(hist + row * kHistBins, (int)min64(kTopK, E), sh);
  if (lower_in && n > kTopK) lower = __ldg(lower_in + row);
  const float* src = scores + row * ld + cs;  // 16-byte aligned: ld and the chunk are multiples of 32
  int K = min(kTopK, n);  // entries in okey / oj
  const int n4 = n >> 2;
  constexpr int kLB = 4;  // 16-byte loads in flight per thread
  for (int v0 = threadIdx.x; v0 < n4; v0 += kLB * NT) {
    float4 f[kLB];
#pragma unroll
    for (int u = 0; u < kLB; ++u)
      if (v0 + u * NT < n4) f[u] = __ldg(reinterpret_cast<const float4*>(src) + v0 + u * NT);
#pragma unroll
    for (int u = 0; u < kLB; ++u)
      if (v0 + u * NT < n4)
        reinterpret_cast<uint4*>(skeys)[v0 + u * NT] =
            make_uint4(score_key(f[u].x), score_key(f[u].y), score_key(f[u].z), score_key(f[u].w));
  }
  for (int i = 4 * n4 + threadIdx.x; i < n; i += NT) skeys[i] = score_key(src[i]);
  if (threadIdx.x == 0) cnt_sh = 0;
  __syncthreads();
  if (n <= kTopK) {  // every candidate is kept, already in position order
    for (int i = threadIdx.x; i < n; i += NT) {
      okey[i] = skeys[i];
      oj[i] = (int32_t)(cs + i);
    }
  } else {
    int cnt = kTopK + 1;
    if (lower > 0u) {
      int m = 0;
      for (int i = threadIdx.x; i < n; i += NT) m += skeys[i] >= lower;
      m = __reduce_add_sync(0xffffffffu, m);
      if ((threadIdx.x & 31) == 0) atomicAdd(&cnt_sh, m);
      __syncthreads();
      cnt = cnt_sh;
    }
    if (cnt <= kTopK) {  // keys >= lower, position order (a single chunk: exactly its top 512)
      compact_selected(skeys, nullptr, cs, n, lower - 1u, 0, sh, okey, oj);
      K = cnt;
    } else {
      uint32_t thr;
      int need_eq;
      radix_select(skeys, n, K, sh, &thr, &need_eq);
      compact_selected(skeys, nullptr, cs, n, thr, need_eq, sh, okey, oj);
    }
  }
  __syncthreads();
  if (nchunks == 1) {
    int32_t* idx = a.idx + ((int64_t)b * a.T + t) * kTopK;
    float* ts = a.top_scores ? a.top_scores + ((int64_t)b * a.T + t) * kTopK : nullptr;
    const int32_t* prow = a.pool_in ? a.pool_in + ((int64_t)b * a.T + t) * kHsiBlocks : nullptr;
    for (int i = threadIdx.x; i < kTopK; i += NT) {
      idx[i] = i < K ? pool_entry(prow, oj[i]) : -1;
      if (ts) ts[i] = i < K ? key_score(okey[i]) : __int_as_float(0x7fc00000);
    }
  } else {
    const int64_t base = (row * nchunks + c) * kTopK;
    for (int i = threadIdx.x; i < K; i += NT) {
      ck[base + i] = okey[i];
      cj[base + i] = oj[i];
    }
    if (threadIdx.x == 0) cn[row * nchunks + c] = K;
  }
}

// Stage 2: grid (rows, nb).  Merge the chunk candidates of one query.
__global__ void __launch_bounds__(kTopkThreads) topk_merge_kernel(IndexArgs a, int b0, int t0, int Tq, int nchunks,
                                                                  const uint32_t* ck, const int32_t* cj, const int* cn) {
  extern __shared__ uint32_t smem[];
  uint32_t* skeys = smem;                                                // [nchunks*512]
  int32_t* sjs = reinterpret_cast<int32_t*>(smem + nchunks * kTopK);    // [nchunks*512]
  __shared__ SelectShared<kTopkThreads> sh;
  __shared__ uint32_t okey[kTopK];
  __shared__ int32_t oj[kTopK];
  __shared__ int offs[kMaxChunks + 1];
  grid_dep_wait();  // launched dependent on the chunk kernel
  grid_dep_trigger();
  const int tl = blockIdx.x, bl = blockIdx.y;
  const int t = t0 + tl;
  if (t >= a.T) return;
  const int b = b0 + bl;
  const int64_t row = (int64_t)bl * Tq + tl;
  __shared__ int cnt_s[kMaxChunks];
  static_assert(kMaxChunks <= 32, "one warp scans the chunk counts");
  if (threadIdx.x < 32) {  // lane c: chunk c's count and its list's end offset
    const int v = threadIdx.x < nchunks ? cn[row * nchunks + threadIdx.x] : 0;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if ((int)threadIdx.x >= o) incl += y;
    }
    if (threadIdx.x < nchunks) {
      cnt_s[threadIdx.x] = v;
      offs[threadIdx.x + 1] = incl;
    }
    if (threadIdx.x == 0) offs[0] = 0;
  }
  __syncthreads();
  const int n = offs[nchunks];
  // all (chunk, slot) loads of a thread are issued before any of its shared-memory stores
  constexpr int kLB = kMaxChunks * kTopK / kTopkThreads;
  uint32_t kk[kLB];
  int32_t jj[kLB];
#pragma unroll
  for (int u = 0; u < kLB; ++u) {
    const int q = threadIdx.x + u * kTopkThreads, c = q / kTopK, i = q % kTopK;
    if (c < nchunks && i < cnt_s[c]) {
      const int64_t src = (row * nchunks + c) * kTopK + i;
      kk[u] = __ldg(ck + src);
      jj[u] = __ldg(cj + src);
    }
  }
#pragma unroll
  for (int u = 0; u < kLB; ++u) {
    const int q = threadIdx.x + u * kTopkThreads, c = q / kTopK, i = q % kTopK;
    if (c < nchunks && i < cnt_s[c]) {
      skeys[offs[c] + i] = kk[u];
      sjs[offs[c] + i] = jj[u];
    }
  }
  __syncthreads();
  const int K = min(kTopK, n);
  if (n <= kTopK) {  // chunk lists are consecutive in position order
    for (int i = threadIdx.x; i < n; i += kTopkThreads) {
      okey[i] = skeys[i];
      oj[i] = sjs[i];
    }
  } else {
    uint32_t thr;
    int need_eq;
    radix_select(skeys, n, K, sh, &thr, &need_eq);
    compact_selected(skeys, sjs, 0, n, thr, need_eq, sh, okey, oj);
  }
  __syncthreads();
  int32_t* idx = a.idx + ((int64_t)b * a.T + t) * kTopK;
  float* ts = a.top_scores ? a.top_scores + ((int64_t)b * a.T + t) * kTopK : nullptr;
  const int32_t* prow = a.pool_in ? a.pool_in + ((int64_t)b * a.T + t) * kHsiBlocks : nullptr;
  for (int i = threadIdx.x; i < kTopK; i += kTopkThreads) {
    idx[i] = i < K ? pool_entry(prow, oj[i]) : -1;
    if (ts) ts[i] = i < K ? key_score(okey[i]) : __int_as_float(0x7fc00000);
  }
}

// K-th largest of the n pairs (key, j) = pair(i) in the order "larger key first, then lower j": as
// the composite V = key * 2^32 + (2^32 - 1 - j), distinct for distinct j, so V >= *thr takes exactly
// the K pairs.  The digits start at the highest bit in which the keys differ (in the position half
// when every key is equal) and stop as soon as a whole bucket is needed.
template <int NT, class Pair>
__device__ void radix_select_pairs(const Pair& pair, int n, int K, SelectShared<NT>& sh, uint64_t* thr) {
  constexpr int kWarps = NT / 32;
  const int tid = threadIdx.x, w = tid >> 5, l = tid & 31;
  const bool one_hist = n <= kSmallSelect;
  const int hw = one_hist ? 0 : w;
  const int nclear = (one_hist ? 1 : kWarps) * 256;
  auto val = [&](int i) -> uint64_t {
    uint32_t k;
    int32_t j;
    pair(i, k, j);
    return ((uint64_t)k << 32) | (uint64_t)(~(uint32_t)j);
  };
  uint32_t mn = 0xffffffffu, mx = 0u;
  for (int i = tid; i < n; i += NT) {
    const uint32_t k = (uint32_t)(val(i) >> 32);
    mn = min(mn, k);
    mx = max(mx, k);
  }
  mn = __reduce_min_sync(0xffffffffu, mn);
  mx = __reduce_max_sync(0xffffffffu, mx);
  if (l == 0) {
    sh.red[0][w] = mn;
    sh.red[1][w] = mx;
  }
  __syncthreads();
  mn = 0xffffffffu;
  mx = 0u;
  for (int x = 0; x < kWarps; ++x) {
    mn = min(mn, sh.red[0][x]);
    mx = max(mx, sh.red[1][x]);
  }
  __syncthreads();
  const int top = mn == mx ? 31 : 63 - __clz(mn ^ mx);
  uint64_t mask = top == 63 ? 0ull : ~((2ull << top) - 1ull);
  uint64_t prefix = ((uint64_t)mx << 32) & mask;
  int krem = K;
  for (int hi = top; hi >= 0; hi -= 8) {
    const int lo = max(hi - 7, 0);
    const uint64_t dmask = (2ull << (hi - lo)) - 1ull;
    for (int i = tid; i < nclear; i += NT) (&sh.hist[0][0])[i] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += NT) {
      const uint64_t v = val(i);
      if ((v & mask) == prefix) atomicAdd(&sh.hist[hw][(uint32_t)((v >> lo) & dmask)], 1u);
    }
    __syncthreads();
    if (!one_hist) {
      for (int b = tid; b < 256; b += NT) {
        uint32_t c = 0;
#pragma unroll
        for (int x = 0; x < kWarps; ++x) c += sh.hist[x][b];
        sh.hist[0][b] = c;
      }
      __syncthreads();
    }
    if (tid < 32) {
      // lane l owns bins 255-8l .. 248-8l (descending)
      uint32_t c[8], tot = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) { c[i] = sh.hist[0][255 - 8 * tid - i]; tot += c[i]; }
      uint32_t incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (tid >= o) incl += v;
      }
      const uint32_t excl = incl - tot;
      if (excl < (uint32_t)krem && incl >= (uint32_t)krem) {
        uint32_t run = excl;
        for (int i = 0; i < 8; ++i) {
          if (run + c[i] >= (uint32_t)krem) {
            sh.bucket = 255 - 8 * tid - i;
            sh.krem = krem - (int)run;
            sh.exact = c[i] == (uint32_t)(krem - (int)run);
            break;
          }
          run += c[i];
        }
      }
    }
    __syncthreads();
    prefix |= (uint64_t)sh.bucket << lo;
    mask |= dmask << lo;
    krem = sh.krem;
    const bool exact = sh.exact;
    __syncthreads();
    if (exact) break;  // the whole bucket is needed: V >= prefix (lower bits 0) takes it and the rest
  }
  *thr = prefix;
}

// Top-512 of a row from its candidate lists (long prefill rows): grid (rows, nb).  The row's four
// segments (counts in cand_n[row * 4 ..], segment s at row * ld + s * ld / 4) hold (score key,
// position) pairs in any order, among them the row's top-K; the K pairs go out in ascending
// position order, each placed by its rank among them.
__global__ void __launch_bounds__(kTopkThreads) topk_cand_kernel(IndexArgs a, SeqPos pos, int b0, int t0, int Tq,
                                                                 const uint32_t* cand_key, const int32_t* cand_j,
                                                                 const int* cand_n, int64_t ld) {
  __shared__ SelectShared<kTopkThreads> sh;
  __shared__ uint32_t okey[kTopK];
  __shared__ int32_t oj[kTopK];
  __shared__ int cnt_sh;
  const int tl = blockIdx.x, bl = blockIdx.y;
  const int t = t0 + tl;
  if (t >= a.T) return;
  const int b = b0 + bl;
  const int tid = threadIdx.x, lane = tid & 31;
  const int64_t row = (int64_t)bl * Tq + tl;
  const int64_t E = (seq_p0(pos, bl) + t + 1) >> a.rshift;
  const int K = (int)min64(kTopK, E);
  int pre[5];  // the segments' starts in the row's numbering of its candidates
  pre[0] = 0;
  for (int q = 0; q < 4; ++q) pre[q + 1] = pre[q] + cand_n[row * 4 + q];
  const int n = pre[4];
  const int64_t seg = ld >> 2;
  auto pair = [&](int i, uint32_t& k, int32_t& j) {
    const int q = (i >= pre[1]) + (i >= pre[2]) + (i >= pre[3]);
    const int64_t at = row * ld + q * seg + (i - pre[q]);
    k = cand_key[at];
    j = cand_j[at];
  };
  uint64_t thr = 0ull;  // n <= K: every candidate
  if (n > K) radix_select_pairs<kTopkThreads>(pair, n, K, sh, &thr);
  if (tid == 0) cnt_sh = 0;
  __syncthreads();
  const int nround = (n + kTopkThreads - 1) / kTopkThreads * kTopkThreads;  // whole warps take part in the ballots
  for (int i = tid; i < nround; i += kTopkThreads) {
    const bool v = i < n;
    uint32_t k = 0u;
    int32_t j = 0;
    if (v) pair(i, k, j);
    const bool take = v && ((((uint64_t)k << 32) | (uint64_t)(~(uint32_t)j)) >= thr);
    const uint32_t bal = __ballot_sync(0xffffffffu, take);
    if (bal) {
      int base = 0;
      if (lane == 0) base = atomicAdd(&cnt_sh, __popc(bal));
      base = __shfl_sync(0xffffffffu, base, 0);
      const int at = base + __popc(bal & ((1u << lane) - 1u));
      if (take && at < kTopK) {
        okey[at] = k;
        oj[at] = j;
      }
    }
  }
  __syncthreads();
  const int m = min(cnt_sh, kTopK);
  int32_t* idx = a.idx + ((int64_t)b * a.T + t) * kTopK;
  float* ts = a.top_scores ? a.top_scores + ((int64_t)b * a.T + t) * kTopK : nullptr;
  for (int i = tid; i < m; i += kTopkThreads) {  // rank by position (positions are distinct)
    const int32_t ji = oj[i];
    int r = 0;
    for (int q = 0; q < m; ++q) r += oj[q] < ji;
    idx[r] = ji;
    if (ts) ts[r] = key_score(okey[i]);
  }
  for (int i = m + tid; i < kTopK; i += kTopkThreads) {
    idx[i] = -1;
    if (ts) ts[i] = __int_as_float(0x7fc00000);
  }
}

// ------------------------------------------------------------------ hierarchical pool
// "Inside DeepSeek V4.1", section "Most layers borrow": blocks of 8 entries scored by their
// best entry, 2048 blocks kept, the block holding the newest entries always among them.
// Pool = the newest block + the kPoolSel best other blocks (block score desc, block asc), or
// every block when there are at most 2048; ascending, -1 padded.  The newest block's key is 0
// (below every finite score) so that the select skips it; it is appended last.
// Stage 1: grid (pool chunks, rows, nb).  A row with a single chunk writes its pool directly.
__global__ void __launch_bounds__(kTopkThreads) pool_chunk_kernel(IndexArgs a, SeqPos pos, int b0, int t0, int Tq,
                                                                  const float* scores, int64_t ld, int pnch,
                                                                  uint32_t* pk, int32_t* pj, int* pn) {
  extern __shared__ uint32_t pkeys[];  // [kPoolChunk] block keys, then okey / oj [kPoolSel]
  uint32_t* okey = pkeys + kPoolChunk;
  int32_t* oj = reinterpret_cast<int32_t*>(okey + kPoolSel);
  __shared__ SelectShared<kTopkThreads> sh;
  const int c = blockIdx.x, tl = blockIdx.y, bl = blockIdx.z;
  const int t = t0 + tl;
  if (t >= a.T || tl >= Tq) return;
  const int b = b0 + bl;
  const int64_t E = (seq_p0(pos, bl) + t + 1) >> a.rshift;
  const int64_t nblk = (E + kHsiBlock - 1) / kHsiBlock;
  int32_t* pool = a.pool_out + ((int64_t)b * a.T + t) * kHsiBlocks;
  if (nblk <= kHsiBlocks) {  // every block
    if (c == 0)
      for (int i = threadIdx.x; i < kHsiBlocks; i += kTopkThreads) pool[i] = i < nblk ? i : -1;
    return;
  }
  const int rnch = (int)((nblk + kPoolChunk - 1) / kPoolChunk);
  if (c >= rnch) return;
  const int64_t row = (int64_t)bl * Tq + tl;
  const int64_t cb = (int64_t)c * kPoolChunk;
  const int n = (int)min64(kPoolChunk, nblk - cb);
  const float4* src = reinterpret_cast<const float4*>(scores + row * ld);  // 32-byte aligned blocks
  for (int i = threadIdx.x; i < n; i += kTopkThreads) {
    const int64_t k = cb + i;
    uint32_t key = 0u;
    if (k != nblk - 1) {  // all 8 entries of an older block are visible
      const float4 u = __ldg(src + 2 * k), v = __ldg(src + 2 * k + 1);
      key = score_key(fmaxf(fmaxf(fmaxf(u.x, u.y), fmaxf(u.z, u.w)), fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w))));
    }
    pkeys[i] = key;
  }
  __syncthreads();
  const int K = min(kPoolSel, n);
  if (n <= kPoolSel) {
    for (int i = threadIdx.x; i < n; i += kTopkThreads) {
      okey[i] = pkeys[i];
      oj[i] = (int32_t)(cb + i);
    }
  } else {
    uint32_t thr;
    int need_eq;
    radix_select(pkeys, n, K, sh, &thr, &need_eq);
    compact_selected(pkeys, nullptr, cb, n, thr, need_eq, sh, okey, oj);
  }
  __syncthreads();
  if (rnch == 1) {  // n = nblk > kPoolSel: the kPoolSel best older blocks, ascending, then the newest
    for (int i = threadIdx.x; i < kHsiBlocks; i += kTopkThreads) pool[i] = i < kPoolSel ? oj[i] : (int32_t)(nblk - 1);
  } else {
    const int64_t base = (row * pnch + c) * kPoolSel;
    for (int i = threadIdx.x; i < K; i += kTopkThreads) {
      pk[base + i] = okey[i];
      pj[base + i] = oj[i];
    }
    if (threadIdx.x == 0) pn[row * pnch + c] = K;
  }
}

// Stage 2: grid (rows, nb).  Rows with more than one pool chunk: select from the chunk lists.
__global__ void __launch_bounds__(kTopkThreads) pool_merge_kernel(IndexArgs a, SeqPos pos, int b0, int t0, int Tq,
                                                                  int pnch, const uint32_t* pk, const int32_t* pj,
                                                                  const int* pn) {
  extern __shared__ uint32_t msm[];
  uint32_t* keys = msm;                                                 // [pnch * kPoolSel]
  int32_t* js = reinterpret_cast<int32_t*>(keys + pnch * kPoolSel);     // [pnch * kPoolSel]
  uint32_t* okey = reinterpret_cast<uint32_t*>(js + pnch * kPoolSel);   // [kPoolSel]
  int32_t* oj = reinterpret_cast<int32_t*>(okey + kPoolSel);            // [kPoolSel]
  __shared__ SelectShared<kTopkThreads> sh;
  __shared__ int offs[kMaxChunks + 1];
  const int tl = blockIdx.x, bl = blockIdx.y;
  const int t = t0 + tl;
  if (t >= a.T || tl >= Tq) return;
  const int b = b0 + bl;
  const int64_t E = (seq_p0(pos, bl) + t + 1) >> a.rshift;
  const int64_t nblk = (E + kHsiBlock - 1) / kHsiBlock;
  const int rnch = (int)((nblk + kPoolChunk - 1) / kPoolChunk);
  if (nblk <= kHsiBlocks || rnch <= 1) return;  // written by stage 1
  const int64_t row = (int64_t)bl * Tq + tl;
  if (threadIdx.x == 0) {
    offs[0] = 0;
    for (int c = 0; c < rnch; ++c) offs[c + 1] = offs[c] + pn[row * pnch + c];
  }
  __syncthreads();
  const int n = offs[rnch];
  for (int q = threadIdx.x; q < rnch * kPoolSel; q += kTopkThreads) {
    const int c = q / kPoolSel, i = q % kPoolSel;
    if (i < offs[c + 1] - offs[c]) {
      const int64_t src = (row * pnch + c) * kPoolSel + i;
      keys[offs[c] + i] = pk[src];
      js[offs[c] + i] = pj[src];
    }
  }
  __syncthreads();
  uint32_t thr;
  int need_eq;
  radix_select(keys, n, kPoolSel, sh, &thr, &need_eq);  // n >= kPoolSel older blocks
  compact_selected(keys, js, 0, n, thr, need_eq, sh, okey, oj);
  __syncthreads();
  int32_t* pool = a.pool_out + ((int64_t)b * a.T + t) * kHsiBlocks;
  for (int i = threadIdx.x; i < kHsiBlocks; i += kTopkThreads) pool[i] = i < kPoolSel ? oj[i] : (int32_t)(nblk - 1);
}

}  // namespace

// Launches take groups of kMaxSeqPerLaunch sequences; a smaller tail group may take more queries
// per pass, so the need is the larger of the two group plans.
size_t index_workspace_bytes(int B, int T, int64_t max_entries, int /*num_sms*/, int mode) {
  size_t need = make_plan(min(B, kMaxSeqPerLaunch), T, max_entries, mode).total;
  if (B > kMaxSeqPerLaunch && B % kMaxSeqPerLaunch)
    need = std::max(need, make_plan(B % kMaxSeqPerLaunch, T, max_entries, mode).total);
  return need;
}

cudaError_t launch_index_topk(const IndexArgs& a, const SeqPos& pos, int b0, int nb, int64_t max_entries, void* ws,
                              size_t ws_bytes, int num_sms, cudaStream_t st, int mode) {
  const IndexPlan p = make_plan(min(nb, kMaxSeqPerLaunch), a.T, max_entries, mode);
  if (ws_bytes < p.total) return cudaErrorInvalidValue;
  char* base = static_cast<char*>(ws);
  float* qdq = reinterpret_cast<float*>(base + p.off_q);
  float* wq = reinterpret_cast<float*>(base + p.off_w);
  const bool so = mode == kIndexScores;  // the caller's score rows (this group's part), no select
  float* sc = so ? a.scores_out + (int64_t)b0 * a.T * a.scores_ld : reinterpret_cast<float*>(base + p.off_s);
  const int64_t ld = so ? a.scores_ld : p.ld;
  uint32_t* ck = reinterpret_cast<uint32_t*>(base + p.off_ck);
  int32_t* cj = reinterpret_cast<int32_t*>(base + p.off_cj);
  int* cn = reinterpret_cast<int*>(base + p.off_cn);
  int* rowlen = mode == kIndexReindex ? reinterpret_cast<int*>(base + p.off_rl) : nullptr;
  uint32_t* hist = p.dec && !so ? reinterpret_cast<uint32_t*>(base + p.off_h) : nullptr;
  // Lower edges from the prefill scorer's histograms pay off only for long rows: with a few
  // thousand keys the select is cheap, and the histograms' set-up per query tile is not.
  int64_t emax_all = 0;  // entries visible to the call's last query, over this launch's sequences
  for (int i = 0; i < nb; ++i) emax_all = max(emax_all, (pos.p0[i] + a.T) >> a.rshift);
  uint32_t* lower = p.tc && !so && emax_all >= kMinHistRow ? reinterpret_cast<uint32_t*>(base + p.off_lo) : nullptr;
  // long rows of csa2_index_topk: candidate lists instead of dense score rows
  const bool use_cand = lower && p.cand;
  int32_t* cand_j = use_cand ? reinterpret_cast<int32_t*>(base + p.off_candj) : nullptr;
  int* cand_n = use_cand ? reinterpret_cast<int*>(base + p.off_candn) : nullptr;
  uint32_t* pk = reinterpret_cast<uint32_t*>(base + p.off_pk);
  int32_t* pj = reinterpret_cast<int32_t*>(base + p.off_pj);
  int* pn = reinterpret_cast<int*>(base + p.off_pn);
  const size_t pool_chunk_smem = (size_t)kPoolChunk * 4 + (size_t)kPoolSel * 8;
  const size_t pool_merge_smem = (size_t)max(p.pnch, 1) * kPoolSel * 8 + (size_t)kPoolSel * 8;
  const size_t score_smem = (size_t)kQT * kHI * kDI * 4;
  const size_t chunk_smem = (size_t)min64(p.chunk, p.ld) * 4;  // a chunk holds at most ld keys
  const size_t merge_smem = (size_t)p.nchunks * kTopK * 8;
  cudaError_t e;
  e = cudaFuncSetAttribute(score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)score_smem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(topk_chunk_kernel<kTopkThreads>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)chunk_smem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(topk_chunk_kernel<kTopkSmall>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)chunk_smem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(topk_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)merge_smem);
  if (e != cudaSuccess) return e;
  if (mode == kIndexPool) {
    e = cudaFuncSetAttribute(pool_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pool_chunk_smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(pool_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pool_merge_smem);
    if (e != cudaSuccess) return e;
  }
  for (int t0 = 0; t0 < a.T; t0 += p.Tq) {
    const int tq = min(p.Tq, a.T - t0);
    int64_t emax = 0;
    for (int i = 0; i < nb; ++i) emax = max(emax, (pos.p0[i] + t0 + tq) >> a.rshift);
    if (mode == kIndexReindex) {  // every query row scans its own pool
      e = launch_index_scores_decode_tc(a, pos, b0, nb, t0, tq, p.Tq, sc, ld, rowlen, hist, num_sms, st);
      if (e != cudaSuccess) return e;
      emax = min64(emax, (int64_t)kHsiBlock * kHsiBlocks);
    } else if (p.tc) {
          e = launch_index_scores_tc(a, pos, b0, nb, t0, tq, p.Tq, emax, emax_all, t0 == 0,
                                 reinterpret_cast<uint8_t*>(base + p.off_img), wq, sc, ld, lower, cand_j, cand_n,
                                 num_sms, st);
      if (e != cudaSuccess) return e;
    } else if (a.T == 1) {
      if (emax > 0) {
        e = launch_index_scores_decode_tc(a, pos, b0, nb, 0, 1, 1, sc, ld, nullptr, hist, num_sms, st);
        if (e != cudaSuccess) return e;
      }
    } else {
      qprep_kernel<<<dim3(tq, nb), kQprepThreads, 0, st>>>(a, b0, t0, p.Tq, qdq, wq);
      note_launch();
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (mode != kIndexReindex && !p.tc && a.T > 1 && emax > 0) {
      dim3 g((unsigned)((emax + kScoreThreads - 1) / kScoreThreads), (unsigned)((tq + kQT - 1) / kQT), (unsigned)nb);
      score_kernel<<<g, kScoreThreads, score_smem, st>>>(a, pos, b0, t0, p.Tq, qdq, wq, sc, ld);
      note_launch();
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (so) continue;
    if (use_cand) {  // the rows' top-512 from their candidate lists
      topk_cand_kernel<<<dim3(tq, nb), kTopkThreads, 0, st>>>(a, pos, b0, t0, p.Tq, reinterpret_cast<const uint32_t*>(sc),
                                                              cand_j, cand_n, p.ld);
      note_launch();
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
      continue;
    }
    const int nch = (int)max64(1, (emax + p.chunk - 1) / p.chunk);
    // rows with a histogram (decode) follow the scorer directly: dependent launches (the
    // launch and block scheduling overlap the previous kernel's end)
    if (hist)
      e = launch_dependent(topk_chunk_kernel<kTopkThreads>, dim3(nch, tq, nb), dim3(kTopkThreads), chunk_smem, st, a,
                           pos, b0, t0, p.Tq, sc, p.ld, p.chunk, nch, ck, cj, cn, rowlen, hist, nullptr);
    else
      topk_chunk_kernel<kTopkSmall><<<dim3(nch, tq, nb), kTopkSmall, chunk_smem, st>>>(
          a, pos, b0, t0, p.Tq, sc, p.ld, p.chunk, nch, ck, cj, cn, rowlen, nullptr, lower);
    note_launch();
    if (e != cudaSuccess || (e = cudaGetLastError()) != cudaSuccess) return e;
    if (nch > 1) {
      e = launch_dependent(topk_merge_kernel, dim3(tq, nb), dim3(kTopkThreads), (size_t)nch * kTopK * 8, st, a, b0, t0,
                           p.Tq, nch, ck, cj, cn);
      note_launch();
      if (e != cudaSuccess || (e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (mode == kIndexPool) {  // the block pool from this pass's score rows
      const int64_t nblk = (emax + kHsiBlock - 1) / kHsiBlock;
      const int pn_launch = nblk > kHsiBlocks ? (int)((nblk + kPoolChunk - 1) / kPoolChunk) : 1;
      pool_chunk_kernel<<<dim3(pn_launch, tq, nb), kTopkThreads, pool_chunk_smem, st>>>(a, pos, b0, t0, p.Tq, sc, p.ld,
                                                                                      p.pnch, pk, pj, pn);
      note_launch();
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
      if (pn_launch > 1) {
        pool_merge_kernel<<<dim3(tq, nb), kTopkThreads, pool_merge_smem, st>>>(a, pos, b0, t0, p.Tq, p.pnch, pk, pj, pn);
        note_launch();
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
      }
    }
  }
  return cudaSuccess;
}

}  // namespace csa2
