// CSA2 oracle: a plain, slow fp64 CPU restatement of one compressed-sparse-attention
// layer (the "Full", ratio-2 source layer).  TEST INFRASTRUCTURE ONLY: the tests, the
// smoke check and the benchmark's CPU-baseline leg call it; the product path never does.
// It shares no code, header, table or helper with the CUDA library.
//
// Sources (pages, by title and section):
//  [PG]  "DeepSeek V4.1 - Pooled group / Source layer, pairs pooled" (atlas page),
//        block "Compressed sparse attention": the equations for w^a, W, k^c, g^c, k^p, c,
//        Z, k^i, k^n, K^I, w^I, S^I, I_t, J^w_t, Y, J, G_t, S, A, O, O-bar; and the
//        paragraph "Between forward calls" (window ring, compressed rows, pair buffer).
//  [RN]  "DeepSeek V4.1 - Window layer / Attention RMSNorm": m2(x), y = gamma*x/sqrt(m2+eps),
//        eps = 1e-20.
//  [IN]  "Inside DeepSeek V4.1" (blog), sections "Attention that looks at 640 places"
//        (128-token FP8 window, pooled pairs, 32x128 FP4 indexer, top 512, 64 heads x 512,
//        sinks) and "890 bytes" (FP4 entries, scales, FP8 window).
//  [KV]  "Inside DeepSeek V4.1 Flash: Deriving the 890-Byte KV Cache", sections
//        "Deriving the 890 bytes per token" and "FP4 is a storage choice ...".
//
// Readings where the pages are silent or garbled (each also listed in the design notes):
//  * FP4 = E2M1 codes, two per byte, element 2i in the low nibble, one UE8M0 scale per 32
//    consecutive values (the OCP MX rule: X = 2^(floor(log2 amax) - 2), elements rounded to
//    nearest, ties to the even code, saturating at +-6).  An all-zero block gets scale byte 0.
//  * FP8 = OCP E4M3 (e4m3fn), round to nearest even, saturating to +-448, no scale.
//  * w^n (lost in the extraction) = gamma_W * RMSNorm(w^a).
//  * RoPE rotates interleaved pairs (2i, 2i+1) of the last 64 dims (or of dims 64..127 of
//    the indexer key) by pos * base^(-2i/64); Z and K^I use pos = 2j, W and Q use the token
//    position t, the output is rotated back by -t.
//  * k^i = c W_IK uses c before RoPE and before FP4.
//  * Q^I is quantised to FP4 (per head row of 128, scale per 32) before the indexer dot.
//  * Top-k: larger score first, equal scores -> lower j first; fewer than k candidates ->
//    all kept, the rest -1; output ascending in j.
//  * Window rows below position 0 do not exist (fewer than 128 rows for t < 127).
//
// Everything is fp64; inputs arrive as float (bf16 inputs widened exactly).
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

namespace {

// E2M1 magnitudes: 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit; exponent 0 is
// subnormal (0.5 * mantissa).  [KV] "FP4 is a storage choice": E2M1 values.
const double kE2M1Mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double e2m1_value(int code) {
  double v = kE2M1Mag[code & 7];
  return (code & 8) ? -v : v;
}

// Nearest E2M1 value; a tie goes to the code whose mantissa bit is 0 ("even").
// Magnitudes above 6 saturate to 6 (nearest representable).
int e2m1_encode(double x) {
  int sign = std::signbit(x) ? 8 : 0;
  double a = std::fabs(x);
  int best = 0;
  double bestd = INFINITY;
  for (int m = 0; m < 8; ++m) {
    double d = std::fabs(a - kE2M1Mag[m]);
    if (d < bestd || (d == bestd && (m & 1) == 0)) {
      best = m;
      bestd = d;
    }
  }
  return sign | best;
}

// OCP E4M3 (e4m3fn): bias 7, exponent 15 with mantissa 7 is NaN, no infinities.
double e4m3_value(int c) {
  int s = (c >> 7) & 1, e = (c >> 3) & 15, m = c & 7;
  if (e == 15 && m == 7) return NAN;
  double v = (e == 0) ? std::ldexp((double)m, -9) : std::ldexp(1.0 + m / 8.0, e - 7);
  return s ? -v : v;
}

// Round to nearest representable finite magnitude, ties to the even code, saturate to 448.
int e4m3_encode(double x) {
  if (std::isnan(x)) return 0x7F;
  int sign = std::signbit(x) ? 0x80 : 0;
  double a = std::fabs(x);
  // magnitudes are increasing in the code for codes 0..126 (126 = 0x7E = 448)
  int lo = 0;
  while (lo < 126 && e4m3_value(lo + 1) <= a) ++lo;
  int best = lo;
  if (lo < 126) {
    double dl = a - e4m3_value(lo), dh = e4m3_value(lo + 1) - a;
    if (dh < dl || (dh == dl && ((lo + 1) & 1) == 0)) best = lo + 1;
  }
  return sign | best;
}

// One MX block of 32 values -> 32 E2M1 codes (returned unpacked) and one UE8M0 scale byte.
void mx_block(const double* v, int* codes, int* scale_byte) {
  double amax = 0.0;
  for (int i = 0; i < 32; ++i) amax = std::max(amax, std::fabs(v[i]));
  int e;
  if (amax == 0.0) {
    e = -127;
  } else {
    int ex;
    std::frexp(amax, &ex);  // amax = f * 2^ex, f in [0.5, 1)  ->  floor(log2 amax) = ex - 1
    e = (ex - 1) - 2;       // emax of E2M1 is 2
    e = std::min(127, std::max(-127, e));
  }
  *scale_byte = e + 127;
  for (int i = 0; i < 32; ++i) codes[i] = e2m1_encode(std::ldexp(v[i], -e));
}

// Quantise a row of n values (n a multiple of 32): codes packed two per byte, element 2i
// in the low nibble; one scale byte per 32 values.
void mx_row(const double* v, int n, uint8_t* codes, uint8_t* scales) {
  int c[32], sb;
  for (int b = 0; b < n / 32; ++b) {
    mx_block(v + 32 * b, c, &sb);
    scales[b] = (uint8_t)sb;
    for (int i = 0; i < 16; ++i) codes[16 * b + i] = (uint8_t)((c[2 * i] & 15) | ((c[2 * i + 1] & 15) << 4));
  }
}

void mx_row_decode(const uint8_t* codes, const uint8_t* scales, int n, double* out) {
  for (int i = 0; i < n; ++i) {
    int byte = codes[i / 2];
    int code = (i & 1) ? (byte >> 4) : (byte & 15);
    out[i] = std::ldexp(e2m1_value(code), (int)scales[i / 32] - 127);
  }
}

// [RN]: y = gamma * x / sqrt(mean(x^2) + eps)
void rmsnorm(const double* x, const float* gamma, int n, double eps, double* y) {
  double ss = 0.0;
  for (int i = 0; i < n; ++i) ss += x[i] * x[i];
  double r = 1.0 / std::sqrt(ss / n + eps);
  for (int i = 0; i < n; ++i) y[i] = (double)gamma[i] * x[i] * r;
}

// Rotate interleaved pairs of x[0..d) by angle pos * base^(-2i/d) (sign = -1: inverse).
void rope(double* x, int d, double pos, double base, double sign) {
  for (int i = 0; i < d / 2; ++i) {
    double theta = std::pow(base, -2.0 * i / d);
    double ang = sign * pos * theta;
    double c = std::cos(ang), s = std::sin(ang);
    double x0 = x[2 * i], x1 = x[2 * i + 1];
    x[2 * i] = x0 * c - x1 * s;
    x[2 * i + 1] = x0 * s + x1 * c;
  }
}

constexpr int D = 512;     // entry / head width
constexpr int DR = 64;     // rotated dims
constexpr int DI = 128;    // indexer key / head width
constexpr int HI = 32;     // indexer heads
constexpr int H = 64;      // attention heads
constexpr int WIN = 128;   // window rows
constexpr int TOPK = 512;  // selected entries

// One compressed entry from its tokens: [PG] k^p, c, Z, k^i, k^n, K^I.  At compression
// ratio 2 the entry j pools tokens (2j, 2j+1) (k0/g0 and k1/g1); at ratio 1 it is token j
// itself (k0 == nullptr: the softmax over one token is 1, so k^p = k^c).  rope_pos is the
// position the entry is rotated by: r * j.
void write_entry(const float* k0, const float* g0, const float* k1, const float* g1, double rope_pos,
                 const float* gamma_c, const float* w_ik, const float* gamma_ik, double base,
                 double eps, uint8_t* zc, uint8_t* zs, uint8_t* kc, uint8_t* ks, double* z_pre,
                 double* ki_pre) {
  double kp[D], c[D], z[D], ki[DI], kn[DI];
  for (int ch = 0; ch < D; ++ch) {
    if (!k0) {
      kp[ch] = k1[ch];
      continue;
    }
    // softmax over the two tokens of the pair, per channel
    double a = g0[ch], b = g1[ch], m = std::max(a, b);
    double ea = std::exp(a - m), eb = std::exp(b - m);
    double w0 = ea / (ea + eb), w1 = eb / (ea + eb);
    kp[ch] = w0 * k0[ch] + w1 * k1[ch];
  }
  rmsnorm(kp, gamma_c, D, eps, c);
  std::memcpy(z, c, sizeof z);
  rope(z + (D - DR), DR, rope_pos, base, 1.0);
  if (z_pre) std::memcpy(z_pre, z, sizeof z);
  mx_row(z, D, zc, zs);
  for (int o = 0; o < DI; ++o) {
    double s = 0.0;
    for (int i = 0; i < D; ++i) s += c[i] * (double)w_ik[(int64_t)i * DI + o];
    ki[o] = s;
  }
  rmsnorm(ki, gamma_ik, DI, eps, kn);
  rope(kn + 64, DI - 64, rope_pos, base, 1.0);
  if (ki_pre) std::memcpy(ki_pre, kn, sizeof kn);
  mx_row(kn, DI, kc, ks);
}

}  // namespace

extern "C" {

// ---------------------------------------------------------------- codecs (for the pins)
double csa2o_e2m1_value(int code) { return e2m1_value(code); }
int csa2o_e2m1_encode(double x) { return e2m1_encode(x); }
double csa2o_e4m3_value(int code) { return e4m3_value(code); }
int csa2o_e4m3_encode(double x) { return e4m3_encode(x); }
void csa2o_e4m3_encode_many(const double* x, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = (uint8_t)e4m3_encode(x[i]);
}
void csa2o_mx_quantize(const double* v, int64_t rows, int n, uint8_t* codes, uint8_t* scales) {
  for (int64_t r = 0; r < rows; ++r) mx_row(v + r * n, n, codes + r * (n / 2), scales + r * (n / 32));
}
void csa2o_mx_dequantize(const uint8_t* codes, const uint8_t* scales, int64_t rows, int n, double* out) {
  for (int64_t r = 0; r < rows; ++r) mx_row_decode(codes + r * (n / 2), scales + r * (n / 32), n, out + r * n);
}
void csa2o_rmsnorm(const double* x, const float* gamma, int n, double eps, double* y) { rmsnorm(x, gamma, n, eps, y); }
void csa2o_rope(double* x, int d, double pos, double base, int inverse) { rope(x, d, pos, base, inverse ? -1.0 : 1.0); }

// ---------------------------------------------------------------- writer, one sequence
// Appends T tokens at absolute positions p0 .. p0+T-1 to a layer of compression ratio
// `ratio` (2: entry j pools tokens 2j, 2j+1; 1: entry j is token j, no pair buffer).
//  kc, gc, wa: [T, 512]; pair_k_in/pair_g_in: the buffered token p0-1 (needed iff p0 odd);
//  pair_k_out/pair_g_out: receive token p0+T-1 iff p0+T is odd (may alias the inputs).
//  z_codes [cap,256], z_scales [cap,16], ki_codes [cap,64], ki_scales [cap,4]: this
//  sequence's caches; entry j is written once token 2j+1 arrives.
//  window [127+T, 512]: row r holds position p0-127+r; rows 127.. are written here.
//  z_pre [n_new,512], ki_pre [n_new,128], win_pre [T,512] (optional): the fp64 values just
//  before FP4 / FP8, for the near-boundary rule of the parity tests.
// Returns the number of entries written; their first index is floor(p0/ratio).
int64_t csa2o_write_seq(int ratio, int T, int64_t p0, const float* kc, const float* gc, const float* wa,
                        const float* gamma_c, const float* w_ik, const float* gamma_ik,
                        const float* gamma_w, double base, double eps, const float* pair_k_in,
                        const float* pair_g_in, float* pair_k_out, float* pair_g_out,
                        int64_t cap, uint8_t* z_codes, uint8_t* z_scales, uint8_t* ki_codes,
                        uint8_t* ki_scales, uint8_t* window, double* z_pre, double* ki_pre,
                        double* win_pre) {
  if (ratio != 1 && ratio != 2) return -1;
  int64_t j0 = p0 / ratio;
  // entries completed by this call: j whose last token ratio*j + ratio-1 is in p0 .. p0+T-1
  std::vector<int64_t> js;
  for (int t = 0; t < T; ++t)
    if ((p0 + t) % ratio == ratio - 1) js.push_back((p0 + t) / ratio);
  for (int64_t j : js)
    if (j >= cap) return -1;
  std::vector<float> keep_k(D), keep_g(D);
  bool have_pair = pair_k_in && pair_g_in;
  if (have_pair) {
    std::memcpy(keep_k.data(), pair_k_in, D * sizeof(float));
    std::memcpy(keep_g.data(), pair_g_in, D * sizeof(float));
  }
#pragma omp parallel for schedule(dynamic)
  for (int64_t n = 0; n < (int64_t)js.size(); ++n) {
    int64_t j = js[n];
    int64_t t1 = ratio * j + ratio - 1 - p0;  // local index of the entry's last token
    const float *k0 = nullptr, *g0 = nullptr;
    if (ratio == 2) {
      if (t1 >= 1) {
        k0 = kc + (t1 - 1) * D;
        g0 = gc + (t1 - 1) * D;
      } else {
        k0 = keep_k.data();
        g0 = keep_g.data();
      }
    }
    write_entry(k0, g0, kc + t1 * D, gc + t1 * D, (double)(ratio * j), gamma_c, w_ik, gamma_ik, base, eps,
                z_codes + j * 256, z_scales + j * 16, ki_codes + j * 64, ki_scales + j * 4,
                z_pre ? z_pre + (j - j0) * D : nullptr, ki_pre ? ki_pre + (j - j0) * DI : nullptr);
  }
  // [PG] W_{t,448:} <- R_t w^n_{t,448:};  W <- FP8(W)
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    double x[D], y[D];
    for (int i = 0; i < D; ++i) x[i] = wa[(int64_t)t * D + i];
    rmsnorm(x, gamma_w, D, eps, y);
    rope(y + (D - DR), DR, (double)(p0 + t), base, 1.0);
    if (win_pre) std::memcpy(win_pre + (int64_t)t * D, y, sizeof y);
    uint8_t* row = window + (int64_t)(127 + t) * D;
    for (int i = 0; i < D; ++i) row[i] = (uint8_t)e4m3_encode(y[i]);
  }
  if (ratio == 2 && (p0 + T) % 2 == 1 && pair_k_out && pair_g_out) {
    std::memcpy(pair_k_out, kc + (int64_t)(T - 1) * D, D * sizeof(float));
    std::memcpy(pair_g_out, gc + (int64_t)(T - 1) * D, D * sizeof(float));
  }
  return (int64_t)js.size();
}

// ---------------------------------------------------------------- indexer scores
// Query rows at absolute positions pos[r]: Q^I qi [nq,32,128], w^I wI [nq,32].
// S^I_{t,j} = sum_h w^I_{t,h} ReLU(Q^I_{h,t} . K^I_j) for j < floor((t+1)/ratio)  ([PG] S^I,
// I_t; an entry is visible once its last token is).
// scores [nq, ld]: row r gets E_r = floor((pos+1)/ratio) values; the rest is left untouched.
// qi_codes [nq,32,64] / qi_scales [nq,32,4] (optional): the FP4 form of Q^I.
int csa2o_index_scores(int ratio, int nq, const int64_t* pos, const float* qi, const float* wI,
                       const uint8_t* ki_codes, const uint8_t* ki_scales, int64_t n_entries,
                       double* scores, int64_t ld, uint8_t* qi_codes, uint8_t* qi_scales) {
  if (ratio != 1 && ratio != 2) return -1;
  for (int r = 0; r < nq; ++r)
    if ((pos[r] + 1) / ratio > n_entries || (pos[r] + 1) / ratio > ld) return -1;
#pragma omp parallel for schedule(dynamic)
  for (int r = 0; r < nq; ++r) {
    std::vector<double> qv(HI * DI), kv(DI), q64(DI);
    for (int h = 0; h < HI; ++h) {
      uint8_t c[64], s[4];
      for (int i = 0; i < DI; ++i) q64[i] = qi[((int64_t)r * HI + h) * DI + i];
      mx_row(q64.data(), DI, c, s);
      mx_row_decode(c, s, DI, qv.data() + h * DI);
      if (qi_codes) std::memcpy(qi_codes + ((int64_t)r * HI + h) * 64, c, 64);
      if (qi_scales) std::memcpy(qi_scales + ((int64_t)r * HI + h) * 4, s, 4);
    }
    int64_t E = (pos[r] + 1) / ratio;
    for (int64_t j = 0; j < E; ++j) {
      mx_row_decode(ki_codes + j * 64, ki_scales + j * 4, DI, kv.data());
      double sc = 0.0;
      for (int h = 0; h < HI; ++h) {
        double dot = 0.0;
        for (int i = 0; i < DI; ++i) dot += qv[h * DI + i] * kv[i];
        sc += (double)wI[(int64_t)r * HI + h] * std::max(0.0, dot);
      }
      scores[(int64_t)r * ld + j] = sc;
    }
  }
  return 0;
}

// ---------------------------------------------------------------- top-k
// For each row: the k largest of scores[r, 0..E_r) (ties: lower j first), ascending in j,
// padded with -1.  kth [nq,2] (optional): the k-th and (k+1)-th largest scores in
// (score desc, j asc) order, NaN where absent.  top [nq,k] (optional): the chosen scores.
int csa2o_topk(int nq, const int64_t* E, const double* scores, int64_t ld, int k, int32_t* idx,
               double* top, double* kth) {
#pragma omp parallel for schedule(dynamic)
  for (int r = 0; r < nq; ++r) {
    const double* s = scores + (int64_t)r * ld;
    std::vector<int64_t> order(E[r]);
    for (int64_t j = 0; j < E[r]; ++j) order[j] = j;
    std::sort(order.begin(), order.end(), [s](int64_t a, int64_t b) {
      if (s[a] != s[b]) return s[a] > s[b];
      return a < b;
    });
    int64_t n = std::min<int64_t>(k, E[r]);
    std::vector<int64_t> chosen(order.begin(), order.begin() + n);
    std::sort(chosen.begin(), chosen.end());
    for (int i = 0; i < k; ++i) {
      idx[(int64_t)r * k + i] = i < n ? (int32_t)chosen[i] : -1;
      if (top) top[(int64_t)r * k + i] = i < n ? s[chosen[i]] : NAN;
    }
    if (kth) {
      kth[2 * r] = E[r] >= k ? s[order[k - 1]] : NAN;
      kth[2 * r + 1] = E[r] > k ? s[order[k]] : NAN;
    }
  }
  return 0;
}

// ---------------------------------------------------------------- hierarchical sparse indexer
// "Inside DeepSeek V4.1", section "Most layers borrow", and "Deriving the 890-Byte KV Cache",
// section "Hierarchical indexing bounds the later searches": the first Full layer groups the
// entries into blocks of 8, scores a block by its best entry score and keeps 2048 blocks
// (16384 candidates), always including the block that holds the newest entries; later
// Reindex layers take their own top-512 inside that pool.
// Reading: block k = entries 8k..8k+7 (visible ones only: j < E); pool = the newest block
// (E-1)/8 plus the 2047 best other blocks (block score desc, block index asc), or every block
// when there are at most 2048; ascending block indices, -1 padded.
constexpr int HSI_BLK = 8, HSI_BLOCKS = 2048;

int csa2o_hsi_pool(int nq, const int64_t* E, const double* scores, int64_t ld, int32_t* pool) {
#pragma omp parallel for schedule(dynamic)
  for (int r = 0; r < nq; ++r) {
    const double* s = scores + (int64_t)r * ld;
    const int64_t nb = (E[r] + HSI_BLK - 1) / HSI_BLK;
    std::vector<int64_t> chosen;
    if (nb <= HSI_BLOCKS) {
      for (int64_t k = 0; k < nb; ++k) chosen.push_back(k);
    } else {
      std::vector<double> bs(nb - 1);
      for (int64_t k = 0; k + 1 < nb; ++k) {
        double m = -INFINITY;
        for (int64_t j = HSI_BLK * k; j < HSI_BLK * (k + 1); ++j) m = std::max(m, s[j]);  // all visible
        bs[k] = m;
      }
      std::vector<int64_t> order(nb - 1);
      for (int64_t k = 0; k + 1 < nb; ++k) order[k] = k;
      std::sort(order.begin(), order.end(), [&bs](int64_t a, int64_t b) {
        if (bs[a] != bs[b]) return bs[a] > bs[b];
        return a < b;
      });
      chosen.assign(order.begin(), order.begin() + (HSI_BLOCKS - 1));
      chosen.push_back(nb - 1);  // the newest block
      std::sort(chosen.begin(), chosen.end());
    }
    for (int i = 0; i < HSI_BLOCKS; ++i)
      pool[(int64_t)r * HSI_BLOCKS + i] = i < (int)chosen.size() ? (int32_t)chosen[i] : -1;
  }
  return 0;
}

// Reindex top-k: the k largest of scores[r, j] over the pool's visible entries j (j < E),
// equal scores -> lower j first; ascending in j, -1 padded.
int csa2o_reindex_topk(int nq, const int64_t* E, const double* scores, int64_t ld, const int32_t* pool, int k,
                       int32_t* idx) {
#pragma omp parallel for schedule(dynamic)
  for (int r = 0; r < nq; ++r) {
    const double* s = scores + (int64_t)r * ld;
    std::vector<int64_t> cand;
    for (int i = 0; i < HSI_BLOCKS; ++i) {
      const int32_t blk = pool[(int64_t)r * HSI_BLOCKS + i];
      if (blk < 0) continue;
      for (int64_t j = (int64_t)HSI_BLK * blk; j < (int64_t)HSI_BLK * (blk + 1) && j < E[r]; ++j) cand.push_back(j);
    }
    std::sort(cand.begin(), cand.end(), [s](int64_t a, int64_t b) {
      if (s[a] != s[b]) return s[a] > s[b];
      return a < b;
    });
    const int64_t n = std::min<int64_t>(k, (int64_t)cand.size());
    std::vector<int64_t> chosen(cand.begin(), cand.begin() + n);
    std::sort(chosen.begin(), chosen.end());
    for (int i = 0; i < k; ++i) idx[(int64_t)r * k + i] = i < n ? (int32_t)chosen[i] : -1;
  }
  return 0;
}

// ---------------------------------------------------------------- sink-softmax MQA
// Query rows at absolute positions pos[r] with Q q [nq,64,512] (already rotated), sinks [64].
// G_t = [window rows for positions max(0,t-127)..t ; Z rows idx[r, i] (>= 0)]   ([PG] J, G_t)
// With a replay start win_start = s ("Inside DeepSeek V4.1 Flash: Deriving the 890-Byte KV
// Cache", section "Bounded replay trades exact state for cheaper resumption") the window
// rows are positions max(s, t-127)..t; s = 0 is the plain window.
// S = Q.G/sqrt(512);  A = exp S / (exp s_h + sum exp S);  O = sum A G;  O[448:] <- R_t^-1 O.
// window: rows of positions win_p0 .. win_p0+win_rows-1 (row r <-> position win_p0 + r).
// out [nq,64,512]; mass [nq,64] (optional) = sum_i A; nrows [nq] (optional) = |G_t|.
int csa2o_attend(int nq, const int64_t* pos, const float* q, const float* sinks,
                 const uint8_t* z_codes, const uint8_t* z_scales, int64_t n_entries,
                 const uint8_t* window, int64_t win_p0, int64_t win_rows, const int32_t* idx,
                 double base, int64_t win_start, double* out, double* mass, int32_t* nrows) {
  for (int r = 0; r < nq; ++r) {
    int64_t lo = std::max<int64_t>(std::max<int64_t>(0, win_start), pos[r] - (WIN - 1));
    if (win_start > pos[r]) return -3;
    if (lo < win_p0 || pos[r] >= win_p0 + win_rows) return -1;
    for (int i = 0; i < TOPK; ++i)
      if (idx[(int64_t)r * TOPK + i] >= n_entries) return -2;
  }
#pragma omp parallel for schedule(dynamic)
  for (int r = 0; r < nq; ++r) {
    int64_t p = pos[r];
    int64_t lo = std::max<int64_t>(std::max<int64_t>(0, win_start), p - (WIN - 1));
    std::vector<double> G;
    for (int64_t x = lo; x <= p; ++x) {
      const uint8_t* row = window + (x - win_p0) * D;
      for (int i = 0; i < D; ++i) G.push_back(e4m3_value(row[i]));
    }
    for (int i = 0; i < TOPK; ++i) {
      int32_t j = idx[(int64_t)r * TOPK + i];
      if (j < 0) continue;
      double tmp[D];
      mx_row_decode(z_codes + (int64_t)j * 256, z_scales + (int64_t)j * 16, D, tmp);
      G.insert(G.end(), tmp, tmp + D);
    }
    int64_t n = (int64_t)G.size() / D;
    if (nrows) nrows[r] = (int32_t)n;
    std::vector<double> S(n);
    const double scale = 1.0 / std::sqrt((double)D);
    for (int h = 0; h < H; ++h) {
      const float* qh = q + ((int64_t)r * H + h) * D;
      double m = sinks[h];
      for (int64_t i = 0; i < n; ++i) {
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += (double)qh[d] * G[i * D + d];
        S[i] = dot * scale;
        m = std::max(m, S[i]);
      }
      double den = std::exp((double)sinks[h] - m);
      for (int64_t i = 0; i < n; ++i) den += std::exp(S[i] - m);
      double o[D] = {0.0}, tot = 0.0;
      for (int64_t i = 0; i < n; ++i) {
        double a = std::exp(S[i] - m) / den;
        tot += a;
        for (int d = 0; d < D; ++d) o[d] += a * G[i * D + d];
      }
      rope(o + (D - DR), DR, (double)p, base, -1.0);
      std::memcpy(out + ((int64_t)r * H + h) * D, o, sizeof o);
      if (mass) mass[(int64_t)r * H + h] = tot;
    }
  }
  return 0;
}

}  // extern "C"
