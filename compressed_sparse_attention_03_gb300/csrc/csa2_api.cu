// C-ABI front end of libcsa2.so: argument validation, the handle, workspace sizing, and the
// split of large batches into launches of at most kMaxSeqPerLaunch sequences.
// The entry points and their contracts are documented in include/csa2.h.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>
#include <new>

#include "../../include/csa2.h"
#include "csa2_internal.h"

struct csa2_handle {
  csa2_config cfg;
  csa2::RopeFreq rf;
  int device;
  int num_sms;
  int rshift;  // log2 of the compression ratio (0: ratio 1, 1: ratio 2)
  // positions read on the device (csa2_set_device_positions): the caller's array and the bound
  // the host plans with
  const int64_t* pos_dev = nullptr;
  int64_t pos_hi = 0;
};

namespace {
// Set by a kernel that read a device position outside 0..bound (every handle's; csa2_check).
__device__ unsigned g_pos_flag;
}  // namespace

namespace {

std::atomic<uint64_t> g_launches{0};

}  // namespace

void csa2::note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

csa2::SeqPos pack_pos(const int64_t* p0, int b0, int nb) {
  csa2::SeqPos s;
  std::memset(&s, 0, sizeof s);
  for (int i = 0; i < nb; ++i) s.p0[i] = p0[b0 + i];
  return s;
}

// The positions of a call's sequences b0 .. b0+nb-1: the host values, or with device positions
// set, the device array (the host copy then holds the bound, for the launchers' planning).
csa2::SeqPos call_pos(const csa2_handle* h, const int64_t* p0, int b0, int nb) {
  if (!h->pos_dev) return pack_pos(p0, b0, nb);
  csa2::SeqPos s;
  std::memset(&s, 0, sizeof s);
  for (int i = 0; i < nb; ++i) s.p0[i] = h->pos_hi;
  s.dev = h->pos_dev + b0;
  s.hi = h->pos_hi;
  void* f = nullptr;
  cudaGetSymbolAddress(&f, g_pos_flag);
  s.flag = static_cast<unsigned*>(f);
  return s;
}

// The host positions a call validates and plans with: its p0 argument, or with device positions
// set, the bound for every sequence (the argument is then not read).
const int64_t* plan_p0(const csa2_handle* h, const int64_t* p0, int B, std::vector<int64_t>& tmp) {
  if (!h->pos_dev) return p0;
  tmp.assign((size_t)B, h->pos_hi);
  return tmp.data();
}

csa2_status cuda_status(cudaError_t e) { return e == cudaSuccess ? CSA2_OK : CSA2_ERR_CUDA; }

csa2::SeqPos no_replay() {
  csa2::SeqPos s;
  std::memset(&s, 0, sizeof s);
  return s;
}

// Largest visible-entry count over the batch for queries p0..p0+T-1: floor((p0+T)/ratio).
int64_t max_visible(const int64_t* p0, int B, int T, int rshift) {
  int64_t m = 0;
  for (int b = 0; b < B; ++b) m = std::max<int64_t>(m, (p0[b] + T) >> rshift);
  return m;
}

// Positions are limited so that every entry index and window row fits int32 arithmetic
// used by the kernels and the top-k candidate domain (at most 2^20 entries per query).
constexpr int64_t kMaxPos = (int64_t(1) << 21) - 2;

csa2_status check_p0(const int64_t* p0, int B, int T) {
  if (!p0) return CSA2_ERR_INVALID_ARG;
  for (int b = 0; b < B; ++b)
    if (p0[b] < 0 || p0[b] + T > kMaxPos) return CSA2_ERR_SHAPE;
  return CSA2_OK;
}

}  // namespace

extern "C" {

void csa2_default_config(csa2_config* c) {
  if (!c) return;
  c->heads = 64;
  c->head_dim = 512;
  c->rope_dims = 64;
  c->idx_heads = 32;
  c->idx_dim = 128;
  c->window = 128;
  c->topk = 512;
  c->ratio = 2;
  c->rope_base = 10000.0;
  c->eps = 1e-20;
}

csa2_status csa2_create(const csa2_config* cfg, csa2_handle** out) {
  if (!out) return CSA2_ERR_INVALID_ARG;
  *out = nullptr;
  if (!cfg) return CSA2_ERR_INVALID_ARG;
  if (cfg->heads != 64 || cfg->head_dim != 512 || cfg->rope_dims != 64 || cfg->idx_heads != 32 || cfg->idx_dim != 128 ||
      cfg->window != 128 || cfg->topk != 512 || (cfg->ratio != 1 && cfg->ratio != 2))
    return CSA2_ERR_UNSUPPORTED;
  if (!(cfg->rope_base > 1.0) || !std::isfinite(cfg->rope_base) || !(cfg->eps >= 0.0) || !std::isfinite(cfg->eps))
    return CSA2_ERR_INVALID_ARG;
  csa2_handle* h = new (std::nothrow) csa2_handle;
  if (!h) return CSA2_ERR_INVALID_ARG;
  h->cfg = *cfg;
  h->rshift = cfg->ratio == 2 ? 1 : 0;
  for (int i = 0; i < csa2::kDR / 2; ++i) h->rf.inv_freq[i] = std::pow(cfg->rope_base, -2.0 * i / csa2::kDR);
  if (cudaGetDevice(&h->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device) != cudaSuccess) {
    delete h;
    return CSA2_ERR_CUDA;
  }
  *out = h;
  return CSA2_OK;
}

void csa2_destroy(csa2_handle* h) { delete h; }

// Positions from device memory (include/csa2.h).
csa2_status csa2_set_device_positions(csa2_handle* h, const int64_t* p0_dev, int64_t p0_max) {
  if (!h) return CSA2_ERR_INVALID_ARG;
  if (!p0_dev) {
    h->pos_dev = nullptr;
    h->pos_hi = 0;
    return CSA2_OK;
  }
  if ((reinterpret_cast<uintptr_t>(p0_dev) & 7u) != 0) return CSA2_ERR_ALIGN;
  if (p0_max < 0 || p0_max + 1 > kMaxPos) return CSA2_ERR_SHAPE;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return CSA2_ERR_CUDA;
  if (dev != h->device) return CSA2_ERR_INVALID_ARG;
  void* f = nullptr;
  if (cudaGetSymbolAddress(&f, g_pos_flag) != cudaSuccess) return CSA2_ERR_CUDA;  // loads the module now
  h->pos_dev = p0_dev;
  h->pos_hi = p0_max;
  return CSA2_OK;
}

uint64_t csa2_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

const char* csa2_status_string(csa2_status s) {
  switch (s) {
    case CSA2_OK: return "ok";
    case CSA2_ERR_INVALID_ARG: return "invalid argument";
    case CSA2_ERR_SHAPE: return "inconsistent sizes";
    case CSA2_ERR_ALIGN: return "pointer not 16-byte aligned";
    case CSA2_ERR_WORKSPACE: return "workspace too small";
    case CSA2_ERR_UNSUPPORTED: return "unsupported configuration";
    case CSA2_ERR_CUDA: return "CUDA error";
    case CSA2_ERR_TOO_LARGE: return "batch exceeds the fixed scratch of csa2_attend_static";
    case CSA2_ERR_TIMEOUT: return "a bounded wait inside a kernel gave up";
  }
  return "unknown status";
}

size_t csa2_workspace_bytes(const csa2_handle* h, int op, int B, int T, int64_t max_entries) {
  if (!h || B <= 0 || T <= 0 || max_entries < 0) return 0;
  switch (op) {
    case CSA2_OP_WRITE_CACHE: return 0;
    case CSA2_OP_INDEX_TOPK: return csa2::index_workspace_bytes(B, T, max_entries, h->num_sms);
    case CSA2_OP_ATTEND: return csa2::attend_workspace_bytes(B, T, h->num_sms);
    case CSA2_OP_INDEX_POOL: return csa2::index_workspace_bytes(B, T, max_entries, h->num_sms, csa2::kIndexPool);
    case CSA2_OP_REINDEX_TOPK: return csa2::index_workspace_bytes(B, T, max_entries, h->num_sms, csa2::kIndexReindex);
    case CSA2_OP_INDEX_SCORES: return csa2::index_workspace_bytes(B, T, max_entries, h->num_sms, csa2::kIndexScores);
  }
  return 0;
}

csa2_status csa2_write_cache(csa2_handle* h, const uint16_t* kc, const uint16_t* gc, const uint16_t* wa,
                             const float* gamma_c, const uint16_t* w_ik, const float* gamma_ik, const float* gamma_w,
                             const int64_t* p0, int B, int T, float* pair_kc, float* pair_gc, uint8_t* z_codes,
                             uint8_t* z_scales, uint8_t* ki_codes, uint8_t* ki_scales, int64_t cap, uint8_t* window,
                             void* /*ws*/, size_t /*ws_bytes*/, csa2_stream_t stream) {
  if (!h || !kc || !gc || !wa || !gamma_c || !w_ik || !gamma_ik || !gamma_w || !z_codes || !z_scales || !ki_codes ||
      !ki_scales || !window)
    return CSA2_ERR_INVALID_ARG;
  if (B <= 0 || T <= 0 || cap < 0 || T > 65535) return CSA2_ERR_INVALID_ARG;
  std::vector<int64_t> bound;
  p0 = plan_p0(h, p0, B, bound);
  csa2_status st = check_p0(p0, B, T);
  if (st != CSA2_OK) return st;
  const int rs = h->rshift;
  // the pair buffer exists at ratio 2 only; with device positions any position may be odd
  bool need_pair = rs == 1 && ((T & 1) != 0 || h->pos_dev);
  for (int b = 0; b < B; ++b) {
    if (rs == 1 && (p0[b] & 1)) need_pair = true;
    if ((p0[b] + T) >> rs > cap) return CSA2_ERR_SHAPE;  // last entry floor((p0+T)/ratio)-1 < cap
  }
  if (need_pair && (!pair_kc || !pair_gc)) return CSA2_ERR_INVALID_ARG;
  const void* ptrs[] = {kc, gc, wa, gamma_c, w_ik, gamma_ik, gamma_w, z_codes, z_scales, ki_codes, ki_scales, window};
  for (const void* p : ptrs)
    if (!aligned16(p)) return CSA2_ERR_ALIGN;
  if ((pair_kc && !aligned16(pair_kc)) || (pair_gc && !aligned16(pair_gc))) return CSA2_ERR_ALIGN;
  csa2::WriterArgs a{};
  for (int b0 = 0; b0 < B; b0 += csa2::kMaxSeqPerLaunch) {
    const int nb = std::min(B - b0, csa2::kMaxSeqPerLaunch);
    a.kc = kc; a.gc = gc; a.wa = wa; a.w_ik = w_ik;
    a.gamma_c = gamma_c; a.gamma_ik = gamma_ik; a.gamma_w = gamma_w;
    a.pair_kc = pair_kc; a.pair_gc = pair_gc;
    a.z_codes = z_codes; a.z_scales = z_scales; a.ki_codes = ki_codes; a.ki_scales = ki_scales; a.window = window;
    a.cap = cap; a.T = T; a.rshift = rs; a.eps = h->cfg.eps;
    st = cuda_status(csa2::launch_writer(a, call_pos(h, p0, b0, nb), b0, nb, h->rf, reinterpret_cast<cudaStream_t>(stream)));
    if (st != CSA2_OK) return st;
  }
  return CSA2_OK;
}

namespace {

// Shared body of the three indexer entry points: mode selects the plain top-512, the top-512
// plus the hierarchical pool, or the top-512 over a given pool.
csa2_status index_call(csa2_handle* h, const uint16_t* qi, const uint16_t* wI, const uint8_t* ki_codes,
                       const uint8_t* ki_scales, int64_t cap, const int64_t* p0, int B, int T, int32_t* idx,
                       float* top_scores, int32_t* pool_out, const int32_t* pool_in, int mode, void* ws,
                       size_t ws_bytes, csa2_stream_t stream, float* scores_out = nullptr, int64_t scores_ld = 0) {
  const bool so = mode == csa2::kIndexScores;
  if (!h || !qi || !wI || !ki_codes || !ki_scales || (!idx && !so) || (so && !scores_out)) return CSA2_ERR_INVALID_ARG;
  if ((mode == csa2::kIndexPool && !pool_out) || (mode == csa2::kIndexReindex && !pool_in)) return CSA2_ERR_INVALID_ARG;
  if (B <= 0 || T <= 0 || cap < 0 || T > 65535) return CSA2_ERR_INVALID_ARG;
  std::vector<int64_t> bound;
  p0 = plan_p0(h, p0, B, bound);
  csa2_status st = check_p0(p0, B, T);
  if (st != CSA2_OK) return st;
  const int64_t emax = max_visible(p0, B, T, h->rshift);
  if (emax > cap) return CSA2_ERR_SHAPE;
  if (emax > (int64_t(1) << 20)) return CSA2_ERR_UNSUPPORTED;
  if (so && (scores_ld < std::max<int64_t>(emax, 1) || scores_ld % 4)) return CSA2_ERR_SHAPE;
  const void* ptrs[] = {qi, wI, ki_codes, ki_scales, so ? static_cast<const void*>(scores_out) : idx};
  for (const void* p : ptrs)
    if (!aligned16(p)) return CSA2_ERR_ALIGN;
  if (top_scores && !aligned16(top_scores)) return CSA2_ERR_ALIGN;
  if ((pool_out && !aligned16(pool_out)) || (pool_in && !aligned16(pool_in))) return CSA2_ERR_ALIGN;
  const size_t need = csa2::index_workspace_bytes(B, T, emax, h->num_sms, mode);
  if (ws_bytes < need || (need && !ws)) return CSA2_ERR_WORKSPACE;
  if (!aligned16(ws)) return CSA2_ERR_ALIGN;
  csa2::IndexArgs a{};
  a.qi = qi; a.wI = wI; a.ki_codes = ki_codes; a.ki_scales = ki_scales; a.cap = cap; a.T = T;
  a.rshift = h->rshift;
  a.idx = idx; a.top_scores = top_scores;
  a.pool_out = mode == csa2::kIndexPool ? pool_out : nullptr;
  a.pool_in = mode == csa2::kIndexReindex ? pool_in : nullptr;
  a.scores_out = scores_out;
  a.scores_ld = scores_ld;
  for (int b0 = 0; b0 < B; b0 += csa2::kMaxSeqPerLaunch) {
    const int nb = std::min(B - b0, csa2::kMaxSeqPerLaunch);
    st = cuda_status(csa2::launch_index_topk(a, call_pos(h, p0, b0, nb), b0, nb, emax, ws, ws_bytes, h->num_sms,
                                             reinterpret_cast<cudaStream_t>(stream), mode));
    if (st != CSA2_OK) return st;
  }
  return CSA2_OK;
}

}  // namespace

csa2_status csa2_index_topk(csa2_handle* h, const uint16_t* qi, const uint16_t* wI, const uint8_t* ki_codes,
                            const uint8_t* ki_scales, int64_t cap, const int64_t* p0, int B, int T, int32_t* idx,
                            float* top_scores, void* ws, size_t ws_bytes, csa2_stream_t stream) {
  return index_call(h, qi, wI, ki_codes, ki_scales, cap, p0, B, T, idx, top_scores, nullptr, nullptr,
                    csa2::kIndexTopk, ws, ws_bytes, stream);
}

// Window roll between calls (include/csa2.h).
csa2_status csa2_roll_window(csa2_handle* h, const uint8_t* window, int B, int T, uint8_t* next, int T_next,
                             csa2_stream_t stream) {
  if (!h || !window || !next) return CSA2_ERR_INVALID_ARG;
  if (B <= 0 || T <= 0 || T_next <= 0 || T > 65535 || T_next > 65535 || B > (1 << 24)) return CSA2_ERR_INVALID_ARG;
  if (!aligned16(window) || !aligned16(next)) return CSA2_ERR_ALIGN;
  // one buffer: only with equal strides (or one sequence) does every block stay within its own rows
  const uintptr_t w0 = reinterpret_cast<uintptr_t>(window), n0 = reinterpret_cast<uintptr_t>(next);
  const uintptr_t w1 = w0 + (uintptr_t)B * (127 + T) * 512, n1 = n0 + (uintptr_t)B * (127 + T_next) * 512;
  const bool overlap = w0 < n1 && n0 < w1;
  if (overlap && !(w0 == n0 && (T == T_next || B == 1))) return CSA2_ERR_INVALID_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return CSA2_ERR_CUDA;
  if (dev != h->device) return CSA2_ERR_INVALID_ARG;
  return cuda_status(csa2::launch_roll_window(window, B, T, next, T_next, reinterpret_cast<cudaStream_t>(stream)));
}

// Indexer scores alone (include/csa2.h): S^I of every visible entry into the caller's rows.
csa2_status csa2_index_scores(csa2_handle* h, const uint16_t* qi, const uint16_t* wI, const uint8_t* ki_codes,
                              const uint8_t* ki_scales, int64_t cap, const int64_t* p0, int B, int T, float* scores,
                              int64_t ld, void* ws, size_t ws_bytes, csa2_stream_t stream) {
  return index_call(h, qi, wI, ki_codes, ki_scales, cap, p0, B, T, nullptr, nullptr, nullptr, nullptr,
                    csa2::kIndexScores, ws, ws_bytes, stream, scores, ld);
}

// Hierarchical Sparse Indexer, owner layer (include/csa2.h): the top-512 plus the block pool.
csa2_status csa2_index_pool(csa2_handle* h, const uint16_t* qi, const uint16_t* wI, const uint8_t* ki_codes,
                            const uint8_t* ki_scales, int64_t cap, const int64_t* p0, int B, int T, int32_t* idx,
                            float* top_scores, int32_t* pool, void* ws, size_t ws_bytes, csa2_stream_t stream) {
  return index_call(h, qi, wI, ki_codes, ki_scales, cap, p0, B, T, idx, top_scores, pool, nullptr, csa2::kIndexPool,
                    ws, ws_bytes, stream);
}

// Hierarchical Sparse Indexer, later layer (include/csa2.h): the top-512 over a given pool.
csa2_status csa2_reindex_topk(csa2_handle* h, const uint16_t* qi, const uint16_t* wI, const uint8_t* ki_codes,
                              const uint8_t* ki_scales, int64_t cap, const int64_t* p0, int B, int T,
                              const int32_t* pool, int32_t* idx, float* top_scores, void* ws, size_t ws_bytes,
                              csa2_stream_t stream) {
  return index_call(h, qi, wI, ki_codes, ki_scales, cap, p0, B, T, idx, top_scores, nullptr, pool,
                    csa2::kIndexReindex, ws, ws_bytes, stream);
}

csa2_status csa2_attend(csa2_handle* h, const uint16_t* q, const float* sinks, const uint8_t* z_codes,
                        const uint8_t* z_scales, int64_t cap, const uint8_t* window, const int32_t* idx,
                        const int64_t* p0, int B, int T, uint16_t* out, void* ws, size_t ws_bytes,
                        csa2_stream_t stream) {
  if (!h || !q || !sinks || !z_codes || !z_scales || !window || !idx || !out) return CSA2_ERR_INVALID_ARG;
  if (B <= 0 || T <= 0 || cap < 0 || T > 65535) return CSA2_ERR_INVALID_ARG;
  std::vector<int64_t> bound;
  p0 = plan_p0(h, p0, B, bound);
  csa2_status st = check_p0(p0, B, T);
  if (st != CSA2_OK) return st;
  const void* ptrs[] = {q, sinks, z_codes, z_scales, window, idx, out};
  for (const void* p : ptrs)
    if (!aligned16(p)) return CSA2_ERR_ALIGN;
  const size_t need = csa2::attend_workspace_bytes(B, T, h->num_sms);
  if (ws_bytes < need || (need && !ws)) return CSA2_ERR_WORKSPACE;
  if (need && !aligned16(ws)) return CSA2_ERR_ALIGN;
  csa2::AttendArgs a{};
  a.q = q; a.sinks = sinks; a.z_codes = z_codes; a.z_scales = z_scales; a.window = window; a.idx = idx;
  a.cap = cap; a.T = T; a.out = out;
  for (int b0 = 0; b0 < B; b0 += csa2::kMaxSeqPerLaunch) {
    const int nb = std::min(B - b0, csa2::kMaxSeqPerLaunch);
    st = cuda_status(csa2::launch_attend(a, call_pos(h, p0, b0, nb), no_replay(), b0, nb, h->rf, ws, ws_bytes, h->num_sms,
                                         reinterpret_cast<cudaStream_t>(stream)));
    if (st != CSA2_OK) return st;
  }
  return CSA2_OK;
}

// csa2_attend with per-sequence replay starts (include/csa2.h): the window rows of query t are
// positions max(win_start[b], t-127)..t.
csa2_status csa2_attend_replay(csa2_handle* h, const uint16_t* q, const float* sinks, const uint8_t* z_codes,
                               const uint8_t* z_scales, int64_t cap, const uint8_t* window, const int32_t* idx,
                               const int64_t* p0, const int64_t* win_start, int B, int T, uint16_t* out, void* ws,
                               size_t ws_bytes, csa2_stream_t stream) {
  if (!h || !q || !sinks || !z_codes || !z_scales || !window || !idx || !out) return CSA2_ERR_INVALID_ARG;
  if (B <= 0 || T <= 0 || cap < 0 || T > 65535) return CSA2_ERR_INVALID_ARG;
  if (h->pos_dev) return CSA2_ERR_UNSUPPORTED;  // win_start <= p0 is checked on the host
  csa2_status st = check_p0(p0, B, T);
  if (st != CSA2_OK) return st;
  if (!win_start) return CSA2_ERR_INVALID_ARG;
  for (int b = 0; b < B; ++b)
    if (win_start[b] < 0 || win_start[b] > p0[b]) return CSA2_ERR_SHAPE;  // 0 <= s <= p0
  const void* ptrs[] = {q, sinks, z_codes, z_scales, window, idx, out};
  for (const void* p : ptrs)
    if (!aligned16(p)) return CSA2_ERR_ALIGN;
  const size_t need = csa2::attend_workspace_bytes(B, T, h->num_sms);
  if (ws_bytes < need || (need && !ws)) return CSA2_ERR_WORKSPACE;
  if (need && !aligned16(ws)) return CSA2_ERR_ALIGN;
  csa2::AttendArgs a{};
  a.q = q; a.sinks = sinks; a.z_codes = z_codes; a.z_scales = z_scales; a.window = window; a.idx = idx;
  a.cap = cap; a.T = T; a.out = out;
  for (int b0 = 0; b0 < B; b0 += csa2::kMaxSeqPerLaunch) {
    const int nb = std::min(B - b0, csa2::kMaxSeqPerLaunch);
    st = cuda_status(csa2::launch_attend(a, pack_pos(p0, b0, nb), pack_pos(win_start, b0, nb), b0, nb, h->rf, ws, ws_bytes, h->num_sms,
                                         reinterpret_cast<cudaStream_t>(stream)));
    if (st != CSA2_OK) return st;
  }
  return CSA2_OK;
}

// Allocation-free variant of csa2_attend (see include/csa2.h): identical validation and
// launches, with the split partials in the library's fixed device array.
csa2_status csa2_attend_static(csa2_handle* h, const uint16_t* q, const float* sinks, const uint8_t* z_codes,
                               const uint8_t* z_scales, int64_t cap, const uint8_t* window, const int32_t* idx,
                               const int64_t* p0, int B, int T, uint16_t* out, csa2_stream_t stream) {
  if (!h || !q || !sinks || !z_codes || !z_scales || !window || !idx || !out) return CSA2_ERR_INVALID_ARG;
  if (B <= 0 || T <= 0 || cap < 0 || T > 65535) return CSA2_ERR_INVALID_ARG;
  std::vector<int64_t> bound;
  p0 = plan_p0(h, p0, B, bound);
  csa2_status st = check_p0(p0, B, T);
  if (st != CSA2_OK) return st;
  const void* ptrs[] = {q, sinks, z_codes, z_scales, window, idx, out};
  for (const void* p : ptrs)
    if (!aligned16(p)) return CSA2_ERR_ALIGN;
  const size_t need = csa2::attend_workspace_bytes(B, T, h->num_sms);
  if (need > csa2::attend_static_scratch_bytes()) return CSA2_ERR_TOO_LARGE;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return CSA2_ERR_CUDA;
  if (dev != h->device) return CSA2_ERR_INVALID_ARG;
  void* ws = nullptr;
  if (need) {  // a batch that is not split needs no scratch and never touches the array
    if (csa2::attend_static_scratch(dev, &ws) != cudaSuccess) return CSA2_ERR_CUDA;
  }
  csa2::AttendArgs a{};
  a.q = q; a.sinks = sinks; a.z_codes = z_codes; a.z_scales = z_scales; a.window = window; a.idx = idx;
  a.cap = cap; a.T = T; a.out = out;
  // Launches of successive groups of sequences reuse the array; they are ordered on `stream`.
  for (int b0 = 0; b0 < B; b0 += csa2::kMaxSeqPerLaunch) {
    const int nb = std::min(B - b0, csa2::kMaxSeqPerLaunch);
    st = cuda_status(csa2::launch_attend(a, call_pos(h, p0, b0, nb), no_replay(), b0, nb, h->rf, ws, need, h->num_sms,
                                         reinterpret_cast<cudaStream_t>(stream)));
    if (st != CSA2_OK) return st;
  }
  return CSA2_OK;
}

}  // extern "C"

// Reports what the bounded waits of earlier kernels recorded (include/csa2.h).
csa2_status csa2_check(csa2_handle* h, csa2_stream_t stream) {
  if (!h) return CSA2_ERR_INVALID_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return CSA2_ERR_CUDA;
  if (dev != h->device) return CSA2_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return CSA2_ERR_CUDA;
  int ea = 0, ei = 0, eo = 0;
  unsigned da = 0, di = 0;
  if (csa2::take_attend_error(&ea) != cudaSuccess || csa2::take_index_error(&ei) != cudaSuccess ||
      csa2::take_outproj_error(&eo) != cudaSuccess || csa2::take_attend_domain(&da) != cudaSuccess ||
      csa2::take_index_domain(&di) != cudaSuccess)
    return CSA2_ERR_CUDA;
  unsigned pf = 0;
  const unsigned zero = 0;
  if (cudaMemcpyFromSymbol(&pf, g_pos_flag, sizeof pf) != cudaSuccess) return CSA2_ERR_CUDA;
  if (pf && cudaMemcpyToSymbol(g_pos_flag, &zero, sizeof zero) != cudaSuccess) return CSA2_ERR_CUDA;
  if (ea || ei || eo) return CSA2_ERR_TIMEOUT;
  if (pf) return CSA2_ERR_SHAPE;
  return (da || di) ? CSA2_ERR_UNSUPPORTED : CSA2_OK;
}

// Test hook for the timeout report (include/csa2.h).
csa2_status csa2_selftest_timeout(csa2_handle* h, csa2_stream_t stream) {
  if (!h) return CSA2_ERR_INVALID_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return CSA2_ERR_CUDA;
  if (dev != h->device) return CSA2_ERR_INVALID_ARG;
  return cuda_status(csa2::launch_wait_probe(reinterpret_cast<cudaStream_t>(stream)));
}

// Tensor-core rate probe (include/csa2.h).
csa2_status csa2_tc_rate(csa2_handle* h, int kind, int iters, double* tflops, csa2_stream_t stream) {
  if (!h || !tflops || kind < 0 || kind > 2 || iters < 1 || iters > 65536) return CSA2_ERR_INVALID_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return CSA2_ERR_CUDA;
  if (dev != h->device) return CSA2_ERR_INVALID_ARG;
  int timed_out = 0;
  const csa2_status s = cuda_status(
      csa2::measure_tc_rate(kind, iters, h->num_sms, reinterpret_cast<cudaStream_t>(stream), tflops, &timed_out));
  if (s != CSA2_OK) return s;
  return timed_out ? CSA2_ERR_TIMEOUT : CSA2_OK;
}

// Grouped output projection W_OA (include/csa2.h).
csa2_status csa2_out_group_proj(csa2_handle* h, const uint16_t* o, const uint16_t* w_oa, int64_t M, uint16_t* out,
                                csa2_stream_t stream) {
  if (!h || !o || !w_oa || !out) return CSA2_ERR_INVALID_ARG;
  if (M <= 0 || M > (int64_t(1) << 31)) return CSA2_ERR_INVALID_ARG;
  if (!aligned16(o) || !aligned16(w_oa) || !aligned16(out)) return CSA2_ERR_ALIGN;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return CSA2_ERR_CUDA;
  if (dev != h->device) return CSA2_ERR_INVALID_ARG;
  return cuda_status(csa2::launch_out_group_proj(o, w_oa, M, out, h->num_sms, reinterpret_cast<cudaStream_t>(stream)));
}
