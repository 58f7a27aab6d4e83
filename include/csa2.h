/* csa2.h - C ABI of the GB300 (sm_103a) CSA2 layer library, libcsa2.so.
 *
 * One DeepSeek-V4.1-style CSA2 ("compressed sparse attention 2") layer of the Full kind at
 * compression ratio 2 (or 1): the compressed-KV writer, the lightning indexer with its top-512
 * select, and 64-head sink-softmax MQA over the 640 gathered rows.  The operations follow
 * the equations of the page "DeepSeek V4.1 - Pooled group / Source layer, pairs pooled",
 * block "Compressed sparse attention" (cited below as [PG]), with the RMSNorm of the page
 * "DeepSeek V4.1 - Window layer / Attention RMSNorm" ([RN], eps = 1e-20) and the storage
 * formats of "Inside DeepSeek V4.1", section "890 bytes" ([IN]).
 *
 * Conventions shared by every call
 *  - Fixed shapes: 64 heads x 512, RoPE on the last 64 dims, indexer 32 heads x 128 (RoPE
 *    on dims 64..127), window 128 rows, top 512.  csa2_create rejects any other value with
 *    CSA2_ERR_UNSUPPORTED.
 *  - Compression ratio r (config.ratio): 2 for the encoder owner layers (entry j pools
 *    tokens 2j, 2j+1), or 1 for the decoder owner layers ("Inside DeepSeek V4.1 Flash:
 *    Deriving the 890-Byte KV Cache", decoder layers of ratio one): entry j is token j
 *    itself (a softmax over one token is 1, so k^p = k^c), there is no pair buffer.  Entry j
 *    is rotated by position r*j and is visible to query t iff j < floor((t+1)/r).
 *  - Tensor arguments are DEVICE pointers, owned by the caller, row-major and densely
 *    packed in the shapes given, 16-byte aligned.  bf16 tensors are passed as uint16_t
 *    bit patterns.  The library allocates no device memory; scratch comes from the caller's
 *    workspace (size from csa2_workspace_bytes), except for csa2_attend_static, whose
 *    scratch is a fixed array of the library (see there).
 *  - p0 is a HOST array of B int64 values: the absolute position of the first of the T new
 *    tokens of each sequence (its cached length before the call), or, after
 *    csa2_set_device_positions, a device array that the kernels read when they run.
 *  - Every call is asynchronous on `stream` and never synchronises.  Argument errors are
 *    returned before anything is launched; launch errors come back as CSA2_ERR_CUDA.
 *  - Every wait inside a kernel is bounded (about 80 ms).  A wait that gives up records a
 *    code in a device error word and lets its kernel finish; csa2_check reports it.
 *  - FP4 scale domain.  The decode indexer (T = 1, and the reindex scan) multiplies the cached
 *    E2M1 codes and UE8M0 scales as stored (block-scaled FP4 MMAs), exactly for every scale
 *    byte.  The other tensor-core kernels decode E2M1 x 2^e exactly into their operands: fp16
 *    (attention) for scale bytes 104..140 (e = -23 .. 13), E5M2 (prefill indexer, T >= 8) for
 *    bytes 112..140 (e = -15 .. 13).  Smaller scales decode with an absolute error under 2^-24
 *    (fp16) or 2^-17 (E5M2) per value, the rest of the row unaffected; bytes 0 with zero codes
 *    are exact zeros.  Bytes above 140 would overflow those operands: a kernel that reads one
 *    (the decode indexer too, so that a call's domain does not depend on the path it takes;
 *    or an indexer query block with e > 13, or an attention query of magnitude 2^16 or more)
 *    records it, and the next csa2_check returns CSA2_ERR_UNSUPPORTED (the outputs since the
 *    previous check are not to be trusted).  Rows this library's writer makes stay
 *    inside: after RMSNorm |value| <= sqrt(512) max|gamma|, so gains of magnitude at most 2^k
 *    give scale bytes <= 129 + k (k <= 11 keeps every byte <= 140).
 *
 * Storage formats (fixed by this library)
 *  - FP4 cache row of n values: n/2 code bytes (E2M1, element 2i in the low nibble of byte
 *    i) and n/32 UE8M0 scale bytes (2^(byte-127)), kept in two separate arrays:
 *      Z   : codes [B, cap, 256], scales [B, cap, 16]   (272 bytes per pooled entry)
 *      K^I : codes [B, cap,  64], scales [B, cap,  4]   ( 68 bytes per pooled entry)
 *    Scale choice follows the OCP MX rule 2^(floor(log2 amax) - 2); codes round to nearest,
 *    ties to even, saturating at +-6.  Entry j pools tokens 2j and 2j+1.
 *  - Window (FP8 E4M3fn, RNE, saturating at +-448, no scale): a per-call view
 *    [B, 127+T, 512] whose row r holds position p0-127+r.  Rows 0..126 are the caller's
 *    (the previous 127 positions; unused where the position is negative); the writer fills
 *    rows 127..126+T.
 */
#ifndef CSA2_H
#define CSA2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* csa2_stream_t; /* a cudaStream_t; NULL = legacy default stream */

typedef enum {
  CSA2_OK = 0,
  CSA2_ERR_INVALID_ARG = 1, /* null pointer, negative size, bad op code */
  CSA2_ERR_SHAPE = 2,       /* sizes inconsistent (cache too small, position too large) */
  CSA2_ERR_ALIGN = 3,       /* a pointer is not 16-byte aligned */
  CSA2_ERR_WORKSPACE = 4,   /* workspace smaller than csa2_workspace_bytes() */
  CSA2_ERR_UNSUPPORTED = 5, /* configuration outside what the kernels implement */
  CSA2_ERR_CUDA = 6,        /* a CUDA launch or device query failed */
  CSA2_ERR_TOO_LARGE = 7,   /* batch needs more than csa2_attend_static's fixed scratch */
  CSA2_ERR_TIMEOUT = 8      /* a bounded wait inside a kernel gave up (csa2_check) */
} csa2_status;

/* Layer configuration.  The integer fields must equal the defaults shown. */
typedef struct {
  int heads;        /* 64 */
  int head_dim;     /* 512 */
  int rope_dims;    /* 64 */
  int idx_heads;    /* 32 */
  int idx_dim;      /* 128 */
  int window;       /* 128 */
  int topk;         /* 512 */
  int ratio;        /* 2 (default) or 1 */
  double rope_base; /* 10000: theta_i = rope_base^(-2i/64) */
  double eps;       /* 1e-20 ([RN]) */
} csa2_config;

typedef struct csa2_handle csa2_handle;

/* Fills `cfg` with the defaults above. */
void csa2_default_config(csa2_config* cfg);

/* Validates `cfg`, records the current CUDA device and its SM count, and precomputes the
 * RoPE frequencies in fp64.  Allocates host memory only.  *out = NULL on error. */
csa2_status csa2_create(const csa2_config* cfg, csa2_handle** out);
void csa2_destroy(csa2_handle* h);
const char* csa2_status_string(csa2_status s);

/* Number of kernels this library has enqueued in this process so far (every handle and
 * device; a launch that failed is counted too).  Host-side counter; never synchronises. */
uint64_t csa2_kernel_launches(void);

enum {
  CSA2_OP_WRITE_CACHE = 0,
  CSA2_OP_INDEX_TOPK = 1,
  CSA2_OP_ATTEND = 2,
  CSA2_OP_INDEX_POOL = 3,
  CSA2_OP_REINDEX_TOPK = 4,
  CSA2_OP_INDEX_SCORES = 5
};

/* Bytes of workspace the call `op` needs for B sequences of T new tokens whose largest
 * visible entry count is at most max_entries (for decode: the cached entries).  Returns 0
 * for a bad op.  A larger workspace is always accepted. */
size_t csa2_workspace_bytes(const csa2_handle* h, int op, int B, int T, int64_t max_entries);

/* (1) Compressed-KV writer, [PG] equations for W, k^p, c, Z, k^i, k^n, K^I.
 *  kc, gc, wa : bf16 [B, T, 512]  per-token k^c, g^c and w^a (the window source).
 *  gamma_c    : f32 [512]   gain of the pooled-key RMSNorm.
 *  w_ik       : bf16 [512, 128]  indexer-key projection, k^i = c W_IK (c before RoPE).
 *  gamma_ik   : f32 [128]   gain of the indexer-key RMSNorm.
 *  gamma_w    : f32 [512]   gain of the window RMSNorm (w^n = gamma_w RMSNorm(w^a)).
 *  p0         : HOST int64 [B].
 *  pair_kc, pair_gc : f32 [B, 512] pair buffer (ratio 2 only).  When p0[b] is odd it must
 *               hold token p0[b]-1; when p0[b]+T is odd the call stores token p0[b]+T-1
 *               there.  May be NULL if every p0[b] and T are even, or at ratio 1.
 *  z_codes/z_scales, ki_codes/ki_scales : the FP4 caches with room for `cap` entries;
 *               entries j whose last token r*j + r-1 is in p0..p0+T-1 are written (j < cap).
 *  window     : u8 [B, 127+T, 512] e4m3 view; rows 127..126+T are written.
 * Per entry: k^p = sum over the pair of softmax(g^c) * k^c per channel (ratio 1: the token's
 * k^c); c = gamma_c RMSNorm(k^p); Z = c with dims 448..511 rotated by position r*j, then
 * FP4.  K^I = gamma_ik RMSNorm(c W_IK) with dims 64..127 rotated by r*j, then FP4.  Per
 * token t: W = gamma_w
 * RMSNorm(w^a) with dims 448..511 rotated by t, then FP8.
 * Workspace: none (ws may be NULL). */
csa2_status csa2_write_cache(csa2_handle* h, const uint16_t* kc, const uint16_t* gc,
                             const uint16_t* wa, const float* gamma_c, const uint16_t* w_ik,
                             const float* gamma_ik, const float* gamma_w, const int64_t* p0,
                             int B, int T, float* pair_kc, float* pair_gc, uint8_t* z_codes,
                             uint8_t* z_scales, uint8_t* ki_codes, uint8_t* ki_scales,
                             int64_t cap, uint8_t* window, void* ws, size_t ws_bytes,
                             csa2_stream_t stream);

/* (1') Window roll between calls ([PG], paragraph "Between forward calls": the layer keeps
 * the window of the last 128 positions).  After a call that appended T tokens at p0, the next
 * call's view must hold positions p0+T-127 .. p0+T-1 in its rows 0..126; these are rows
 * T .. T+126 of this call's view, and this call copies them:
 *  window : u8 [B, 127+T, 512]  this call's view (rows 127.. written by csa2_write_cache).
 *  next   : u8 [B, 127+T_next, 512]  the next call's view; rows 0..126 are written, the rest
 *           is untouched (the next csa2_write_cache fills rows 127..).
 * `next` may be `window` itself when T_next == T or B == 1: each sequence's rows then move
 * within its own rows.  Any other overlap of the two views is CSA2_ERR_INVALID_ARG.  Rows of
 * negative positions (p0+T < 127) are copied as they are; no call reads them.
 * Workspace: none. */
csa2_status csa2_roll_window(csa2_handle* h, const uint8_t* window, int B, int T, uint8_t* next,
                             int T_next, csa2_stream_t stream);

/* (2)+(3) Lightning indexer and top-512, [PG] equations for S^I and I_t.
 *  qi  : bf16 [B, T, 32, 128]  indexer queries Q^I (quantised here to FP4, scale per 32).
 *  wI  : bf16 [B, T, 32]       head weights w^I (already divided by sqrt(128*32)).
 *  ki_codes/ki_scales : the K^I cache (cap entries per sequence).
 * For query t (absolute position p0+t) the candidates are j < floor((p0+t+1)/2), which
 * must not exceed cap.  S^I_{t,j} = sum_h w^I_h ReLU(Q^I_h . K^I_j) in fp32.
 *  idx        : int32 [B, T, 512] the 512 largest scores (equal scores: lower j first),
 *               ascending in j; when fewer candidates exist all are kept and the rest is -1.
 *  top_scores : f32 [B, T, 512] or NULL: the scores of idx (NaN where idx is -1).
 * Workspace: csa2_workspace_bytes(h, CSA2_OP_INDEX_TOPK, B, T, max_entries). */
csa2_status csa2_index_topk(csa2_handle* h, const uint16_t* qi, const uint16_t* wI,
                            const uint8_t* ki_codes, const uint8_t* ki_scales, int64_t cap,
                            const int64_t* p0, int B, int T, int32_t* idx, float* top_scores,
                            void* ws, size_t ws_bytes, csa2_stream_t stream);

/* (2) Lightning-indexer scores alone, [PG] equation for S^I: the fp32 values that
 * csa2_index_topk selects from, for a caller that needs every score (a different select, a
 * check of the scores themselves).  Arguments as csa2_index_topk, plus
 *  scores : f32 [B, T, ld]; row (b, t) receives S^I_{t,j} for every visible j <
 *           floor((p0[b]+t+1)/ratio) in the same fp32 arithmetic as csa2_index_topk; the
 *           rest of the row is left untouched.  16-byte aligned.
 *  ld     : row stride in floats, a multiple of 4 and at least the largest visible count
 *           (CSA2_ERR_SHAPE otherwise).
 * All T queries are scored in one pass, so the caller holds B*T*ld floats at once.
 * Workspace: csa2_workspace_bytes(h, CSA2_OP_INDEX_SCORES, B, T, max_entries). */
csa2_status csa2_index_scores(csa2_handle* h, const uint16_t* qi, const uint16_t* wI,
                              const uint8_t* ki_codes, const uint8_t* ki_scales, int64_t cap,
                              const int64_t* p0, int B, int T, float* scores, int64_t ld,
                              void* ws, size_t ws_bytes, csa2_stream_t stream);

/* (2)+(3) Hierarchical Sparse Indexer, owner layer ("Inside DeepSeek V4.1", section "Most
 * layers borrow"; "Deriving the 890-Byte KV Cache", section "Hierarchical indexing bounds the
 * later searches").  Arguments and idx / top_scores as csa2_index_topk, plus
 *  pool : int32 [B, T, 2048] per query the entry blocks (block k = entries 8k..8k+7) that
 *         later layers search: the newest block (the one holding entry E-1, E the visible
 *         entries) and the 2047 other blocks with the largest block score (the maximum of
 *         S^I over its 8 entries; equal scores: lower block first).  With at most 2048 blocks
 *         every block is kept.  Ascending, -1 padded.
 * Workspace: csa2_workspace_bytes(h, CSA2_OP_INDEX_POOL, B, T, max_entries). */
csa2_status csa2_index_pool(csa2_handle* h, const uint16_t* qi, const uint16_t* wI,
                            const uint8_t* ki_codes, const uint8_t* ki_scales, int64_t cap,
                            const int64_t* p0, int B, int T, int32_t* idx, float* top_scores,
                            int32_t* pool, void* ws, size_t ws_bytes, csa2_stream_t stream);

/* (2)+(3) Hierarchical Sparse Indexer, later layer: S^I of this layer's queries over the
 * entries of `pool` only (same pages and sections as csa2_index_pool), and their top-512.
 *  pool : int32 [B, T, 2048] as written by csa2_index_pool for the same p0 and T: ascending
 *         blocks, -1 padded, every block but the last fully visible.  A block outside that
 *         rule gives unspecified idx (entries it names beyond E-1 are scored as zero keys)
 *         but no access outside the caches.
 *  idx / top_scores : as csa2_index_topk, over the pool's visible entries (at most 16384).
 * Workspace: csa2_workspace_bytes(h, CSA2_OP_REINDEX_TOPK, B, T, max_entries). */
csa2_status csa2_reindex_topk(csa2_handle* h, const uint16_t* qi, const uint16_t* wI,
                              const uint8_t* ki_codes, const uint8_t* ki_scales, int64_t cap,
                              const int64_t* p0, int B, int T, const int32_t* pool,
                              int32_t* idx, float* top_scores, void* ws, size_t ws_bytes,
                              csa2_stream_t stream);

/* Grouped output projection W_OA ("Inside DeepSeek V4.1", section "Attention that looks at
 * 640 places": 8 groups of a 1,024-wide bottleneck; [PG] o^g_{t,r} = [O-bar_{h,t}]_{h in r} W_OA,r).
 *  o    : bf16 [M, 64, 512]  attention outputs (M = B*T rows, e.g. csa2_attend's `out`).
 *  w_oa : bf16 [8, 1024, 4096]  per group r the weights as [output i][input k], input
 *         k = 512 (h - 8r) + d for head h of group r (heads 8r .. 8r+7, one after another).
 *  out  : bf16 [M, 8, 1024]  o^g; fp32 accumulation, rounded to bf16 once.
 * The model width that W_OB maps o^g back to is not on the pages, so W_OB is not provided.
 * Workspace: none. */
csa2_status csa2_out_group_proj(csa2_handle* h, const uint16_t* o, const uint16_t* w_oa,
                                int64_t M, uint16_t* out, csa2_stream_t stream);

/* Tensor-core rate probe (no counterpart on the pages): the peak that the tensor-bound
 * kernels here are quoted against, measured on this device for each operand kind they use.
 * One block per SM; its elected thread issues `iters` MMAs of M = 128, N = 256 back to back on
 * fixed shared-memory operands into one tensor-memory accumulator (no memory traffic):
 *   kind 0: tcgen05.mma kind::f16 (fp16, K = 16 per MMA)
 *   kind 1: kind::f8f6f4 (E5M2, K = 32)
 *   kind 2: kind::mxf4 (packed E2M1 with UE8M0 scales per 32 values, K = 64)
 * Times three launches with CUDA events on `stream` (synchronising it) and writes the best
 * rate, 2 * 128 * 256 * K * iters * SMs / time, in TFLOP/s to *tflops (host).  1 <= iters <=
 * 65536 and 0 <= kind <= 2, else CSA2_ERR_INVALID_ARG; CSA2_ERR_TIMEOUT if a block's bounded
 * wait gave up (the number is then not to be trusted).  Not for use inside stream capture. */
csa2_status csa2_tc_rate(csa2_handle* h, int kind, int iters, double* tflops, csa2_stream_t stream);

/* Failure report (no counterpart on the pages).  Synchronises `stream`, then reports whether
 * a bounded wait inside any kernel of this library gave up since the last check:
 * CSA2_ERR_TIMEOUT (the outputs of the calls since then are not to be trusted); else
 * CSA2_ERR_SHAPE if a kernel read a device position outside 0..p0_max (see
 * csa2_set_device_positions); else CSA2_ERR_UNSUPPORTED if a kernel read an FP4 scale or query
 * outside the fp16 domain (see the conventions above); CSA2_ERR_CUDA if synchronising or
 * reading the words failed; CSA2_OK otherwise.  Clears the error words and flags.  Call with
 * the handle's device current; while an error word is set, later waits that stay pending give
 * up early, so check before trusting further results.  Not for use inside stream capture (it
 * synchronises). */
csa2_status csa2_check(csa2_handle* h, csa2_stream_t stream);

/* Positions from device memory, for a step captured once in a CUDA graph and replayed at every
 * position (no counterpart on the pages; the positions are the p0 of the calls above).
 *  - p0_dev: DEVICE array of B int64 (8-byte aligned, owned by the caller) with sequence b's
 *    p0 at p0_dev[b], for the largest B of the calls that follow; NULL returns the handle to
 *    host positions.  p0_max: a bound, 0 <= p0_dev[b] <= p0_max (CSA2_ERR_SHAPE unless
 *    p0_max + 1 <= 2^21 - 2).
 *  - While set, csa2_write_cache, the indexer calls and csa2_attend / csa2_attend_static do not
 *    read their p0 argument (it may be NULL): their kernels read p0_dev when they run, and the
 *    host validates and sizes everything (cache capacity, workspace, grids) as if every p0 were
 *    p0_max, so workspaces are sized with max_entries = floor((p0_max + T) / ratio).  At ratio 2
 *    csa2_write_cache then needs the pair buffers for every T.  csa2_attend_replay returns
 *    CSA2_ERR_UNSUPPORTED.
 *  - The calls enqueue the same kernels for every position, so a stream capture of one step
 *    (after one uncaptured step, which loads the library's kernels) replays correctly at any
 *    positions written to p0_dev before each replay.  Results are bit-identical to the calls
 *    with those positions on the host.
 *  - A value outside 0..p0_max is clamped into that range, so that every access stays within
 *    what was validated, and csa2_check returns CSA2_ERR_SHAPE.
 *  - Call outside stream capture, with the handle's device current. */
csa2_status csa2_set_device_positions(csa2_handle* h, const int64_t* p0_dev, int64_t p0_max);

/* Test hook for csa2_check (no counterpart on the pages): enqueues one kernel whose single
 * bounded wait can never complete (nothing arrives at its barrier), so that the next
 * csa2_check returns CSA2_ERR_TIMEOUT.  The kernel ends by itself after the wait's bound
 * (about 80 ms); it faults nothing and the device stays usable. */
csa2_status csa2_selftest_timeout(csa2_handle* h, csa2_stream_t stream);

/* (4) Sink-softmax MQA, [PG] equations for J^w_t, Y, J, G_t, S, A, O and O-bar.
 *  q      : bf16 [B, T, 64, 512] queries, RoPE already applied to dims 448..511.
 *  sinks  : f32 [64] per-head sink logits s_h.
 *  z_codes/z_scales : the Z cache (cap entries); window: the e4m3 view [B, 127+T, 512].
 *  idx    : int32 [B, T, 512] entry indices (any source: this layer's csa2_index_topk or a
 *           shared layer's); -1 entries are skipped, others must be < cap.
 * G_t = window rows of positions max(0,t-127)..t followed by the Z rows idx[t] (at most
 * 640 rows), dequantised exactly.  S = Q.G/sqrt(512), A = exp S / (exp s_h + sum exp S),
 * O = sum A G, then dims 448..511 of O rotated by -t.
 *  out    : bf16 [B, T, 64, 512].
 * Workspace: csa2_workspace_bytes(h, CSA2_OP_ATTEND, B, T, 0). */
csa2_status csa2_attend(csa2_handle* h, const uint16_t* q, const float* sinks,
                        const uint8_t* z_codes, const uint8_t* z_scales, int64_t cap,
                        const uint8_t* window, const int32_t* idx, const int64_t* p0, int B,
                        int T, uint16_t* out, void* ws, size_t ws_bytes, csa2_stream_t stream);

/* (4') csa2_attend after a bounded replay ("Inside DeepSeek V4.1 Flash: Deriving the 890-Byte
 * KV Cache", section "Bounded replay trades exact state for cheaper resumption"): local
 * state was rebuilt only from position s on, so query t sees the window positions
 * max(s, t-127)..t instead of max(0, t-127)..t.
 *  win_start : HOST int64 [B], the replay start s of each sequence, 0 <= s <= p0[b]
 *              (CSA2_ERR_SHAPE otherwise).  Window-view rows of positions < s are not read.
 * Every other argument, the result for s = 0, the workspace and the errors are those of
 * csa2_attend. */
csa2_status csa2_attend_replay(csa2_handle* h, const uint16_t* q, const float* sinks,
                               const uint8_t* z_codes, const uint8_t* z_scales, int64_t cap,
                               const uint8_t* window, const int32_t* idx, const int64_t* p0,
                               const int64_t* win_start, int B, int T, uint16_t* out, void* ws,
                               size_t ws_bytes, csa2_stream_t stream);

/* csa2_attend with no workspace argument.  Not an operation of the pages (they have no
 * counterpart): an interface for callers that cannot allocate device memory at call time,
 * e.g. a serving process that hands all free HBM to its KV-cache pool at start-up, or code
 * that must not call cudaMalloc/cudaFree because those can synchronise the device and stall
 * the work of other streams.
 * Same arguments, results and launches as csa2_attend (bit-identical output), but the split
 * partials live in one fixed device array of the library: 152 rows x 64 heads x 514 fp32 =
 * 20,000,768 bytes, enough for every batch on a device with at most 152 SMs.  A batch whose
 * split partials need more (only possible on a larger device) is rejected with
 * CSA2_ERR_TOO_LARGE before anything is launched.  Nothing in the array has to start at
 * zero: every split writes all of its partial row, also when it received no rows.
 *  - Set-up: the first call on a device resolves the array's address there with
 *    cudaGetSymbolAddress (which may load the library's module and so allocate the array);
 *    later calls reuse the cached address and make no allocating call at all.  Make the
 *    first call on each device before any stream capture.  The handle's device must be the
 *    current device (else CSA2_ERR_INVALID_ARG).
 *  - The cached address belongs to this process and to the device's current context: it is
 *    kept with the context's ID, and a call made in another context (after cudaDeviceReset
 *    ended the old one) resolves the address again, so that first call after a reset is a
 *    set-up call like the very first one.  Without the driver's context-ID query (CUDA
 *    drivers before 12.0) every call resolves the address, which allocates only once.
 *  - The array is shared: calls that may overlap in time (different streams, or different
 *    threads without ordering) race on it and corrupt each other's output.  Calls queued on
 *    one stream are ordered and safe. */
csa2_status csa2_attend_static(csa2_handle* h, const uint16_t* q, const float* sinks,
                               const uint8_t* z_codes, const uint8_t* z_scales, int64_t cap,
                               const uint8_t* window, const int32_t* idx, const int64_t* p0,
                               int B, int T, uint16_t* out, csa2_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* CSA2_H */
