// Internal declarations shared by the C-ABI front end (csa2_api.cu) and the kernel files.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace csa2 {

constexpr int kD = 512;      // entry / head width
constexpr int kDR = 64;      // rotated dims (last 64 of Z, W, Q, O)
constexpr int kDI = 128;     // indexer key width
constexpr int kHI = 32;      // indexer heads
constexpr int kH = 64;       // attention heads
constexpr int kWin = 128;    // window rows
constexpr int kTopK = 512;   // selected entries
constexpr int kMaxSeqPerLaunch = 128;  // sequences whose p0 travels in one launch's params

// Absolute start positions of up to kMaxSeqPerLaunch sequences, passed by value, or (dev not
// null) read by the kernels from device memory when they run: dev[bl] for the launch's sequence
// bl, planned for on the host as if it were hi.  A device value outside 0..hi is clamped into it
// (so every access stays within what the host validated) and sets *flag.
struct SeqPos {
  int64_t p0[kMaxSeqPerLaunch];
  const int64_t* dev;
  int64_t hi;
  unsigned* flag;
};

#ifdef __CUDACC__
__device__ __forceinline__ int64_t seq_p0(const SeqPos& s, int bl) {
  if (s.dev == nullptr) return s.p0[bl];
  int64_t v = s.dev[bl];
  if (v < 0 || v > s.hi) {
    atomicOr(s.flag, 1u);
    v = v < 0 ? 0 : s.hi;
  }
  return v;
}
#endif

// RoPE frequencies theta_i = base^(-2i/64), i < 32, computed on the host in fp64.
struct RopeFreq {
  double inv_freq[kDR / 2];
};

struct WriterArgs {
  const uint16_t *kc, *gc, *wa, *w_ik;
  const float *gamma_c, *gamma_ik, *gamma_w;
  float *pair_kc, *pair_gc;
  uint8_t *z_codes, *z_scales, *ki_codes, *ki_scales, *window;
  int64_t cap;
  int T;
  int rshift;  // log2 of the compression ratio: entry j covers tokens (j << rshift) .. + ratio-1
  double eps;
};

struct IndexArgs {
  const uint16_t *qi, *wI;
  const uint8_t *ki_codes, *ki_scales;
  int64_t cap;
  int T;
  int rshift;  // log2 of the compression ratio: query t sees entries j < (t+1) >> rshift
  int32_t* idx;
  float* top_scores;
  // hierarchical indexer: pool_out [B, T, 2048] receives the block pool (csa2_index_pool);
  // pool_in [B, T, 2048] restricts the scan to a pool (csa2_reindex_topk)
  int32_t* pool_out;
  const int32_t* pool_in;
  // csa2_index_scores: the fp32 score rows go to the caller's [B, T, scores_ld] array
  float* scores_out;
  int64_t scores_ld;
};

constexpr int kHsiBlock = 8, kHsiBlocks = 2048;  // blocks of 8 entries, 2048 blocks per pool
enum IndexMode { kIndexTopk = 0, kIndexPool = 1, kIndexReindex = 2, kIndexScores = 3 };

struct AttendArgs {
  const uint16_t* q;
  const float* sinks;
  const uint8_t *z_codes, *z_scales, *window;
  const int32_t* idx;
  int64_t cap;
  int T;
  uint16_t* out;
};

// Tiled 2-D tensor map (cuTensorMapEncodeTiled through the runtime's driver entry point) over
// [rows][cols] elements of elem_bytes with a row pitch of pitch_bytes, box [box_rows][box_cols],
// rows outside the tensor read as zero.  False if the entry point is missing or the base, pitch
// or box width breaks the 16-byte rules.
bool encode_tiled_2d(CUtensorMap* map, CUtensorMapDataType dtype, int elem_bytes, const void* base, uint64_t cols,
                     uint64_t rows, uint64_t pitch_bytes, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle swizzle);

// The same for n elements in one dimension, box of `box` elements (box * elem_bytes a multiple of 16).
bool encode_tiled_1d(CUtensorMap* map, CUtensorMapDataType dtype, int elem_bytes, const void* base, uint64_t n,
                     uint32_t box);

// Tensor-core rate (csa2_tc_rate): best of three launches of `iters` MMAs per SM, in TFLOP/s;
// *timed_out is set if a block's bounded wait gave up.
cudaError_t measure_tc_rate(int kind, int iters, int num_sms, cudaStream_t st, double* tflops, int* timed_out);

// Launchers: each enqueues on `st` and returns the first CUDA launch error (or success).
// `b0` is the batch index of the first sequence in `pos`, `nb` how many follow.
cudaError_t launch_writer(const WriterArgs& a, const SeqPos& pos, int b0, int nb, const RopeFreq& rf,
                          cudaStream_t st);
// Window roll: rows T .. T+126 of each sequence's view [B, 127+T, 512] -> rows 0 .. 126 of the
// next view [B, 127+T_next, 512] (one block per sequence; its rows may move within one buffer).
cudaError_t launch_roll_window(const uint8_t* window, int B, int T, uint8_t* next, int T_next, cudaStream_t st);
size_t index_workspace_bytes(int B, int T, int64_t max_entries, int num_sms, int mode = kIndexTopk);
cudaError_t launch_index_topk(const IndexArgs& a, const SeqPos& pos, int b0, int nb, int64_t max_entries,
                              void* ws, size_t ws_bytes, int num_sms, cudaStream_t st, int mode = kIndexTopk);
size_t index_tc_image_bytes(int nb, int Tq, int64_t max_entries);
// Prefill score GEMM for the pass t0 .. t0+tq-1: emax = visible entries of the pass's last query,
// emax_all = of the call's last query (the key-image stride); build_keys: write the key images
// (once per call, on its first pass).  lower (optional) [nb * Tq] receives per query row the
// lower edge of the score-key histogram bin that holds its 512th largest score.
cudaError_t launch_index_scores_tc(const IndexArgs& a, const SeqPos& pos, int b0, int nb, int t0, int tq, int Tq,
                                   int64_t emax, int64_t emax_all, bool build_keys, uint8_t* img, float* wq,
                                   float* scores, int64_t ld, uint32_t* lower, int32_t* cand_j, int* cand_n,
                                   int num_sms, cudaStream_t st);
// One query row per (sequence, t) of the pass t0 .. t0+tq-1 (T == 1, or a pool scan); row r =
// bl * Tq + tl.  With a.pool_in, row r's positions are its pool's entries and rowlen[r]
// receives the number of visible ones.
cudaError_t launch_index_scores_decode_tc(const IndexArgs& a, const SeqPos& pos, int b0, int nb, int t0, int tq,
                                          int Tq, float* scores, int64_t ld, int* rowlen, uint32_t* hist, int num_sms,
                                          cudaStream_t st);
// Device error words of the bounded waits: read and cleared (synchronous; the caller has
// synchronised the work it checks).
cudaError_t take_attend_error(int* code);
cudaError_t take_index_error(int* code);
cudaError_t take_outproj_error(int* code);
// Domain flags: set when a kernel read an FP4 scale above 2^13 (or a value that overflows an fp16
// operand); read and cleared like the error words.
cudaError_t take_index_domain(unsigned* flag);
cudaError_t take_attend_domain(unsigned* flag);
// Grouped output projection: o [M, 64, 512] bf16, w [8, 1024, 4096] bf16 (group, output,
// input), out [M, 8, 1024] bf16.
cudaError_t launch_out_group_proj(const uint16_t* o, const uint16_t* w, int64_t M, uint16_t* out, int num_sms,
                                  cudaStream_t st);
// A kernel whose one bounded wait can never complete (a test of the timeout report).
cudaError_t launch_wait_probe(cudaStream_t st);
// Counts one kernel enqueued by this library (read back by csa2_kernel_launches).
void note_launch();

size_t attend_workspace_bytes(int B, int T, int num_sms);
// wst: per-sequence replay starts of the window (zeros: the plain window of 128 positions).
cudaError_t launch_attend(const AttendArgs& a, const SeqPos& pos, const SeqPos& wst, int b0, int nb, const RopeFreq& rf,
                          void* ws, size_t ws_bytes, int num_sms, cudaStream_t st);

// Fixed device scratch of csa2_attend_static: room for this many split-partial rows (one row =
// 64 heads x 514 fp32), the most a launch needs on a device with at most 152 SMs.
constexpr size_t kStaticAttendRows = 152;
size_t attend_static_scratch_bytes();
cudaError_t attend_static_scratch(int device, void** out);

}  // namespace csa2
