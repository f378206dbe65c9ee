// Internal definitions shared by the host entry points and the kernels:
// workspace layout, per-sequence plan, and the launch parameter block.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace sv {

// Streaming pass (row statistics): a row is cut into `nseg` segments of
// `seg_elems` elements; one (row, segment) pair is a unit of work for one warp.
// A call small enough to be one unit per resident warp (152 SMs x 8 CTAs x 4
// warps) is cut that way, so that it streams in a single wave; larger calls
// aim for at least kTargetUnits units, for balance across waves.
constexpr long long kWarpsPerWave = 152 * 8 * 4;
constexpr long long kTargetUnits = 16384;
constexpr long long kSegMinBytes = 2048;   // four 16-byte vectors per lane
constexpr long long kSegMaxBytes = 32768;  // eight rounds of eight 16-byte vectors per lane

// Sampling pass: rows are cut into chunks (one CTA of 256 threads), each
// chunk into 8 sub-chunks (one warp each) of 512 elements, or of 256 when
// 4096-element chunks would give fewer than two CTAs per SM (152 SMs).
constexpr int kSubPerChunk = 8;
constexpr long long kMinDrawCtas = 2 * 152;

constexpr int kMaxK = 64;

enum : int { kModeResidual = 0, kModeBonus = 1, kModeFailed = -1 };

// What the scan decided for one sequence; read by the sampling kernels.
struct Plan {
  int j;        // accepted drafts (index of the first rejection, or K)
  int mode;     // kModeResidual, kModeBonus or kModeFailed
  long long row_q;  // target row to draw from (global row index into target_logits)
  long long row_p;  // draft row of the residual (global row index into draft_logits)
  float m_q, m_p;   // maxima of those rows (raw logits)
  float s_q, s_p;   // streaming-pass sums of exp((l - m) / T) of those rows
  float u;          // uniform of the draw
  int pad;
};

struct Layout {
  int es;                // element bytes
  int rows_per_seq;      // 2K+1
  long long rows_total;  // B (2K+1)
  int nseg;              // segments per row
  int seg_elems;         // elements per segment (multiple of 8)
  long long n_units;     // rows_total * nseg
  int nchunk;            // sampling chunks per row
  int sub_elems;         // elements per sub-chunk (512 or 256)
  size_t off_status, off_ctrl, ctrl_bytes, off_seg, off_row, off_plan, off_sub, total;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Pure host computation of the workspace layout for B sequences of
// `rows_per_seq` rows of V elements; false for invalid sizes.
inline bool make_layout_rows(int B, int rows_per_seq, int V, int dtype, Layout* L) {
  if (B < 0 || rows_per_seq < 1 || V < 1) return false;
  if (dtype != 0 && dtype != 1) return false;
  L->es = dtype == 0 ? 2 : 4;
  L->rows_per_seq = rows_per_seq;
  L->rows_total = (long long)B * L->rows_per_seq;
  const long long row_bytes = (long long)V * L->es;
  const long long total_bytes = L->rows_total * row_bytes;
  if (total_bytes > (1LL << 46)) return false;
  long long target = total_bytes <= kWarpsPerWave * kSegMaxBytes ? kWarpsPerWave : kTargetUnits;
  if (L->rows_total > target) target = L->rows_total;
  long long seg_bytes = target > 0 ? total_bytes / target : kSegMaxBytes;
  if (seg_bytes < kSegMinBytes) seg_bytes = kSegMinBytes;
  if (seg_bytes > kSegMaxBytes) seg_bytes = kSegMaxBytes;
  long long nseg = (row_bytes + seg_bytes - 1) / seg_bytes;
  if (nseg < 1) nseg = 1;
  long long seg_elems = ((V + nseg - 1) / nseg + 7) / 8 * 8;
  nseg = (V + seg_elems - 1) / seg_elems;
  L->nseg = (int)nseg;
  L->seg_elems = (int)seg_elems;
  L->n_units = L->rows_total * nseg;
  L->sub_elems = (long long)B * ((V + 4095) / 4096) < kMinDrawCtas ? 256 : 512;
  const long long chunk = (long long)kSubPerChunk * L->sub_elems;
  L->nchunk = (int)(((long long)V + chunk - 1) / chunk);
  size_t off = 0;
  L->off_status = off;  // status word (read by the host), then the control block
  L->off_ctrl = off;
  // status, abort, ticket (12 B, then 4 reserved), then done_s [B], done_p
  // [B], ready [B] and done_r [B rows_per_seq]
  L->ctrl_bytes = align_up(16 + (size_t)B * 12 + (size_t)L->rows_total * 4, 16);
  off = align_up(off + L->ctrl_bytes, 256);
  L->off_seg = off;
  off = align_up(off + (size_t)L->n_units * sizeof(float2), 256);
  L->off_row = off;
  off = align_up(off + (size_t)L->rows_total * sizeof(float2), 256);
  L->off_plan = off;
  off = align_up(off + (size_t)B * sizeof(Plan), 256);
  L->off_sub = off;
  off = align_up(off + (size_t)B * L->nchunk * kSubPerChunk * 4 * sizeof(float2), 256);
  L->total = off;
  return true;
}

// The verification step: B sequences of 2K+1 rows (K+1 target, K draft).
inline bool make_layout(int B, int K, int V, int dtype, Layout* L) {
  if (K < 1 || K > kMaxK) return false;
  return make_layout_rows(B, 2 * K + 1, V, dtype, L);
}

// Greedy mode: B sequences of the K+1 target rows only.
inline bool make_greedy_layout(int B, int K, int V, int dtype, Layout* L) {
  if (K < 1 || K > kMaxK) return false;
  return make_layout_rows(B, K + 1, V, dtype, L);
}

// Top-k filtered verification: the control block (status), then per row of
// the B (2K+1) rows a flag word, the probability of the row's drafted token,
// and its k kept (id, probability) pairs.
constexpr int kTopKMax = 256;
struct TopKLayout {
  int es, rows_per_seq;
  long long rows;
  size_t ctrl_bytes, off_flag, off_at, off_idx, off_prob, total;
};
inline bool make_topk_layout(int B, int K, int V, int dtype, int top_k, TopKLayout* L) {
  if (B < 0 || K < 1 || K > kMaxK || V < 1 || top_k < 1 || top_k > kTopKMax) return false;
  if (dtype != 0 && dtype != 1) return false;
  L->es = dtype == 0 ? 2 : 4;
  L->rows_per_seq = 2 * K + 1;
  L->rows = (long long)B * L->rows_per_seq;
  size_t off = 0;
  L->ctrl_bytes = 16;
  off = align_up(off + L->ctrl_bytes, 256);
  L->off_flag = off;
  off = align_up(off + (size_t)L->rows * 4, 256);
  L->off_at = off;
  off = align_up(off + (size_t)L->rows * 8, 256);
  L->off_idx = off;
  off = align_up(off + (size_t)L->rows * top_k * 4, 256);
  L->off_prob = off;
  off = align_up(off + (size_t)L->rows * top_k * 8, 256);
  L->total = off;
  return true;
}

// The draft-side sampler: N independent rows, each its own "sequence".
inline bool make_sample_layout(int N, int V, int dtype, Layout* L) {
  return make_layout_rows(N, 1, V, dtype, L);
}

struct Params {
  const void* target;
  const void* draft;
  const int32_t* tokens;
  const float* uniforms;
  int B, K, V, dtype, es;
  float c2;        // log2(e) / T in fp32 (streaming pass)
  float ih, il;    // 1/T as a float-float (sampling pass)
  float d_inv, d_ch, d_cli;  // the draw's fast reduction: 1024/(T ln2), fp32(T ln2/1024),
                             // the rest of T ln2/1024 over T
  int unit_t;      // T == 1 exactly
  int sampler;     // 1: draft-side sampler (one row per sequence, K = 0, no scan)
  int fused;       // 1: the fused kernel runs (plans are published with a release flag)
  int withhold;    // test hook: 1 = never publish the flag, so the draw's waits run out
  int top_k;       // top-k path: entries kept per row
  double temp_d;   // top-k path: the temperature, widened to fp64
  int key_ibits;   // top-k path: bits of the (V-1-id) tie-break below the value key
  unsigned* topk_flag;  // top-k path: [B (2K+1)] row flags (nonfinite, empty row)
  double* topk_at;      // top-k path: [B (2K+1)] probability of the row's drafted token
  int* topk_idx;        // top-k path: [B (2K+1), k] kept ids, ascending
  double* topk_prob;    // top-k path: [B (2K+1), k] their probabilities over the kept set
  float top_p;                   // nucleus path: the probability mass kept per row
  unsigned long long* topp_cut;  // nucleus path: [B (2K+1)] keys >= cut are kept
  int* topp_kept;                // nucleus path: [B (2K+1)] kept entries per row, or null
  long long nsi;   // fused kernel: streaming items (of up to 8 units) per sequence
  long long lag;   // fused kernel: sequences between a sequence's streaming and draw tickets
  double inv_t;    // 1/T in fp64 (scan)
  int rows_per_seq;
  int nseg, seg_elems;
  long long n_units;
  int nchunk;
  int sub_elems;   // elements per sub-chunk of the draw (512 or 256)
  long long ns;    // streaming units per sequence ((2K+1) * nseg)
  long long np;    // draw chunks per sequence (nchunk)
  void* ctrl;      // control block, zeroed before every launch
  size_t ctrl_bytes;
  unsigned* abort;   // set by the first bounded wait that runs out (fused kernel)
  unsigned* ticket;  // work items handed out (fused kernel)
  unsigned* done_s;  // [B] rows whose statistics are complete, per sequence
  unsigned* done_p;  // [B] draw chunks counted per sequence
  unsigned* ready;   // [B] the sequence's plan is published
  unsigned* done_r;  // [B (2K+1)] streamed segments counted per row
  float2* seg_part;  // [n_units] (max, sum) per segment
  float2* row_stat;  // [B (2K+1)] (max, sum) per row
  Plan* plans;
  float2* sub_part;
  unsigned* status;
  int32_t* out_tokens;
  int32_t* n_acc;
  double* dbg_lse;
  double* dbg_thr;
  double* dbg_prob;
  double* dbg_max;    // [B (2K+1)] row maximum of l / T
  double* dbg_ratio;  // [B K] q(x~)/p(x~), not clamped
};

// Launchers (sv_kernels.cu). `aligned`: 16-byte aligned rows (vector-load path).
cudaError_t prepare_device(int device);
// Optional events recorded around the step (any may be null): `start` before
// the streaming kernel, `stats_done` between it and the draw kernel, `end`
// after the draw kernel.
struct Events {
  cudaEvent_t start = nullptr, stats_done = nullptr, end = nullptr;
};
cudaError_t launch_all(Params P, bool aligned, cudaStream_t stream, const Events& ev);
// Greedy mode: one kernel over the K+1 target rows of each sequence.
cudaError_t launch_greedy(const Params& P, bool aligned, cudaStream_t stream);
// Top-k filtered verification: the row selection kernel, then the sparse
// verification kernel.
cudaError_t launch_topk(const Params& P, bool aligned, cudaStream_t stream);
// Nucleus-filtered verification: the per-row cut (with each row's kept-set
// statistics), the scan, then the draw with the kept sets applied on load.
cudaError_t launch_topp(Params P, bool aligned, cudaStream_t stream);
cudaError_t fill_int(int* p, long long n, int v, cudaStream_t stream);
// Kernels one call over B sequences of rows_per_seq rows of V elements of
// `es` bytes launches: 1 when the fused kernel is taken, else 2.
int kernels_per_call(long long B, int rows_per_seq, long long V, int es);
// Test hook: 0 chooses the kernels by size, 1 forces the kernel pair, 2 the
// fused kernel.
void force_path(int path);
// Test hook: withhold the plans' release flag (the fused kernel's waits run out).
void withhold_plans(int on);

}  // namespace sv
