// C-ABI entry points (declared in include/spec_verify.h): argument checks,
// workspace layout and the launch of the verification kernels.
#include <cmath>
#include <cstdint>
#include <cstring>

#include <cuda_runtime.h>

#include "../../include/spec_verify.h"
#include "sv_internal.h"

static void fill_params(sv::Params& P, const sv::Layout& L, int B, int K, int V, int dtype,
                        float temperature, void* workspace);

namespace {

bool misaligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) != 0; }

// Checks that need no device. Returns SV_OK or a host error code.
int validate(const void* target, const void* draft, const void* tokens, const void* uniforms,
             int B, int K, int V, int dtype, float temperature, const void* out,
             const void* n_acc, const void* workspace, size_t workspace_bytes, sv::Layout* L) {
  if (dtype != SV_BF16 && dtype != SV_F32) return SV_ERR_DTYPE;
  if (!sv::make_layout(B, K, V, dtype, L)) return SV_ERR_SHAPE;
  if (!std::isfinite(temperature) || !(temperature > 0.0f)) return SV_ERR_TEMPERATURE;
  if (B == 0) return SV_OK;
  if (!target || !draft || !tokens || !uniforms || !out || !n_acc || !workspace) return SV_ERR_NULL;
  const size_t es = dtype == SV_BF16 ? 2 : 4;
  if (misaligned(target, es) || misaligned(draft, es) || misaligned(tokens, 4) ||
      misaligned(uniforms, 4) || misaligned(out, 4) || misaligned(n_acc, 4) ||
      misaligned(workspace, 256))
    return SV_ERR_ALIGN;
  if (workspace_bytes < L->total) return SV_ERR_WORKSPACE;
  return SV_OK;
}

int run(const void* target, const void* draft, const int32_t* tokens, const float* uniforms,
        int B, int K, int V, int dtype, float temperature, int32_t* out, int32_t* n_acc,
        void* workspace, size_t workspace_bytes, void* stream, double* dbg_lse, double* dbg_thr,
        double* dbg_prob, const sv::Events& ev = sv::Events(), double* dbg_max = nullptr,
        double* dbg_ratio = nullptr) {
  sv::Layout L;
  int rc = validate(target, draft, tokens, uniforms, B, K, V, dtype, temperature, out, n_acc,
                    workspace, workspace_bytes, &L);
  if (rc != SV_OK || B == 0) return rc;

  sv::Params P{};
  fill_params(P, L, B, K, V, dtype, temperature, workspace);
  P.target = target;
  P.draft = draft;
  P.tokens = tokens;
  P.uniforms = uniforms;
  P.out_tokens = out;
  P.n_acc = n_acc;
  P.dbg_lse = dbg_lse;
  P.dbg_thr = dbg_thr;
  P.dbg_prob = dbg_prob;
  P.dbg_max = dbg_max;
  P.dbg_ratio = dbg_ratio;
  const bool aligned = !misaligned(target, 16) && !misaligned(draft, 16) &&
                       ((size_t)V * L.es) % 16 == 0;
  cudaError_t e = sv::launch_all(P, aligned, static_cast<cudaStream_t>(stream), ev);
  return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

// Checks of the sampler's arguments that need no device.
int validate_sample(const void* logits, const void* uniforms, int N, int V, int dtype,
                    float temperature, const void* out, const void* workspace,
                    size_t workspace_bytes, sv::Layout* L) {
  if (dtype != SV_BF16 && dtype != SV_F32) return SV_ERR_DTYPE;
  if (!sv::make_sample_layout(N, V, dtype, L)) return SV_ERR_SHAPE;
  if (!std::isfinite(temperature) || !(temperature > 0.0f)) return SV_ERR_TEMPERATURE;
  if (N == 0) return SV_OK;
  if (!logits || !uniforms || !out || !workspace) return SV_ERR_NULL;
  const size_t es = dtype == SV_BF16 ? 2 : 4;
  if (misaligned(logits, es) || misaligned(uniforms, 4) || misaligned(out, 4) ||
      misaligned(workspace, 256))
    return SV_ERR_ALIGN;
  if (workspace_bytes < L->total) return SV_ERR_WORKSPACE;
  return SV_OK;
}

}  // namespace

// Parameter fields shared by the verification and the sampler: sizes, the
// temperature constants, the layout and the workspace's pointers.
static void fill_params(sv::Params& P, const sv::Layout& L, int B, int K, int V, int dtype,
                        float temperature, void* workspace) {
  P.B = B;
  P.K = K;
  P.V = V;
  P.dtype = dtype;
  P.es = L.es;
  const double T = (double)temperature;
  const double inv = 1.0 / T;
  P.c2 = (float)(1.4426950408889634074 / T);
  P.ih = (float)inv;
  P.il = (float)(inv - (double)P.ih);
  P.unit_t = temperature == 1.0f ? 1 : 0;
  P.inv_t = inv;
  {
    const double C = T * 0.69314718055994530942 / 1024.0;
    P.d_ch = (float)C;
    P.d_cli = (float)((C - (double)P.d_ch) * inv);
    P.d_inv = (float)(1.0 / C);
  }
  P.rows_per_seq = L.rows_per_seq;
  P.nseg = L.nseg;
  P.seg_elems = L.seg_elems;
  P.n_units = L.n_units;
  P.nchunk = L.nchunk;
  P.sub_elems = L.sub_elems;
  P.ns = (long long)L.rows_per_seq * L.nseg;
  P.np = L.nchunk;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  // Control block: status, abort, ticket (4 B each, 4 reserved), then done_s,
  // done_p, ready [B] each and done_r [B rows_per_seq]; zeroed before every
  // launch.
  P.ctrl = ws + L.off_ctrl;
  P.ctrl_bytes = L.ctrl_bytes;
  P.status = reinterpret_cast<unsigned*>(ws + L.off_ctrl);
  P.abort = P.status + 1;
  P.ticket = P.status + 2;
  P.done_s = reinterpret_cast<unsigned*>(ws + L.off_ctrl + 16);
  P.done_p = P.done_s + B;
  P.ready = P.done_p + B;
  P.done_r = P.ready + B;
  P.seg_part = reinterpret_cast<float2*>(ws + L.off_seg);
  P.row_stat = reinterpret_cast<float2*>(ws + L.off_row);
  P.plans = reinterpret_cast<sv::Plan*>(ws + L.off_plan);
  P.sub_part = reinterpret_cast<float2*>(ws + L.off_sub);
}

namespace {

struct Staging {
  size_t target, draft, tokens, uniforms, out, nacc, total;
};

bool staging_layout(int B, int K, int V, int dtype, Staging* S) {
  sv::Layout L;
  if (!sv::make_layout(B, K, V, dtype, &L)) return false;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = sv::align_up(off + bytes, 256);
    return at;
  };
  S->target = take((size_t)B * (K + 1) * V * L.es);
  S->draft = take((size_t)B * K * V * L.es);
  S->tokens = take((size_t)B * K * 4);
  S->uniforms = take((size_t)B * (K + 2) * 4);
  S->out = take((size_t)B * (K + 1) * 4);
  S->nacc = take((size_t)B * 4);
  S->total = off;
  return true;
}

}  // namespace

extern "C" {

size_t sv_workspace_size(int B, int K, int V, int dtype) {
  sv::Layout L;
  if (!sv::make_layout(B, K, V, dtype, &L)) return 0;
  return L.total;
}

int spec_verify(const void* target_logits, const void* draft_logits, const int32_t* draft_tokens,
                const float* uniforms, int B, int K, int V, int dtype, float temperature,
                int32_t* out_tokens, int32_t* n_accepted, void* workspace, size_t workspace_bytes,
                void* stream) {
  return run(target_logits, draft_logits, draft_tokens, uniforms, B, K, V, dtype, temperature,
             out_tokens, n_accepted, workspace, workspace_bytes, stream, nullptr, nullptr, nullptr);
}

int spec_verify_debug(const void* target_logits, const void* draft_logits,
                      const int32_t* draft_tokens, const float* uniforms, int B, int K, int V,
                      int dtype, float temperature, int32_t* out_tokens, int32_t* n_accepted,
                      void* workspace, size_t workspace_bytes, void* stream, double* row_lse,
                      double* thresholds, double* sample_prob, double* row_max,
                      double* ratios) {
  return run(target_logits, draft_logits, draft_tokens, uniforms, B, K, V, dtype, temperature,
             out_tokens, n_accepted, workspace, workspace_bytes, stream, row_lse, thresholds,
             sample_prob, sv::Events(), row_max, ratios);
}

int spec_verify_profiled(const void* target_logits, const void* draft_logits,
                         const int32_t* draft_tokens, const float* uniforms, int B, int K, int V,
                         int dtype, float temperature, int32_t* out_tokens, int32_t* n_accepted,
                         void* workspace, size_t workspace_bytes, void* stream, void* ev_start,
                         void* ev_stats_done, void* ev_end) {
  sv::Events ev;
  ev.start = static_cast<cudaEvent_t>(ev_start);
  ev.stats_done = static_cast<cudaEvent_t>(ev_stats_done);
  ev.end = static_cast<cudaEvent_t>(ev_end);
  return run(target_logits, draft_logits, draft_tokens, uniforms, B, K, V, dtype, temperature,
             out_tokens, n_accepted, workspace, workspace_bytes, stream, nullptr, nullptr, nullptr,
             ev);
}

size_t sv_staging_size(int B, int K, int V, int dtype) {
  Staging S;
  if (!staging_layout(B, K, V, dtype, &S)) return 0;
  return S.total;
}

}  // extern "C"

namespace {

// The host-buffer step: inputs host -> device into `staging`, the step, the
// outputs device -> host; nothing waits when `sync` is false.
int host_step(const void* h_target_logits, const void* h_draft_logits,
              const int32_t* h_draft_tokens, const float* h_uniforms, int B, int K, int V,
              int dtype, float temperature, int32_t* h_out_tokens, int32_t* h_n_accepted,
              void* staging, size_t staging_bytes, void* workspace, size_t workspace_bytes,
              void* stream, bool sync) {
  sv::Layout L;
  int rc = validate(h_target_logits, h_draft_logits, h_draft_tokens, h_uniforms, B, K, V, dtype,
                    temperature, h_out_tokens, h_n_accepted, workspace, workspace_bytes, &L);
  if (rc != SV_OK || B == 0) return rc;
  Staging S;
  if (!staging_layout(B, K, V, dtype, &S)) return SV_ERR_SHAPE;
  if (!staging) return SV_ERR_NULL;
  if (misaligned(staging, 256)) return SV_ERR_ALIGN;
  if (staging_bytes < S.total) return SV_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned char* d = static_cast<unsigned char*>(staging);
  const size_t es = L.es;
  const size_t nt = (size_t)B * (K + 1) * V * es, nd = (size_t)B * K * V * es;
  if (cudaMemcpyAsync(d + S.target, h_target_logits, nt, cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaMemcpyAsync(d + S.draft, h_draft_logits, nd, cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaMemcpyAsync(d + S.tokens, h_draft_tokens, (size_t)B * K * 4, cudaMemcpyHostToDevice,
                      st) != cudaSuccess ||
      cudaMemcpyAsync(d + S.uniforms, h_uniforms, (size_t)B * (K + 2) * 4, cudaMemcpyHostToDevice,
                      st) != cudaSuccess)
    return SV_ERR_CUDA;
  rc = spec_verify(d + S.target, d + S.draft, reinterpret_cast<const int32_t*>(d + S.tokens),
                   reinterpret_cast<const float*>(d + S.uniforms), B, K, V, dtype, temperature,
                   reinterpret_cast<int32_t*>(d + S.out), reinterpret_cast<int32_t*>(d + S.nacc),
                   workspace, workspace_bytes, stream);
  if (rc != SV_OK) return rc;
  if (cudaMemcpyAsync(h_out_tokens, d + S.out, (size_t)B * (K + 1) * 4, cudaMemcpyDeviceToHost,
                      st) != cudaSuccess ||
      cudaMemcpyAsync(h_n_accepted, d + S.nacc, (size_t)B * 4, cudaMemcpyDeviceToHost, st) !=
          cudaSuccess)
    return SV_ERR_CUDA;
  if (!sync) return SV_OK;
  unsigned status = 0;
  if (cudaMemcpyAsync(&status, static_cast<unsigned char*>(workspace) + L.off_status,
                      sizeof(status), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return SV_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return SV_ERR_CUDA;
  return (int)status;
}

}  // namespace

extern "C" {

int spec_verify_host(const void* h_target_logits, const void* h_draft_logits,
                     const int32_t* h_draft_tokens, const float* h_uniforms, int B, int K, int V,
                     int dtype, float temperature, int32_t* h_out_tokens, int32_t* h_n_accepted,
                     void* staging, size_t staging_bytes, void* workspace,
                     size_t workspace_bytes, void* stream) {
  return host_step(h_target_logits, h_draft_logits, h_draft_tokens, h_uniforms, B, K, V, dtype,
                   temperature, h_out_tokens, h_n_accepted, staging, staging_bytes, workspace,
                   workspace_bytes, stream, true);
}

int spec_verify_host_async(const void* h_target_logits, const void* h_draft_logits,
                           const int32_t* h_draft_tokens, const float* h_uniforms, int B, int K,
                           int V, int dtype, float temperature, int32_t* h_out_tokens,
                           int32_t* h_n_accepted, void* staging, size_t staging_bytes,
                           void* workspace, size_t workspace_bytes, void* stream) {
  return host_step(h_target_logits, h_draft_logits, h_draft_tokens, h_uniforms, B, K, V, dtype,
                   temperature, h_out_tokens, h_n_accepted, staging, staging_bytes, workspace,
                   workspace_bytes, stream, false);
}

size_t sv_sample_workspace_size(int N, int V, int dtype) {
  sv::Layout L;
  if (!sv::make_sample_layout(N, V, dtype, &L)) return 0;
  return L.total;
}

int spec_draft_sample(const void* logits, const float* uniforms, int N, int V, int dtype,
                      float temperature, int32_t* out_tokens, double* sample_prob,
                      void* workspace, size_t workspace_bytes, void* stream) {
  sv::Layout L;
  const int rc = validate_sample(logits, uniforms, N, V, dtype, temperature, out_tokens,
                                 workspace, workspace_bytes, &L);
  if (rc != SV_OK || N == 0) return rc;
  sv::Params P{};
  fill_params(P, L, N, 0, V, dtype, temperature, workspace);
  P.sampler = 1;
  P.target = logits;
  P.uniforms = uniforms;
  P.out_tokens = out_tokens;
  P.dbg_prob = sample_prob;
  const bool aligned = !misaligned(logits, 16) && ((size_t)V * L.es) % 16 == 0;
  const cudaError_t e = sv::launch_all(P, aligned, static_cast<cudaStream_t>(stream), sv::Events());
  return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

size_t sv_greedy_workspace_size(int B, int K, int V, int dtype) {
  sv::Layout L;
  if (!sv::make_greedy_layout(B, K, V, dtype, &L)) return 0;
  return L.total;
}

int spec_verify_greedy(const void* target_logits, const int32_t* draft_tokens, int B, int K,
                       int V, int dtype, int32_t* out_tokens, int32_t* n_accepted,
                       void* workspace, size_t workspace_bytes, void* stream) {
  if (dtype != SV_BF16 && dtype != SV_F32) return SV_ERR_DTYPE;
  sv::Layout L;
  if (!sv::make_greedy_layout(B, K, V, dtype, &L)) return SV_ERR_SHAPE;
  if (B == 0) return SV_OK;
  if (!target_logits || !draft_tokens || !out_tokens || !n_accepted || !workspace)
    return SV_ERR_NULL;
  if (misaligned(target_logits, L.es) || misaligned(draft_tokens, 4) ||
      misaligned(out_tokens, 4) || misaligned(n_accepted, 4) || misaligned(workspace, 256))
    return SV_ERR_ALIGN;
  if (workspace_bytes < L.total) return SV_ERR_WORKSPACE;
  sv::Params P{};
  fill_params(P, L, B, K, V, dtype, 1.0f, workspace);
  P.target = target_logits;
  P.tokens = draft_tokens;
  P.out_tokens = out_tokens;
  P.n_acc = n_accepted;
  const bool aligned = !misaligned(target_logits, 16) && ((size_t)V * L.es) % 16 == 0;
  const cudaError_t e = sv::launch_greedy(P, aligned, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

size_t sv_topk_workspace_size(int B, int K, int V, int dtype, int top_k) {
  if (top_k >= V) return sv_workspace_size(B, K, V, dtype);
  sv::TopKLayout L;
  if (!sv::make_topk_layout(B, K, V, dtype, top_k, &L)) return 0;
  return L.total;
}

int spec_verify_topk(const void* target_logits, const void* draft_logits,
                     const int32_t* draft_tokens, const float* uniforms, int B, int K, int V,
                     int dtype, float temperature, int top_k, int32_t* out_tokens,
                     int32_t* n_accepted, void* workspace, size_t workspace_bytes, void* stream) {
  if (top_k >= V && V >= 1)  // keeps every entry: the unfiltered verification
    return run(target_logits, draft_logits, draft_tokens, uniforms, B, K, V, dtype, temperature,
               out_tokens, n_accepted, workspace, workspace_bytes, stream, nullptr, nullptr,
               nullptr);
  if (dtype != SV_BF16 && dtype != SV_F32) return SV_ERR_DTYPE;
  sv::TopKLayout L;
  if (!sv::make_topk_layout(B, K, V, dtype, top_k, &L)) return SV_ERR_SHAPE;
  if (!std::isfinite(temperature) || !(temperature > 0.0f)) return SV_ERR_TEMPERATURE;
  if (B == 0) return SV_OK;
  if (!target_logits || !draft_logits || !draft_tokens || !uniforms || !out_tokens ||
      !n_accepted || !workspace)
    return SV_ERR_NULL;
  if (misaligned(target_logits, L.es) || misaligned(draft_logits, L.es) ||
      misaligned(draft_tokens, 4) || misaligned(uniforms, 4) || misaligned(out_tokens, 4) ||
      misaligned(n_accepted, 4) || misaligned(workspace, 256))
    return SV_ERR_ALIGN;
  if (workspace_bytes < L.total) return SV_ERR_WORKSPACE;
  sv::Params P{};
  P.B = B;
  P.K = K;
  P.V = V;
  P.dtype = dtype;
  P.es = L.es;
  P.rows_per_seq = L.rows_per_seq;
  P.top_k = top_k;
  P.temp_d = (double)temperature;
  int ib = 1;
  while (ib < 31 && ((long long)(V - 1) >> ib) != 0) ++ib;
  P.key_ibits = ib;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  P.ctrl = ws;
  P.ctrl_bytes = L.ctrl_bytes;
  P.status = reinterpret_cast<unsigned*>(ws);
  P.topk_flag = reinterpret_cast<unsigned*>(ws + L.off_flag);
  P.topk_at = reinterpret_cast<double*>(ws + L.off_at);
  P.topk_idx = reinterpret_cast<int*>(ws + L.off_idx);
  P.topk_prob = reinterpret_cast<double*>(ws + L.off_prob);
  P.target = target_logits;
  P.draft = draft_logits;
  P.tokens = draft_tokens;
  P.uniforms = uniforms;
  P.out_tokens = out_tokens;
  P.n_acc = n_accepted;
  const bool aligned = !misaligned(target_logits, 16) && !misaligned(draft_logits, 16) &&
                       ((size_t)V * L.es) % 16 == 0;
  const cudaError_t e = sv::launch_topk(P, aligned, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

}  // extern "C"

namespace {

// Nucleus path workspace: the unfiltered layout, then one cut key per row.
struct ToppLayout {
  sv::Layout L;
  size_t off_cut, total;
};

bool make_topp_layout(int B, int K, int V, int dtype, ToppLayout* T) {
  if (!sv::make_layout(B, K, V, dtype, &T->L)) return false;
  size_t off = sv::align_up(T->L.total, 256);
  T->off_cut = off;
  off = sv::align_up(off + (size_t)B * (2 * K + 1) * 8, 256);
  T->total = off;
  return true;
}

}  // namespace

extern "C" {

size_t sv_topp_workspace_size(int B, int K, int V, int dtype) {
  ToppLayout T;
  if (!make_topp_layout(B, K, V, dtype, &T)) return 0;
  return T.total;
}

int spec_verify_topp(const void* target_logits, const void* draft_logits,
                     const int32_t* draft_tokens, const float* uniforms, int B, int K, int V,
                     int dtype, float temperature, float top_p, int32_t* out_tokens,
                     int32_t* n_accepted, int32_t* kept_counts, void* workspace,
                     size_t workspace_bytes, void* stream) {
  if (dtype != SV_BF16 && dtype != SV_F32) return SV_ERR_DTYPE;
  if (!(top_p > 0.0f)) return SV_ERR_SHAPE;
  ToppLayout TL;
  if (!make_topp_layout(B, K, V, dtype, &TL)) return SV_ERR_SHAPE;
  sv::Layout L;
  int rc = validate(target_logits, draft_logits, draft_tokens, uniforms, B, K, V, dtype,
                    temperature, out_tokens, n_accepted, workspace, workspace_bytes, &L);
  if (rc != SV_OK || B == 0) return rc;
  if (misaligned(kept_counts, 4)) return SV_ERR_ALIGN;
  if (workspace_bytes < TL.total) return SV_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const long long rows = (long long)B * (2 * K + 1);
  if (top_p >= 1.0f) {  // keeps every entry: the unfiltered call
    rc = run(target_logits, draft_logits, draft_tokens, uniforms, B, K, V, dtype, temperature,
             out_tokens, n_accepted, workspace, workspace_bytes, stream, nullptr, nullptr,
             nullptr);
    if (rc == SV_OK && kept_counts && sv::fill_int(kept_counts, rows, V, st) != cudaSuccess)
      return SV_ERR_CUDA;
    return rc;
  }
  sv::Params P{};
  fill_params(P, TL.L, B, K, V, dtype, temperature, workspace);
  P.target = target_logits;
  P.draft = draft_logits;
  P.tokens = draft_tokens;
  P.uniforms = uniforms;
  int ib = 1;
  while (ib < 31 && ((long long)(V - 1) >> ib) != 0) ++ib;
  P.key_ibits = ib;
  P.top_p = top_p;
  P.temp_d = (double)temperature;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  P.topp_cut = reinterpret_cast<unsigned long long*>(ws + TL.off_cut);
  P.topp_kept = kept_counts;
  P.out_tokens = out_tokens;
  P.n_acc = n_accepted;
  const bool aligned = !misaligned(target_logits, 16) && !misaligned(draft_logits, 16) &&
                       ((size_t)V * TL.L.es) % 16 == 0;
  return sv::launch_topp(P, aligned, st) == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

int sv_read_device_status(const void* workspace, void* stream, int* status) {
  if (!workspace || !status) return SV_ERR_NULL;
  if (misaligned(workspace, 256)) return SV_ERR_ALIGN;
  unsigned v = 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return SV_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return SV_ERR_CUDA;
  *status = (int)v;
  return SV_OK;
}

const char* sv_status_string(int status) {
  switch (status) {
    case SV_OK: return "ok";
    case SV_ERR_NULL: return "a required pointer is NULL";
    case SV_ERR_SHAPE: return "invalid shape (B < 0, K outside [1,64], V < 1, or too large)";
    case SV_ERR_TEMPERATURE: return "temperature must be finite and > 0";
    case SV_ERR_DTYPE: return "dtype must be SV_BF16 or SV_F32";
    case SV_ERR_ALIGN: return "pointer misaligned (elements, or 256 bytes for workspace/staging)";
    case SV_ERR_WORKSPACE: return "workspace or staging buffer too small";
    case SV_ERR_CUDA: return "a CUDA runtime call failed";
    case SV_ERR_SCRATCH_LIMIT: return "problem needs more scratch than spec_verify_static holds";
    default: break;
  }
  if (status & SV_DEV_TIMEOUT) return "device: a bounded wait ran out (results invalid)";
  if (status & SV_DEV_NONFINITE) return "device: a logit row holds NaN or +inf";
  if (status & SV_DEV_EMPTY_ROW) return "device: a logit row is entirely -inf";
  if (status & SV_DEV_TOKEN_RANGE) return "device: a draft token lies outside [0, V)";
  if (status & SV_DEV_UNIFORM_RANGE) return "device: a uniform is NaN or outside [0, 1]";
  return "unknown status";
}

int sv_kernels_per_call(int B, int K, int V, int dtype) {
  sv::Layout L;
  if (!sv::make_layout(B, K, V, dtype, &L) || B == 0) return 0;
  return sv::kernels_per_call(B, L.rows_per_seq, V, L.es);
}

int sv_topp_kernels_per_call(int B, int K, int V, int dtype) {
  sv::Layout L;
  if (!sv::make_layout(B, K, V, dtype, &L) || B == 0) return 0;
  return L.sub_elems == 512 ? 4 : 3;
}

void sv_force_path(int path) { sv::force_path(path); }

void sv_test_withhold_plans(int on) { sv::withhold_plans(on); }

}  // extern "C"
