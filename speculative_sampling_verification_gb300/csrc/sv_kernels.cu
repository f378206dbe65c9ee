// Kernel of the verification step of speculative sampling (modified rejection
// sampling: §4.2 and Algorithm 2 of "Accelerating Large Language Model
// Decoding with Speculative Sampling", wikillm.com paper card).
//
// One persistent kernel per call. CTAs take tickets from a counter; a ticket
// is one of two kinds of work item, dispensed in sequence-major order:
//
//   stats(b, u)   one segment of one of the 2K+1 logit rows of sequence b,
//                 streamed HBM -> shared memory by 1-D bulk copies
//                 (cp.async.bulk, mbarrier completion): per segment the
//                 maximum m and sum_i 2^((l_i - m) log2(e)/T), the
//                 temperature transform of §4.2 "Decoding transforms".
//                 The CTA that completes the last segment of b runs the scan
//                 of b: combine segments, gather the logits at the drafted
//                 tokens, thresholds min(1, q/p) in fp64, first rejection j
//                 (Algorithm 2 step 3), and publishes the plan of b.
//   draw(b, c)    one 4096-element chunk of the row pair the draw of b needs
//                 (target and draft row j for the residual (q - p)_+, or
//                 target row K for the bonus token, Algorithm 2 step 4):
//                 float-float sums of exp((l - m)/T) and of the residual's
//                 positive part per 512-element sub-chunk. The CTA that
//                 completes the last chunk of b runs the exact inverse-CDF
//                 search and writes the drawn token.
//
// draw(b, .) tickets come `lag` sequences after stats(b, .) tickets, so the
// plan of b is normally ready when they are taken and the two rows they
// re-read are still in L2; their float-float arithmetic overlaps the HBM
// streaming of later sequences. A draw ticket never waits on a ticket handed
// out after it, so the schedule cannot deadlock; every wait is bounded.
#include <cfloat>
#include <climits>
#include <cstdint>
#include <mutex>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {

constexpr unsigned kDevTokenRange = 16, kDevNonfinite = 32, kDevEmptyRow = 64,
                   kDevUniformRange = 128, kDevTimeout = 256;
constexpr float kLn2 = 0.693147180559945309f;

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kStageBytes = 16384;
constexpr int kStages = 4;
constexpr int kVecPerThread = kStageBytes / 16 / kThreads;  // 4
constexpr int kCtasPerSm = 3;
static_assert(kSegMaxBytes <= (long long)kStages * kStageBytes, "a segment must fit the ring");

// ---------------------------------------------------------------- addressing and loads

// Row r of sequence b: target rows r = 0..K, then draft rows r = K+1..2K.
SV_DEVINL const unsigned char* row_base(const Params& P, long long b, int r) {
  if (r <= P.K)
    return static_cast<const unsigned char*>(P.target) +
           ((size_t)b * (P.K + 1) + r) * (size_t)P.V * P.es;
  return static_cast<const unsigned char*>(P.draft) +
         ((size_t)b * P.K + (r - P.K - 1)) * (size_t)P.V * P.es;
}

template <int DT>
SV_DEVINL float load_elem(const unsigned char* row, long long i) {
  if constexpr (DT == 0) {
    const unsigned short h = __ldg(reinterpret_cast<const unsigned short*>(row) + i);
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
  } else {
    return __ldg(reinterpret_cast<const float*>(row) + i);
  }
}

SV_DEVINL uint32_t ld_acquire(const unsigned* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

SV_DEVINL void st_release(unsigned* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Bounded wait for a flag another CTA sets (200 ms of wall time at most).
SV_DEVINL bool wait_flag(const unsigned* p) {
  if (ld_acquire(p)) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
    __nanosleep(100);
    if (ld_acquire(p)) return true;
    if (global_ns() - t0 > kWaitLimitNs) return false;
  }
}

// ---------------------------------------------------------------- per-CTA shared state

struct CtaShared {
  float2 tab[256];  // 2^(j/256), head + tail
  uint64_t full[kStages];
  float red_m[kWarps], red_s[kWarps];
  float s_m[2 * kMaxK + 1], s_s[2 * kMaxK + 1];
  double s_lse[2 * kMaxK + 1];
  double s_thr[kMaxK];
  float s_u[kMaxK + 2];
  int s_tok[kMaxK];
  ff red_f[kWarps];
  ff s_pref;
  Plan plan;
  unsigned long long ticket, next;
  unsigned bits;
  int j, g, flag;
};

// ---------------------------------------------------------------- (max, sum) pairs
// A pair (m, s) stands for the sum s * 2^(m c2) of 2^(l_i c2) terms; s is
// NaN when a NaN (or +inf) entry was seen; m = -inf with s = 0 means "no
// finite entry yet".

SV_DEVINL void ms_combine(float& m, float& s, float m2, float s2, float c2) {
  const float M = fmaxf(m, m2);
  if (M == neg_inf()) {
    s = s + s2;
    return;
  }
  const float a = (m == neg_inf()) ? 0.0f : ex2_fast((m - M) * c2);
  const float b = (m2 == neg_inf()) ? 0.0f : ex2_fast((m2 - M) * c2);
  s = s * a + s2 * b;
  m = M;
}

// Block-wide combine (kThreads threads). Result in thread 0.
SV_DEVINL void block_combine(float& m, float& s, float c2, CtaShared& sh) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    ms_combine(m, s, m2, s2, c2);
  }
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) {
    sh.red_m[w] = m;
    sh.red_s[w] = s;
  }
  __syncthreads();
  if (w == 0) {
    m = l < kWarps ? sh.red_m[l] : neg_inf();
    s = l < kWarps ? sh.red_s[l] : 0.0f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
      const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
      ms_combine(m, s, m2, s2, c2);
    }
  }
  __syncthreads();
}

// ---------------------------------------------------------------- stats: one segment
//
// Per thread: the stage's local max (packed bf16x2 max for bf16), a rescale
// of the four running sums only when the max grows, then one FFMA and one
// MUFU ex2 per element against H = fl(m * c2); the rounding residual of H is
// folded back in once per segment.

template <int DT>
SV_DEVINL bool any_nan(const uint4 (&v)[kVecPerThread]) {
  bool bad = false;
#pragma unroll
  for (int i = 0; i < kVecPerThread; ++i) {
    const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if constexpr (DT == 0) {
        bad |= ((w[k] & 0x7fffu) > 0x7f80u) || (((w[k] >> 16) & 0x7fffu) > 0x7f80u);
      } else {
        bad |= (w[k] & 0x7fffffffu) > 0x7f800000u;
      }
    }
  }
  return bad;
}

template <int DT>
SV_DEVINL void stats_consume(const uint4 (&v)[kVecPerThread], float& m_run, float& H,
                             float (&acc)[4], bool& nan_seen, float c2) {
  float lm;
  if constexpr (DT == 0) {
    uint32_t mx = bf16x2_max(bf16x2_max(v[0].x, v[0].y), bf16x2_max(v[0].z, v[0].w));
#pragma unroll
    for (int i = 1; i < kVecPerThread; ++i)
      mx = bf16x2_max(mx, bf16x2_max(bf16x2_max(v[i].x, v[i].y), bf16x2_max(v[i].z, v[i].w)));
    lm = fmaxf(bf16_lo(mx), bf16_hi(mx));
  } else {
    lm = neg_inf();
#pragma unroll
    for (int i = 0; i < kVecPerThread; ++i)
      lm = fmaxf(lm, fmaxf(fmaxf(__uint_as_float(v[i].x), __uint_as_float(v[i].y)),
                           fmaxf(__uint_as_float(v[i].z), __uint_as_float(v[i].w))));
  }
  if (lm > m_run) {
    const float Hn = lm * c2;
    const float f = ex2_fast(H - Hn);
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[k] *= f;
    m_run = lm;
    H = Hn;
  }
  if (m_run == neg_inf()) {  // only -inf (or NaN) entries so far
    nan_seen |= any_nan<DT>(v);
    return;
  }
#pragma unroll
  for (int i = 0; i < kVecPerThread; ++i) {
    const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
    if constexpr (DT == 0) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        acc[k] += ex2_fast(__fmaf_rn(bf16_lo(w[k]), c2, -H));
        acc[k] += ex2_fast(__fmaf_rn(bf16_hi(w[k]), c2, -H));
      }
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[k] += ex2_fast(__fmaf_rn(__uint_as_float(w[k]), c2, -H));
    }
  }
}

// Per-thread sum of a finished segment, with H's rounding residual folded in.
SV_DEVINL float thread_sum(float m_run, float H, const float (&acc)[4], bool nan_seen, float c2) {
  if (m_run == neg_inf()) return nan_seen ? __int_as_float(0x7fc00000) : 0.0f;
  float s = (acc[0] + acc[1]) + (acc[2] + acc[3]);
  const float L = __fmaf_rn(m_run, c2, -H);  // m*c2 - H exactly (to fp32)
  s *= __fmaf_rn(-L, kLn2, 1.0f);            // 2^-L to first order (|L| < 1e-5)
  return nan_seen ? __int_as_float(0x7fc00000) : s;
}

SV_DEVINL int unit_len(const Params& P, long long u) {
  const int seg = (int)(u % P.nseg);
  return seg == P.nseg - 1 ? P.V - seg * P.seg_elems : P.seg_elems;
}

SV_DEVINL const unsigned char* unit_row(const Params& P, long long u) {
  const long long row = u / P.nseg;
  return row_base(P, row / P.rows_per_seq, (int)(row % P.rows_per_seq));
}

// Bulk-copy path, producer side (thread 0): issue the segment's 16 KB pieces
// (at most two: segments are at most 32 KB) into the next ring stages.
// `issued` counts pieces issued over the CTA's life.
template <int DT>
SV_DEVINL void stats_issue(const Params& P, long long u, unsigned char* ring, CtaShared& sh,
                           uint32_t& issued) {
  constexpr int kEs = DT == 0 ? 2 : 4;
  constexpr int kStageElems = kStageBytes / kEs;
  const int len = unit_len(P, u);
  const int npieces = (len + kStageElems - 1) / kStageElems;
  const unsigned char* src = unit_row(P, u) + (size_t)(u % P.nseg) * P.seg_elems * kEs;
  for (int i = 0; i < npieces; ++i) {
    const int st = (int)((issued + i) % kStages);
    const int n = min(kStageElems, len - i * kStageElems);
    const uint32_t bytes = (uint32_t)n * kEs;
    mbar_arrive_expect_tx(&sh.full[st], bytes);
    bulk_copy_g2s(ring + st * kStageBytes, src + (size_t)i * kStageBytes, bytes, &sh.full[st]);
  }
  issued += npieces;
}

// Bulk-copy path, consumer side (all threads): the segment's pieces are the
// next ones in ring order. `piece` counts consumed pieces (mbarrier phases).
// Returns false, with every thread agreeing, if a wait ran out.
template <int DT>
SV_DEVINL bool stats_consume_unit(const Params& P, long long u, const unsigned char* ring,
                                  CtaShared& sh, uint32_t& piece) {
  constexpr int kEs = DT == 0 ? 2 : 4;
  constexpr int kStageElems = kStageBytes / kEs;
  const int tid = threadIdx.x;
  const int len = unit_len(P, u);
  const int npieces = (len + kStageElems - 1) / kStageElems;
  const float c2 = P.c2;
  float m_run = neg_inf(), H = neg_inf();
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  bool nan_seen = false, timed_out = false;
  const uint32_t fill = DT == 0 ? 0xff80ff80u : 0xff800000u;  // -inf
  for (int i = 0; i < npieces; ++i) {
    const uint32_t p = piece + i;
    const int st = (int)(p % kStages);
    if (!mbar_wait(&sh.full[st], (p / kStages) & 1u)) timed_out = true;
    const unsigned char* buf = ring + st * kStageBytes;
    const int nvec = min(kStageElems, len - i * kStageElems) * kEs / 16;
    uint4 v[kVecPerThread];
#pragma unroll
    for (int k = 0; k < kVecPerThread; ++k) {
      const int idx = tid + k * kThreads;
      v[k] = idx < nvec ? ld_shared_v4(buf + idx * 16) : make_uint4(fill, fill, fill, fill);
    }
    stats_consume<DT>(v, m_run, H, acc, nan_seen, c2);
  }
  piece += npieces;
  float s = thread_sum(m_run, H, acc, nan_seen, c2);
  float m = m_run;
  block_combine(m, s, c2, sh);  // its barriers also free the segment's stages
  if (tid == 0) P.seg_part[u] = make_float2(m, s);
  return !__syncthreads_or(timed_out);
}

// Plain-load path for rows that are not 16-byte aligned: two passes (max, sum).
template <int DT>
SV_DEVINL void stats_unit_plain(const Params& P, long long u, CtaShared& sh) {
  const float c2 = P.c2;
  const int len = unit_len(P, u);
  const unsigned char* rb = unit_row(P, u);
  const long long e0 = (long long)(u % P.nseg) * P.seg_elems;
  float m = neg_inf();
  bool nan_seen = false;
  for (int i = threadIdx.x; i < len; i += kThreads) {
    const float l = load_elem<DT>(rb, e0 + i);
    nan_seen |= (l != l);
    m = fmaxf(m, l);
  }
  float s = 0.f;
  if (m != neg_inf()) {
    for (int i = threadIdx.x; i < len; i += kThreads)
      s += ex2_fast((load_elem<DT>(rb, e0 + i) - m) * c2);
  }
  if (nan_seen) s = __int_as_float(0x7fc00000);
  block_combine(m, s, c2, sh);
  if (threadIdx.x == 0) P.seg_part[u] = make_float2(m, s);
}

// ---------------------------------------------------------------- scan of one sequence

SV_DEVINL void scan_seq(const Params& P, long long b, CtaShared& sh) {
  const int tid = threadIdx.x, K = P.K, R = P.rows_per_seq;
  if (tid == 0) sh.bits = 0;
  // Stage the drafted tokens and uniforms of the sequence.
  for (int t = tid; t < K + 2; t += kThreads) {
    if (t < K) sh.s_tok[t] = P.tokens[b * K + t];
    sh.s_u[t] = P.uniforms[b * (K + 2) + t];
  }
  __syncthreads();

  // Row statistics: m = max over segments, S = sum of rescaled segment sums
  // (one pass, rescaling the running sum when the maximum grows).
  for (int r = tid; r < R; r += kThreads) {
    const float2* part = P.seg_part + ((long long)b * R + r) * P.nseg;
    float m = neg_inf();
    double S = 0.0;
    bool nan_seen = false;
    for (int g = 0; g < P.nseg; ++g) {
      const float2 ps = __ldcg(part + g);
      nan_seen |= (ps.y != ps.y);
      if (ps.x == neg_inf()) continue;
      if (ps.x > m) {
        if (m != neg_inf()) S *= (double)exp2f((m - ps.x) * P.c2);
        m = ps.x;
      }
      S += (double)ps.y * (double)exp2f((ps.x - m) * P.c2);
    }
    unsigned bits = 0;
    if (nan_seen) {
      bits = kDevNonfinite;
    } else if (m == neg_inf()) {
      bits = kDevEmptyRow;
    }
    if (bits) atomicOr(&sh.bits, bits);
    sh.s_m[r] = m;
    sh.s_s[r] = (float)S;
    sh.s_lse[r] = bits ? __longlong_as_double(0x7ff8000000000000LL) : (double)m * P.inv_t + log(S);
  }
  for (int t = tid; t < K; t += kThreads) {
    const int x = sh.s_tok[t];
    if (x < 0 || x >= P.V) atomicOr(&sh.bits, kDevTokenRange);
  }
  for (int t = tid; t < K + 2; t += kThreads) {
    const float u = sh.s_u[t];
    if (!(u >= 0.0f && u <= 1.0f)) atomicOr(&sh.bits, kDevUniformRange);
  }
  __syncthreads();
  const unsigned bits = sh.bits;
  if (P.dbg_lse)
    for (int r = tid; r < R; r += kThreads) P.dbg_lse[b * R + r] = sh.s_lse[r];

  if (!bits) {
    // Thresholds min(1, q(x~)/p(x~)) at the drafted tokens (§4.2), in fp64:
    // log q(x) - log p(x) = (lq - lp)/T - (lse_q - lse_p).
    for (int t = tid; t < K; t += kThreads) {
      const int x = sh.s_tok[t];
      float lq, lp;
      if (P.dtype == 0) {
        lq = load_elem<0>(row_base(P, b, t), x);
        lp = load_elem<0>(row_base(P, b, K + 1 + t), x);
      } else {
        lq = load_elem<1>(row_base(P, b, t), x);
        lp = load_elem<1>(row_base(P, b, K + 1 + t), x);
      }
      double thr;
      if (lq == neg_inf()) {
        thr = 0.0;  // q(x~) = 0 rejects
      } else if (lp == neg_inf()) {
        thr = 1.0;  // p(x~) = 0 < q(x~) accepts
      } else {
        const double lr =
            ((double)lq - (double)lp) * P.inv_t - (sh.s_lse[t] - sh.s_lse[K + 1 + t]);
        thr = lr >= 0.0 ? 1.0 : exp(lr);
      }
      sh.s_thr[t] = thr;
      if (P.dbg_thr) P.dbg_thr[b * K + t] = thr;
    }
  }
  __syncthreads();

  if (tid == 0) {
    Plan pl{};
    if (bits) {
      atomicOr(P.status, bits);
      pl.j = -1;
      pl.mode = kModeFailed;
      P.n_acc[b] = -1;
      if (P.dbg_prob) P.dbg_prob[b] = __longlong_as_double(0x7ff8000000000000LL);
    } else {
      // Left-to-right scan: accept while u_t < thr_t (Algorithm 2 step 3).
      int j = K;
      for (int t = 0; t < K; ++t) {
        if (!((double)sh.s_u[t] < sh.s_thr[t])) {
          j = t;
          break;
        }
      }
      pl.j = j;
      if (j < K) {
        pl.mode = kModeResidual;
        pl.row_q = b * (K + 1) + j;
        pl.row_p = b * K + j;
        pl.m_q = sh.s_m[j];
        pl.s_q = sh.s_s[j];
        pl.m_p = sh.s_m[K + 1 + j];
        pl.s_p = sh.s_s[K + 1 + j];
        pl.u = sh.s_u[K];
      } else {
        pl.mode = kModeBonus;
        pl.row_q = b * (K + 1) + K;
        pl.row_p = -1;
        pl.m_q = sh.s_m[K];
        pl.s_q = sh.s_s[K];
        pl.u = sh.s_u[K + 1];
      }
      P.n_acc[b] = j;
    }
    P.plans[b] = pl;
    sh.j = pl.j;
  }
  __syncthreads();
  const int j = sh.j;
  for (int t = tid; t <= K; t += kThreads) {
    if (j < 0 || t > j)
      P.out_tokens[b * (K + 1) + t] = -1;
    else if (t < j)
      P.out_tokens[b * (K + 1) + t] = sh.s_tok[t];
  }
  if (P.dbg_thr && bits)
    for (int t = tid; t < K; t += kThreads)
      P.dbg_thr[b * K + t] = __longlong_as_double(0x7ff8000000000000LL);
  // Publish the plan: every thread's writes first, then the flag (release).
  __threadfence();
  __syncthreads();
  if (tid == 0) st_release(P.ready + b, 1u);
}

// ---------------------------------------------------------------- draw: shared element code

// Element weights of the draw, in float-float. For the residual,
// w = e_q * S_p - e_p * S_q on the positive set (q > p judged with the
// streaming-pass sums), which is the residual max(0, q - p) scaled by S_q S_p
// > 0; for the bonus (or the zero-residual fallback) w = e_q.
struct DrawRow {
  const unsigned char* rq;
  const unsigned char* rp;
  float mq, mp, sq, sp;
  float ih, il;
  bool unit_t;
};

SV_DEVINL DrawRow draw_row(const Params& P, const Plan& pl) {
  DrawRow d;
  d.rq = static_cast<const unsigned char*>(P.target) + (size_t)pl.row_q * P.V * P.es;
  d.rp = pl.mode == kModeResidual
             ? static_cast<const unsigned char*>(P.draft) + (size_t)pl.row_p * P.V * P.es
             : nullptr;
  d.mq = pl.m_q;
  d.mp = pl.m_p;
  d.sq = pl.s_q;
  d.sp = pl.s_p;
  d.ih = P.ih;
  d.il = P.il;
  d.unit_t = P.unit_t != 0;
  return d;
}

template <bool RESID>
SV_DEVINL void element_exps(const DrawRow& d, float lq, float lp, const float2* tab, ff& eq,
                            ff& ep, bool& in_pos) {
  const ff xq = scaled_diff(lq, d.mq, d.ih, d.il, d.unit_t);
  eq = exp_ff(xq.hi, xq.lo, tab);
  if constexpr (RESID) {
    const ff xp = scaled_diff(lp, d.mp, d.ih, d.il, d.unit_t);
    ep = exp_ff(xp.hi, xp.lo, tab);
    in_pos = __fmul_rn(eq.hi, d.sp) > __fmul_rn(ep.hi, d.sq);
  } else {
    ep = {0.f, 0.f};
    in_pos = false;
  }
}

template <int DT>
SV_DEVINL void load_run(const unsigned char* row, long long e, int V, bool vec_ok,
                        float (&x)[16 / (DT == 0 ? 2 : 4)]) {
  constexpr int kVec = 16 / (DT == 0 ? 2 : 4);
  if (vec_ok && e + kVec <= V) {
    const uint4 q = ld_global_nc_v4(row + e * (DT == 0 ? 2 : 4));
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
    if constexpr (DT == 0) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        x[2 * k] = bf16_lo(w[k]);
        x[2 * k + 1] = bf16_hi(w[k]);
      }
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k) x[k] = __uint_as_float(w[k]);
    }
  } else {
#pragma unroll
    for (int k = 0; k < kVec; ++k) x[k] = (e + k < V) ? load_elem<DT>(row, e + k) : neg_inf();
  }
}

// ---------------------------------------------------------------- draw: one chunk

template <int DT, bool RESID>
SV_DEVINL void partial_body(const Params& P, const DrawRow& d, const float2* tab, bool aligned,
                            long long b, int c) {
  constexpr int kVec = 16 / (DT == 0 ? 2 : 4);
  constexpr int kRuns = kSubElems / (32 * kVec);
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long e0 = ((long long)c * kSubPerChunk + w) * kSubElems;
  ff Sq{0.f, 0.f}, Sp{0.f, 0.f}, A{0.f, 0.f}, Bs{0.f, 0.f};
  if (e0 < P.V) {
#pragma unroll
    for (int r = 0; r < kRuns; ++r) {
      const long long e = e0 + (long long)r * 32 * kVec + lane * kVec;
      float xq[kVec], xp[kVec] = {};
      load_run<DT>(d.rq, e, P.V, aligned, xq);
      if constexpr (RESID) load_run<DT>(d.rp, e, P.V, aligned, xp);
#pragma unroll
      for (int k = 0; k < kVec; ++k) {
        ff eq, ep;
        bool pos;
        element_exps<RESID>(d, xq[k], xp[k], tab, eq, ep, pos);
        ff_accumulate(Sq, eq);
        if constexpr (RESID) {
          ff_accumulate(Sp, ep);
          if (pos) {
            ff_accumulate(A, eq);
            ff_accumulate(Bs, ep);
          }
        }
      }
    }
  }
  Sq = ff_warp_sum(ff_normalize(Sq));
  if constexpr (RESID) {
    Sp = ff_warp_sum(ff_normalize(Sp));
    A = ff_warp_sum(ff_normalize(A));
    Bs = ff_warp_sum(ff_normalize(Bs));
  }
  if (lane == 0) {
    float4* out = reinterpret_cast<float4*>(
        P.sub_part + (((size_t)b * P.nchunk + c) * kSubPerChunk + w) * 4);
    out[0] = make_float4(Sq.hi, Sq.lo, Sp.hi, Sp.lo);
    out[1] = make_float4(A.hi, A.lo, Bs.hi, Bs.lo);
  }
}

// ---------------------------------------------------------------- draw: finish of one sequence
// All arithmetic here is float-float (fp32 pairs): fp64 throughput is low on
// this part, and a block-wide fp64 operation costs as much as hundreds of
// fp32 ones.

SV_DEVINL ff ff_of(float x, float y) { return {x, y}; }

// Block sum of float-float values; result in every thread.
SV_DEVINL ff block_sum_ff(ff x, CtaShared& sh) {
  x = ff_warp_sum(x);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) sh.red_f[w] = x;
  __syncthreads();
  ff t{0.f, 0.f};
  for (int i = 0; i < kWarps; ++i) t = ff_add(t, sh.red_f[i]);
  return t;
}

// Block exclusive prefix of float-float values in thread order.
SV_DEVINL ff block_exclusive_ff(ff x, CtaShared& sh, ff* total) {
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  ff inc = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const ff y = ff_shfl_up(inc, o);
    if (l >= o) inc = ff_add(inc, y);
  }
  ff exc = ff_shfl_up(inc, 1);
  if (l == 0) exc = {0.f, 0.f};
  __syncthreads();
  if (l == 31) sh.red_f[w] = inc;
  __syncthreads();
  ff base{0.f, 0.f}, all{0.f, 0.f};
  for (int i = 0; i < kWarps; ++i) {
    if (i < w) base = ff_add(base, sh.red_f[i]);
    all = ff_add(all, sh.red_f[i]);
  }
  *total = all;
  return ff_add(base, exc);
}

// Weight of element e in the draw (0 outside the row or the positive set).
template <int DT>
SV_DEVINL ff draw_weight(const DrawRow& d, bool use_res, ff Sq, ff Sp, long long e, int V,
                         const float2* tab) {
  if (e >= V) return {0.f, 0.f};
  const float lq = load_elem<DT>(d.rq, e);
  ff eq, ep;
  bool pos;
  if (use_res) {
    const float lp = load_elem<DT>(d.rp, e);
    element_exps<true>(d, lq, lp, tab, eq, ep, pos);
    return pos ? ff_sub(ff_mul(ff_normalize(eq), Sp), ff_mul(ff_normalize(ep), Sq))
               : ff{0.f, 0.f};
  }
  element_exps<false>(d, lq, 0.f, tab, eq, ep, pos);
  return ff_normalize(eq);
}

template <int DT>
SV_DEVINL void finish_seq(const Params& P, long long b, const Plan& pl, CtaShared& sh) {
  const int tid = threadIdx.x;
  const int nsub = P.nchunk * kSubPerChunk;
  const float4* part = reinterpret_cast<const float4*>(P.sub_part + (size_t)b * nsub * 4);
  const bool resid = pl.mode == kModeResidual;
  const int run = (nsub + kThreads - 1) / kThreads;
  const int g0 = min(nsub, tid * run), g1 = min(nsub, g0 + run);

  // Totals over the row(s): S_q, S_p and the positive-set sums A, B.
  ff tq{0.f, 0.f}, tp{0.f, 0.f}, ta{0.f, 0.f}, tb{0.f, 0.f};
  for (int g = g0; g < g1; ++g) {
    const float4 x = __ldcg(part + 2 * g);
    tq = ff_add(tq, ff_of(x.x, x.y));
    if (resid) {
      const float4 y = __ldcg(part + 2 * g + 1);
      tp = ff_add(tp, ff_of(x.z, x.w));
      ta = ff_add(ta, ff_of(y.x, y.y));
      tb = ff_add(tb, ff_of(y.z, y.w));
    }
  }
  const ff Sq = block_sum_ff(tq, sh);
  ff Sp{0.f, 0.f}, A{0.f, 0.f}, Bt{0.f, 0.f};
  if (resid) {
    Sp = block_sum_ff(tp, sh);
    A = block_sum_ff(ta, sh);
    Bt = block_sum_ff(tb, sh);
  }
  // Residual mass sum max(0, q - p), scaled by S_q S_p; zero -> fall back to q.
  const bool use_res = resid && ff_sub(ff_mul(Sp, A), ff_mul(Sq, Bt)).hi > 0.f;
  auto mass = [&](int g) -> ff {
    if (use_res) {
      const float4 y = __ldcg(part + 2 * g + 1);
      return ff_sub(ff_mul(Sp, ff_of(y.x, y.y)), ff_mul(Sq, ff_of(y.z, y.w)));
    }
    const float4 x = __ldcg(part + 2 * g);
    return ff_of(x.x, x.y);
  };
  ff run_sum{0.f, 0.f};
  for (int g = g0; g < g1; ++g) run_sum = ff_add(run_sum, mass(g));
  ff total;
  const ff run_pref = block_exclusive_ff(run_sum, sh, &total);
  const ff tau = ff_mul_f(total, pl.u);

  // First sub-chunk whose cumulative mass passes tau.
  if (tid == 0) sh.g = INT_MAX;
  __syncthreads();
  {
    ff cum = run_pref;
    for (int g = g0; g < g1; ++g) {
      const ff mg = mass(g);
      const ff next = ff_add(cum, mg);
      if (mg.hi > 0.f && ff_gt(next, tau)) {
        atomicMin(&sh.g, g);
        break;
      }
      cum = next;
    }
  }
  __syncthreads();
  int gs = sh.g;
  const bool last_mode = gs == INT_MAX;
  __syncthreads();
  if (last_mode) {
    // u * total reached the end (u = 1): the last sub-chunk with positive mass.
    if (tid == 0) sh.g = -1;
    __syncthreads();
    for (int g = g1 - 1; g >= g0; --g) {
      if (mass(g).hi > 0.f) {
        atomicMax(&sh.g, g);
        break;
      }
    }
    __syncthreads();
    gs = sh.g;
  } else {
    ff cum = run_pref;
    for (int g = g0; g < g1; ++g) {
      if (g == gs) sh.s_pref = cum;
      cum = ff_add(cum, mass(g));
    }
    __syncthreads();
  }
  if (tid < 32 && gs >= 0) {
    // Warp 0: exact search inside sub-chunk gs, 16 consecutive elements per lane.
    const int lane = tid;
    const DrawRow d = draw_row(P, pl);
    const long long eb = (long long)gs * kSubElems + lane * 16;
    ff lsum{0.f, 0.f};
    for (int k = 0; k < 16; ++k)
      lsum = ff_add(lsum, draw_weight<DT>(d, use_res, Sq, Sp, eb + k, P.V, sh.tab));
    ff inc = lsum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const ff y = ff_shfl_up(inc, o);
      if (lane >= o) inc = ff_add(inc, y);
    }
    ff lpre = ff_shfl_up(inc, 1);
    if (lane == 0) lpre = {0.f, 0.f};
    int found = -1, lastk = -1;
    ff wfound{0.f, 0.f}, wlast{0.f, 0.f};
    ff cum = ff_add(sh.s_pref, lpre);
    for (int k = 0; k < 16; ++k) {
      const ff wk = draw_weight<DT>(d, use_res, Sq, Sp, eb + k, P.V, sh.tab);
      cum = ff_add(cum, wk);
      if (wk.hi > 0.f) {
        lastk = k;
        wlast = wk;
        if (!last_mode && found < 0 && ff_gt(cum, tau)) {
          found = k;
          wfound = wk;
        }
      }
    }
    const unsigned hit = __ballot_sync(0xffffffffu, found >= 0);
    int token;
    ff wt;
    if (hit) {
      const int src = __ffs(hit) - 1;
      token = (int)((long long)gs * kSubElems + src * 16 + __shfl_sync(0xffffffffu, found, src));
      wt = {__shfl_sync(0xffffffffu, wfound.hi, src), __shfl_sync(0xffffffffu, wfound.lo, src)};
    } else {
      // Last positive element of the sub-chunk (u = 1, or rounding at its end).
      const unsigned any = __ballot_sync(0xffffffffu, lastk >= 0);
      const int src = any ? 31 - __clz(any) : 0;
      const int kk = __shfl_sync(0xffffffffu, lastk, src);
      wt = {__shfl_sync(0xffffffffu, wlast.hi, src), __shfl_sync(0xffffffffu, wlast.lo, src)};
      token = (int)((long long)gs * kSubElems + src * 16 + (kk < 0 ? 0 : kk));
    }
    if (lane == 0) {
      P.out_tokens[b * (P.K + 1) + pl.j] = token;
      if (P.dbg_prob) P.dbg_prob[b] = ff_to_double(wt) / ff_to_double(total);
    }
  }
}

// ---------------------------------------------------------------- the persistent kernel

struct Item {
  bool stats;
  long long b;
  long long idx;
};

// Ticket -> work item: stats tickets of sequence s, then (after `lag`
// sequences) the draw tickets of sequence s - lag.
SV_DEVINL Item decode(const Params& P, unsigned long long t) {
  const long long NS = P.ns, NP = P.np, L = P.lag, B = P.B;
  const unsigned long long ph1 = (unsigned long long)(L * NS);
  if (t < ph1) return {true, (long long)(t / NS), (long long)(t % NS)};
  t -= ph1;
  const unsigned long long ph2 = (unsigned long long)((B - L) * (NS + NP));
  if (t < ph2) {
    const long long s = L + (long long)(t / (NS + NP));
    const long long o = (long long)(t % (NS + NP));
    if (o < NS) return {true, s, o};
    return {false, s - L, o - NS};
  }
  t -= ph2;
  return {false, (B - L) + (long long)(t / NP), (long long)(t % NP)};
}

SV_DEVINL unsigned atomic_add_acq_rel(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

template <int DT, bool ALIGNED>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) verify_kernel(Params P) {
  extern __shared__ __align__(128) unsigned char ring[];
  __shared__ CtaShared sh;
  const int tid = threadIdx.x;
  sh.tab[tid] = kSvExp2Table[tid];
  const unsigned long long total = (unsigned long long)P.B * (P.ns + P.np);
  uint32_t piece = 0, issued = 0;  // consumed / issued ring pieces (thread 0 issues)
  if (tid == 0) {
    if (ALIGNED) {
      for (int s = 0; s < kStages; ++s) mbar_init(&sh.full[s], 1);
      fence_barrier_init();
    }
    // One ticket of lookahead: the next streaming unit's bytes are in flight
    // while the current item is processed.
    sh.next = atomicAdd(P.ticket, 1ull);
    if (ALIGNED && sh.next < total) {
      const Item it = decode(P, sh.next);
      if (it.stats) stats_issue<DT>(P, it.b * P.ns + it.idx, ring, sh, issued);
    }
  }
  __syncthreads();
  for (;;) {
    const unsigned long long t = sh.next;
    if (t >= total) break;
    __syncthreads();  // everyone has read sh.next
    if (tid == 0) {
      const unsigned long long n = atomicAdd(P.ticket, 1ull);
      sh.next = n;
      if (ALIGNED && n < total) {
        const Item nt = decode(P, n);
        if (nt.stats) stats_issue<DT>(P, nt.b * P.ns + nt.idx, ring, sh, issued);
      }
    }
    const Item it = decode(P, t);
    const long long b = it.b;
    if (it.stats) {
      const long long u = b * P.ns + it.idx;
      if constexpr (ALIGNED) {
        if (!stats_consume_unit<DT>(P, u, ring, sh, piece)) {
          if (tid == 0) {
            atomicOr(P.status, kDevTimeout);
            // The current segment's pieces and the prefetched ones may still be
            // in flight: give them a bounded chance to land before exiting.
            for (uint32_t q = piece >= 2 ? piece - 2 : 0; q < issued; ++q)
              (void)mbar_wait(&sh.full[q % kStages], (q / kStages) & 1u);
          }
          return;
        }
      } else {
        stats_unit_plain<DT>(P, u, sh);
      }
      if (tid == 0) sh.flag = atomic_add_acq_rel(P.done_s + b, 1u) == (unsigned)(P.ns - 1);
      __syncthreads();
      if (sh.flag) scan_seq(P, b, sh);
    } else {
      if (tid == 0) {
        if (wait_flag(P.ready + b)) {
          const Plan* src = P.plans + b;
          Plan pl;
          pl.j = __ldcg(&src->j);
          pl.mode = __ldcg(&src->mode);
          pl.row_q = __ldcg(&src->row_q);
          pl.row_p = __ldcg(&src->row_p);
          pl.m_q = __ldcg(&src->m_q);
          pl.m_p = __ldcg(&src->m_p);
          pl.s_q = __ldcg(&src->s_q);
          pl.s_p = __ldcg(&src->s_p);
          pl.u = __ldcg(&src->u);
          sh.plan = pl;
        } else {
          atomicOr(P.status, kDevTimeout);
          sh.plan.mode = kModeFailed;
        }
      }
      __syncthreads();
      const Plan pl = sh.plan;
      if (pl.mode != kModeFailed) {
        const DrawRow d = draw_row(P, pl);
        if (pl.mode == kModeResidual)
          partial_body<DT, true>(P, d, sh.tab, ALIGNED, b, (int)it.idx);
        else
          partial_body<DT, false>(P, d, sh.tab, ALIGNED, b, (int)it.idx);
      }
      __syncthreads();  // all partial writes of this CTA precede the release below
      if (tid == 0) sh.flag = atomic_add_acq_rel(P.done_p + b, 1u) == (unsigned)(P.np - 1);
      __syncthreads();
      if (sh.flag && pl.mode != kModeFailed) finish_seq<DT>(P, b, pl, sh);
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------- host-side launch

namespace {
struct DeviceInfo {
  int sms = 0;
  int blocks_per_sm[4] = {0, 0, 0, 0};
  bool ready = false;
};
DeviceInfo g_dev[64];
std::mutex g_dev_mu;

template <int DT, bool AL>
cudaError_t setup_kernel(int* occ) {
  const int smem = AL ? kStages * kStageBytes : 0;
  cudaError_t e = cudaFuncSetAttribute(verify_kernel<DT, AL>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, verify_kernel<DT, AL>, kThreads, smem);
  if (e == cudaSuccess && *occ < 1) *occ = 1;
  return e;
}
}  // namespace

cudaError_t prepare_device(int device) {
  if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DeviceInfo& di = g_dev[device];
  if (di.ready) return cudaSuccess;
  cudaError_t e = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, device);
  if (e == cudaSuccess) e = setup_kernel<0, true>(&di.blocks_per_sm[0]);
  if (e == cudaSuccess) e = setup_kernel<0, false>(&di.blocks_per_sm[1]);
  if (e == cudaSuccess) e = setup_kernel<1, true>(&di.blocks_per_sm[2]);
  if (e == cudaSuccess) e = setup_kernel<1, false>(&di.blocks_per_sm[3]);
  if (e != cudaSuccess) return e;
  di.ready = true;
  return cudaSuccess;
}

int kernels_per_call() { return 1; }

cudaError_t launch_all(Params P, bool aligned, cudaStream_t st, const Events& ev) {
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return e;
  e = prepare_device(device);
  if (e != cudaSuccess) return e;
  const DeviceInfo& di = g_dev[device];
  const int variant = (P.dtype == 0 ? 0 : 2) + (aligned ? 0 : 1);
  long long grid = (long long)di.sms * di.blocks_per_sm[variant];
  const long long tickets = (long long)P.B * (P.ns + P.np);
  if (grid > tickets) grid = tickets;
  // Draw tickets of sequence b follow its stats tickets by about one wave of
  // the grid, so that its plan is normally ready when they are taken.
  long long lag = (grid + P.ns - 1) / P.ns + 1;
  P.lag = lag < P.B ? (int)lag : P.B;
  e = cudaMemsetAsync(P.ctrl, 0, P.ctrl_bytes, st);
  if (e != cudaSuccess) return e;
  // External records, so that the events become timing nodes when the stream
  // is being captured into a graph.
  if (ev.start) {
    e = cudaEventRecordWithFlags(ev.start, st, cudaEventRecordExternal);
    if (e != cudaSuccess) return e;
  }
  const int smem = aligned ? kStages * kStageBytes : 0;
  if (P.dtype == 0) {
    if (aligned)
      verify_kernel<0, true><<<(unsigned)grid, kThreads, smem, st>>>(P);
    else
      verify_kernel<0, false><<<(unsigned)grid, kThreads, smem, st>>>(P);
  } else {
    if (aligned)
      verify_kernel<1, true><<<(unsigned)grid, kThreads, smem, st>>>(P);
    else
      verify_kernel<1, false><<<(unsigned)grid, kThreads, smem, st>>>(P);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (ev.stats_done) e = cudaEventRecordWithFlags(ev.stats_done, st, cudaEventRecordExternal);
  if (e == cudaSuccess && ev.end) e = cudaEventRecordWithFlags(ev.end, st, cudaEventRecordExternal);
  return e;
}

}  // namespace sv
