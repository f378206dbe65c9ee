// Kernels of the verification step of speculative sampling (modified
// rejection sampling: §4.2 and Algorithm 2 of "Accelerating Large Language
// Model Decoding with Speculative Sampling", wikillm.com paper card).
//
// One call runs four kernels on the caller's stream:
//   1. stats      one streaming pass over all B(2K+1) logit rows: per (row,
//                 segment) the maximum m and sum_i 2^((l_i - m) log2(e)/T), the
//                 temperature transform of §4.2 "Decoding transforms";
//   2. scan       per sequence: combine the segments, gather the logits at the
//                 drafted tokens, thresholds min(1, q/p), first rejection j;
//   3. partials   per (sequence, 4096-element chunk) of the one row pair that
//                 the draw needs: float-float sums of exp((l - m)/T) (and of
//                 the residual's positive part), per 512-element sub-chunk;
//   4. finish     per sequence: exact inverse-CDF search for the drawn token.
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

// Block-wide combine; blockDim.x a multiple of 32, at most 1024. Result in thread 0.
SV_DEVINL void block_combine(float& m, float& s, float c2, float* red_m, float* red_s) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    ms_combine(m, s, m2, s2, c2);
  }
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) {
    red_m[w] = m;
    red_s[w] = s;
  }
  __syncthreads();
  if (w == 0) {
    const int nw = blockDim.x >> 5;
    m = l < nw ? red_m[l] : neg_inf();
    s = l < nw ? red_s[l] : 0.0f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
      const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
      ms_combine(m, s, m2, s2, c2);
    }
  }
  __syncthreads();
}

// ---------------------------------------------------------------- 1. stats, bulk-copy path
//
// Persistent CTAs, each owning a contiguous range of units (row segments) in
// sequence-major order. Thread 0 streams the range through a ring of kStages
// 16 KB shared-memory stages with 1-D bulk copies (cp.async.bulk, completion
// on an mbarrier); all 256 threads consume each stage with 16-byte shared
// loads. Per thread: the stage's local max (packed bf16x2 max for bf16), a
// rescale of the four running sums only when the max grows, then one FFMA and
// one MUFU ex2 per element against H = fl(m * c2). The rounding residual of H
// is folded back in once per unit.

constexpr int kStatsThreads = 256;
constexpr int kStageBytes = 16384;
constexpr int kStages = 4;
constexpr int kVecPerThread = kStageBytes / 16 / kStatsThreads;  // 4

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

// Per-thread (m, s) of a finished unit, with H's rounding residual folded in.
SV_DEVINL float thread_sum(float m_run, float H, const float (&acc)[4], bool nan_seen, float c2) {
  if (m_run == neg_inf()) return nan_seen ? __int_as_float(0x7fc00000) : 0.0f;
  float s = (acc[0] + acc[1]) + (acc[2] + acc[3]);
  const float L = __fmaf_rn(m_run, c2, -H);  // m*c2 - H exactly (to fp32)
  s *= __fmaf_rn(-L, kLn2, 1.0f);            // 2^-L to first order (|L| < 1e-5)
  return nan_seen ? __int_as_float(0x7fc00000) : s;
}

template <int DT>
__global__ void __launch_bounds__(kStatsThreads) stats_tma_kernel(Params P) {
  extern __shared__ __align__(128) unsigned char sbuf[];
  __shared__ __align__(8) uint64_t full[kStages];
  __shared__ float red_m[kStatsThreads / 32], red_s[kStatsThreads / 32];
  constexpr int kEs = DT == 0 ? 2 : 4;
  constexpr int kStageElems = kStageBytes / kEs;
  const int tid = threadIdx.x;
  const long long u0 = (long long)blockIdx.x * P.n_units / gridDim.x;
  const long long u1 = (long long)(blockIdx.x + 1) * P.n_units / gridDim.x;
  if (u0 >= u1) return;

  auto unit_len = [&](long long u) -> int {
    const int seg = (int)(u % P.nseg);
    return seg == P.nseg - 1 ? P.V - seg * P.seg_elems : P.seg_elems;
  };

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&full[s], 1);
    fence_barrier_init();
  }
  __syncthreads();

  // Producer cursor (thread 0): next piece = unit pu, element offset poff.
  long long pu = u0;
  int poff = 0;
  uint32_t issued = 0;
  auto issue = [&](int stage) {
    if (pu >= u1) return;
    ++issued;
    const int len = unit_len(pu);
    const int n = min(kStageElems, len - poff);
    const long long row = pu / P.nseg;
    const int seg = (int)(pu % P.nseg);
    const unsigned char* src = row_base(P, row / P.rows_per_seq, (int)(row % P.rows_per_seq)) +
                               ((size_t)seg * P.seg_elems + poff) * kEs;
    const uint32_t bytes = (uint32_t)n * kEs;
    mbar_arrive_expect_tx(&full[stage], bytes);
    bulk_copy_g2s(sbuf + stage * kStageBytes, src, bytes, &full[stage]);
    poff += n;
    if (poff >= len) {
      ++pu;
      poff = 0;
    }
  };
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) issue(s);
  }

  const float c2 = P.c2;
  long long cu = u0;
  int coff = 0;
  uint32_t piece = 0;
  float m_run = neg_inf(), H = neg_inf();
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  bool nan_seen = false, timed_out = false;
  const uint32_t fill = DT == 0 ? 0xff80ff80u : 0xff800000u;  // -inf

  while (cu < u1) {
    const int stage = (int)(piece % kStages);
    const uint32_t parity = (piece / kStages) & 1u;
    const int len = unit_len(cu);
    const int n = min(kStageElems, len - coff);
    if (!mbar_wait(&full[stage], parity)) timed_out = true;
    const unsigned char* buf = sbuf + stage * kStageBytes;
    const int nvec = n * kEs / 16;
    uint4 v[kVecPerThread];
#pragma unroll
    for (int i = 0; i < kVecPerThread; ++i) {
      const int idx = tid + i * kStatsThreads;
      v[i] = idx < nvec ? ld_shared_v4(buf + idx * 16) : make_uint4(fill, fill, fill, fill);
    }
    stats_consume<DT>(v, m_run, H, acc, nan_seen, c2);
    coff += n;
    if (coff >= len) {
      float s = thread_sum(m_run, H, acc, nan_seen, c2);
      float m = m_run;
      block_combine(m, s, c2, red_m, red_s);
      if (tid == 0) P.seg_part[cu] = make_float2(m, s);
      m_run = neg_inf();
      H = neg_inf();
      acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
      nan_seen = false;
      ++cu;
      coff = 0;
    }
    // Every thread is done with this stage; a timed-out wait anywhere aborts the CTA.
    if (__syncthreads_or(timed_out)) {
      if (tid == 0) {
        atomicOr(P.status, kDevTimeout);
        // Give the copies still in flight a bounded chance to land before exiting.
        for (uint32_t p = piece; p < issued; ++p)
          (void)mbar_wait(&full[p % kStages], (p / kStages) & 1u);
      }
      return;
    }
    if (tid == 0) issue(stage);
    ++piece;
  }
}

// ---------------------------------------------------------------- 1'. stats, plain-load path
// For rows that are not 16-byte aligned: one CTA per unit at a time, two
// passes over the unit with element loads (max, then sum).

template <int DT>
__global__ void __launch_bounds__(kStatsThreads) stats_plain_kernel(Params P) {
  __shared__ float red_m[kStatsThreads / 32], red_s[kStatsThreads / 32];
  const float c2 = P.c2;
  for (long long u = blockIdx.x; u < P.n_units; u += gridDim.x) {
    const long long row = u / P.nseg;
    const int seg = (int)(u % P.nseg);
    const int len = seg == P.nseg - 1 ? P.V - seg * P.seg_elems : P.seg_elems;
    const unsigned char* rb = row_base(P, row / P.rows_per_seq, (int)(row % P.rows_per_seq));
    const long long e0 = (long long)seg * P.seg_elems;
    float m = neg_inf();
    bool nan_seen = false;
    for (int i = threadIdx.x; i < len; i += blockDim.x) {
      const float l = load_elem<DT>(rb, e0 + i);
      nan_seen |= (l != l);
      m = fmaxf(m, l);
    }
    float s = 0.f;
    if (m != neg_inf()) {
      for (int i = threadIdx.x; i < len; i += blockDim.x)
        s += ex2_fast((load_elem<DT>(rb, e0 + i) - m) * c2);
    }
    if (nan_seen) s = __int_as_float(0x7fc00000);
    block_combine(m, s, c2, red_m, red_s);
    if (threadIdx.x == 0) P.seg_part[u] = make_float2(m, s);
  }
}

// ---------------------------------------------------------------- 2. scan

constexpr int kScanThreads = 128;

__global__ void __launch_bounds__(kScanThreads) scan_kernel(Params P) {
  __shared__ float s_m[2 * kMaxK + 1];
  __shared__ float s_s[2 * kMaxK + 1];
  __shared__ double s_lse[2 * kMaxK + 1];
  __shared__ double s_thr[kMaxK];
  __shared__ unsigned s_bits;
  __shared__ int s_j;
  const long long b = blockIdx.x;
  const int tid = threadIdx.x, K = P.K, R = P.rows_per_seq;
  if (tid == 0) s_bits = 0;
  __syncthreads();

  // Row statistics: m = max over segments, S = sum of rescaled segment sums.
  for (int r = tid; r < R; r += blockDim.x) {
    const float2* part = P.seg_part + ((long long)b * R + r) * P.nseg;
    float m = neg_inf();
    bool nan_seen = false;
    for (int g = 0; g < P.nseg; ++g) {
      const float2 ps = part[g];
      m = fmaxf(m, ps.x);
      nan_seen |= (ps.y != ps.y);
    }
    double S = 0.0;
    unsigned bits = 0;
    if (nan_seen) {
      bits = kDevNonfinite;
    } else if (m == neg_inf()) {
      bits = kDevEmptyRow;
    } else {
      for (int g = 0; g < P.nseg; ++g) {
        const float2 ps = part[g];
        if (ps.x != neg_inf()) S += (double)ps.y * (double)exp2f((ps.x - m) * P.c2);
      }
    }
    if (bits) atomicOr(&s_bits, bits);
    s_m[r] = m;
    s_s[r] = (float)S;
    s_lse[r] = bits ? __longlong_as_double(0x7ff8000000000000LL) : (double)m * P.inv_t + log(S);
  }
  for (int t = tid; t < K; t += blockDim.x) {
    const int x = P.tokens[b * K + t];
    if (x < 0 || x >= P.V) atomicOr(&s_bits, kDevTokenRange);
  }
  for (int t = tid; t < K + 2; t += blockDim.x) {
    const float u = P.uniforms[b * (K + 2) + t];
    if (!(u >= 0.0f && u <= 1.0f)) atomicOr(&s_bits, kDevUniformRange);
  }
  __syncthreads();
  const unsigned bits = s_bits;
  if (P.dbg_lse)
    for (int r = tid; r < R; r += blockDim.x) P.dbg_lse[b * R + r] = s_lse[r];
  if (bits) {
    for (int t = tid; t <= K; t += blockDim.x) P.out_tokens[b * (K + 1) + t] = -1;
    if (P.dbg_thr)
      for (int t = tid; t < K; t += blockDim.x)
        P.dbg_thr[b * K + t] = __longlong_as_double(0x7ff8000000000000LL);
    if (tid == 0) {
      atomicOr(P.status, bits);
      Plan pl{};
      pl.j = -1;
      pl.mode = kModeFailed;
      P.plans[b] = pl;
      P.n_acc[b] = -1;
      if (P.dbg_prob) P.dbg_prob[b] = __longlong_as_double(0x7ff8000000000000LL);
    }
    return;
  }

  // Thresholds min(1, q(x~)/p(x~)) at the drafted tokens (§4.2), in fp64:
  // log q(x) - log p(x) = (lq - lp)/T - (lse_q - lse_p).
  for (int t = tid; t < K; t += blockDim.x) {
    const int x = P.tokens[b * K + t];
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
      const double lr = ((double)lq - (double)lp) * P.inv_t - (s_lse[t] - s_lse[K + 1 + t]);
      thr = lr >= 0.0 ? 1.0 : exp(lr);
    }
    s_thr[t] = thr;
    if (P.dbg_thr) P.dbg_thr[b * K + t] = thr;
  }
  __syncthreads();

  // Left-to-right scan: accept while u_t < thr_t (Algorithm 2 step 3).
  if (tid == 0) {
    const float* u = P.uniforms + b * (K + 2);
    int j = K;
    for (int t = 0; t < K; ++t) {
      if (!((double)u[t] < s_thr[t])) {
        j = t;
        break;
      }
    }
    Plan pl{};
    pl.j = j;
    if (j < K) {
      pl.mode = kModeResidual;
      pl.row_q = b * (K + 1) + j;
      pl.row_p = b * K + j;
      pl.m_q = s_m[j];
      pl.s_q = s_s[j];
      pl.m_p = s_m[K + 1 + j];
      pl.s_p = s_s[K + 1 + j];
      pl.u = u[K];
    } else {
      pl.mode = kModeBonus;
      pl.row_q = b * (K + 1) + K;
      pl.row_p = -1;
      pl.m_q = s_m[K];
      pl.s_q = s_s[K];
      pl.m_p = 0.f;
      pl.s_p = 0.f;
      pl.u = u[K + 1];
    }
    P.plans[b] = pl;
    P.n_acc[b] = j;
    s_j = j;
  }
  __syncthreads();
  const int j = s_j;
  for (int t = tid; t <= K; t += blockDim.x) {
    if (t < j)
      P.out_tokens[b * (K + 1) + t] = P.tokens[b * K + t];
    else if (t > j)
      P.out_tokens[b * (K + 1) + t] = -1;
  }
}

// ---------------------------------------------------------------- 3./4. draw: shared element code

constexpr int kSampleThreads = 256;

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

template <int DT, bool RESID>
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

// ---------------------------------------------------------------- 3. partials

template <int DT, bool RESID>
SV_DEVINL void partial_body(const Params& P, const Plan& pl, const float2* tab, bool aligned,
                            long long b, int c) {
  constexpr int kVec = 16 / (DT == 0 ? 2 : 4);
  constexpr int kRuns = kSubElems / (32 * kVec);
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long e0 = ((long long)c * kSubPerChunk + w) * kSubElems;
  DrawRow d;
  d.rq = static_cast<const unsigned char*>(P.target) + (size_t)pl.row_q * P.V * P.es;
  d.rp = RESID ? static_cast<const unsigned char*>(P.draft) + (size_t)pl.row_p * P.V * P.es
               : nullptr;
  d.mq = pl.m_q;
  d.mp = pl.m_p;
  d.sq = pl.s_q;
  d.sp = pl.s_p;
  d.ih = P.ih;
  d.il = P.il;
  d.unit_t = P.unit_t != 0;
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
        element_exps<DT, RESID>(d, xq[k], RESID ? xp[k] : 0.f, tab, eq, ep, pos);
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
    float2* out = P.sub_part + (((size_t)b * P.nchunk + c) * kSubPerChunk + w) * 4;
    out[0] = make_float2(Sq.hi, Sq.lo);
    out[1] = make_float2(Sp.hi, Sp.lo);
    out[2] = make_float2(A.hi, A.lo);
    out[3] = make_float2(Bs.hi, Bs.lo);
  }
}

template <int DT>
__global__ void __launch_bounds__(kSampleThreads) partials_kernel(Params P, int aligned) {
  __shared__ float2 tab[256];
  const long long b = blockIdx.x / P.nchunk;
  const int c = (int)(blockIdx.x % P.nchunk);
  const Plan pl = P.plans[b];
  if (pl.mode == kModeFailed) return;
  tab[threadIdx.x] = kSvExp2Table[threadIdx.x];
  __syncthreads();
  if (pl.mode == kModeResidual)
    partial_body<DT, true>(P, pl, tab, aligned != 0, b, c);
  else
    partial_body<DT, false>(P, pl, tab, aligned != 0, b, c);
}

// ---------------------------------------------------------------- 4. finish

SV_DEVINL double ffd(float2 v) { return (double)v.x + (double)v.y; }

SV_DEVINL double warp_sum_d(double x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Block sum of doubles (256 threads); result in every thread.
SV_DEVINL double block_sum_d(double x, double* red) {
  x = warp_sum_d(x);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = x;
  __syncthreads();
  double t = 0.0;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) t += red[i];
  return t;
}

// Block exclusive prefix of doubles in thread order (256 threads).
SV_DEVINL double block_exclusive_d(double x, double* red, double* total) {
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  double inc = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double y = __shfl_up_sync(0xffffffffu, inc, o);
    if (l >= o) inc += y;
  }
  __syncthreads();
  if (l == 31) red[w] = inc;
  __syncthreads();
  double base = 0.0, all = 0.0;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) {
    if (i < w) base += red[i];
    all += red[i];
  }
  *total = all;
  return base + inc - x;
}

template <int DT>
__global__ void __launch_bounds__(kSampleThreads) finish_kernel(Params P, int aligned) {
  __shared__ float2 tab[256];
  __shared__ double red[kSampleThreads / 32];
  __shared__ int s_g;
  __shared__ double s_pref;
  const long long b = blockIdx.x;
  const Plan pl = P.plans[b];
  if (pl.mode == kModeFailed) return;
  const int tid = threadIdx.x;
  tab[tid] = kSvExp2Table[tid];
  if (tid == 0) s_g = INT_MAX;
  __syncthreads();

  const int nsub = P.nchunk * kSubPerChunk;
  const float2* part = P.sub_part + (size_t)b * nsub * 4;
  const bool resid = pl.mode == kModeResidual;
  const int run = (nsub + kSampleThreads - 1) / kSampleThreads;
  const int g0 = min(nsub, tid * run), g1 = min(nsub, g0 + run);

  // Totals over the row(s): S_q, S_p and the positive-set sums A, B.
  double tq = 0, tp = 0, ta = 0, tb = 0;
  for (int g = g0; g < g1; ++g) {
    tq += ffd(part[g * 4 + 0]);
    if (resid) {
      tp += ffd(part[g * 4 + 1]);
      ta += ffd(part[g * 4 + 2]);
      tb += ffd(part[g * 4 + 3]);
    }
  }
  const double Sq = block_sum_d(tq, red);
  double Sp = 0, A = 0, Bt = 0;
  if (resid) {
    Sp = block_sum_d(tp, red);
    A = block_sum_d(ta, red);
    Bt = block_sum_d(tb, red);
  }
  // Residual mass sum max(0, q - p), scaled by S_q S_p; zero -> fall back to q.
  const bool use_res = resid && (Sp * A - Sq * Bt > 0.0);
  auto mass = [&](int g) -> double {
    return use_res ? Sp * ffd(part[g * 4 + 2]) - Sq * ffd(part[g * 4 + 3]) : ffd(part[g * 4 + 0]);
  };
  double run_sum = 0.0;
  for (int g = g0; g < g1; ++g) run_sum += mass(g);
  double total;
  const double run_pref = block_exclusive_d(run_sum, red, &total);
  const double tau = (double)pl.u * total;

  // First sub-chunk whose cumulative mass passes tau.
  {
    double cum = run_pref;
    for (int g = g0; g < g1; ++g) {
      const double mg = mass(g);
      if (mg > 0.0 && cum + mg > tau) {
        atomicMin(&s_g, g);
        break;
      }
      cum += mg;
    }
  }
  __syncthreads();
  int gs = s_g;
  bool last_mode = gs == INT_MAX;
  if (last_mode) {
    // u * total reached the end (u = 1): the last sub-chunk with positive mass.
    __syncthreads();
    if (tid == 0) s_g = -1;
    __syncthreads();
    for (int g = g1 - 1; g >= g0; --g) {
      if (mass(g) > 0.0) {
        atomicMax(&s_g, g);
        break;
      }
    }
    __syncthreads();
    gs = s_g;
  } else {
    double cum = run_pref;
    for (int g = g0; g < g1; ++g) {
      if (g == gs) s_pref = cum;
      cum += mass(g);
    }
  }
  __syncthreads();
  if (tid >= 32 || gs < 0) return;

  // Warp 0: exact search inside sub-chunk gs, 16 consecutive elements per lane.
  const int lane = tid;
  DrawRow d;
  d.rq = static_cast<const unsigned char*>(P.target) + (size_t)pl.row_q * P.V * P.es;
  d.rp = resid ? static_cast<const unsigned char*>(P.draft) + (size_t)pl.row_p * P.V * P.es
               : nullptr;
  d.mq = pl.m_q;
  d.mp = pl.m_p;
  d.sq = pl.s_q;
  d.sp = pl.s_p;
  d.ih = P.ih;
  d.il = P.il;
  d.unit_t = P.unit_t != 0;
  const long long eb = (long long)gs * kSubElems + lane * 16;
  double wv[16];
  double lsum = 0.0;
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const long long e = eb + k;
    double wk = 0.0;
    if (e < P.V) {
      const float lq = load_elem<DT>(d.rq, e);
      ff eq, ep;
      bool pos;
      if (use_res) {
        const float lp = load_elem<DT>(d.rp, e);
        element_exps<DT, true>(d, lq, lp, tab, eq, ep, pos);
        if (pos) wk = ff_to_double(eq) * Sp - ff_to_double(ep) * Sq;
      } else {
        element_exps<DT, false>(d, lq, 0.f, tab, eq, ep, pos);
        wk = ff_to_double(eq);
      }
    }
    wv[k] = wk;
    lsum += wk;
  }
  double lpre = lsum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double y = __shfl_up_sync(0xffffffffu, lpre, o);
    if (lane >= o) lpre += y;
  }
  lpre -= lsum;  // exclusive

  int found = -1;
  double wfound = 0.0;
  if (!last_mode) {
    double cum = s_pref + lpre;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      cum += wv[k];
      if (found < 0 && wv[k] > 0.0 && cum > tau) {
        found = k;
        wfound = wv[k];
      }
    }
  }
  unsigned hit = __ballot_sync(0xffffffffu, found >= 0);
  int token;
  double wt;
  if (hit) {
    const int src = __ffs(hit) - 1;
    token = (int)((long long)gs * kSubElems + src * 16 + __shfl_sync(0xffffffffu, found, src));
    wt = __shfl_sync(0xffffffffu, wfound, src);
  } else {
    // Last positive element of the sub-chunk (u = 1, or rounding at its end).
    int lastk = -1;
#pragma unroll
    for (int k = 0; k < 16; ++k)
      if (wv[k] > 0.0) lastk = k;
    const unsigned any = __ballot_sync(0xffffffffu, lastk >= 0);
    const int src = any ? 31 - __clz(any) : 0;
    const int kk = __shfl_sync(0xffffffffu, lastk, src);
    double wl = 0.0;
#pragma unroll
    for (int k = 0; k < 16; ++k)
      if (k == lastk) wl = wv[k];
    wt = __shfl_sync(0xffffffffu, wl, src);
    token = (int)((long long)gs * kSubElems + src * 16 + (kk < 0 ? 0 : kk));
  }
  if (lane == 0) {
    P.out_tokens[b * (P.K + 1) + pl.j] = token;
    if (P.dbg_prob) P.dbg_prob[b] = wt / total;
  }
}

// ---------------------------------------------------------------- host-side launch

namespace {
struct DeviceInfo {
  int sms = 0;
  int stats_blocks_per_sm = 0;
  bool ready = false;
};
DeviceInfo g_dev[64];
std::mutex g_dev_mu;
}  // namespace

cudaError_t prepare_device(int device) {
  if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DeviceInfo& di = g_dev[device];
  if (di.ready) return cudaSuccess;
  cudaError_t e = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, device);
  if (e != cudaSuccess) return e;
  const int smem = kStages * kStageBytes;
  e = cudaFuncSetAttribute(stats_tma_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(stats_tma_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int occ = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, stats_tma_kernel<0>, kStatsThreads, smem);
  if (e != cudaSuccess) return e;
  di.stats_blocks_per_sm = occ > 0 ? occ : 1;
  di.ready = true;
  return cudaSuccess;
}

int kernels_per_call() { return 4; }

template <int DT>
static cudaError_t launch_typed(const Params& P, bool aligned, cudaStream_t st, const DeviceInfo& di,
                                const Events& ev) {
  if (aligned) {
    long long grid = (long long)di.sms * di.stats_blocks_per_sm;
    if (grid > P.n_units) grid = P.n_units;
    stats_tma_kernel<DT><<<(unsigned)grid, kStatsThreads, kStages * kStageBytes, st>>>(P);
  } else {
    long long grid = (long long)di.sms * 4;
    if (grid > P.n_units) grid = P.n_units;
    stats_plain_kernel<DT><<<(unsigned)grid, kStatsThreads, 0, st>>>(P);
  }
  if (ev.stats_done && cudaEventRecord(ev.stats_done, st) != cudaSuccess) return cudaGetLastError();
  scan_kernel<<<(unsigned)P.B, kScanThreads, 0, st>>>(P);
  partials_kernel<DT><<<(unsigned)((long long)P.B * P.nchunk), kSampleThreads, 0, st>>>(P, aligned ? 1 : 0);
  finish_kernel<DT><<<(unsigned)P.B, kSampleThreads, 0, st>>>(P, aligned ? 1 : 0);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess && ev.end) e = cudaEventRecord(ev.end, st);
  return e;
}

cudaError_t launch_all(const Params& P, bool aligned, cudaStream_t st, const Events& ev) {
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return e;
  e = prepare_device(device);
  if (e != cudaSuccess) return e;
  if (ev.start) {
    e = cudaEventRecord(ev.start, st);
    if (e != cudaSuccess) return e;
  }
  e = cudaMemsetAsync(P.status, 0, sizeof(unsigned), st);
  if (e != cudaSuccess) return e;
  const DeviceInfo& di = g_dev[device];
  return P.dtype == 0 ? launch_typed<0>(P, aligned, st, di, ev)
                      : launch_typed<1>(P, aligned, st, di, ev);
}

}  // namespace sv
