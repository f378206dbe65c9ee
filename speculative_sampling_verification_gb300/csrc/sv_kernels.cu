// Kernels of the verification step of speculative sampling (modified
// rejection sampling: §4.2 and Algorithm 2 of "Accelerating Large Language
// Model Decoding with Speculative Sampling", wikillm.com paper card).
//
// The verification step takes one of two launch shapes, chosen per call by
// the bytes it streams:
//
//   stats_kernel, then the draw (small and very large calls). stats_kernel has
//       one warp per row segment (at most 32 KB, sequence-major so that
//       sequences complete one after another): each lane keeps eight 16-byte
//       loads in flight per round and reduces its share to the segment's
//       maximum m and sum_i 2^((l_i - m) log2(e)/T), the temperature transform
//       of §4.2 "Decoding transforms", with no shared memory and no barrier.
//       The warp that counts a row's last segment combines the row; the warp
//       that counts a sequence's last row runs its scan (scan_warp): logits at
//       the drafted tokens, thresholds min(1, q/p) in float-float, the first
//       rejection j (Algorithm 2 step 3) and the plan of the draw.
//       draw_sum_kernel, a programmatic dependent of stats_kernel, has one
//       CTA per chunk of the row pair the draw needs (target and draft row j
//       for the residual (q - p)_+, or target row K for the bonus token,
//       Algorithm 2 step 4): each warp sums one sub-chunk in float-float and
//       leaves. draw_finish_kernel, one CTA per sequence, then runs the
//       inverse-CDF search for the token.
//   fused_kernel (mid-sized calls). The same warp and chunk code in one
//       launch: CTAs take tickets, streaming items first, then draw chunks,
//       each of which waits (bounded) for its sequence's plan.
//
// Hand-offs use acquire-release counters ("the last to arrive does the
// follow-up"); only the fused kernel's draw CTAs ever wait, and every wait
// gives up after a fixed time.
#include <cfloat>
#include <math_constants.h>
#include <climits>
#include <type_traits>
#include <cstdint>
#include <atomic>
#include <map>
#include <mutex>

#include "sv_device.cuh"
#include "sv_internal.h"

// This file is compiled as several translation units, in parallel: SV_TU
// selects which host launchers (and so which kernel instantiations) a unit
// holds: 1 the verification and the sampler, 2 greedy mode and top-k, 3 the
// nucleus path; 0 (the default) all of them.
#ifndef SV_TU
#define SV_TU 0
#endif
#define SV_TU_HAS(n) (SV_TU == 0 || SV_TU == (n))

namespace sv {

constexpr unsigned kDevTokenRange = 16, kDevNonfinite = 32, kDevEmptyRow = 64,
                   kDevUniformRange = 128, kDevTimeout = 256;
constexpr float kLn2 = 0.693147180559945309f;

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

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

// ---------------------------------------------------------------- per-CTA shared state of the draw

struct CtaShared {
  float2 tab[256];  // 2^(j/256), head + tail
  float2 tab1k[1024];  // 2^(j/1024), head + tail (the fast exponential)
  ff red4[kWarps][4];
  ff s_pref;
  Plan plan;
  unsigned bits;
  int j, g, flag;
};

// ---------------------------------------------------------------- (max, sum) pairs
// A pair (m, s) stands for the sum s * 2^(m c2) of 2^(l_i c2) terms; s is
// NaN when a NaN (or +inf) entry was seen; m = -inf with s = 0 means "no
// finite entry yet".

// Warp-wide combine of one pair per lane with the accurate exp2f: the
// maximum first, then every lane's sum rescaled to it. All lanes get the
// result.
SV_DEVINL float2 warp_combine_pairs(float m, float s, float c2) {
  float M = m;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  if (M != neg_inf() && M != m) s = (m == neg_inf()) ? s * 0.0f : s * exp2f((m - M) * c2);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  return make_float2(M, s);
}

// ---------------------------------------------------------------- stats: one warp, one segment
//
// A unit is one segment (at most 32 KB) of one row, reduced by one warp with
// no shared memory and no barrier. Per round each lane holds eight 16-byte
// vectors. It takes their max (packed bf16x2 max for bf16), rescales its
// four running sums when the max grows, then spends one FFMA and one MUFU
// ex2 per element against H = fl(m * c2). The lanes are then combined: the
// warp maximum M first, then every lane's sum scaled by 2^(H - M c2), which
// also folds the rounding residual of H back in.

constexpr int kStatsThreads = 128;
constexpr int kStatsWarps = kStatsThreads / 32;
constexpr int kStatsCtasPerSm = 8;
constexpr int kStatsVec = 8;  // 16-byte vectors per lane per round

template <int DT, int N>
SV_DEVINL bool any_nan(const uint4 (&v)[N]) {
  bool bad = false;
#pragma unroll
  for (int i = 0; i < N; ++i) {
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

template <int DT, int N>
SV_DEVINL void stats_consume(const uint4 (&v)[N], float& m_run, float& H,
                             float2 (&acc)[2], bool& nan_seen, float c2) {
  float lm;
  if constexpr (DT == 0) {
    uint32_t mx = bf16x2_max(bf16x2_max(v[0].x, v[0].y), bf16x2_max(v[0].z, v[0].w));
#pragma unroll
    for (int i = 1; i < N; ++i)
      mx = bf16x2_max(mx, bf16x2_max(bf16x2_max(v[i].x, v[i].y), bf16x2_max(v[i].z, v[i].w)));
    lm = fmaxf(bf16_lo(mx), bf16_hi(mx));
  } else {
    lm = neg_inf();
#pragma unroll
    for (int i = 0; i < N; ++i)
      lm = fmaxf(lm, fmaxf(fmaxf(__uint_as_float(v[i].x), __uint_as_float(v[i].y)),
                           fmaxf(__uint_as_float(v[i].z), __uint_as_float(v[i].w))));
  }
  if (lm > m_run) {
    const float Hn = lm * c2;
    const float2 f = f2(ex2_fast(H - Hn));
    acc[0] = f2_mul(acc[0], f);
    acc[1] = f2_mul(acc[1], f);
    m_run = lm;
    H = Hn;
  }
  if (m_run == neg_inf()) {  // only -inf (or NaN) entries so far
    nan_seen |= any_nan<DT, N>(v);
    return;
  }
  const float2 c2p = f2(c2), nH = f2(-H);
#pragma unroll
  for (int i = 0; i < N; ++i) {
    const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
    if constexpr (DT == 0) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 a = f2_fma(make_float2(bf16_lo(w[k]), bf16_hi(w[k])), c2p, nH);
        acc[k & 1] = f2_add(acc[k & 1], make_float2(ex2_fast(a.x), ex2_fast(a.y)));
      }
    } else {
#pragma unroll
      for (int k = 0; k < 4; k += 2) {
        const float2 a =
            f2_fma(make_float2(__uint_as_float(w[k]), __uint_as_float(w[k + 1])), c2p, nH);
        acc[k >> 1] = f2_add(acc[k >> 1], make_float2(ex2_fast(a.x), ex2_fast(a.y)));
      }
    }
  }
}

// Warp-wide (max, sum) of the lanes' running statistics; all lanes get it.
SV_DEVINL float2 warp_stats(float m_run, float H, const float2 (&acc)[2], bool nan_seen, float c2) {
  float M = m_run;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float s = 0.0f;
  if (m_run != neg_inf()) {
    s = (acc[0].x + acc[0].y) + (acc[1].x + acc[1].y);
    // 2^(H - M c2): to first order when m_run is the maximum (|H - M c2| is
    // below an ulp of H), else by the hardware exp2.
    const float E = __fmaf_rn(-M, c2, H);
    s *= (m_run == M) ? __fmaf_rn(E, kLn2, 1.0f) : ex2_fast(E);
  }
  if (nan_seen) s = __int_as_float(0x7fc00000);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  return make_float2(M, s);
}

SV_DEVINL int unit_len(const Params& P, long long u) {
  const int seg = (int)(u % P.nseg);
  return seg == P.nseg - 1 ? P.V - seg * P.seg_elems : P.seg_elems;
}

SV_DEVINL const unsigned char* unit_row(const Params& P, long long u) {
  const long long row = u / P.nseg;
  return row_base(P, row / P.rows_per_seq, (int)(row % P.rows_per_seq));
}

// Vector-load path (16-byte aligned rows): the segment's 16-byte vectors,
// eight per lane in flight at a time, streamed past L1.
template <int DT>
SV_DEVINL float2 stats_warp_vec(const Params& P, long long u, int lane) {
  constexpr int kEs = DT == 0 ? 2 : 4;
  const int len = unit_len(P, u);
  const unsigned char* base = unit_row(P, u) + (size_t)(u % P.nseg) * P.seg_elems * kEs;
  const int nvec = len * kEs / 16;
  const float c2 = P.c2;
  const uint32_t fill = DT == 0 ? 0xff80ff80u : 0xff800000u;  // -inf
  float m_run = neg_inf(), H = neg_inf();
  float2 acc[2] = {f2(0.0f), f2(0.0f)};
  bool nan_seen = false;
  if constexpr (DT == 0) {
    // bf16 carries twice the elements per byte of fp32, so a round's arithmetic
    // takes twice as long: two half-rounds of four vectors alternate, the next
    // one's loads issued before the current one's arithmetic, so that the
    // lane's loads stay in flight through it.
    constexpr int kHalf = kStatsVec / 2;
    constexpr int kH = kHalf * 32;
    const int nh = nvec / kH;  // whole half-rounds
    uint4 va[kHalf], vb[kHalf];
    if (nh > 0) {
#pragma unroll
      for (int k = 0; k < kHalf; ++k) va[k] = ld_global_nc_v4(base + (size_t)(k * 32 + lane) * 16);
    }
    int h = 0;
    for (; h + 1 < nh; h += 2) {
#pragma unroll
      for (int k = 0; k < kHalf; ++k)
        vb[k] = ld_global_nc_v4(base + (size_t)((h + 1) * kH + k * 32 + lane) * 16);
      stats_consume<DT, kHalf>(va, m_run, H, acc, nan_seen, c2);
      if (h + 2 < nh) {
#pragma unroll
        for (int k = 0; k < kHalf; ++k)
          va[k] = ld_global_nc_v4(base + (size_t)((h + 2) * kH + k * 32 + lane) * 16);
      }
      stats_consume<DT, kHalf>(vb, m_run, H, acc, nan_seen, c2);
    }
    if (h < nh) stats_consume<DT, kHalf>(va, m_run, H, acc, nan_seen, c2);
    const int done = nh * kH;
    if (done < nvec) {  // the last, partial half-round, padded with -inf
      uint4 v[kHalf];
#pragma unroll
      for (int k = 0; k < kHalf; ++k) {
        const int idx = done + k * 32 + lane;
        v[k] = idx < nvec ? ld_global_nc_v4(base + (size_t)idx * 16) : make_uint4(fill, fill, fill, fill);
      }
      stats_consume<DT, kHalf>(v, m_run, H, acc, nan_seen, c2);
    }
    return warp_stats(m_run, H, acc, nan_seen, c2);
  }
  constexpr int kRound = kStatsVec * 32;
  const int nfull = nvec / kRound * kRound;
  for (int i0 = 0; i0 < nfull; i0 += kRound) {  // whole rounds: no bounds tests
    uint4 v[kStatsVec];
#pragma unroll
    for (int k = 0; k < kStatsVec; ++k) v[k] = ld_global_nc_v4(base + (size_t)(i0 + k * 32 + lane) * 16);
    stats_consume<DT, kStatsVec>(v, m_run, H, acc, nan_seen, c2);
  }
  if (nfull < nvec) {  // the last, partial round, padded with -inf
    uint4 v[kStatsVec];
#pragma unroll
    for (int k = 0; k < kStatsVec; ++k) {
      const int idx = nfull + k * 32 + lane;
      v[k] = idx < nvec ? ld_global_nc_v4(base + (size_t)idx * 16) : make_uint4(fill, fill, fill, fill);
    }
    stats_consume<DT, kStatsVec>(v, m_run, H, acc, nan_seen, c2);
  }
  return warp_stats(m_run, H, acc, nan_seen, c2);
}

// Plain-load path for rows that are not 16-byte aligned: two passes (the
// warp maximum, then the sum against it).
template <int DT>
SV_DEVINL float2 stats_warp_plain(const Params& P, long long u, int lane) {
  const float c2 = P.c2;
  const int len = unit_len(P, u);
  const unsigned char* rb = unit_row(P, u);
  const long long e0 = (long long)(u % P.nseg) * P.seg_elems;
  float m = neg_inf();
  bool nan_seen = false;
  for (int i = lane; i < len; i += 32) {
    const float l = load_elem<DT>(rb, e0 + i);
    nan_seen |= (l != l);
    m = fmaxf(m, l);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float s = 0.f;
  if (m != neg_inf()) {
    for (int i = lane; i < len; i += 32) s += ex2_fast((load_elem<DT>(rb, e0 + i) - m) * c2);
  }
  if (nan_seen) s = __int_as_float(0x7fc00000);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  return make_float2(m, s);
}

// (max, sum) of a whole row from its segments' pairs, one warp; all lanes
// get it.
SV_DEVINL float2 row_combine(const Params& P, long long row, int lane) {
  const float2* part = P.seg_part + row * P.nseg;
  float m = neg_inf(), s = 0.0f;
  if (P.nseg <= 32) {
    if (lane < P.nseg) {
      const float2 ps = __ldcg(part + lane);
      m = ps.x;
      s = ps.y;
    }
    return warp_combine_pairs(m, s, P.c2);
  }
  // More segments than lanes: each lane first combines its own.
  float2 ps[4];
  for (int g0 = 0; g0 < P.nseg; g0 += 4 * 32) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int g = g0 + k * 32 + lane;
      ps[k] = g < P.nseg ? __ldcg(part + g) : make_float2(neg_inf(), 0.0f);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float M = fmaxf(m, ps[k].x);
      if (M != neg_inf()) {
        const float a = (m == neg_inf()) ? 0.0f : exp2f((m - M) * P.c2);
        const float c = (ps[k].x == neg_inf()) ? 0.0f : exp2f((ps[k].x - M) * P.c2);
        s = s * a + ps[k].y * c;
        m = M;
      } else {
        s += ps[k].y;
      }
    }
  }
  return warp_combine_pairs(m, s, P.c2);
}

// ---------------------------------------------------------------- keys and kept sets of nucleus-filtered rows

// Order-preserving map of a bf16 (16-bit) or f32 bit pattern to an unsigned
// key: unsigned order is numeric order, -0 folded into +0.
template <int DT>
SV_DEVINL uint32_t value_key(uint32_t bits) {
  if constexpr (DT == 0) {
    if (bits == 0x8000u) bits = 0;
    return (bits & 0x8000u) ? (~bits & 0xffffu) : (bits | 0x8000u);
  } else {
    if (bits == 0x80000000u) bits = 0;
    return (bits & 0x80000000u) ? ~bits : (bits | 0x80000000u);
  }
}

// The logit back from a key (value_key above the low `ib` id bits).
template <int DT>
SV_DEVINL float key_value(unsigned long long key, int ib) {
  const uint32_t vk = (uint32_t)(key >> ib);
  if constexpr (DT == 0) {
    const uint32_t h = (vk & 0x8000u) ? (vk & 0x7fffu) : (~vk & 0xffffu);
    return __uint_as_float(h << 16);
  } else {
    return __uint_as_float((vk & 0x80000000u) ? (vk & 0x7fffffffu) : ~vk);
  }
}

// The kept set of a nucleus-filtered row as a test on the loaded value: the
// entry (x, id) is kept iff its key (value, then smaller id first) is at or
// above the row's cut, i.e. x > xc, or x == xc and id <= imax (xc the cut
// entry's value; -0.0 equals +0.0 in both orders). A row without a cut keeps
// everything (xc = -inf, imax the largest id).
struct RowMask {
  float xc;
  long long imax;
};

SV_DEVINL float masked(float x, long long id, const RowMask& k) {
  return (x > k.xc || (x == k.xc && id <= k.imax)) ? x : neg_inf();
}

// Row r (0..K target, K+1..2K draft) of sequence b: its cut as a RowMask.
SV_DEVINL RowMask row_mask(const Params& P, long long b, int r) {
  RowMask k{neg_inf(), 0x7fffffffffffffffLL};
  if (!P.topp_cut) return k;
  const unsigned long long cut = __ldcg(P.topp_cut + b * P.rows_per_seq + r);
  if (cut == 0) return k;
  k.xc = P.dtype == 0 ? key_value<0>(cut, P.key_ibits) : key_value<1>(cut, P.key_ibits);
  k.imax = (long long)P.V - 1 - (long long)(cut & ((1ull << P.key_ibits) - 1));
  return k;
}

// Whether the entry (x, id) of a row with cut `cut` is kept (cut 0: every
// entry), by the key itself.
template <int DT>
SV_DEVINL bool kept_by_key(float x, int id, unsigned long long cut, int ib, int V) {
  const uint32_t bits = DT == 0 ? (__float_as_uint(x) >> 16) : __float_as_uint(x);
  const unsigned long long key =
      ((unsigned long long)value_key<DT>(bits) << ib) | (unsigned long long)(V - 1 - id);
  return key >= cut;
}

// ---------------------------------------------------------------- scan of one sequence, one warp

struct WarpScan {
  float m[2 * kMaxK + 1], s[2 * kMaxK + 1];
  double thr[kMaxK];
  float u[kMaxK + 2];
  int tok[kMaxK];
};

SV_DEVINL void scan_warp(const Params& P, long long b, int lane, WarpScan& ws) {
  const int K = P.K, R = P.rows_per_seq;
  unsigned bits = 0;
  // The drafted tokens, the uniforms and the row statistics, one lane per
  // entry.
  for (int t = lane; t < K + 2; t += 32) {
    if (t < K) {
      const int x = P.tokens[b * K + t];
      ws.tok[t] = x;
      if (x < 0 || x >= P.V) bits |= kDevTokenRange;
    }
    const float u = P.uniforms[b * (K + 2) + t];
    ws.u[t] = u;
    if (!(u >= 0.0f && u <= 1.0f)) bits |= kDevUniformRange;
  }
  for (int r = lane; r < R; r += 32) {
    const float2 st = __ldcg(P.row_stat + b * R + r);
    unsigned rb = 0;
    if (st.y != st.y) {
      rb = kDevNonfinite;
    } else if (st.x == neg_inf()) {
      rb = kDevEmptyRow;
    }
    bits |= rb;
    ws.m[r] = st.x;
    ws.s[r] = st.y;
    if (P.dbg_lse)  // lse = m/T + ln S, only for the debug export
      P.dbg_lse[b * R + r] = rb ? __longlong_as_double(0x7ff8000000000000LL)
                                : (double)st.x * P.inv_t + log((double)st.y);
    if (P.dbg_max)  // max_i l_i / T
      P.dbg_max[b * R + r] = rb ? __longlong_as_double(0x7ff8000000000000LL)
                                : (double)st.x * P.inv_t;
  }
  bits = __reduce_or_sync(0xffffffffu, bits);
  __syncwarp();

  if (!bits) {
    // Thresholds min(1, q(x~)/p(x~)) at the drafted tokens (§4.2):
    // q(x)/p(x) = e_q(x) S_p / (e_p(x) S_q), e(x) = exp((l(x) - m)/T) <= 1 in
    // float-float against each row's own maximum, S the streaming sums. When
    // an e(x) underflows fp32, the log-space form is used in fp64 instead.
    for (int t = lane; t < K; t += 32) {
      const int x = ws.tok[t];
      float lq, lp;
      if (P.dtype == 0) {
        lq = load_elem<0>(row_base(P, b, t), x);
        lp = load_elem<0>(row_base(P, b, K + 1 + t), x);
      } else {
        lq = load_elem<1>(row_base(P, b, t), x);
        lp = load_elem<1>(row_base(P, b, K + 1 + t), x);
      }
      if (P.topp_cut) {  // nucleus-filtered rows: an entry outside the kept set is -inf
        const unsigned long long cq = __ldcg(P.topp_cut + b * R + t);
        const unsigned long long cp = __ldcg(P.topp_cut + b * R + K + 1 + t);
        const bool kq = P.dtype == 0 ? kept_by_key<0>(lq, x, cq, P.key_ibits, P.V)
                                     : kept_by_key<1>(lq, x, cq, P.key_ibits, P.V);
        const bool kp = P.dtype == 0 ? kept_by_key<0>(lp, x, cp, P.key_ibits, P.V)
                                     : kept_by_key<1>(lp, x, cp, P.key_ibits, P.V);
        if (!kq) lq = neg_inf();
        if (!kp) lp = neg_inf();
      }
      const float mq = ws.m[t], mp = ws.m[K + 1 + t];
      const float sq = ws.s[t], sp = ws.s[K + 1 + t];
      double thr, ratio = 0.0;
      if (lq == neg_inf()) {
        thr = 0.0;  // q(x~) = 0 rejects
        ratio = 0.0;
      } else if (lp == neg_inf()) {
        thr = 1.0;  // p(x~) = 0 < q(x~) accepts
        ratio = __longlong_as_double(0x7ff0000000000000LL);
      } else {
        const bool unit_t = P.unit_t != 0;
        const ff xq = scaled_diff(lq, mq, P.ih, P.il, unit_t);
        const ff xp = scaled_diff(lp, mp, P.ih, P.il, unit_t);
        const ff eq = exp_ff(xq.hi, xq.lo, kSvExp2Table);
        const ff ep = exp_ff(xp.hi, xp.lo, kSvExp2Table);
        if (eq.hi > 1e-30f && ep.hi > 1e-30f) {
          // q/p = (e_q S_p) / (e_p S_q) in float-float: the fp32 quotient and
          // one correction from the float-float remainder.
          const ff num = ff_mul_f(eq, sp), den = ff_mul_f(ep, sq);
          const float q1 = __fdiv_rn(num.hi, den.hi);
          const ff rem = ff_sub(num, ff_mul_f(den, q1));
          const double r = ff_to_double(fast_two_sum(q1, __fdiv_rn(rem.hi, den.hi)));
          thr = r >= 1.0 ? 1.0 : r;
          ratio = r;
        } else {
          const double lr = ((double)lq - (double)lp) * P.inv_t -
                            (((double)mq - (double)mp) * P.inv_t + log((double)sq / (double)sp));
          thr = lr >= 0.0 ? 1.0 : exp(lr);
          if (P.dbg_ratio) ratio = exp(lr);
        }
      }
      ws.thr[t] = thr;
      if (P.dbg_thr) P.dbg_thr[b * K + t] = thr;
      if (P.dbg_ratio) P.dbg_ratio[b * K + t] = ratio;
    }
  }
  __syncwarp();

  // Left-to-right scan: accept while u_t < thr_t (Algorithm 2 step 3); the
  // first rejection is the lowest lane (of each group of 32) that rejects.
  int j = bits ? -1 : K;
  if (!bits) {
    for (int t0 = 0; t0 < K; t0 += 32) {
      const int t = t0 + lane;
      const bool rej = t < K && !((double)ws.u[t] < ws.thr[t]);
      const unsigned mask = __ballot_sync(0xffffffffu, rej);
      if (mask) {
        j = t0 + __ffs(mask) - 1;
        break;
      }
    }
  }
  // Outputs other than the drawn token. Position j also gets -1 here, before
  // the plan is released: the draw overwrites it, so a draw that never
  // completes (the fused kernel's bounded wait ran out) leaves -1 there
  // rather than whatever the buffer held.
  for (int t = lane; t <= K; t += 32) {
    if (j < 0 || t >= j)
      P.out_tokens[b * (K + 1) + t] = -1;
    else
      P.out_tokens[b * (K + 1) + t] = ws.tok[t];
  }
  __syncwarp();
  if (lane == 0) {
    Plan pl{};
    if (bits) {
      atomicOr(P.status, bits);
      pl.j = -1;
      pl.mode = kModeFailed;
      P.n_acc[b] = -1;
      if (P.dbg_prob) P.dbg_prob[b] = __longlong_as_double(0x7ff8000000000000LL);
    } else {
      pl.j = j;
      if (j < K) {
        pl.mode = kModeResidual;
        pl.row_q = b * (K + 1) + j;
        pl.row_p = b * K + j;
        pl.m_q = ws.m[j];
        pl.s_q = ws.s[j];
        pl.m_p = ws.m[K + 1 + j];
        pl.s_p = ws.s[K + 1 + j];
        pl.u = ws.u[K];
      } else {
        pl.mode = kModeBonus;
        pl.row_q = b * (K + 1) + K;
        pl.row_p = -1;
        pl.m_q = ws.m[K];
        pl.s_q = ws.s[K];
        pl.u = ws.u[K + 1];
      }
      P.n_acc[b] = j;
    }
    P.plans[b] = pl;
    // The release is cumulative: with the warp barrier above it also orders
    // the other lanes' output stores before the draw CTAs' acquire.
    if (P.fused && !P.withhold) st_release_u32(P.ready + b, 1u);  // for the fused kernel's draw CTAs
  }
  if (bits) {
    for (int t = lane; t < K; t += 32) {
      if (P.dbg_thr) P.dbg_thr[b * K + t] = __longlong_as_double(0x7ff8000000000000LL);
      if (P.dbg_ratio) P.dbg_ratio[b * K + t] = __longlong_as_double(0x7ff8000000000000LL);
    }
  }
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
  // The fast form (rows whose maximum has |m/T| below about 1386): weights
  // exp(l/T) 2^-q0 per row, qb = 127 - q0; alpha / beta put the streaming
  // pass's test e_q S_p > e_p S_q (e = exp((l - m)/T)) on these weights, and
  // lmin is the clamp that keeps every argument inside the reduction's range.
  bool fast;
  int2 qb;
  float alpha, beta, lmin;
  DrawConst dc;
  // Nucleus-filtered rows: the kept set of each row (RowMask), applied to
  // every element as it is loaded.
  RowMask kq, kp;
};

// Exponent shift of one row in the fast form, and its factor 2^(q0 - m c2)
// (the ratio of exp((l - m)/T) to the row's weight exp(l/T) 2^-q0).
SV_DEVINL int row_q0(float m, float c2) { return (int)floorf(m * c2) + 1; }

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
  const bool resid = pl.mode == kModeResidual;
  const float cq = pl.m_q * P.c2, cp = resid ? pl.m_p * P.c2 : 0.0f;
  d.fast = fabsf(cq) <= 2000.0f && fabsf(cp) <= 2000.0f;
  const int q0q = row_q0(pl.m_q, P.c2), q0p = resid ? row_q0(pl.m_p, P.c2) : q0q;
  d.qb = make_int2(127 - q0q, 127 - q0p);
  d.alpha = pl.s_p * exp2f((float)q0q - cq);
  d.beta = resid ? pl.s_q * exp2f((float)q0p - cp) : 0.0f;
  d.lmin = -2048.0f * __fdividef(1.0f, P.ih);
  d.dc = DrawConst{P.d_inv, P.d_ch, P.d_cli, P.ih};
  d.kq = row_mask(P, pl.row_q / (P.K + 1), (int)(pl.row_q % (P.K + 1)));
  d.kp = resid ? row_mask(P, pl.row_p / P.K, P.K + 1 + (int)(pl.row_p % P.K)) : d.kq;
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

template <int DT, bool RESID, int SUB, bool MASK = false>
SV_DEVINL void partial_body(const Params& P, const DrawRow& d, const float2* tab,
                            const float2* tab1k, bool aligned, long long b, int c) {
  constexpr int kVec = 16 / (DT == 0 ? 2 : 4);
  constexpr int kRuns = SUB / (32 * kVec);
  static_assert(kRuns >= 1 && kRuns * 32 * kVec == SUB, "sub-chunk must be whole runs");
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long e0 = ((long long)c * kSubPerChunk + w) * SUB;
  ff Sq = ff_bias_start(), Sp = ff_bias_start(), A = ff_bias_start(), Bs = ff_bias_start();
  if (e0 < P.V && d.fast) {
    // The fast form: weights exp(l/T) 2^-q0 from exp_draw2 (~5e-11).
    const float2 lmin = f2(d.lmin);
    if constexpr (RESID) {
      ff2 S = {f2(1.0f), f2(0.0f)}, AB = {f2(1.0f), f2(0.0f)};
      const float2 ab = make_float2(d.alpha, d.beta);
#pragma unroll
      for (int r = 0; r < kRuns; ++r) {
        const long long e = e0 + (long long)r * 32 * kVec + lane * kVec;
        float xq[kVec], xp[kVec];
        load_run<DT>(d.rq, e, P.V, aligned, xq);
        load_run<DT>(d.rp, e, P.V, aligned, xp);
        if constexpr (MASK) {
#pragma unroll
          for (int k = 0; k < kVec; ++k) {
            xq[k] = masked(xq[k], e + k, d.kq);
            xp[k] = masked(xp[k], e + k, d.kp);
          }
        }
#pragma unroll
        for (int k = 0; k < kVec; ++k) {
          const float2 l = make_float2(fmaxf(xq[k], lmin.x), fmaxf(xp[k], lmin.y));
          const ff2 ex = exp_draw2(l, d.qb, d.dc, tab1k);
          ff_accumulate_biased2(S, ex);
          const float2 v = f2_mul(f2_add(ex.hi, ex.lo), ab);
          if (v.x > v.y) ff_accumulate_biased2(AB, ex);
        }
      }
      Sq = {S.hi.x, S.lo.x};
      Sp = {S.hi.y, S.lo.y};
      A = {AB.hi.x, AB.lo.x};
      Bs = {AB.hi.y, AB.lo.y};
    } else {
      const int2 qb = make_int2(d.qb.x, d.qb.x);
#pragma unroll
      for (int r = 0; r < kRuns; ++r) {
        const long long e = e0 + (long long)r * 32 * kVec + lane * kVec;
        float xq[kVec];
        load_run<DT>(d.rq, e, P.V, aligned, xq);
        if constexpr (MASK) {
#pragma unroll
          for (int k = 0; k < kVec; ++k) xq[k] = masked(xq[k], e + k, d.kq);
        }
#pragma unroll
        for (int k = 0; k < kVec; k += 2) {
          const float2 l = make_float2(fmaxf(xq[k], lmin.x), fmaxf(xq[k + 1], lmin.x));
          const ff2 ex = exp_draw2(l, qb, d.dc, tab1k);
          ff_accumulate_biased(Sq, {ex.hi.x, ex.lo.x});
          ff_accumulate_biased(Sq, {ex.hi.y, ex.lo.y});
        }
      }
    }
  } else if (e0 < P.V) {
    // The shifted form (rows with an extreme maximum): weights exp((l - m)/T).
    if constexpr (RESID) {
      // The target and draft elements side by side in the two lanes of
      // packed fp32 pairs: (S_q, S_p) and (A, B) accumulate together.
      ff2 S = {f2(1.0f), f2(0.0f)}, AB = {f2(1.0f), f2(0.0f)};
      const float2 nm = make_float2(-d.mq, -d.mp);
#pragma unroll
      for (int r = 0; r < kRuns; ++r) {
        const long long e = e0 + (long long)r * 32 * kVec + lane * kVec;
        float xq[kVec], xp[kVec];
        load_run<DT>(d.rq, e, P.V, aligned, xq);
        load_run<DT>(d.rp, e, P.V, aligned, xp);
        if constexpr (MASK) {
#pragma unroll
          for (int k = 0; k < kVec; ++k) {
            xq[k] = masked(xq[k], e + k, d.kq);
            xp[k] = masked(xp[k], e + k, d.kp);
          }
        }
#pragma unroll
        for (int k = 0; k < kVec; ++k) {
          const ff2 x = scaled_diff2(make_float2(xq[k], xp[k]), nm, d.ih, d.il, d.unit_t);
          const ff2 ex = exp_ff2(x.hi, x.lo, tab);
          ff_accumulate_biased2(S, ex);
          if (__fmul_rn(ex.hi.x, d.sp) > __fmul_rn(ex.hi.y, d.sq)) ff_accumulate_biased2(AB, ex);
        }
      }
      Sq = {S.hi.x, S.lo.x};
      Sp = {S.hi.y, S.lo.y};
      A = {AB.hi.x, AB.lo.x};
      Bs = {AB.hi.y, AB.lo.y};
    } else {
      // Exponentials two elements at a time; the sum keeps element order.
      const float2 nm = f2(-d.mq);
#pragma unroll
      for (int r = 0; r < kRuns; ++r) {
        const long long e = e0 + (long long)r * 32 * kVec + lane * kVec;
        float xq[kVec];
        load_run<DT>(d.rq, e, P.V, aligned, xq);
        if constexpr (MASK) {
#pragma unroll
          for (int k = 0; k < kVec; ++k) xq[k] = masked(xq[k], e + k, d.kq);
        }
#pragma unroll
        for (int k = 0; k < kVec; k += 2) {
          const ff2 x = scaled_diff2(make_float2(xq[k], xq[k + 1]), nm, d.ih, d.il, d.unit_t);
          const ff2 ex = exp_ff2(x.hi, x.lo, tab);
          ff_accumulate_biased(Sq, {ex.hi.x, ex.lo.x});
          ff_accumulate_biased(Sq, {ex.hi.y, ex.lo.y});
        }
      }
    }
  }
  Sq = ff_warp_sum(ff_bias_end(Sq));
  if constexpr (RESID) {
    Sp = ff_warp_sum(ff_bias_end(Sp));
    A = ff_warp_sum(ff_bias_end(A));
    Bs = ff_warp_sum(ff_bias_end(Bs));
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

// One block pass over per-thread float-float values, in thread order: the
// exclusive prefixes of (s1, s2), the block totals of (s1, s2) and of (t1, t2).
struct BlockScan2 {
  ff pre1, pre2, tot1, tot2, sum1, sum2;
};

SV_DEVINL BlockScan2 block_scan2(ff s1, ff s2, ff t1, ff t2, CtaShared& sh) {
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  ff i1 = s1, i2 = s2;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const ff y1 = ff_shfl_up(i1, o), y2 = ff_shfl_up(i2, o);
    if (l >= o) {
      i1 = ff_add(i1, y1);
      i2 = ff_add(i2, y2);
    }
  }
  ff e1 = ff_shfl_up(i1, 1), e2 = ff_shfl_up(i2, 1);
  if (l == 0) e1 = e2 = {0.f, 0.f};
  t1 = ff_warp_sum(t1);
  t2 = ff_warp_sum(t2);
  __syncthreads();  // red4 may still be read from an earlier use
  if (l == 31) {
    sh.red4[w][0] = i1;
    sh.red4[w][1] = i2;
    sh.red4[w][2] = t1;
    sh.red4[w][3] = t2;
  }
  __syncthreads();
  BlockScan2 r{};
  ff b1{0.f, 0.f}, b2{0.f, 0.f};
  for (int i = 0; i < kWarps; ++i) {
    if (i < w) {
      b1 = ff_add(b1, sh.red4[i][0]);
      b2 = ff_add(b2, sh.red4[i][1]);
    }
    r.tot1 = ff_add(r.tot1, sh.red4[i][0]);
    r.tot2 = ff_add(r.tot2, sh.red4[i][1]);
    r.sum1 = ff_add(r.sum1, sh.red4[i][2]);
    r.sum2 = ff_add(r.sum2, sh.red4[i][3]);
  }
  r.pre1 = ff_add(b1, e1);
  r.pre2 = ff_add(b2, e2);
  return r;
}

// Block exclusive prefix of float-float values in thread order.
SV_DEVINL ff block_exclusive_ff(ff x, CtaShared& sh) {
  const ff z{0.f, 0.f};
  return block_scan2(x, z, z, z, sh).pre1;
}

// The finish runs in the CTA that counted the last draw chunk of sequence b.
// Sub-chunk g holds float-float sums S_q[g], S_p[g] over its elements and
// A[g], B[g] over its elements of the positive set; for the residual the
// weight before sub-chunk g is S_p * (A[0] + .. + A[g-1]) - S_q * (B[0] + ..
// + B[g-1]) with S_p, S_q the row totals (at the end: R = S_p A - S_q B), for
// the bonus draw (or the zero-residual fallback) it is S_q[0] + .. + S_q[g-1].
template <int DT, int SUB, bool MASK = false>
SV_DEVINL void finish_seq(const Params& P, long long b, const Plan& pl, CtaShared& sh,
                          bool aligned) {
  constexpr int kPer = SUB / kThreads;  // elements per thread in the exact search
  static_assert(kPer * kThreads == SUB, "sub-chunk must split evenly over the CTA");
  const int tid = threadIdx.x;
  const int nsub = P.nchunk * kSubPerChunk;
  const float4* part = reinterpret_cast<const float4*>(P.sub_part + (size_t)b * nsub * 4);
  const bool resid = pl.mode == kModeResidual;
  const int run = (nsub + kThreads - 1) / kThreads;
  const int g0 = min(nsub, tid * run), g1 = min(nsub, g0 + run);

  // This thread's sub-chunk sums, read once (kept in registers when the run
  // is short, i.e. V up to 2^19; otherwise re-read from L2 below).
  constexpr int kCache = 4;
  float4 cx[kCache], cy[kCache];
  const bool cached = run <= kCache;
  auto load_sub = [&](int g, float4& x, float4& y) {
    if (cached) {
#pragma unroll
      for (int i = 0; i < kCache; ++i)
        if (g - g0 == i) {
          x = cx[i];
          y = cy[i];
        }
    } else {
      x = __ldcg(part + 2 * g);
      y = resid ? __ldcg(part + 2 * g + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };
  ff tq{0.f, 0.f}, tp{0.f, 0.f}, ta{0.f, 0.f}, tb{0.f, 0.f};
  for (int g = g0; g < g1; ++g) {
    const float4 x = __ldcg(part + 2 * g);
    const float4 y = resid ? __ldcg(part + 2 * g + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
    if (cached) {
#pragma unroll
      for (int i = 0; i < kCache; ++i)
        if (g - g0 == i) {
          cx[i] = x;
          cy[i] = y;
        }
    }
    tq = ff_add(tq, ff_of(x.x, x.y));
    tp = ff_add(tp, ff_of(x.z, x.w));
    ta = ff_add(ta, ff_of(y.x, y.y));
    tb = ff_add(tb, ff_of(y.z, y.w));
  }
  // Residual: prefixes of (A, B) and totals of (S_q, S_p); bonus: prefix of S_q.
  BlockScan2 bs = resid ? block_scan2(ta, tb, tq, tp, sh)
                        : block_scan2(tq, ff{0.f, 0.f}, ff{0.f, 0.f}, ff{0.f, 0.f}, sh);
  const ff Sq = resid ? bs.sum1 : bs.tot1;
  const ff Sp = bs.sum2;
  // Residual mass sum max(0, q - p), scaled by S_q S_p; zero -> fall back to
  // q. R is the difference of two float-float products; when the positive
  // set's q and p agree exactly (e.g. one-hot rows on the same token), their
  // rounding leaves a residue near 2^-48 of the terms, so a residual below
  // 2^-40 of them counts as zero.
  const ff SA = ff_mul(Sp, bs.tot1), SB = ff_mul(Sq, bs.tot2);
  const ff R = ff_sub(SA, SB);
  const bool res_first = resid && R.hi > 0x1p-40f * (SA.hi + SB.hi);
  const BlockScan2 bs_res = bs;
  const DrawRow d = draw_row(P, pl);
  // Element loads of the two rows (the kept set applied, for filtered rows).
  auto ld_q = [&](long long e) {
    const float x = load_elem<DT>(d.rq, e);
    if constexpr (MASK) return masked(x, e, d.kq);
    return x;
  };
  auto ld_p = [&](long long e) {
    const float x = load_elem<DT>(d.rp, e);
    if constexpr (MASK) return masked(x, e, d.kp);
    return x;
  };

  // One search: the sub-chunk holding u * total, then the element within it.
  // Returns whether a token was written (uniform across the CTA).
  auto search = [&](bool use_res) -> bool {
    const BlockScan2 bsx = use_res ? bs_res
                                   : (resid ? block_scan2(tq, ff{0.f, 0.f}, ff{0.f, 0.f},
                                                          ff{0.f, 0.f}, sh)
                                            : bs_res);
    const ff total = use_res ? R : Sq;
    const ff tau = ff_mul_f(total, pl.u);
    auto weight_before = [&](ff pa, ff pb) {
      return use_res ? ff_sub(ff_mul(Sp, pa), ff_mul(Sq, pb)) : pa;
    };
    auto sub_sums = [&](int g, ff& a, ff& bb) {
      float4 x, y;
      load_sub(g, x, y);
      if (use_res) {
        a = ff_of(y.x, y.y);
        bb = ff_of(y.z, y.w);
      } else {
        a = ff_of(x.x, x.y);
        bb = {0.f, 0.f};
      }
    };

    // The first sub-chunk with positive weight whose cumulative weight passes
    // tau, and the last sub-chunk with positive weight.
    __syncthreads();  // sh.g / sh.j may still be read by an earlier search
    if (tid == 0) {
      sh.g = INT_MAX;
      sh.j = -1;
    }
    __syncthreads();
    {
      ff pa = bsx.pre1, pb = bsx.pre2;
      int found = -1, lastpos = -1;
      for (int g = g0; g < g1; ++g) {
        ff a, bb;
        sub_sums(g, a, bb);
        pa = ff_add(pa, a);
        pb = ff_add(pb, bb);
        const ff next = weight_before(pa, pb);
        const bool positive =
            use_res ? ff_sub(ff_mul(Sp, a), ff_mul(Sq, bb)).hi > 0.f : a.hi > 0.f;
        if (positive) {
          lastpos = g;
          if (found < 0 && ff_gt(next, tau)) found = g;
        }
      }
      if (found >= 0) atomicMin(&sh.g, found);
      if (lastpos >= 0) atomicMax(&sh.j, lastpos);
    }
    __syncthreads();
    const bool last_mode = sh.g == INT_MAX;
    const int gs = last_mode ? sh.j : sh.g;
    if (gs < 0) return false;  // uniform across the CTA: no positive weight at all
    // The weight before sub-chunk gs, from the thread that holds it.
    if (!last_mode && gs >= g0 && gs < g1) {
      ff pa = bsx.pre1, pb = bsx.pre2;
      for (int g = g0; g < gs; ++g) {
        ff a, bb;
        sub_sums(g, a, bb);
        pa = ff_add(pa, a);
        pb = ff_add(pb, bb);
      }
      sh.s_pref = weight_before(pa, pb);
    }
    // Exact search inside sub-chunk gs: kPer consecutive elements per thread,
    // with the chunk pass's own element weights (so that the search agrees
    // with the sub-chunk sums it starts from).
    const long long e0 = (long long)gs * SUB + kPer * tid;
    ff w[kPer];
    ff wsum{0.f, 0.f};
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const long long e = e0 + k;
      w[k] = {0.f, 0.f};
      if (e < P.V) {
        const float lq = ld_q(e);
        ff eq, ep;
        bool pos;
        if (d.fast) {
          const float lqc = fmaxf(lq, d.lmin);
          const ff fq = exp_draw(lqc, d.qb.x, d.dc, sh.tab1k);
          if (use_res) {
            const float lpc = fmaxf(ld_p(e), d.lmin);
            const ff fp = exp_draw(lpc, d.qb.y, d.dc, sh.tab1k);
            pos = __fmul_rn(__fadd_rn(fq.hi, fq.lo), d.alpha) >
                  __fmul_rn(__fadd_rn(fp.hi, fp.lo), d.beta);
            if (pos) w[k] = ff_sub(ff_mul(ff_normalize(fq), Sp), ff_mul(ff_normalize(fp), Sq));
          } else {
            w[k] = ff_normalize(fq);
          }
        } else if (use_res) {
          const float lp = ld_p(e);
          element_exps<true>(d, lq, lp, sh.tab, eq, ep, pos);
          if (pos) w[k] = ff_sub(ff_mul(ff_normalize(eq), Sp), ff_mul(ff_normalize(ep), Sq));
        } else {
          element_exps<false>(d, lq, 0.f, sh.tab, eq, ep, pos);
          w[k] = ff_normalize(eq);
        }
      }
      wsum = ff_add(wsum, w[k]);
    }
    // block_exclusive_ff's barriers also publish s_pref.
    const ff tpre = block_exclusive_ff(wsum, sh);
    if (tid == 0) {
      sh.g = INT_MAX;
      sh.j = -1;
    }
    __syncthreads();
    ff cum = ff_add(sh.s_pref, tpre);
    int found = -1, lastk = -1;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      cum = ff_add(cum, w[k]);
      if (!last_mode && found < 0 && w[k].hi > 0.f && ff_gt(cum, tau)) found = k;
      if (w[k].hi > 0.f) lastk = k;
    }
    if (found >= 0) atomicMin(&sh.g, kPer * tid + found);
    if (lastk >= 0) atomicMax(&sh.j, kPer * tid + lastk);
    __syncthreads();
    // The first element whose cumulative weight passes tau; else (u = 1, or
    // rounding at the sub-chunk's end) the last positive element.
    const int pick = sh.g != INT_MAX ? sh.g : sh.j;
    if (pick < 0) return false;
    if (pick / kPer == tid) {
      const long long e = (long long)gs * SUB + pick;
      P.out_tokens[b * (P.K + 1) + pl.j] = (int)e;
      if (P.dbg_prob) {
        // The drawn token's probability for the debug export, its weight
        // taken with the precise exponential in the same scaling.
        ff wt = w[pick % kPer];
        if (d.fast) {
          const float lqc = fmaxf(ld_q(e), d.lmin);
          const ff pq = ff_normalize(exp_precise(lqc, d.qb.x, d.ih, d.il, sh.tab));
          if (use_res) {
            const float lpc = fmaxf(ld_p(e), d.lmin);
            const ff pp = ff_normalize(exp_precise(lpc, d.qb.y, d.ih, d.il, sh.tab));
            wt = ff_sub(ff_mul(pq, Sp), ff_mul(pp, Sq));
          } else {
            wt = pq;
          }
        }
        P.dbg_prob[b] = ff_to_double(wt) / ff_to_double(total);
      }
    }
    return true;
  };
  // The residual first (when it is not zero); if its search finds no positive
  // weight, the zero-residual fallback to q.
  if (search(res_first)) return;
  if (res_first) search(false);
}

// ---------------------------------------------------------------- the two kernels

SV_DEVINL unsigned atomic_add_acq_rel(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// Draft-side sampler: once row b's statistics are complete, its plan is a
// bonus-mode draw from the row with the row's uniform (or, for a bad row or
// uniform, the failure outputs) -- there is no acceptance scan.
SV_DEVINL void sample_plan(const Params& P, long long b, float2 st, int lane) {
  if (lane != 0) return;
  unsigned bits = 0;
  if (st.y != st.y) {
    bits = kDevNonfinite;
  } else if (st.x == neg_inf()) {
    bits = kDevEmptyRow;
  }
  const float u = P.uniforms[b];
  if (!(u >= 0.0f && u <= 1.0f)) bits |= kDevUniformRange;
  if (P.dbg_lse)
    P.dbg_lse[b] = bits ? __longlong_as_double(0x7ff8000000000000LL)
                        : (double)st.x * P.inv_t + log((double)st.y);
  Plan pl{};
  if (bits) {
    atomicOr(P.status, bits);
    pl.j = -1;
    pl.mode = kModeFailed;
    P.out_tokens[b] = -1;
    if (P.dbg_prob) P.dbg_prob[b] = __longlong_as_double(0x7ff8000000000000LL);
  } else {
    pl.j = 0;
    pl.mode = kModeBonus;
    pl.row_q = b;
    pl.row_p = -1;
    pl.m_q = st.x;
    pl.s_q = st.y;
    pl.u = u;
  }
  P.plans[b] = pl;
  if (P.fused && !P.withhold) st_release_u32(P.ready + b, 1u);
}

// One warp per row segment u. The warp that counts the last segment of a row
// combines the row; the warp that completes the last row of a sequence scans
// it. The counters are acquire-release atomics taken by lane 0; __syncwarp
// then orders the other lanes' reads (through L2) after lane 0's acquire.
template <int DT, bool VEC>
SV_DEVINL void stats_warp_unit(const Params& P, long long u, int lane, WarpScan& ws) {
  const long long row = u / P.nseg;
  const long long b = row / P.rows_per_seq;
  float2 st;
  if constexpr (VEC)
    st = stats_warp_vec<DT>(P, u, lane);
  else
    st = stats_warp_plain<DT>(P, u, lane);
  if (P.nseg > 1) {
    unsigned last = 0;
    if (lane == 0) {
      P.seg_part[u] = st;
      last = atomic_add_acq_rel(P.done_r + row, 1u) == (unsigned)(P.nseg - 1);
    }
    if (!__shfl_sync(0xffffffffu, last, 0)) return;
    __syncwarp();
    st = row_combine(P, row, lane);
  }
  if (P.sampler) {
    sample_plan(P, row, st, lane);
    return;
  }
  unsigned last = 0;
  if (lane == 0) {
    P.row_stat[row] = st;
    last = atomic_add_acq_rel(P.done_s + b, 1u) == (unsigned)(P.rows_per_seq - 1);
  }
  if (!__shfl_sync(0xffffffffu, last, 0)) return;
  __syncwarp();
  scan_warp(P, b, lane, ws);
}

template <int DT, bool VEC>
__global__ void __launch_bounds__(kStatsThreads, kStatsCtasPerSm) stats_kernel(Params P) {
  __shared__ WarpScan scan_sh[kStatsWarps];
  // Let the draw kernel be launched once every CTA of this grid has started.
  asm volatile("griddepcontrol.launch_dependents;");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long u = (long long)blockIdx.x * kStatsWarps + warp;
  if (u < P.n_units) stats_warp_unit<DT, VEC>(P, u, lane, scan_sh[warp]);
}

// Chunk c of sequence b's draw, by one CTA whose table is loaded and whose
// view of the plan is current: the sub-chunk sums, and the finish in the CTA
// that counts the sequence's last chunk.
template <int DT, bool VEC, int SUB, bool MASK = false>
SV_DEVINL void draw_chunk(const Params& P, long long b, int c, CtaShared& sh) {
  const int tid = threadIdx.x;
  if (tid == 0) {
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
  }
  __syncthreads();
  const Plan pl = sh.plan;
  if (pl.mode == kModeFailed) return;  // outputs already written by the scan
  const DrawRow d = draw_row(P, pl);
  if (pl.mode == kModeResidual)
    partial_body<DT, true, SUB, MASK>(P, d, sh.tab, sh.tab1k, VEC, b, c);
  else
    partial_body<DT, false, SUB, MASK>(P, d, sh.tab, sh.tab1k, VEC, b, c);
  __syncthreads();  // all sub-chunk writes of this CTA precede the release below
  if (tid == 0) sh.flag = atomic_add_acq_rel(P.done_p + b, 1u) == (unsigned)(P.np - 1);
  __syncthreads();
  if (sh.flag) finish_seq<DT, SUB, MASK>(P, b, pl, sh, VEC);  // the barrier above orders its reads
}


// The kernel pair's draw for small calls (2048-element chunks): one launch,
// one CTA per draw chunk; the CTA that counts the last chunk of a sequence
// runs its inverse-CDF search. For such calls the finish kernel's launch
// would cost more than the CTA barrier it saves.
template <int DT, bool VEC, int SUB, bool MASK = false>
__global__ void __launch_bounds__(kThreads, 5) draw_kernel(Params P) {
  __shared__ CtaShared sh;
  sh.tab[threadIdx.x] = kSvExp2Table[threadIdx.x];
#pragma unroll
  for (int i = 0; i < 4; ++i) sh.tab1k[threadIdx.x + i * kThreads] = kSvExp2Table1024[threadIdx.x + i * kThreads];
  // Wait until the streaming grid has completed and its writes are visible
  // (immediate when this kernel was launched as an ordinary dependent).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  draw_chunk<DT, VEC, SUB, MASK>(P, blockIdx.x / P.np, (int)(blockIdx.x % P.np), sh);
}

// ---------------------------------------------------------------- the kernel pair's draw
//
// After stats_kernel, the draw of the kernel pair takes two launches. In
// draw_sum_kernel (one CTA per draw chunk) each warp sums its sub-chunk and
// leaves, without waiting for the CTA's other warps; draw_finish_kernel (one
// CTA per sequence) then runs each sequence's inverse-CDF search once every
// chunk's sums are in memory. Both are programmatic dependents of the launch
// before them: they become resident while it ends, load their tables, and
// wait on the device for it to complete.

template <int DT, bool VEC, int SUB, bool MASK = false>
__global__ void __launch_bounds__(kThreads, 5) draw_sum_kernel(Params P) {
  __shared__ float2 tab[256];
  __shared__ float2 tab1k[1024];
  __shared__ Plan plan;
  const int tid = threadIdx.x;
  tab[tid] = kSvExp2Table[tid];
#pragma unroll
  for (int i = 0; i < 4; ++i) tab1k[tid + i * kThreads] = kSvExp2Table1024[tid + i * kThreads];
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const long long b = blockIdx.x / P.np;
  const int c = (int)(blockIdx.x % P.np);
  if (tid == 0) {
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
    plan = pl;
  }
  __syncthreads();  // the tables and the plan
  const Plan pl = plan;
  if (pl.mode == kModeFailed) return;  // outputs already written by the scan
  const DrawRow d = draw_row(P, pl);
  if (pl.mode == kModeResidual)
    partial_body<DT, true, SUB, MASK>(P, d, tab, tab1k, VEC, b, c);
  else
    partial_body<DT, false, SUB, MASK>(P, d, tab, tab1k, VEC, b, c);
}

template <int DT, bool VEC, int SUB, bool MASK = false>
__global__ void __launch_bounds__(kThreads) draw_finish_kernel(Params P) {
  __shared__ CtaShared sh;
  const int tid = threadIdx.x;
  sh.tab[tid] = kSvExp2Table[tid];
#pragma unroll
  for (int i = 0; i < 4; ++i) sh.tab1k[tid + i * kThreads] = kSvExp2Table1024[tid + i * kThreads];
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const long long b = blockIdx.x;
  if (tid == 0) sh.plan = P.plans[b];
  __syncthreads();
  const Plan pl = sh.plan;
  if (pl.mode == kModeFailed) return;
  finish_seq<DT, SUB, MASK>(P, b, pl, sh, VEC);
}

// ---------------------------------------------------------------- the draft-side sampler
//
// One token per row drawn from softmax(l/T) in a single read of the row.
// sample_sum_kernel: each warp loads its sub-chunk into registers, takes the
// sub-chunk's own maximum m_g, and sums its weights exp(l/T) 2^-q0_g in
// float-float with the fast exponential, q0_g = floor(m_g log2(e)/T) + 1; it
// records (sum, m_g, flags). sample_finish_kernel (one CTA per row): the row
// maximum is the largest m_g; each sub-chunk sum times 2^(q0_g - q0_row) is an
// exact power-of-two rescaling to the row's own shift, after which the
// verifier's finish draws the token as its bonus draw does. A row whose
// maximum lies beyond the fast form's range has its sums recomputed by the
// finish CTA in the shifted form.

constexpr unsigned kSubNonfinite = 1u, kSubExtreme = 2u;

template <int DT, bool VEC, int SUB>
__global__ void __launch_bounds__(kThreads, 5) sample_sum_kernel(Params P) {
  constexpr int kVec = 16 / (DT == 0 ? 2 : 4);
  constexpr int kRuns = SUB / (32 * kVec);
  __shared__ float2 tab1k[1024];
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
#pragma unroll
  for (int i = 0; i < 4; ++i) tab1k[tid + i * kThreads] = kSvExp2Table1024[tid + i * kThreads];
  __syncthreads();
  const long long r = blockIdx.x / P.np;
  const int c = (int)(blockIdx.x % P.np);
  const long long e0 = ((long long)c * kSubPerChunk + w) * SUB;
  const unsigned char* row = static_cast<const unsigned char*>(P.target) + (size_t)r * P.V * P.es;
  float x[kRuns][kVec];
  float mx = neg_inf();
  bool bad = false;
#pragma unroll
  for (int k = 0; k < kRuns; ++k) {
    const long long e = e0 + (long long)k * 32 * kVec + lane * kVec;
    if (e0 < P.V) {
      load_run<DT>(row, e, P.V, VEC, x[k]);
    } else {
#pragma unroll
      for (int j = 0; j < kVec; ++j) x[k][j] = neg_inf();
    }
#pragma unroll
    for (int j = 0; j < kVec; ++j) {
      bad |= x[k][j] != x[k][j] || x[k][j] == -neg_inf();
      mx = fmaxf(mx, x[k][j]);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  bad = __any_sync(0xffffffffu, bad);
  unsigned flags = bad ? kSubNonfinite : 0u;
  ff S = ff_bias_start();
  if (!bad && mx != neg_inf()) {
    const float cm = mx * P.c2;
    if (fabsf(cm) <= 2000.0f) {
      const int q0 = row_q0(mx, P.c2);
      const int2 qb = make_int2(127 - q0, 127 - q0);
      const DrawConst dc{P.d_inv, P.d_ch, P.d_cli, P.ih};
      const float lmin = -2048.0f * __fdividef(1.0f, P.ih);
#pragma unroll
      for (int k = 0; k < kRuns; ++k) {
#pragma unroll
        for (int j = 0; j < kVec; j += 2) {
          const float2 l = make_float2(fmaxf(x[k][j], lmin), fmaxf(x[k][j + 1], lmin));
          const ff2 ex = exp_draw2(l, qb, dc, tab1k);
          ff_accumulate_biased(S, {ex.hi.x, ex.lo.x});
          ff_accumulate_biased(S, {ex.hi.y, ex.lo.y});
        }
      }
    } else {
      flags |= kSubExtreme;
    }
  }
  S = ff_warp_sum(ff_bias_end(S));
  if (lane == 0) {
    float4* out = reinterpret_cast<float4*>(
        P.sub_part + (((size_t)r * P.nchunk + c) * kSubPerChunk + w) * 4);
    out[0] = make_float4(S.hi, S.lo, mx, __uint_as_float(flags));
    out[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

template <int DT, bool VEC, int SUB>
__global__ void __launch_bounds__(kThreads) sample_finish_kernel(Params P) {
  __shared__ CtaShared sh;
  __shared__ float s_m[kWarps];
  __shared__ unsigned s_f[kWarps];
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  sh.tab[tid] = kSvExp2Table[tid];
#pragma unroll
  for (int i = 0; i < 4; ++i) sh.tab1k[tid + i * kThreads] = kSvExp2Table1024[tid + i * kThreads];
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const long long r = blockIdx.x;
  const int nsub = P.nchunk * kSubPerChunk;
  float4* part = reinterpret_cast<float4*>(P.sub_part + (size_t)r * nsub * 4);
  // The row's maximum and flags.
  float m = neg_inf();
  unsigned flags = 0;
  for (int g = tid; g < nsub; g += kThreads) {
    const float4 rec = __ldcg(part + 2 * g);
    m = fmaxf(m, rec.z);
    flags |= __float_as_uint(rec.w);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    flags |= __shfl_xor_sync(0xffffffffu, flags, o);
  }
  if (lane == 0) {
    s_m[w] = m;
    s_f[w] = flags;
  }
  __syncthreads();
  m = s_m[0];
  flags = s_f[0];
  for (int i = 1; i < kWarps; ++i) {
    m = fmaxf(m, s_m[i]);
    flags |= s_f[i];
  }
  unsigned bits = 0;
  if (flags & kSubNonfinite) {
    bits = kDevNonfinite;
  } else if (m == neg_inf()) {
    bits = kDevEmptyRow;
  }
  const float u = P.uniforms[r];
  if (!(u >= 0.0f && u <= 1.0f)) bits |= kDevUniformRange;
  if (bits) {
    if (tid == 0) {
      atomicOr(P.status, bits);
      P.out_tokens[r] = -1;
      if (P.dbg_prob) P.dbg_prob[r] = __longlong_as_double(0x7ff8000000000000LL);
      if (P.dbg_lse) P.dbg_lse[r] = __longlong_as_double(0x7ff8000000000000LL);
    }
    return;
  }
  Plan pl{};
  pl.j = 0;
  pl.mode = kModeBonus;
  pl.row_q = r;
  pl.row_p = -1;
  pl.m_q = m;
  pl.s_q = 1.0f;
  pl.u = u;
  const float cm = m * P.c2;
  double lse_scale;  // log of the factor the row's weights carry: exp(l/T) = w * e^lse_scale
  if ((flags & kSubExtreme) || fabsf(cm) > 2000.0f) {
    // Beyond the fast form's range: the row's sums again, in the shifted form
    // (weights exp((l - m)/T)), one sub-chunk per warp.
    __syncthreads();
    const DrawRow d = draw_row(P, pl);
    for (int c = 0; c < P.nchunk; ++c) partial_body<DT, false, SUB>(P, d, sh.tab, sh.tab1k, VEC, r, c);
    lse_scale = (double)m * P.inv_t;
  } else {
    // Exact rescaling of every sub-chunk sum to the row's shift.
    const int q0r = row_q0(m, P.c2);
    for (int g = tid; g < nsub; g += kThreads) {
      const float4 rec = __ldcg(part + 2 * g);
      float f = 0.0f;
      if (rec.z != neg_inf()) {
        const int e = row_q0(rec.z, P.c2) - q0r;  // <= 0
        f = e < -126 ? 0.0f : __int_as_float((e + 127) << 23);
      }
      part[2 * g] = make_float4(rec.x * f, rec.y * f, 0.f, 0.f);
    }
    lse_scale = (double)q0r * 0.69314718055994530942;
  }
  __threadfence_block();
  __syncthreads();
  if (P.dbg_lse) {  // log sum_i exp(l_i / T), from the row's float-float total
    ff t{0.f, 0.f};
    for (int g = tid; g < nsub; g += kThreads) {
      const float4 rec = __ldcg(part + 2 * g);
      t = ff_add(t, ff{rec.x, rec.y});
    }
    t = ff_warp_sum(t);
    __syncthreads();
    if (lane == 0) sh.red4[w][0] = t;
    __syncthreads();
    if (tid == 0) {
      ff tot{0.f, 0.f};
      for (int i = 0; i < kWarps; ++i) tot = ff_add(tot, sh.red4[i][0]);
      P.dbg_lse[r] = lse_scale + log(ff_to_double(tot));
    }
  }
  finish_seq<DT, SUB>(P, r, pl, sh, VEC);
}

// ---------------------------------------------------------------- the fused kernel
//
// For mid-sized calls one launch does the whole step. Each CTA takes a ticket when it starts: tickets below
// ceil(n_units / 8) are streaming items (eight warp-units, as stats_kernel's
// warps), the rest draw chunks in sequence order (draw_chunk). A
// draw CTA waits for its sequence's plan, which the sequence's scan releases;
// every streaming ticket precedes every draw ticket and streaming never
// waits, so each awaited plan is being computed by a CTA already running. The
// wait is bounded: after kWaitLimitNs it sets kDevTimeout and the abort flag
// and the CTA returns. Compared with the kernel pair, a sequence's draw starts
// as soon as its own scan is done, during the last streaming wave instead of
// after the grid boundary. Measured on GB300 it wins between a few tens of MB
// and a GB of logits; below, the ticket's round trip at every CTA's start
// costs more than it saves, and above, the draw's 4 CTAs per SM (64 registers
// for the streaming role) lose to the draw kernel's 5.

constexpr long long kFusedMinBytes = 16ll << 20;   // calls streaming from this much ...
constexpr long long kFusedMaxBytes = 1ll << 30;    // ... up to this take the fused kernel

union FusedShared {
  WarpScan scan[kWarps];
  CtaShared draw;
};

SV_DEVINL void note_timeout(const Params& P) {
  atomicOr(P.status, kDevTimeout);
  atomicExch(P.abort, 1u);
}

// Bounded wait (one thread) for sequence b's plan.
SV_DEVINL bool wait_ready(const Params& P, long long b) {
  if (ld_acquire_u32(P.ready + b)) return true;
  const uint64_t t0 = global_ns();
  unsigned ns = 64;
  for (;;) {
    __nanosleep(ns);
    if (ns < 1024) ns <<= 1;
    if (ld_acquire_u32(P.ready + b)) return true;
    if (ld_acquire_u32(P.abort)) return false;
    if (global_ns() - t0 > kWaitLimitNs) {
      note_timeout(P);
      return false;
    }
  }
}

// Ticket t -> work item. Sequence s has nsi streaming items (up to eight of
// its units each) and np draw chunks. The streaming items of sequences
// 0 .. lag-1 come first; then, for s = lag .. B-1, the streaming items of s
// followed by the draw chunks of s - lag; then the draw chunks of the last lag
// sequences. So every streaming ticket of a sequence precedes its draw
// tickets, whatever the lag (lag = B: all streaming first).
struct FusedItem {
  bool stream;
  long long b, idx;
};

SV_DEVINL FusedItem fused_item(const Params& P, long long t) {
  const long long NS = P.nsi, NP = P.np, L = P.lag, B = P.B;
  if (t < L * NS) return {true, t / NS, t % NS};
  t -= L * NS;
  if (t < (B - L) * (NS + NP)) {
    const long long s = L + t / (NS + NP), o = t % (NS + NP);
    if (o < NS) return {true, s, o};
    return {false, s - L, o - NS};
  }
  t -= (B - L) * (NS + NP);
  return {false, (B - L) + t / NP, t % NP};
}

template <int DT, bool VEC, int SUB>
__global__ void __launch_bounds__(kThreads, 4) fused_kernel(Params P) {
  __shared__ FusedShared sh;
  __shared__ unsigned s_ticket;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) s_ticket = atomicAdd(P.ticket, 1u);
  __syncthreads();
  const FusedItem it = fused_item(P, (long long)s_ticket);
  if (it.stream) {
    const long long k = it.idx * kWarps + warp;  // the sequence's k-th unit
    if (k < P.ns) stats_warp_unit<DT, VEC>(P, it.b * P.ns + k, lane, sh.scan[warp]);
    return;
  }
  const long long b = it.b;
  sh.draw.tab[tid] = kSvExp2Table[tid];
#pragma unroll
  for (int i = 0; i < 4; ++i) sh.draw.tab1k[tid + i * kThreads] = kSvExp2Table1024[tid + i * kThreads];
  if (tid == 0) sh.draw.flag = wait_ready(P, b) ? 1 : 0;
  __syncthreads();
  if (!sh.draw.flag) return;
  draw_chunk<DT, VEC, SUB>(P, b, (int)it.idx, sh.draw);
}

// ---------------------------------------------------------------- greedy mode (T = 0)
//
// The card's inferred greedy rule (Pitfalls, "Greedy mode is not specified"):
// accept x~_t while it equals argmax q_t, ties to the smallest token id, else
// emit argmax q_j; all K accepted emits argmax q_K. Only the K+1 target rows
// are read, once: one warp per segment finds the segment's maximum and the
// first index holding it; the warp that counts a row's last segment combines
// the row; the warp that completes a sequence's last row compares.
// A pair (v, i) holds the value and the first index of the maximum; v is NaN
// when a NaN or +inf entry was seen (the sequence fails, U12).

SV_DEVINL uint32_t bf16x2_max_nan(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

SV_DEVINL float fmax_nan(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}

// Warp-wide (max, first index of the max) of one pair per lane; NaN wins.
SV_DEVINL void warp_argmax(float& v, long long& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float v2 = __shfl_xor_sync(0xffffffffu, v, o);
    const long long i2 = __shfl_xor_sync(0xffffffffu, i, o);
    const bool take = (v2 != v2) ? !(v != v) || i2 < i
                      : (v != v) ? false
                                 : (v2 > v || (v2 == v && i2 < i));
    if (take) {
      v = v2;
      i = i2;
    }
  }
}

template <int DT>
SV_DEVINL float vec_elem(const uint4& q, int e) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  if constexpr (DT == 0)
    return (e & 1) ? bf16_hi(w[e >> 1]) : bf16_lo(w[e >> 1]);
  else
    return __uint_as_float(w[e]);
}

// Vector-load path: per round, the round's maximum with a NaN-propagating
// packed max; only when it beats the lane's best is the round searched (in
// index order) for the first element equal to it.
template <int DT>
SV_DEVINL void greedy_warp_vec(const Params& P, long long u, int lane, float& bv, long long& bi) {
  constexpr int kEs = DT == 0 ? 2 : 4;
  constexpr int kPerVec = 16 / kEs;
  const int len = unit_len(P, u);
  const long long e_base = (long long)(u % P.nseg) * P.seg_elems;
  const unsigned char* base = unit_row(P, u) + (size_t)e_base * kEs;
  const int nvec = len * kEs / 16;
  const uint32_t fill = DT == 0 ? 0xff80ff80u : 0xff800000u;  // -inf
  bv = neg_inf();
  bi = e_base;
  for (int i0 = 0; i0 < nvec; i0 += kStatsVec * 32) {
    uint4 v[kStatsVec];
#pragma unroll
    for (int k = 0; k < kStatsVec; ++k) {
      const int idx = i0 + k * 32 + lane;
      v[k] = idx < nvec ? ld_global_nc_v4(base + (size_t)idx * 16) : make_uint4(fill, fill, fill, fill);
    }
    // Each vector's maximum, then the round's.
    float vmax[kStatsVec];
#pragma unroll
    for (int k = 0; k < kStatsVec; ++k) {
      if constexpr (DT == 0) {
        const uint32_t m2 = bf16x2_max_nan(bf16x2_max_nan(v[k].x, v[k].y),
                                           bf16x2_max_nan(v[k].z, v[k].w));
        vmax[k] = fmax_nan(bf16_lo(m2), bf16_hi(m2));
      } else {
        vmax[k] = fmax_nan(fmax_nan(__uint_as_float(v[k].x), __uint_as_float(v[k].y)),
                           fmax_nan(__uint_as_float(v[k].z), __uint_as_float(v[k].w)));
      }
    }
    float lm = vmax[0];
#pragma unroll
    for (int k = 1; k < kStatsVec; ++k) lm = fmax_nan(lm, vmax[k]);
    if (lm != lm) {  // a NaN: the sequence fails, the index no longer matters
      bv = lm;
    } else if (bv == bv && lm > bv) {
      // The first vector holding lm, then the first element of it that does.
      int kk = 0;
#pragma unroll
      for (int k = kStatsVec - 1; k >= 0; --k)
        if (vmax[k] == lm) kk = k;
      uint4 q = v[0];
#pragma unroll
      for (int k = 1; k < kStatsVec; ++k)
        if (k == kk) q = v[k];
      int ee = 0;
#pragma unroll
      for (int e = kPerVec - 1; e >= 0; --e)
        if (vec_elem<DT>(q, e) == lm) ee = e;
      bi = e_base + (long long)(i0 + kk * 32 + lane) * kPerVec + ee;
      bv = lm;
    }
  }
  warp_argmax(bv, bi);
}

// Plain-load path for rows that are not 16-byte aligned.
template <int DT>
SV_DEVINL void greedy_warp_plain(const Params& P, long long u, int lane, float& bv, long long& bi) {
  const int len = unit_len(P, u);
  const unsigned char* rb = unit_row(P, u);
  const long long e0 = (long long)(u % P.nseg) * P.seg_elems;
  bv = neg_inf();
  bi = e0;
  for (int i = lane; i < len; i += 32) {
    const float l = load_elem<DT>(rb, e0 + i);
    if (l != l) {
      bv = l;
    } else if (bv == bv && l > bv) {
      bv = l;
      bi = e0 + i;
    }
  }
  warp_argmax(bv, bi);
}

// (max, first index) of a whole row from its segments' pairs.
SV_DEVINL void greedy_row_combine(const Params& P, long long row, int lane, float& bv,
                                  long long& bi) {
  const float2* part = P.seg_part + row * P.nseg;
  bv = neg_inf();
  bi = LLONG_MAX;
  for (int g = lane; g < P.nseg; g += 32) {
    const float2 ps = __ldcg(part + g);
    const long long i = (long long)__float_as_int(ps.y);
    const bool take = (ps.x != ps.x) ? true : (bv != bv) ? false : (ps.x > bv || (ps.x == bv && i < bi));
    if (take && !(bv != bv)) {
      bv = ps.x;
      bi = i;
    }
  }
  warp_argmax(bv, bi);
}

SV_DEVINL void greedy_scan(const Params& P, long long b, int lane) {
  const int K = P.K, R = P.rows_per_seq;  // R = K + 1
  unsigned bits = 0;
  for (int r = lane; r < R; r += 32) {
    const float2 st = __ldcg(P.row_stat + b * R + r);
    if (st.x != st.x || st.x == __int_as_float(0x7f800000)) {
      bits |= kDevNonfinite;
    } else if (st.x == neg_inf()) {
      bits |= kDevEmptyRow;
    }
  }
  for (int t = lane; t < K; t += 32) {
    const int x = P.tokens[b * K + t];
    if (x < 0 || x >= P.V) bits |= kDevTokenRange;
  }
  bits = __reduce_or_sync(0xffffffffu, bits);
  int j = K;
  if (!bits) {
    for (int t0 = 0; t0 < K; t0 += 32) {
      const int t = t0 + lane;
      bool mismatch = false;
      if (t < K) {
        const int am = __float_as_int(__ldcg(P.row_stat + b * R + t).y);
        mismatch = P.tokens[b * K + t] != am;
      }
      const unsigned mask = __ballot_sync(0xffffffffu, mismatch);
      if (mask) {
        j = t0 + __ffs(mask) - 1;
        break;
      }
    }
  } else {
    j = -1;
  }
  if (lane == 0) {
    if (bits) atomicOr(P.status, bits);
    P.n_acc[b] = j;
  }
  for (int t = lane; t <= K; t += 32) {
    int o = -1;
    if (j >= 0 && t < j) o = P.tokens[b * K + t];
    if (j >= 0 && t == j) o = __float_as_int(__ldcg(P.row_stat + b * R + j).y);
    P.out_tokens[b * (K + 1) + t] = o;
  }
}

template <int DT, bool VEC>
__global__ void __launch_bounds__(kStatsThreads, kStatsCtasPerSm) greedy_kernel(Params P) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long u = (long long)blockIdx.x * kStatsWarps + warp;
  if (u >= P.n_units) return;
  const long long row = u / P.nseg;
  const long long b = row / P.rows_per_seq;
  float bv;
  long long bi;
  if constexpr (VEC)
    greedy_warp_vec<DT>(P, u, lane, bv, bi);
  else
    greedy_warp_plain<DT>(P, u, lane, bv, bi);
  if (P.nseg > 1) {
    unsigned last = 0;
    if (lane == 0) {
      P.seg_part[u] = make_float2(bv, __int_as_float((int)bi));
      last = atomic_add_acq_rel(P.done_r + row, 1u) == (unsigned)(P.nseg - 1);
    }
    if (!__shfl_sync(0xffffffffu, last, 0)) return;
    __syncwarp();
    greedy_row_combine(P, row, lane, bv, bi);
  }
  unsigned last = 0;
  if (lane == 0) {
    P.row_stat[row] = make_float2(bv, __int_as_float((int)bi));
    last = atomic_add_acq_rel(P.done_s + b, 1u) == (unsigned)(P.rows_per_seq - 1);
  }
  if (!__shfl_sync(0xffffffffu, last, 0)) return;
  __syncwarp();
  greedy_scan(P, b, lane);
}

// ---------------------------------------------------------------- top-k filtered verification
//
// The card's §4.2 "Decoding transforms": top-k is applied to both p and q,
// then the rejection scheme runs on the filtered distributions. Each of the
// 2K+1 rows keeps its k largest logits (ties to the smaller token id, -0
// equal to +0). A row is reduced to its k kept entries in one streaming pass
// (one CTA per row): elements are compared against a running threshold, the
// k-th largest key known so far, and the few that beat it are appended to a
// candidate buffer in shared memory, which is cut back to its k largest (a
// radix select over the buffer) once it holds more than a few times k. For
// rows in random order the threshold rises fast, so nearly every element
// costs one packed max and one compare, and the row is read from memory
// once. A row whose candidates overflow the buffer (an adversarial order,
// such as ascending logits) is selected exactly by a radix select over the
// row itself instead. The kept entries' softmax is taken in fp64 and stored
// as (id, q) pairs in ascending id, and the verification runs on those pairs.

constexpr int kSelThreads = 256;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSelTile = kSelThreads * 8;  // elements per tile: 8 consecutive per thread
constexpr int kSelCap = 5120;              // candidate buffer entries
static_assert(kTopKMax == kSelThreads, "the final stage gives one kept entry per thread");

template <int DT>
SV_DEVINL bool nan_or_pos_inf(uint32_t bits) {
  if constexpr (DT == 0)
    return ((bits & 0x7fffu) > 0x7f80u) || bits == 0x7f80u;
  else
    return ((bits & 0x7fffffffu) > 0x7f800000u) || bits == 0x7f800000u;
}

// Words per thread per tile: 8 bf16 in 4 words, or 8 f32 in 8.
template <int DT>
struct SelWords {
  static constexpr int n = DT == 0 ? 4 : 8;
};

template <int DT>
SV_DEVINL uint32_t elem_bits(const uint32_t (&w)[SelWords<DT>::n], int j) {
  if constexpr (DT == 0)
    return (w[j >> 1] >> ((j & 1) * 16)) & 0xffffu;
  else
    return w[j];
}

// This thread's 8 elements of the tile starting at e0 (elements past V read
// as -inf and are marked invalid by the returned count). VEC: 16-byte loads
// (the row is 16-byte aligned and V * element size a multiple of 16).
template <int DT, bool VEC>
SV_DEVINL int load_sel_tile(const unsigned char* rb, long long e0, int V,
                            uint32_t (&w)[SelWords<DT>::n]) {
  const long long left = (long long)V - e0;
  const int nv = left <= 0 ? 0 : (left >= 8 ? 8 : (int)left);
  constexpr uint32_t kNegInf = DT == 0 ? 0xff80ff80u : 0xff800000u;
  if constexpr (VEC) {
    if constexpr (DT == 0) {
      uint4 v = make_uint4(kNegInf, kNegInf, kNegInf, kNegInf);
      if (nv > 0) v = ld_global_nc_v4(rb + e0 * 2);
      w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
    } else {
      uint4 a = make_uint4(kNegInf, kNegInf, kNegInf, kNegInf), b = a;
      if (nv > 0) a = ld_global_nc_v4(rb + e0 * 4);
      if (nv > 4) b = ld_global_nc_v4(rb + (e0 + 4) * 4);
      w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
      w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
    }
  } else {
    if constexpr (DT == 0) {
      const unsigned short* r = reinterpret_cast<const unsigned short*>(rb) + e0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t lo = 2 * j < nv ? __ldg(r + 2 * j) : 0xff80u;
        const uint32_t hi = 2 * j + 1 < nv ? __ldg(r + 2 * j + 1) : 0xff80u;
        w[j] = lo | (hi << 16);
      }
    } else {
      const uint32_t* r = reinterpret_cast<const uint32_t*>(rb) + e0;
#pragma unroll
      for (int j = 0; j < 8; ++j) w[j] = j < nv ? __ldg(r + j) : kNegInf;
    }
  }
  return nv;
}

// This thread's 8 elements of a tile that lies wholly inside the row.
template <int DT, bool VEC>
SV_DEVINL void load_full_tile(const unsigned char* rb, unsigned e0, uint32_t (&w)[SelWords<DT>::n]) {
  if constexpr (VEC) {
    if constexpr (DT == 0) {
      const uint4 v = ld_global_nc_v4(rb + (size_t)e0 * 2);
      w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
    } else {
      const uint4 a = ld_global_nc_v4(rb + (size_t)e0 * 4);
      const uint4 b = ld_global_nc_v4(rb + (size_t)e0 * 4 + 16);
      w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
      w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
    }
  } else {
    if constexpr (DT == 0) {
      const unsigned short* r = reinterpret_cast<const unsigned short*>(rb) + e0;
#pragma unroll
      for (int j = 0; j < 4; ++j) w[j] = (uint32_t)__ldg(r + 2 * j) | ((uint32_t)__ldg(r + 2 * j + 1) << 16);
    } else {
      const uint32_t* r = reinterpret_cast<const uint32_t*>(rb) + e0;
#pragma unroll
      for (int j = 0; j < 8; ++j) w[j] = __ldg(r + j);
    }
  }
}

SV_DEVINL double warp_max_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmax(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

SV_DEVINL double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Bit pattern (bf16: 16 bits) of the NaN-propagating max of one thread's 8
// values of a tile.
template <int DT>
SV_DEVINL uint32_t sel_max_bits(const uint32_t (&w)[SelWords<DT>::n]) {
  if constexpr (DT == 0) {
    const uint32_t m2 = bf16x2_max_nan(bf16x2_max_nan(w[0], w[1]), bf16x2_max_nan(w[2], w[3]));
    return __float_as_uint(fmax_nan(bf16_lo(m2), bf16_hi(m2))) >> 16;
  } else {
    return __float_as_uint(
        fmax_nan(fmax_nan(fmax_nan(__uint_as_float(w[0]), __uint_as_float(w[1])),
                          fmax_nan(__uint_as_float(w[2]), __uint_as_float(w[3]))),
                 fmax_nan(fmax_nan(__uint_as_float(w[4]), __uint_as_float(w[5])),
                          fmax_nan(__uint_as_float(w[6]), __uint_as_float(w[7])))));
  }
}

struct SelShared {
  unsigned long long buf[kSelCap];    // candidate keys
  unsigned long long keep[kTopKMax];  // the k largest, while the buffer is cut back
  unsigned hist[256];
  unsigned wsum[kSelWarps];
  unsigned long long prefix, tau, kmax;
  unsigned count, remaining, in_bucket, next_remaining, found_bin, n_keep, overflow, bad;
  unsigned cnt[3];
  double ssum;
};
// Within the default dynamic shared memory limit (no opt-in attribute needed).
static_assert(sizeof(SelShared) <= 48 * 1024, "select kernel shared memory");

// The k largest of n distinct keys key(0..n-1) of `bits` bits into buf[0, k):
// a radix select over 8-bit digits from the top key bit (the key is padded
// with zeros at the bottom to a whole number of digits), stopping once the
// selected bucket is taken whole, then one pass that keeps every key whose
// resolved digits reach the selected prefix (exactly k of them). Sets count
// = k and tau = the smallest kept key. `get(i, key)` returns false for NaN /
// +inf (sets sh.bad and returns early).
template <typename GetKey>
SV_DEVINL void sel_radix(SelShared& sh, long long n, int k, int bits, GetKey get) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int pad = (8 - bits % 8) % 8, top = bits + pad;
  if (tid == 0) {
    sh.prefix = 0;
    sh.remaining = (unsigned)k;
    sh.n_keep = 0;
    sh.tau = ~0ull;
  }
  int resolved = 0;
  unsigned bad = 0;
  for (;;) {
    const int shift = top - resolved - 8;
    sh.hist[tid] = 0;
    __syncthreads();
    const bool all = shift + 8 >= 64;
    const unsigned long long pre = all ? 0ull : (sh.prefix >> (shift + 8));
    for (long long base = 0; base < n; base += kSelThreads) {
      const long long i = base + tid;
      unsigned bin = 256u;
      if (i < n) {
        unsigned long long key;
        bad |= get(i, key) ? 0u : 1u;
        key <<= pad;
        if (all || (key >> (shift + 8)) == pre) bin = (unsigned)((key >> shift) & 255u);
      }
      const unsigned grp = __match_any_sync(0xffffffffu, bin);
      if (bin < 256u && lane == __ffs(grp) - 1) atomicAdd(&sh.hist[bin], __popc(grp));
    }
    if (__syncthreads_or(bad)) {
      if (tid == 0) sh.bad = 1;
      __syncthreads();
      return;
    }
    // Thread t holds bin 255 - t; the inclusive scan over t counts the
    // matching keys at or above each bin.
    const unsigned tot = sh.hist[255 - tid];
    unsigned inc = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += y;
    }
    if (lane == 31) sh.wsum[warp] = inc;
    __syncthreads();
    for (int w = 0; w < warp; ++w) inc += sh.wsum[w];
    const unsigned rem = sh.remaining;
    if (inc >= rem && inc - tot < rem) {
      sh.found_bin = 255u - (unsigned)tid;
      sh.in_bucket = tot;
      sh.next_remaining = rem - (inc - tot);
    }
    __syncthreads();
    if (tid == 0) {
      sh.prefix |= (unsigned long long)sh.found_bin << shift;
      sh.remaining = sh.next_remaining;
    }
    resolved += 8;
    __syncthreads();
    if (sh.in_bucket == sh.remaining || resolved >= top) break;
  }
  const int lo = top - resolved;
  const unsigned long long thr = sh.prefix >> lo;
  for (long long i = tid; i < n; i += kSelThreads) {
    unsigned long long key;
    get(i, key);
    if (((key << pad) >> lo) >= thr) {
      const unsigned s = atomicAdd(&sh.n_keep, 1u);
      if (s < (unsigned)kTopKMax) sh.keep[s] = key;
    }
  }
  __syncthreads();
  if (tid < k) {
    const unsigned long long key = sh.keep[tid];
    sh.buf[tid] = key;
    atomicMin(&sh.tau, key);
  }
  if (tid == 0) sh.count = (unsigned)k;
  __syncthreads();
}

// The largest 16-bit x such that at least k of the threads' values m[0..3]
// (those with ok set) are >= x, by a radix select over two 8-bit digits with
// block-wide histograms; 0 when fewer than k values are given.
SV_DEVINL uint32_t sel_kth16(SelShared& sh, const uint32_t (&m)[4], const bool (&ok)[4], int k) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t prefix = 0;
  unsigned rem = (unsigned)k;
  for (int pass = 0; pass < 2; ++pass) {
    const int shift = pass == 0 ? 8 : 0;
    sh.hist[tid] = 0;
    __syncthreads();
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const bool in = ok[u] && (pass == 0 || (m[u] >> 8) == prefix);
      const unsigned bin = in ? ((m[u] >> shift) & 255u) : 256u;
      const unsigned grp = __match_any_sync(0xffffffffu, bin);
      if (bin < 256u && lane == __ffs(grp) - 1) atomicAdd(&sh.hist[bin], __popc(grp));
    }
    __syncthreads();
    const unsigned tot = sh.hist[255 - tid];
    unsigned inc = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += y;
    }
    if (lane == 31) sh.wsum[warp] = inc;
    __syncthreads();
    for (int w = 0; w < warp; ++w) inc += sh.wsum[w];
    if (pass == 0 && tid == kSelThreads - 1) sh.found_bin = inc;  // all the values
    if (inc >= rem && inc - tot < rem) {
      sh.in_bucket = 255u - (unsigned)tid;
      sh.next_remaining = rem - (inc - tot);
    }
    __syncthreads();
    if (pass == 0 && sh.found_bin < (unsigned)k) return 0;
    prefix = pass == 0 ? sh.in_bucket : ((prefix << 8) | sh.in_bucket);
    rem = sh.next_remaining;
    __syncthreads();
  }
  return prefix;
}

template <int DT>
struct TileWords {
  uint32_t v[SelWords<DT>::n];
};

// The rare path of the collecting pass, for a thread whose tile maximum
// reached the threshold value (or is NaN): appends its elements (the first
// nv of 8, from element e0) whose key beats thr to the candidate buffer, and
// returns whether one of them is NaN or +inf. Out of line, so that the
// streaming loop stays small.
template <int DT>
__device__ __noinline__ bool sel_slow(SelShared& sh, TileWords<DT> t, int nv, unsigned e0, int V,
                                      int ib, unsigned long long thr) {
  bool bad = false;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (j >= nv) break;
    const uint32_t bits = elem_bits<DT>(t.v, j);
    if (nan_or_pos_inf<DT>(bits)) {
      bad = true;
      continue;
    }
    const unsigned long long key =
        ((unsigned long long)value_key<DT>(bits) << ib) | (unsigned long long)(V - 1 - (int)(e0 + j));
    if (key > thr) {
      const unsigned pos = atomicAdd(&sh.count, 1u);
      if (pos < (unsigned)kSelCap)
        sh.buf[pos] = key;
      else
        sh.overflow = 1;
    }
  }
  return bad;
}

// Float value (NaN-propagating max) of one thread's 8 values of a tile.
template <int DT>
SV_DEVINL float sel_max_f(const uint32_t (&w)[SelWords<DT>::n]) {
  const uint32_t mb = sel_max_bits<DT>(w);
  return __uint_as_float(DT == 0 ? mb << 16 : mb);
}

// One CTA per row of the B (2K+1) rows: the row's k kept entries, as token
// ids in ascending order with their fp64 probabilities softmax(l / T) over
// the kept set, and the probability of the row's drafted token; the row's
// flag is 0, kDevNonfinite (NaN or +inf anywhere in the row) or kDevEmptyRow
// (every kept entry -inf).
//
// A first pass over a leading sample of the row (at least kSelSampleTiles
// tiles, at least an eighth of the row) takes every thread's maxima over its
// elements of it (4 per thread), and x, the k-th largest of them (to 16 bits
// of the value key), bounds the candidates from below: at least k elements
// are at least x, so none below x is among the row's k largest. The second
// pass reads the whole row (the sample again from L2) and appends the
// elements at or above x to the buffer; about k times the row/sample ratio
// of them for rows in random order. Neither pass has a block-wide barrier,
// so every warp keeps its loads in flight.
constexpr int kSelSampleTiles = 16;

template <int DT, bool VEC>
__global__ void __launch_bounds__(kSelThreads, DT == 0 ? 5 : 4) topk_select_kernel(Params P) {
  extern __shared__ __align__(16) unsigned char sel_smem[];
  SelShared& sh = *reinterpret_cast<SelShared*>(sel_smem);
  constexpr int W = SelWords<DT>::n;
  constexpr int NB = DT == 0 ? 16 : 32;  // value key bits
  constexpr int S = DT == 0 ? 4 : 2;      // tiles loaded per step: 64 bytes per thread
  const int tid = threadIdx.x, lane = tid & 31;
  const long long row = blockIdx.x;
  const unsigned char* rb = row_base(P, row / P.rows_per_seq, (int)(row % P.rows_per_seq));
  const int V = P.V, k = P.top_k, ib = P.key_ibits;
  const int top = NB + ib;  // key bits
  const unsigned long long idmask = (1ull << ib) - 1;
  if (tid == 0) {
    sh.count = 0;
    sh.overflow = 0;
    sh.bad = 0;
    sh.kmax = 0;
    sh.ssum = 0.0;
  }
  bool bad = false;
  const unsigned ntiles = (unsigned)(((long long)V + kSelTile - 1) / kSelTile);
  const unsigned nfull = (unsigned)V / kSelTile;  // tiles wholly inside the row
  const unsigned nsample = min(ntiles, max((unsigned)kSelSampleTiles, (ntiles + 7) / 8));
  // Pass 1 over the sample: NaN-propagating maxima in 4 slots (tile mod 4).
  float mx[4] = {-CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F};
  bool ok[4] = {false, false, false, false};
  const unsigned sfull = min(nsample, nfull) / 4 * 4;
  for (unsigned t = 0; t < sfull; t += 4) {
    uint32_t w[4][W];
#pragma unroll
    for (int u = 0; u < 4; ++u) load_full_tile<DT, VEC>(rb, (t + u) * kSelTile + tid * 8, w[u]);
#pragma unroll
    for (int u = 0; u < 4; ++u) mx[u] = fmax_nan(mx[u], sel_max_f<DT>(w[u]));
  }
  if (sfull > 0) ok[0] = ok[1] = ok[2] = ok[3] = true;
  for (unsigned t = sfull; t < nsample; ++t) {
    uint32_t w[W];
    const int nv = load_sel_tile<DT, VEC>(rb, (long long)t * kSelTile + tid * 8, V, w);
    mx[t % 4] = fmax_nan(mx[t % 4], sel_max_f<DT>(w));
    ok[t % 4] |= nv > 0;
  }
  uint32_t m16[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const uint32_t mb = DT == 0 ? (__float_as_uint(mx[u]) >> 16) : __float_as_uint(mx[u]);
    ok[u] = ok[u] && !nan_or_pos_inf<DT>(mb);  // a failing row is caught by pass 2
    m16[u] = value_key<DT>(mb) >> (NB - 16);
  }
  __syncthreads();  // the shared counters above
  const uint32_t x16 = sel_kth16(sh, m16, ok, k);
  // Candidates: value key >= xv = x16 << (NB - 16), i.e. key > thr; a tile is
  // looked at element by element only when its maximum reaches xv's value.
  const uint32_t xv = x16 << (NB - 16);
  const unsigned long long thr = x16 ? ((unsigned long long)xv << ib) - 1 : 0ull;
  const float tvf = x16 ? key_value<DT>((unsigned long long)xv, 0) : -CUDART_INF_F;
  // Pass 2 over the row, appending the candidates.
  const unsigned rfull = nfull / S * S;
  for (unsigned t = 0; t < rfull; t += S) {
    uint32_t w[S][W];
#pragma unroll
    for (int u = 0; u < S; ++u) load_full_tile<DT, VEC>(rb, (t + u) * kSelTile + tid * 8, w[u]);
#pragma unroll
    for (int u = 0; u < S; ++u) {
      if (!(sel_max_f<DT>(w[u]) < tvf)) {  // at or above the threshold value, or NaN
        TileWords<DT> tw;
#pragma unroll
        for (int i = 0; i < W; ++i) tw.v[i] = w[u][i];
        bad |= sel_slow<DT>(sh, tw, 8, (t + u) * kSelTile + tid * 8, V, ib, thr);
      }
    }
  }
  for (unsigned t = rfull; t < ntiles; ++t) {
    uint32_t w[W];
    const unsigned e0 = t * kSelTile + tid * 8;
    const int nv = load_sel_tile<DT, VEC>(rb, (long long)e0, V, w);
    if (nv > 0 && !(sel_max_f<DT>(w) < tvf)) {
      TileWords<DT> tw;
#pragma unroll
      for (int i = 0; i < W; ++i) tw.v[i] = w[i];
      bad |= sel_slow<DT>(sh, tw, nv, e0, V, ib, thr);
    }
  }
  if (__syncthreads_or(bad)) {
    if (tid == 0) P.topk_flag[row] = kDevNonfinite;
    return;
  }
  if (sh.overflow) {
    // Exact selection over the row itself (NaN / +inf are checked again, as
    // the streaming pass stopped early).
    sel_radix(sh, V, k, top, [&](long long i, unsigned long long& key) {
      uint32_t bits;
      if constexpr (DT == 0)
        bits = __ldg(reinterpret_cast<const unsigned short*>(rb) + i);
      else
        bits = __ldg(reinterpret_cast<const uint32_t*>(rb) + i);
      key = ((unsigned long long)value_key<DT>(bits) << ib) | (unsigned long long)(V - 1 - i);
      return !nan_or_pos_inf<DT>(bits);
    });
    if (sh.bad) {
      if (tid == 0) P.topk_flag[row] = kDevNonfinite;
      return;
    }
  } else if (sh.count > (unsigned)k) {
    sel_radix(sh, sh.count, k, top, [&](long long i, unsigned long long& key) {
      key = sh.buf[i];
      return true;
    });
  }
  // buf[0, k): the kept keys. Softmax(l / T) over them in fp64: the max is
  // the largest key's value (division by T > 0 keeps the order).
  unsigned long long key = 0;
  if (tid < k) {
    key = sh.buf[tid];
    atomicMax(&sh.kmax, key);
  }
  __syncthreads();
  const double m = (double)key_value<DT>(sh.kmax, ib) / P.temp_d;
  if (m == -CUDART_INF) {
    if (tid == 0) P.topk_flag[row] = kDevEmptyRow;
    return;
  }
  const int id = V - 1 - (int)(key & idmask);
  const double e = tid < k ? exp((double)key_value<DT>(key, ib) / P.temp_d - m) : 0.0;
  const double ws = warp_sum_d(e);
  if (lane == 0) atomicAdd(&sh.ssum, ws);
  // Position in ascending id: the kept entries with a smaller id, i.e. a
  // larger low (V-1-id) part.
  int pos = 0;
  if (tid < k) {
    const unsigned long long mine = key & idmask;
    for (int s = 0; s < k; ++s) pos += (sh.buf[s] & idmask) > mine ? 1 : 0;
  }
  __syncthreads();
  const double q = e / sh.ssum;
  const int r = (int)(row % P.rows_per_seq), K = P.K;
  const long long b = row / P.rows_per_seq;
  // The drafted token this row is tested at: x_t for target row t < K and for
  // draft row K+1+t; the bonus row K has none.
  const int x = r == K ? -1 : __ldg(P.tokens + b * K + (r < K ? r : r - K - 1));
  if (tid < k) {
    P.topk_idx[row * k + pos] = id;
    P.topk_prob[row * k + pos] = q;
    if (id == x) P.topk_at[row] = q;
  }
  if (tid == 0) P.topk_flag[row] = 0;
  // A drafted token outside the kept set has probability 0 in this row.
  if (!__syncthreads_or(tid < k && id == x) && tid == 0) P.topk_at[row] = 0.0;
}

// Position of `x` in ascending ids[0, n), or -1.
SV_DEVINL int sorted_find(const int* ids, int n, int x) {
  int lo = 0, hi = n - 1;
  while (lo <= hi) {
    const int mid = (lo + hi) >> 1;
    const int v = ids[mid];
    if (v == x) return mid;
    if (v < x)
      lo = mid + 1;
    else
      hi = mid - 1;
  }
  return -1;
}

constexpr int kTvThreads = kTopKMax;  // one kept entry per thread

struct TopKVerifyShared {
  int pid[kTopKMax];
  double pprob[kTopKMax];
  double wsum[kTvThreads / 32];
  unsigned bits;
  int j, first, last;
};

// One CTA per sequence: the verification of `verify` on the kept entries.
// The thresholds use the per-row probabilities of the drafted tokens; the
// draw walks the k kept entries of the drawn row in ascending id, one per
// thread, with the draft row's kept list in shared memory for the residual.
#if SV_TU_HAS(2)
__global__ void __launch_bounds__(kTvThreads) topk_verify_kernel(Params P) {
  __shared__ TopKVerifyShared sh;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long b = blockIdx.x;
  const int K = P.K, R = P.rows_per_seq, k = P.top_k;
  const long long row0 = b * R;
  if (tid == 0) {
    sh.bits = 0;
    sh.j = K;
    sh.first = INT_MAX;
    sh.last = -1;
  }
  __syncthreads();
  unsigned bits = 0;
  for (int r = tid; r < R; r += kTvThreads) bits |= __ldcg(P.topk_flag + row0 + r);
  for (int t = tid; t < K; t += kTvThreads) {
    const int x = P.tokens[b * K + t];
    if (x < 0 || x >= P.V) bits |= kDevTokenRange;
  }
  for (int t = tid; t < K + 2; t += kTvThreads) {
    const float u = P.uniforms[b * (K + 2) + t];
    if (!(u >= 0.0f && u <= 1.0f)) bits |= kDevUniformRange;
  }
  bits = __reduce_or_sync(0xffffffffu, bits);
  if (lane == 0 && bits) atomicOr(&sh.bits, bits);
  __syncthreads();
  bits = sh.bits;
  if (bits) {
    if (tid == 0) {
      atomicOr(P.status, bits);
      P.n_acc[b] = -1;
    }
    for (int t = tid; t <= K; t += kTvThreads) P.out_tokens[b * (K + 1) + t] = -1;
    return;
  }
  // Acceptance tests: the first t whose u_t < min(1, q/p) fails.
  for (int t = tid; t < K; t += kTvThreads) {
    const double q = __ldcg(P.topk_at + row0 + t), p = __ldcg(P.topk_at + row0 + K + 1 + t);
    const double thr = p > 0.0 ? fmin(1.0, q / p) : (q > 0.0 ? 1.0 : 0.0);
    if (!((double)P.uniforms[b * (K + 2) + t] < thr)) atomicMin(&sh.j, t);
  }
  __syncthreads();
  const int j = sh.j;
  const bool resid = j < K;
  const long long qrow = row0 + (resid ? j : K), prow = row0 + K + 1 + j;
  if (resid && tid < k) {
    sh.pid[tid] = __ldcg(P.topk_idx + prow * k + tid);
    sh.pprob[tid] = __ldcg(P.topk_prob + prow * k + tid);
  }
  const int id = tid < k ? __ldcg(P.topk_idx + qrow * k + tid) : 0;
  const double q = tid < k ? __ldcg(P.topk_prob + qrow * k + tid) : 0.0;
  __syncthreads();
  double w = q;
  if (resid && tid < k) {
    const int pos = sorted_find(sh.pid, k, id);
    w = fmax(0.0, q - (pos >= 0 ? sh.pprob[pos] : 0.0));
  }
  // Inclusive scan of the weights in ascending id; the last entry is the total.
  auto block_scan = [&](double v) -> double {
    double inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += y;
    }
    if (lane == 31) sh.wsum[warp] = inc;
    __syncthreads();
    for (int w2 = 0; w2 < warp; ++w2) inc += sh.wsum[w2];
    return inc;
  };
  double c = block_scan(w);
  double total = 0.0;
#pragma unroll
  for (int w2 = 0; w2 < kTvThreads / 32; ++w2) total += sh.wsum[w2];
  if (resid && !(total > 0.0)) {  // zero residual: fall back to q (U5)
    __syncthreads();
    w = q;
    c = block_scan(w);
    total = 0.0;
#pragma unroll
    for (int w2 = 0; w2 < kTvThreads / 32; ++w2) total += sh.wsum[w2];
  }
  const double target = (double)P.uniforms[b * (K + 2) + (resid ? K : K + 1)] * total;
  if (tid < k && w > 0.0) {
    atomicMax(&sh.last, tid);
    if (c > target) atomicMin(&sh.first, tid);
  }
  __syncthreads();
  const int pick = sh.first != INT_MAX ? sh.first : sh.last;
  if (tid == pick) P.out_tokens[b * (K + 1) + j] = id;
  if (tid == 0) {
    P.n_acc[b] = j;
    if (pick < 0) P.out_tokens[b * (K + 1) + j] = -1;
  }
  for (int t = tid; t <= K; t += kTvThreads) {
    if (t < j) P.out_tokens[b * (K + 1) + t] = P.tokens[b * K + t];
    if (t > j) P.out_tokens[b * (K + 1) + t] = -1;
  }
}
#endif  // SV_TU_HAS(2)

// ---------------------------------------------------------------- nucleus (top-p) filtered verification
//
// The card's §4.2 "Decoding transforms" with the nucleus rule: each of the
// 2K+1 rows keeps the shortest prefix of its entries, in (logit descending,
// id ascending) order, whose probability softmax(l / T) reaches top_p. The cut
// is found per row without a sort, as a key K* (the order-preserving value key
// above V-1-id): an entry is kept iff its key is >= K*. One CTA per row:
//   1. the row maximum m (and NaN / +inf);
//   2. levels of mass histograms over d = (m - l) / T: level L bins d at width
//      4 / 16^(L-1), so a level-L bin splits into 16 level-(L+1) bins exactly
//      (d * 2^j is exact); each level keeps the bin in which the running mass,
//      from the top, reaches p * S (S, the row's total, from level 1), and
//      adds the bins above it to the mass above;
//   3. once that bin holds at most kTpCap entries, they are gathered with
//      their weights and K* is found among them by a radix select on the key
//      weighted by mass; a bin that never gets that small (heavy ties) is
//      resolved bit by bit over the key with a pass per bit.
// Weights are exp((l - m) / T) in float-float (the same exp as the unfiltered
// path, ~1e-12 relative); masses are summed as float-float per thread and in
// fp64 across threads. This kernel re-reads the row from global memory for
// every pass; it serves rows too long for a cluster's shared memory (the
// cluster kernel below takes the others). Like that kernel it leaves the row's
// statistics (m, S_kept) for the verification.

constexpr int kTpThreads = 256;
constexpr int kTpBins = 16;
constexpr int kTpCap = 1024;
constexpr int kTpMaxLevels = 6;

struct TopPShared {
  float2 tab[256];
  union {
    struct {  // level histograms: per-thread float-float masses and counts
      float bhi[kTpBins][kTpThreads], blo[kTpBins][kTpThreads];
      unsigned bcnt[kTpBins][kTpThreads];
    } lv;
    struct {  // the cut bin's entries, and the mass-weighted radix select over them
      unsigned long long ckey[kTpCap];
      double cw[kTpCap];
      double mh[256];
      unsigned ch[256];
    } rs;
  } u;
  double red[kTpThreads / 32];
  double wsum[kTpThreads / 32];
  double binmass[kTpBins];
  unsigned bincount[kTpBins];
  unsigned n_cand, wcnt[kTpThreads / 32];
  unsigned long long cutmin, prefix;
  int sel;
  double sel_above;
  unsigned sel_count;
};

SV_DEVINL double tp_block_sum(TopPShared& sh, double v) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum_d(v);
  __syncthreads();
  if (lane == 0) sh.red[warp] = v;
  __syncthreads();
  double r = 0.0;
#pragma unroll
  for (int w = 0; w < kTpThreads / 32; ++w) r += sh.red[w];
  return r;
}

// Level-L bins of d have width 16^-(L-1): index floor(d * 16^(L-1)) (exact:
// the product is a power-of-two scaling), clamped far above any real index.
SV_DEVINL float tp_scale(int level) { return ldexpf(1.0f, 4 * (level - 1)); }
SV_DEVINL long long tp_index(float d, float sc) { return (long long)floorf(fminf(d * sc, 1e15f)); }

template <int DT>
SV_DEVINL float tp_float(uint32_t b) { return __uint_as_float(DT == 0 ? b << 16 : b); }

// Element j of a tile's words, selected without indexing the array at run time.
template <int DT>
SV_DEVINL uint32_t tp_pick(const uint32_t (&w)[SelWords<DT>::n], int j) {
  uint32_t r = elem_bits<DT>(w, 0);
#pragma unroll
  for (int k = 1; k < 8; ++k) r = j == k ? elem_bits<DT>(w, k) : r;
  return r;
}

template <int DT, bool VEC>
__global__ void __launch_bounds__(kTpThreads, 3) topp_cut_kernel(Params P) {
  extern __shared__ __align__(16) unsigned char tp_smem[];
  TopPShared& sh = *reinterpret_cast<TopPShared*>(tp_smem);
  constexpr int W = SelWords<DT>::n;
  constexpr int NB = DT == 0 ? 16 : 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long row = blockIdx.x;
  const unsigned char* rb = row_base(P, row / P.rows_per_seq, (int)(row % P.rows_per_seq));
  const int V = P.V, ib = P.key_ibits;
  const int bits = NB + ib;
  const bool unit_t = P.unit_t != 0;
  sh.tab[tid] = kSvExp2Table[tid];
  const unsigned ntiles = (unsigned)(((long long)V + kSelTile - 1) / kSelTile);
  auto key_of = [&](uint32_t b, unsigned i) -> unsigned long long {
    return ((unsigned long long)value_key<DT>(b) << ib) | (unsigned long long)(V - 1 - (int)i);
  };
  // Visit the row 4 tiles at a time (4 loads in flight per thread); fn(w, nv,
  // e0) gets one tile's words, its valid count and its first element.
  auto for_tiles = [&](auto&& fn) {
    for (unsigned t = 0; t < ntiles; t += 4) {
      uint32_t w[4][W];
      int nv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        nv[u] = load_sel_tile<DT, VEC>(rb, (long long)(t + u) * kSelTile + tid * 8, V, w[u]);
#pragma unroll
      for (int u = 0; u < 4; ++u) fn(w[u], nv[u], (t + u) * kSelTile + tid * 8);
    }
  };
  // 1. The maximum, and NaN / +inf (NaN-propagating packed maxima).
  float mf = -CUDART_INF_F;
  for_tiles([&](const uint32_t (&w)[W], int, unsigned) {
    mf = fmax_nan(mf, tp_float<DT>(sel_max_bits<DT>(w)));
  });
  bool bad = isnan(mf) || mf == CUDART_INF_F;
  float m = mf;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) sh.red[warp] = m;
  const bool any_bad = __syncthreads_or(bad);
  m = (float)sh.red[0];
  for (int w2 = 1; w2 < kTpThreads / 32; ++w2) m = fmaxf(m, (float)sh.red[w2]);
  if (any_bad || m == -CUDART_INF_F) {
    // A failing row: the verification reports it from the statistics.
    if (tid == 0) {
      P.topp_cut[row] = 0;
      if (P.topp_kept) P.topp_kept[row] = V;
      P.row_stat[row] = any_bad ? make_float2(0.0f, __int_as_float(0x7fc00000))
                                : make_float2(-CUDART_INF_F, 0.0f);
    }
    return;
  }
  // Entries of the bin `parent` at scale sc: index(d) == parent (>= parent
  // for an open bin, the last bin of a level holding everything below), with
  // d = (m - l) / T, i.e. l in (m - T (parent+1)/sc, m - T parent/sc]. A
  // widened value window screens elements before the exact test.
  auto window = [&](float sc, long long parent, bool open, float& lo, float& hi) {
    const double T = P.temp_d;
    const double a = (double)m - T * (double)(parent + 1) / (double)sc;
    const double b = (double)m - T * (double)parent / (double)sc;
    const double slack = (fabs((double)m) + T * (double)(parent + 1) / (double)sc) * 1e-5 + 1e-30;
    lo = open ? -CUDART_INF_F : (float)(a - slack);
    hi = (float)(b + slack);
  };
  auto member = [&](float d, float sc, long long parent, bool open) {
    const long long i = tp_index(d, sc);
    return open ? i >= parent : i == parent;
  };
  double target = 0.0, above = 0.0;
  unsigned count_above = 0;  // entries in the bins above the cut bin, over the levels
  unsigned long long cut = 0;
  int level = 1;
  long long parent = 0;  // the bin, at level - 1, that holds the cut
  bool open = false;     // that bin is the open last bin of its level
  bool gathered = false;
  for (; level <= kTpMaxLevels; ++level) {
    const float sc = tp_scale(level), psc = tp_scale(level - 1);
#pragma unroll
    for (int b = 0; b < kTpBins; ++b) {
      sh.u.lv.bhi[b][tid] = 0.0f;
      sh.u.lv.blo[b][tid] = 0.0f;
      sh.u.lv.bcnt[b][tid] = 0;
    }
    auto add = [&](float d, ff wt) {
      const long long r = tp_index(d, sc) - (level > 1 ? 16 * parent : 0);
      const int bin = (int)(r < 15 ? r : 15);
      ff acc = {sh.u.lv.bhi[bin][tid], sh.u.lv.blo[bin][tid]};
      ff_accumulate(acc, wt);
      sh.u.lv.bhi[bin][tid] = acc.hi;
      sh.u.lv.blo[bin][tid] = acc.lo;
      sh.u.lv.bcnt[bin][tid] += 1;
    };
    if (level == 1) {
      // Every entry: the weights of element pairs with the packed (f32x2)
      // exponential, lane for lane the same operations as exp_ff.
      const float2 nm2 = make_float2(-m, -m);
      for_tiles([&](const uint32_t (&w)[W], int nv, unsigned) {
#pragma unroll
        for (int j = 0; j < 8; j += 2) {
          const float2 l2 = make_float2(tp_float<DT>(elem_bits<DT>(w, j)),
                                        tp_float<DT>(elem_bits<DT>(w, j + 1)));
          const ff2 x = scaled_diff2(l2, nm2, P.ih, P.il, unit_t);
          const ff2 wt = exp_ff2(x.hi, x.lo, sh.tab);
          if (j < nv) add(-x.hi.x, ff{wt.hi.x, wt.lo.x});
          if (j + 1 < nv) add(-x.hi.y, ff{wt.hi.y, wt.lo.y});
        }
      });
    } else {
      float lo, hi;
      window(psc, parent, open, lo, hi);
      for_tiles([&](const uint32_t (&w)[W], int nv, unsigned) {
        unsigned cand = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float l = tp_float<DT>(elem_bits<DT>(w, j));
          if (j < nv && l >= lo && l <= hi) cand |= 1u << j;
        }
        while (cand) {
          const int j = __ffs(cand) - 1;
          cand &= cand - 1;
          const ff x = scaled_diff(tp_float<DT>(tp_pick<DT>(w, j)), m, P.ih, P.il, unit_t);
          const float d = -x.hi;
          if (!member(d, psc, parent, open)) continue;
          add(d, exp_ff(x.hi, x.lo, sh.tab));
        }
      });
    }
    __syncthreads();
    // Bin totals: warp w sums bins 2w and 2w+1 over the threads.
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int b = 2 * warp + h;
      double s = 0.0;
      unsigned c = 0;
      for (int t = lane; t < kTpThreads; t += 32) {
        s += (double)sh.u.lv.bhi[b][t] + (double)sh.u.lv.blo[b][t];
        c += sh.u.lv.bcnt[b][t];
      }
      s = warp_sum_d(s);
      c = __reduce_add_sync(0xffffffffu, c);
      if (lane == 0) {
        sh.binmass[b] = s;
        sh.bincount[b] = c;
      }
    }
    __syncthreads();
    if (level == 1) {  // S: every entry is in one of the level-1 bins
      double S = 0.0;
      for (int b = 0; b < kTpBins; ++b) S += sh.binmass[b];
      target = (double)P.top_p * S;
    }
    // The bin where the running mass from the top reaches the target. If
    // rounding (the bins re-sum the parent bin in another order) leaves the
    // target just out of reach, the cut is at the end of the parent bin: its
    // last non-empty bin.
    int bstar = -1, last = -1;
    double a = above;
    for (int b = 0; b < kTpBins; ++b) {
      if (sh.bincount[b] == 0) continue;
      last = b;
      if (a + sh.binmass[b] >= target) {
        bstar = b;
        break;
      }
      a += sh.binmass[b];
    }
    if (bstar < 0) {
      bstar = last;
      a -= sh.binmass[last];
    }
    above = a;
    for (int b = 0; b < bstar; ++b) count_above += sh.bincount[b];
    const unsigned count = sh.bincount[bstar];
    parent = (level > 1 ? 16 * parent : 0) + bstar;
    open = bstar == kTpBins - 1 && (level == 1 || open);
    __syncthreads();
    if (count <= (unsigned)kTpCap) {
      gathered = true;
      break;
    }
  }
  if (gathered) {
    // 3. Gather the bin's entries with their weights (the level histograms'
    // memory is reused from here).
    const float sc = tp_scale(level);
    if (tid == 0) {
      sh.n_cand = 0;
      sh.cutmin = ~0ull;
    }
    __syncthreads();
    float lo, hi;
    window(sc, parent, open, lo, hi);
    for_tiles([&](const uint32_t (&w)[W], int nv, unsigned e0) {
      unsigned cand = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float l = tp_float<DT>(elem_bits<DT>(w, j));
        if (j < nv && l >= lo && l <= hi) cand |= 1u << j;
      }
      while (cand) {
        const int j = __ffs(cand) - 1;
        cand &= cand - 1;
        const uint32_t b = tp_pick<DT>(w, j);
        const ff x = scaled_diff(tp_float<DT>(b), m, P.ih, P.il, unit_t);
        if (!member(-x.hi, sc, parent, open)) continue;
        const unsigned s = atomicAdd(&sh.n_cand, 1u);
        if (s < (unsigned)kTpCap) {
          sh.u.rs.ckey[s] = key_of(b, e0 + j);
          sh.u.rs.cw[s] = ff_to_double(exp_ff(x.hi, x.lo, sh.tab));
        }
      }
    });
    __syncthreads();
    const unsigned n = min(sh.n_cand, (unsigned)kTpCap);
    // Radix select over the candidates' keys, 8-bit digits from the top,
    // weighted by mass: the largest key K* with above + mass(key >= K*) >=
    // target. Thread t holds bin 255 - t; an fp64 scan over the threads gives
    // the mass at or above each bin.
    const int pad = (8 - bits % 8) % 8, top = bits + pad;
    unsigned long long prefix = 0;
    double abv = above;
    int resolved = 0;
    while (resolved < top) {
      const int shift = top - resolved - 8;
      sh.u.rs.mh[tid] = 0.0;
      sh.u.rs.ch[tid] = 0;
      if (tid == 0) sh.sel = -1;
      __syncthreads();
      for (unsigned i = tid; i < n; i += kTpThreads) {
        const unsigned long long k = sh.u.rs.ckey[i] << pad;
        if (resolved == 0 || (k >> (shift + 8)) == (prefix >> (shift + 8))) {
          const unsigned bin = (unsigned)((k >> shift) & 255u);
          atomicAdd(&sh.u.rs.mh[bin], sh.u.rs.cw[i]);
          atomicAdd(&sh.u.rs.ch[bin], 1u);
        }
      }
      __syncthreads();
      const double mk = sh.u.rs.mh[255 - tid];
      const unsigned ck = sh.u.rs.ch[255 - tid];
      double inc = mk;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const double y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
      }
      if (lane == 31) sh.wsum[warp] = inc;
      __syncthreads();
      for (int w2 = 0; w2 < warp; ++w2) inc += sh.wsum[w2];
      if (ck > 0 && abv + inc >= target && abv + inc - mk < target) {
        sh.sel = 255 - tid;
        sh.sel_above = abv + inc - mk;
        sh.sel_count = ck;
      }
      __syncthreads();
      if (tid == 0 && sh.sel < 0) {
        // Rounding: the target is just out of reach; the cut is the last key.
        double a2 = abv;
        int last = -1;
        for (int b = 255; b >= 0; --b) {
          if (sh.u.rs.ch[b] == 0) continue;
          last = b;
          a2 += sh.u.rs.mh[b];
        }
        if (last >= 0) {
          sh.sel = last;
          sh.sel_above = a2 - sh.u.rs.mh[last];
          sh.sel_count = sh.u.rs.ch[last];
        } else {
          sh.sel_count = 0;
        }
      }
      __syncthreads();
      const int sel = sh.sel;
      prefix |= (unsigned long long)(sel < 0 ? 0 : sel) << shift;
      abv = sh.sel_above;
      resolved += 8;
      if (sh.sel_count <= 1) break;
      __syncthreads();
    }
    // The single key under the prefix.
    const int lo_bits = top - resolved;
    for (unsigned i = tid; i < n; i += kTpThreads) {
      const unsigned long long k = sh.u.rs.ckey[i] << pad;
      if ((k >> lo_bits) == (prefix >> lo_bits)) atomicMin(&sh.cutmin, sh.u.rs.ckey[i]);
    }
    __syncthreads();
    cut = sh.cutmin;
    // Kept: the entries above the cut bin, and the candidates at or above K*;
    // their mass is the row's kept total S_kept.
    unsigned c = 0;
    double kmass = 0.0;
    for (unsigned i = tid; i < n; i += kTpThreads)
      if (sh.u.rs.ckey[i] >= cut) {
        ++c;
        kmass += sh.u.rs.cw[i];
      }
    c = __reduce_add_sync(0xffffffffu, c);
    if (lane == 0) sh.wcnt[warp] = c;
    kmass = tp_block_sum(sh, kmass);
    if (tid == 0) {
      unsigned tot = count_above;
      for (int w2 = 0; w2 < kTpThreads / 32; ++w2) tot += sh.wcnt[w2];
      P.topp_cut[row] = cut;
      if (P.topp_kept) P.topp_kept[row] = (int)tot;
      P.row_stat[row] = make_float2(m, (float)(above + kmass));
    }
    return;
  }
  // Heavy ties around the cut: bit by bit over the key, one pass per bit,
  // with the exact mass of the keys at or above the trial cut.
  unsigned long long x = 0;
  for (int bit = bits - 1; bit >= 0; --bit) {
    const unsigned long long y = x | (1ull << bit);
    ff part = {0.0f, 0.0f};
    for_tiles([&](const uint32_t (&w)[W], int nv, unsigned e0) {
      for (int j = 0; j < nv; ++j) {
        const uint32_t b = tp_pick<DT>(w, j);
        if (key_of(b, e0 + j) >= y) {
          const ff xx = scaled_diff(tp_float<DT>(b), m, P.ih, P.il, unit_t);
          ff_accumulate(part, exp_ff(xx.hi, xx.lo, sh.tab));
        }
      }
    });
    if (tp_block_sum(sh, ff_to_double(part)) >= target) x = y;
  }
  cut = x;
  // The kept count and mass, for the caller (a pass over the row on this path).
  unsigned kept = 0;
  ff kpart = {0.0f, 0.0f};
  for_tiles([&](const uint32_t (&w)[W], int nv, unsigned e0) {
    for (int j = 0; j < nv; ++j) {
      const uint32_t b = tp_pick<DT>(w, j);
      if (key_of(b, e0 + j) >= cut) {
        ++kept;
        const ff xx = scaled_diff(tp_float<DT>(b), m, P.ih, P.il, unit_t);
        ff_accumulate(kpart, exp_ff(xx.hi, xx.lo, sh.tab));
      }
    }
  });
  kept = __reduce_add_sync(0xffffffffu, kept);
  if (lane == 0) sh.wcnt[warp] = kept;
  const double kmass = tp_block_sum(sh, ff_to_double(kpart));
  if (tid == 0) {
    unsigned tot = 0;
    for (int w2 = 0; w2 < kTpThreads / 32; ++w2) tot += sh.wcnt[w2];
    P.topp_cut[row] = cut;
    if (P.topp_kept) P.topp_kept[row] = (int)tot;
    P.row_stat[row] = make_float2(m, (float)kmass);
  }
}

// ---------------------------------------------------------------- nucleus: the cut on a thread-block cluster
//
// The cut of topp_cut_kernel with the row held on chip. A cluster of NC CTAs
// takes one row; each CTA copies its slice of the row (at most one slice
// budget of bytes) into its shared memory once, so the row crosses HBM once
// and every later pass reads shared memory. After each pass the CTAs publish
// per-bin totals in their own shared memory; after a cluster barrier every
// CTA sums all CTAs' totals in rank order, so all of them take the same
// decision. Passes:
//   0. the row maximum m (a NaN or +inf entry fails the row);
//   1. float-float masses of 16 bins of D = fl(fl(m - l) log2(e) / (4T)),
//      bin floor(D), the last one open; S, the row's total, is their sum;
//   2.. the cut bin split 16 ways (bin floor(D 16^(L-1)), an exact scaling),
//      over the entries whose value lies in its window, counting them;
//   once the bin just split held at most kTcCap entries (so its cut sub-bin
//   does too), a last pass gathers the cut bin's keys and weights into the
//   first CTA and counts the entries above it; the first CTA then finds the
//   cut key bit by bit below the candidates' common key prefix, with one
//   block-wide float-float sum per bit and no atomics. A cut bin that never
//   gets that small (heavy ties) is resolved the same way over the row.
// D is a monotone function of the logit, so bins above the cut bin hold only
// larger keys. Weights are the draw's: exp(l/T) 2^-q0 from the fast
// exponential (~5e-11) for rows whose maximum has |m/T| below ~1386, else
// exp((l - m)/T) (exp_ff, ~1e-12). The kernel leaves the row's statistics
// (m, S_kept) for the verification, which reads the unfiltered rows and
// applies each row's kept set as it loads them.

constexpr int kTcThreads = 256;
constexpr int kTcWarps = kTcThreads / 32;
constexpr int kTcCap = 1024;
constexpr int kTcMaxLevels = 7;
constexpr int kTcMaxCluster = 8;  // portable cluster sizes; longer rows take topp_cut_kernel

struct TcShared {
  union {
    float2 bin[kTpBins][kTcThreads];  // per-thread float-float bin masses, each biased by 1
    struct {  // the first CTA's gathered candidates: keys and float-float weights
      unsigned long long ckey[kTcCap];
      float2 cw[kTcCap];
    } rs;
  } u;
  float2 tab1k[1024];
  float2 tab[256];
  // Each CTA's totals of a pass, written by every CTA of the cluster into
  // every CTA's inbox (by pass parity): 16 bin masses, then a count.
  float2 inbox[2][kTcMaxCluster][kTpBins + 1];
  float inmax[kTcMaxCluster];
  float wmax[kTcWarps];
  ff wff[kTcWarps];
  ff wff2[2][kTcWarps];
  unsigned long long wkey[2][kTcWarps];
  unsigned wcnt[kTcWarps], wcnt2[kTcWarps];
  double binmass[kTpBins];
  unsigned members;  // entries of the bin just split, over the cluster
  float queue[kTcWarps][64];  // per warp: window entries waiting to be weighed
  unsigned off_cand, tot_cand, tot_above;
  // the decision after each pass (the same in every CTA of the cluster)
  double above, target;
  long long parent;
  int open, state;
  float m;
  unsigned n_cand, n_above;  // the first CTA's counters of the gather pass
  unsigned copied;
  unsigned long long bar;
};

constexpr size_t kTcSliceOffset = (sizeof(TcShared) + 127) / 128 * 128;
// Two CTAs per SM (the 64 KB slice budget) need both CTAs' shared memory, with
// the 1 KB each the driver reserves, within the SM's 228 KB.
static_assert(2 * (kTcSliceOffset + (64u << 10) + 1024) <= 228u * 1024u,
              "the nucleus cut kernel must fit two CTAs per SM");

template <int DT>
SV_DEVINL void tc_unpack(const uint4& q, float (&x)[DT == 0 ? 8 : 4]) {
  if constexpr (DT == 0) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      x[2 * k] = bf16_lo(w[k]);
      x[2 * k + 1] = bf16_hi(w[k]);
    }
  } else {
    x[0] = __uint_as_float(q.x);
    x[1] = __uint_as_float(q.y);
    x[2] = __uint_as_float(q.z);
    x[3] = __uint_as_float(q.w);
  }
}

// Float-float add of a weight into this thread's bin b (biased accumulator:
// every weight is at most 1).
SV_DEVINL void tc_bin_add(TcShared& sh, int b, float hi, float lo) {
  float2 a = sh.u.bin[b][threadIdx.x];
  const float s = __fadd_rn(a.x, hi);
  const float e = __fsub_rn(hi, __fsub_rn(s, a.x));
  a.y = __fadd_rn(a.y, __fadd_rn(e, lo));
  a.x = s;
  sh.u.bin[b][threadIdx.x] = a;
}

template <int DT, bool VEC>
__global__ void __launch_bounds__(kTcThreads, 2) topp_cluster_kernel(Params P, int nc,
                                                                      int slice_elems) {
  extern __shared__ __align__(128) unsigned char tc_smem[];
  TcShared& sh = *reinterpret_cast<TcShared*>(tc_smem);
  constexpr int kEs = DT == 0 ? 2 : 4;
  constexpr int kEpv = 16 / kEs;  // elements per 16-byte vector
  uint4* sl4 = reinterpret_cast<uint4*>(tc_smem + kTcSliceOffset);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned rank = cluster_ctarank();
  const long long row = blockIdx.x / nc;
  const unsigned char* rb = row_base(P, row / P.rows_per_seq, (int)(row % P.rows_per_seq));
  const int V = P.V, ib = P.key_ibits;
  const long long e_begin = (long long)rank * slice_elems;
  const int n = (int)max(0LL, min((long long)slice_elems, (long long)V - e_begin));
  const int nvec = (n + kEpv - 1) / kEpv;
  const unsigned bar = smem_u32(&sh.bar);
  // Every CTA of the cluster must have started before another writes into
  // its shared memory: the arrival here, the wait before the first write.
  cluster_arrive_relaxed();

  // ---- the slice into shared memory
  if constexpr (VEC) {
    if (tid == 0) {
      mbar_init(bar, 1);
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (tid == 0) {
      // n * kEs is a multiple of 16 (the row and V * kEs are 16-byte aligned,
      // and slices start at multiples of 8 elements).
      const unsigned bytes = (unsigned)n * kEs;
      mbar_arrive_expect_tx(bar, bytes);
      for (unsigned off = 0; off < bytes; off += 16384u)
        bulk_copy_g2s(smem_u32(sl4) + off, rb + e_begin * kEs + off, min(16384u, bytes - off), bar);
    }
  } else {
    using E = typename std::conditional<DT == 0, unsigned short, uint32_t>::type;
    E* se = reinterpret_cast<E*>(sl4);
    const E kNegInf = DT == 0 ? (E)0xff80u : (E)0xff800000u;
    const E* src = reinterpret_cast<const E*>(rb) + e_begin;
    for (int i = tid; i < nvec * kEpv; i += kTcThreads) se[i] = i < n ? src[i] : kNegInf;
  }
  sh.tab[tid] = kSvExp2Table[tid];
#pragma unroll
  for (int i = 0; i < 4; ++i) sh.tab1k[tid + i * kTcThreads] = kSvExp2Table1024[tid + i * kTcThreads];
  // One thread waits for the copy (with a backoff, so that the CTA sharing
  // the SM keeps its issue slots); the barrier passes the completion on.
  if constexpr (VEC) {
    if (tid == 0) {
      unsigned ok = 1;
      if (!mbar_test_parity(bar, 0)) {
        const uint64_t t0 = global_ns();
        unsigned ns = 32;
        for (;;) {
          __nanosleep(ns);
          if (ns < 256) ns <<= 1;
          if (mbar_test_parity(bar, 0)) break;
          if (global_ns() - t0 > kWaitLimitNs) {
            ok = 0;
            break;
          }
        }
      }
      sh.copied = ok;
    }
  }
  __syncthreads();
  const bool copied = VEC ? sh.copied != 0 : true;

  // ---- pass 0: the maximum (NaN-propagating; +inf is caught as well)
  float mx = neg_inf();
  if constexpr (DT == 0) {
    uint32_t mm = 0xff80ff80u;
    for (int v = tid; v < nvec; v += kTcThreads) {
      const uint4 q = sl4[v];
      mm = bf16x2_max_nan(mm, bf16x2_max_nan(bf16x2_max_nan(q.x, q.y), bf16x2_max_nan(q.z, q.w)));
    }
    mx = fmax_nan(bf16_lo(mm), bf16_hi(mm));
  } else {
    for (int v = tid; v < nvec; v += kTcThreads) {
      const uint4 q = sl4[v];
      mx = fmax_nan(mx, fmax_nan(fmax_nan(__uint_as_float(q.x), __uint_as_float(q.y)),
                                 fmax_nan(__uint_as_float(q.z), __uint_as_float(q.w))));
    }
  }
  if (!copied) mx = __int_as_float(0x7fc00000);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmax_nan(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (lane == 0) sh.wmax[warp] = mx;
  __syncthreads();
  cluster_wait();
  if (tid < nc) {  // this CTA's maximum into every CTA's inbox
    float c = sh.wmax[0];
    for (int w2 = 1; w2 < kTcWarps; ++w2) c = fmax_nan(c, sh.wmax[w2]);
    dsmem_st_f32(dsmem_map(smem_u32(&sh.inmax[rank]), tid), c);
  }
  cluster_sync();
  if (warp == 0) {
    float c = lane < nc ? sh.inmax[lane] : neg_inf();
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c = fmax_nan(c, __shfl_xor_sync(0xffffffffu, c, o));
    if (lane == 0) sh.m = c;
  }
  __syncthreads();
  const float m = sh.m;
  if (!copied && tid == 0) atomicOr(P.status, kDevTimeout);
  if (isnan(m) || m == CUDART_INF_F || m == neg_inf()) {
    // A failing row: the verification reports it from the statistics.
    if (rank == 0 && tid == 0) {
      P.topp_cut[row] = 0;
      if (P.topp_kept) P.topp_kept[row] = V;
      P.row_stat[row] = m == neg_inf() ? make_float2(neg_inf(), 0.0f)
                                       : make_float2(0.0f, __int_as_float(0x7fc00000));
    }
    return;
  }

  // ---- row constants: D's scale, the weights' form
  const float c2q = P.c2 * 0.25f;
  const bool unit_t = P.unit_t != 0;
  const float mc = m * P.c2;
  const bool fast = fabsf(mc) <= 2000.0f;
  const int q0 = row_q0(m, P.c2);
  const int qb = 127 - q0;
  const float lmin = -2048.0f * __fdividef(1.0f, P.ih);
  const DrawConst dc{P.d_inv, P.d_ch, P.d_cli, P.ih};
  auto weight = [&](float l) -> ff {
    if (fast) return exp_draw(fmaxf(l, lmin), qb, dc, sh.tab1k);
    const ff x = scaled_diff(l, m, P.ih, P.il, unit_t);
    return exp_ff(x.hi, x.lo, sh.tab);
  };
  auto dval = [&](float l) { return __fmul_rn(__fsub_rn(m, l), c2q); };
  // The value window of bin `parent` at scale sc (open: everything below too),
  // widened by far more than D's rounding.
  // (fp32: its rounding, ~1e-7 of |m| + D, is far inside the slack.)
  auto window = [&](float sc, long long parent, bool open, float& lo, float& hi) {
    const float w = 1.0f / (sc * c2q);
    const float s0 = (float)parent * w, s1 = (float)(parent + 1) * w;
    const float slack = (fabsf(m) + s1) * 1e-5f + 1e-30f;
    lo = open ? neg_inf() : m - s1 - slack;
    hi = m - s0 + slack;
  };
  // floor(D sc) (D >= 0; the product is exact; an infinite or huge D
  // saturates). Indices stay below 2^28 for D < 16 and scales up to 16^6.
  auto bin_index = [&](float d, float sc) -> long long {
    return (long long)__float2int_rz(__fmul_rn(d, sc));
  };

  // Per-pass reduction: this CTA's 16 bin totals (float-float, each thread's
  // bias removed) and the entries it split (`members`, one count per
  // thread), published at parity `par`; after the cluster barrier, warp 0
  // sums the CTAs' totals in rank order into binmass and members.
  auto reduce_and_share = [&](int par, unsigned members) {
    members = __reduce_add_sync(0xffffffffu, members);
    if (lane == 0) sh.wcnt[warp] = members;
    __syncthreads();
    {
      // Thread (b, part) sums bin b over 16 threads' columns; after the
      // butterfly all 16 hold the total, and thread (b, r) writes it into
      // CTA r's inbox.
      const int b = tid >> 4, part = tid & 15;
      ff acc{0.0f, 0.0f};
      for (int t = part; t < kTcThreads; t += 16) {
        const float2 a = sh.u.bin[b][t];
        acc = ff_add(acc, fast_two_sum(__fsub_rn(a.x, 1.0f), a.y));
      }
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) acc = ff_add(acc, ff_shfl_xor(acc, o));
      if (part < nc)
        dsmem_st_f32x2(dsmem_map(smem_u32(&sh.inbox[par][rank][b]), part), acc.hi, acc.lo);
      if (tid < nc) {
        unsigned c = 0;
        for (int w2 = 0; w2 < kTcWarps; ++w2) c += sh.wcnt[w2];
        dsmem_st_f32x2(dsmem_map(smem_u32(&sh.inbox[par][rank][kTpBins]), tid),
                       __uint_as_float(c), 0.0f);
      }
    }
    cluster_sync();
    if (warp == 0) {
      ff tot{0.0f, 0.0f};
      unsigned c = 0;
      if (lane < kTpBins) {
        for (int r = 0; r < nc; ++r) {
          const float2 v = sh.inbox[par][r][lane];
          tot = ff_add(tot, ff{v.x, v.y});
        }
        sh.binmass[lane] = ff_to_double(tot);
      } else if (lane == kTpBins) {
        for (int r = 0; r < nc; ++r) c += __float_as_uint(sh.inbox[par][r][kTpBins].x);
        sh.members = c;
      }
    }
    __syncthreads();
  };
  // (Each thread writes only its own column; the last pass's reads of
  // other columns ended before the barriers that closed it.)
  auto zero_bins = [&]() {
#pragma unroll
    for (int b = 0; b < kTpBins; ++b) sh.u.bin[b][tid] = make_float2(1.0f, 0.0f);
  };
  // The bin where the running mass from the top reaches the target; if
  // rounding leaves the target just out of reach, the last bin with mass.
  // Warp 0 decides (a scan over the 16 bins, lane b holding bin b); the
  // caller synchronises.
  auto decide = [&](int level) {
    if (warp != 0) return;
    const double M = lane < kTpBins ? sh.binmass[lane] : 0.0;
    if (level == 1) {
      double S = M;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) S += __shfl_xor_sync(0xffffffffu, S, o);
      if (lane == 0) {
        sh.target = (double)P.top_p * S;
        sh.above = 0.0;
        sh.parent = 0;
        sh.open = 0;
      }
      __syncwarp();
    }
    const double above0 = sh.above, target = sh.target;
    double Pb = M;  // inclusive prefix over the bins
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double y = __shfl_up_sync(0xffffffffu, Pb, o);
      if (lane >= o) Pb += y;
    }
    const unsigned nonempty = __ballot_sync(0xffffffffu, lane < kTpBins && M > 0.0);
    const unsigned reach = __ballot_sync(0xffffffffu, lane < kTpBins && M > 0.0 && above0 + Pb >= target);
    const int bstar = reach ? __ffs(reach) - 1 : (nonempty ? 31 - __clz(nonempty) : 0);
    const double before = __shfl_sync(0xffffffffu, Pb - M, bstar);  // mass of the bins above bstar
    if (lane == 0) {
      sh.above = above0 + before;
      const long long parent = (level > 1 ? 16 * sh.parent : 0) + bstar;
      sh.open = (bstar == kTpBins - 1 && (level == 1 || sh.open)) ? 1 : 0;
      sh.parent = parent;
      // state: 0 split the new cut bin, 1 gather it (it holds at most as many
      // entries as the bin just split), 2 heavy ties
      if (sh.members <= (unsigned)kTcCap)
        sh.state = 1;
      else
        sh.state = level >= kTcMaxLevels ? 2 : 0;
    }
  };

  // ---- pass 1: every entry, float-float masses of the 16 level-1 bins
  zero_bins();
  {
    const float2 mm2 = f2(m), cq2 = f2(c2q);
    const int2 qb2 = make_int2(qb, qb);
    const float2 nm2 = f2(-m);
    for (int v = tid; v < nvec; v += kTcThreads) {
      float x[kEpv];
      tc_unpack<DT>(sl4[v], x);
#pragma unroll
      for (int j = 0; j < kEpv; j += 2) {
        const float2 l = make_float2(x[j], x[j + 1]);
        ff2 w;
        if (fast) {
          w = exp_draw2(make_float2(fmaxf(l.x, lmin), fmaxf(l.y, lmin)), qb2, dc, sh.tab1k);
        } else {
          const ff2 xs = scaled_diff2(l, nm2, P.ih, P.il, unit_t);
          w = exp_ff2(xs.hi, xs.lo, sh.tab);
        }
        const float2 D = f2_mul(f2_sub(mm2, l), cq2);
        // floor(D) (D >= 0) as the low bits of D + 2^23 rounded toward zero:
        // exact below 2^23, and at least 2^23 (clamped to the last bin) above.
        const float2 Dz = f2_add_rz(D, f2(8388608.0f));
        const int b0 = min(kTpBins - 1, __float_as_int(Dz.x) - 0x4b000000);
        const int b1 = min(kTpBins - 1, __float_as_int(Dz.y) - 0x4b000000);
        tc_bin_add(sh, b0, w.hi.x, w.lo.x);
        tc_bin_add(sh, b1, w.hi.y, w.lo.y);
      }
    }
  }
  reduce_and_share(1, tid == 0 ? (unsigned)n : 0u);  // level 1 splits the whole slice
  decide(1);
  __syncthreads();

  // ---- passes 2..: the cut bin at 16 times the resolution
  int level = 1;
  while (sh.state == 0) {
    ++level;
    const float psc = ldexpf(1.0f, 4 * (level - 2)), sc = ldexpf(1.0f, 4 * (level - 1));
    const long long parent = sh.parent;
    const bool open = sh.open != 0;
    float lo, hi;
    window(psc, parent, open, lo, hi);
    zero_bins();
    unsigned members = 0;
    // The entries inside the window go through a per-warp queue and are
    // weighed 32 at a time, one per lane, so that the exponentials do not
    // diverge with the lanes' candidate counts.
    float* wq = sh.queue[warp];
    int qn = 0;  // queued entries (the same in every lane)
    auto weigh = [&](int cnt) {
      if (lane < cnt) {
        const float l = wq[lane];
        const float d = dval(l);
        const long long ip = bin_index(d, psc);
        if (open ? ip >= parent : ip == parent) {
          const long long r = bin_index(d, sc) - 16 * parent;
          const int b = (int)(r < kTpBins - 1 ? r : kTpBins - 1);
          const ff w = weight(l);
          tc_bin_add(sh, b, w.hi, w.lo);
          ++members;
        }
      }
    };
    for (int v0 = 0; v0 < nvec; v0 += kTcThreads) {  // the same trip count in every lane
      const int v = v0 + tid;
      float x[kEpv];
      unsigned cand = 0;
      if (v < nvec) {
        tc_unpack<DT>(sl4[v], x);
#pragma unroll
        for (int j = 0; j < kEpv; ++j)
          if (x[j] >= lo && x[j] <= hi && (VEC || v * kEpv + j < n)) cand |= 1u << j;
      }
      while (__any_sync(0xffffffffu, cand != 0)) {
        const bool has = cand != 0;
        float l = 0.0f;
        if (has) {
          const int j = __ffs(cand) - 1;
          cand &= cand - 1;
          l = x[0];
#pragma unroll
          for (int k = 1; k < kEpv; ++k) l = j == k ? x[k] : l;
        }
        const unsigned bal = __ballot_sync(0xffffffffu, has);
        if (has) wq[qn + __popc(bal & ((1u << lane) - 1u))] = l;
        qn += __popc(bal);
        if (qn >= 32) {  // at most 63 queued
          __syncwarp();
          weigh(32);
          __syncwarp();
          if (lane < qn - 32) wq[lane] = wq[32 + lane];
          __syncwarp();
          qn -= 32;
        }
      }
    }
    __syncwarp();
    weigh(qn);
    reduce_and_share(level & 1, members);
    decide(level);
    __syncthreads();
  }

  const float sc = ldexpf(1.0f, 4 * (level - 1));
  const long long parent = sh.parent;
  const bool open = sh.open != 0;
  float lo, hi;
  window(sc, parent, open, lo, hi);
  // Class of an entry against the cut bin: 1 above it, 0 in it, -1 below.
  auto classify = [&](float l, float& d) -> int {
    if (l > hi) return 1;
    if (l < lo) return -1;
    d = dval(l);
    const long long i = bin_index(d, sc);
    if (i < parent) return 1;
    return (open || i == parent) ? 0 : -1;
  };

  if (sh.state == 1) {
    // ---- the gather pass: this CTA's entries of the cut bin (keys and
    // weights) into its own shared memory, the entries above the bin counted;
    // then each CTA copies its entries into the first CTA after those of the
    // lower ranks.
    if (tid == 0) {
      sh.n_cand = 0;
      sh.n_above = 0;
    }
    __syncthreads();  // the bins (whose memory the candidates reuse) are no longer read
    unsigned n_ab = 0;
    for (int v0 = 0; v0 < nvec; v0 += kTcThreads) {  // the same trip count in every lane
      const int v = v0 + tid;
      float x[kEpv];
      if (v < nvec) {
        tc_unpack<DT>(sl4[v], x);
      } else {
#pragma unroll
        for (int k = 0; k < kEpv; ++k) x[k] = neg_inf();
      }
      // Entries above the window are counted at once; those inside it (rare)
      // take the exact test, slot by slot, only when some lane has one.
      unsigned win = 0;
#pragma unroll
      for (int j = 0; j < kEpv; ++j) {
        const bool valid = v < nvec && (VEC || v * kEpv + j < n);
        if (valid && x[j] > hi)
          ++n_ab;
        else if (valid && x[j] >= lo)
          win |= 1u << j;
      }
      if (!__any_sync(0xffffffffu, win != 0)) continue;
#pragma unroll
      for (int j = 0; j < kEpv; ++j) {
        const int e = v * kEpv + j;
        float d;
        const int cls = ((win >> j) & 1u) ? classify(x[j], d) : -1;
        n_ab += cls > 0 ? 1u : 0u;
        const unsigned bal = __ballot_sync(0xffffffffu, cls == 0);
        if (bal) {
          const int first = __ffs(bal) - 1;
          unsigned base = 0;
          if (lane == first) base = atomicAdd(&sh.n_cand, (unsigned)__popc(bal));
          base = __shfl_sync(0xffffffffu, base, first);
          const unsigned s = base + (unsigned)__popc(bal & ((1u << lane) - 1u));
          if (cls == 0 && s < (unsigned)kTcCap) {
            const uint32_t bits = DT == 0 ? (__float_as_uint(x[j]) >> 16) : __float_as_uint(x[j]);
            sh.u.rs.ckey[s] = ((unsigned long long)value_key<DT>(bits) << ib) |
                              (unsigned long long)(V - 1 - (int)(e_begin + e));
            const ff w = ff_normalize(weight(x[j]));
            sh.u.rs.cw[s] = make_float2(w.hi, w.lo);
          }
        }
      }
    }
    n_ab = __reduce_add_sync(0xffffffffu, n_ab);
    if (lane == 0 && n_ab) atomicAdd(&sh.n_above, n_ab);
    __syncthreads();
    // (The other parity than the last level's, whose inboxes may still be
    // read.)
    const int gpar = (level + 1) & 1;
    if (tid < nc)  // this CTA's counts into every CTA's inbox
      dsmem_st_f32x2(dsmem_map(smem_u32(&sh.inbox[gpar][rank][0]), tid),
                     __uint_as_float(sh.n_cand), __uint_as_float(sh.n_above));
    cluster_sync();  // every CTA's counts and entries are final
    if (warp == 0) {
      unsigned off = 0, tot = 0, tab = 0;
      if (lane < nc) {
        const float2 c = sh.inbox[gpar][lane][0];
        off = lane < (int)rank ? __float_as_uint(c.x) : 0u;
        tot = __float_as_uint(c.x);
        tab = __float_as_uint(c.y);
      }
      off = __reduce_add_sync(0xffffffffu, off);
      tot = __reduce_add_sync(0xffffffffu, tot);
      tab = __reduce_add_sync(0xffffffffu, tab);
      if (lane == 0) {
        sh.off_cand = off;
        sh.tot_cand = tot;
        sh.tot_above = tab;
      }
    }
    __syncthreads();
    if (rank != 0) {
      const unsigned off = sh.off_cand, mine = min(sh.n_cand, (unsigned)kTcCap);
      const unsigned ckey_a = dsmem_map(smem_u32(&sh.u.rs.ckey[0]), 0);
      const unsigned cw_a = dsmem_map(smem_u32(&sh.u.rs.cw[0]), 0);
      for (unsigned i = tid; i < mine && off + i < (unsigned)kTcCap; i += kTcThreads) {
        dsmem_st_u64(ckey_a + 8u * (off + i), sh.u.rs.ckey[i]);
        const float2 w = sh.u.rs.cw[i];
        dsmem_st_f32x2(cw_a + 8u * (off + i), w.x, w.y);
      }
    }
    cluster_sync();  // every entry is in the first CTA
    if (rank != 0) return;

    // ---- the first CTA: the cut key K*, the largest candidate key with
    // above + mass(keys >= K*) >= target, found bit by bit below the
    // candidates' common prefix with one block reduction (float-float) per
    // bit; no atomics.
    const unsigned ncand = min(sh.tot_cand, (unsigned)kTcCap);
    auto to_ff = [](double d) -> ff {
      const float h = (float)d;
      return {h, (float)(d - (double)h)};
    };
    const ff above_ff = to_ff(sh.above), target_ff = to_ff(sh.target);
    auto reaches = [&](ff part) {  // above + part >= target
      const ff a = ff_add(above_ff, part);
      return a.hi > target_ff.hi || (a.hi == target_ff.hi && a.lo >= target_ff.lo);
    };
    // Block sums alternate between two slot arrays, so one barrier per sum
    // suffices: a slot is rewritten only after every thread has passed the
    // barrier of the sum in between.
    int fpar = 0;
    auto block_ff = [&](ff v) -> ff {
      const int par = fpar;
      fpar ^= 1;
      v = ff_warp_sum(v);
      if (lane == 0) sh.wff2[par][warp] = v;
      __syncthreads();
      ff t{0.0f, 0.0f};
#pragma unroll
      for (int w2 = 0; w2 < kTcWarps; ++w2) t = ff_add(t, sh.wff2[par][w2]);
      return t;
    };
    // max (mode 0) or min (mode 1) of the keys over the block
    auto block_key = [&](unsigned long long k, int mode, int par) -> unsigned long long {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long y = __shfl_xor_sync(0xffffffffu, k, o);
        k = mode == 0 ? (y > k ? y : k) : (y < k ? y : k);
      }
      if (lane == 0) sh.wkey[par][warp] = k;
      __syncthreads();
      unsigned long long r = sh.wkey[par][0];
#pragma unroll
      for (int w2 = 1; w2 < kTcWarps; ++w2) {
        const unsigned long long y = sh.wkey[par][w2];
        r = mode == 0 ? (y > r ? y : r) : (y < r ? y : r);
      }
      return r;
    };
    auto write_out = [&](unsigned long long cut, unsigned kept_c, ff kept_mass) {
      const double S_kept = sh.above + ff_to_double(kept_mass);
      P.topp_cut[row] = cut;
      if (P.topp_kept) P.topp_kept[row] = (int)(sh.tot_above + kept_c);
      const double f = fast ? exp((double)q0 * 0.69314718055994530942 - (double)m * P.inv_t) : 1.0;
      P.row_stat[row] = make_float2(m, (float)(S_kept * f));
    };
    if (ncand <= (unsigned)kTcThreads) {
      // Few candidates (the usual case): each thread takes one, with the
      // mass and count of the candidates at or above its key; K* is the
      // largest key whose mass reaches the target.
      const bool has = tid < ncand;
      unsigned long long ki = 0;
      ff mi{0.0f, 0.0f};
      unsigned ci = 0;
      float wi = 0.0f;
      if (has) {
        ki = sh.u.rs.ckey[tid];
        wi = sh.u.rs.cw[tid].x;
        for (unsigned j = 0; j < ncand; ++j)
          if (sh.u.rs.ckey[j] >= ki) {
            const float2 w = sh.u.rs.cw[j];
            mi = ff_add(mi, ff{w.x, w.y});
            ++ci;
          }
      }
      const bool q = has && reaches(mi);
      unsigned long long cut;
      if (__syncthreads_or(q)) {
        cut = block_key(q ? ki : 0ull, 0, 0);
      } else {
        // Rounding leaves the target just out of reach: every entry with
        // mass is kept, so the cut is the smallest candidate key with mass.
        cut = block_key((has && wi > 0.0f) ? ki : ~0ull, 1, 0);
        if (cut == ~0ull) cut = block_key(has ? ki : 0ull, 0, 1);
      }
      if (has && ki == cut) write_out(cut, ci, mi);
      return;
    }
    unsigned long long kmax = 0, kmin = ~0ull, kpos = ~0ull;
    ff total{0.0f, 0.0f};
    for (unsigned i = tid; i < ncand; i += kTcThreads) {
      const unsigned long long k = sh.u.rs.ckey[i];
      const float2 w = sh.u.rs.cw[i];
      kmax = k > kmax ? k : kmax;
      kmin = k < kmin ? k : kmin;
      if (w.x > 0.0f) kpos = k < kpos ? k : kpos;
      total = ff_add(total, ff{w.x, w.y});
    }
    kmax = block_key(kmax, 0, 0);
    kmin = block_key(kmin, 1, 1);
    kpos = block_key(kpos, 1, 0);
    total = block_ff(total);
    unsigned long long cut;
    if (!reaches(total)) {
      // Rounding leaves the target just out of reach: every entry with mass
      // is kept, so the cut is the smallest candidate key with mass.
      cut = kpos != ~0ull ? kpos : kmax;
    } else {
      const unsigned long long diff = kmin ^ kmax;
      const int hb = diff ? 63 - __clzll((long long)diff) : -1;
      unsigned long long x = hb < 0 ? kmax : (hb == 63 ? 0ull : (kmax >> (hb + 1)) << (hb + 1));
      for (int bit = hb; bit >= 0; --bit) {
        const unsigned long long y = x | (1ull << bit);
        ff part{0.0f, 0.0f};
        for (unsigned i = tid; i < ncand; i += kTcThreads)
          if (sh.u.rs.ckey[i] >= y) {
            const float2 w = sh.u.rs.cw[i];
            part = ff_add(part, ff{w.x, w.y});
          }
        part = block_ff(part);
        if (reaches(part)) x = y;
      }
      cut = x;
    }
    // Kept: the entries above the cut bin, and the candidates at or above the
    // cut; their mass is the row's kept total S_kept.
    unsigned c = 0;
    ff kmass{0.0f, 0.0f};
    for (unsigned i = tid; i < ncand; i += kTcThreads)
      if (sh.u.rs.ckey[i] >= cut) {
        ++c;
        const float2 w = sh.u.rs.cw[i];
        kmass = ff_add(kmass, ff{w.x, w.y});
      }
    c = __reduce_add_sync(0xffffffffu, c);
    if (lane == 0) sh.wcnt[warp] = c;
    const ff km = block_ff(kmass);  // its barrier also publishes wcnt
    if (tid == 0) {
      unsigned tot = 0;
      for (int w2 = 0; w2 < kTcWarps; ++w2) tot += sh.wcnt[w2];
      write_out(cut, tot, km);
    }
    return;
  }

  // ---- heavy ties: the cut key bit by bit, with the exact mass of the cut
  // bin's keys at or above the trial key (the bins above it are all kept)
  const int bits = (DT == 0 ? 16 : 32) + ib;
  unsigned long long x = 0;
  auto mass_at_or_above = [&](unsigned long long y, int par, double& mass, unsigned& n_ge,
                              unsigned& n_ab) {
    ff part{0.0f, 0.0f};
    unsigned cge = 0, cab = 0;
    for (int v = tid; v < nvec; v += kTcThreads) {
      float xv[kEpv];
      tc_unpack<DT>(sl4[v], xv);
#pragma unroll
      for (int j = 0; j < kEpv; ++j) {
        const int e = v * kEpv + j;
        if (e >= n) continue;
        float d;
        const int cls = classify(xv[j], d);
        if (cls > 0) {
          ++cab;
          continue;
        }
        if (cls < 0) continue;
        const uint32_t bb = DT == 0 ? (__float_as_uint(xv[j]) >> 16) : __float_as_uint(xv[j]);
        const unsigned long long key = ((unsigned long long)value_key<DT>(bb) << ib) |
                                       (unsigned long long)(V - 1 - (int)(e_begin + e));
        if (key >= y) {
          ff_accumulate(part, weight(xv[j]));
          ++cge;
        }
      }
    }
    part = ff_warp_sum(part);
    cge = __reduce_add_sync(0xffffffffu, cge);
    cab = __reduce_add_sync(0xffffffffu, cab);
    if (lane == 0) {
      sh.wff[warp] = part;
      sh.wcnt[warp] = cge;
      sh.wcnt2[warp] = cab;
    }
    __syncthreads();
    if (tid < nc) {  // this CTA's totals into every CTA's inbox
      ff t{0.0f, 0.0f};
      unsigned a1 = 0, a2 = 0;
      for (int w2 = 0; w2 < kTcWarps; ++w2) {
        t = ff_add(t, sh.wff[w2]);
        a1 += sh.wcnt[w2];
        a2 += sh.wcnt2[w2];
      }
      dsmem_st_f32x2(dsmem_map(smem_u32(&sh.inbox[par][rank][0]), tid), t.hi, t.lo);
      dsmem_st_f32x2(dsmem_map(smem_u32(&sh.inbox[par][rank][1]), tid), __uint_as_float(a1),
                     __uint_as_float(a2));
    }
    cluster_sync();
    if (tid == 0) {
      ff t{0.0f, 0.0f};
      unsigned a1 = 0, a2 = 0;
      for (int r = 0; r < nc; ++r) {
        const float2 v = sh.inbox[par][r][0], c = sh.inbox[par][r][1];
        t = ff_add(t, ff{v.x, v.y});
        a1 += __float_as_uint(c.x);
        a2 += __float_as_uint(c.y);
      }
      sh.binmass[0] = ff_to_double(t);
      sh.wcnt[0] = a1;
      sh.wcnt2[0] = a2;
    }
    __syncthreads();
    mass = sh.above + sh.binmass[0];
    n_ge = sh.wcnt[0];
    n_ab = sh.wcnt2[0];
    __syncthreads();
  };
  int par = (level + 1) & 1;
  for (int bit = bits - 1; bit >= 0; --bit) {
    const unsigned long long y = x | (1ull << bit);
    double mass;
    unsigned n_ge, n_ab;
    mass_at_or_above(y, par, mass, n_ge, n_ab);
    par ^= 1;
    if (mass >= sh.target) x = y;
  }
  double S_kept;
  unsigned n_ge, n_ab;
  mass_at_or_above(x, par, S_kept, n_ge, n_ab);
  cluster_sync();  // no CTA leaves while another may still read its totals
  if (rank == 0 && tid == 0) {
    P.topp_cut[row] = x;
    if (P.topp_kept) P.topp_kept[row] = (int)(n_ge + n_ab);
    const double f = fast ? exp((double)q0 * 0.69314718055994530942 - (double)m * P.inv_t) : 1.0;
    P.row_stat[row] = make_float2(m, (float)(S_kept * f));
  }
}

// ---------------------------------------------------------------- host-side launch

#if SV_TU_HAS(1)
namespace {
struct DeviceInfo {
  bool ready = false;
};
DeviceInfo g_dev[64];
std::mutex g_dev_mu;
std::atomic<int> g_force_path{0};
std::atomic<int> g_withhold{0};

bool take_fused(long long B, int rows_per_seq, long long V, int es, bool sampler = false) {
  const int path = g_force_path.load();
  if (path == 1) return false;
  if (path == 2) return true;
  // The sampler draws every row, so its draw kernel's occupancy decides: the pair.
  const long long bytes = B * rows_per_seq * V * es;
  return !sampler && bytes >= kFusedMinBytes && bytes <= kFusedMaxBytes;
}
}  // namespace

void force_path(int path) { g_force_path.store(path); }

// Sequences between a sequence's streaming tickets and its draw tickets in
// the fused kernel (B: every streaming ticket first).
long long fused_lag(long long B) { return B; }

void withhold_plans(int on) { g_withhold.store(on ? 1 : 0); }

int kernels_per_call(long long B, int rows_per_seq, long long V, int es) {
  if (take_fused(B, rows_per_seq, V, es)) return 1;
  // 2048-element draw chunks (small calls): the one-launch draw.
  return B * ((V + 4095) / 4096) < kMinDrawCtas ? 2 : 3;
}

template <int DT, bool VEC, int SUB>
cudaError_t launch_fused(Params P, cudaStream_t st, const Events& ev) {
  P.nsi = (P.ns + kWarps - 1) / kWarps;
  P.lag = fused_lag(P.B);
  fused_kernel<DT, VEC, SUB><<<(unsigned)((long long)P.B * (P.nsi + P.np)), kThreads, 0, st>>>(P);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess && ev.stats_done)
    e = cudaEventRecordWithFlags(ev.stats_done, st, cudaEventRecordExternal);
  return e;
}

template <int DT, bool VEC, int SUB>
cudaError_t launch_sampler(const Params& P, cudaStream_t st) {
  sample_sum_kernel<DT, VEC, SUB><<<(unsigned)((long long)P.B * P.np), kThreads, 0, st>>>(P);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)P.B);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, sample_finish_kernel<DT, VEC, SUB>, P);
}

template <int DT, bool VEC, int SUB>
cudaError_t launch_pair(const Params& P, cudaStream_t st, const Events& ev) {
  const unsigned stats_grid = (unsigned)((P.n_units + kStatsWarps - 1) / kStatsWarps);
  stats_kernel<DT, VEC><<<stats_grid, kStatsThreads, 0, st>>>(P);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // The draw kernel is a programmatic dependent of the streaming kernel: it
  // may be launched while the last streaming CTAs still run, and waits on the
  // device for the streaming grid to complete. An event recorded between the
  // two (the profiled entry point) makes it an ordinary launch.
  if (ev.stats_done) {
    e = cudaEventRecordWithFlags(ev.stats_done, st, cudaEventRecordExternal);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((long long)P.B * P.np));
  cfg.blockDim = dim3(kThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = ev.stats_done ? 0 : 1;
  if constexpr (SUB == 256) return cudaLaunchKernelEx(&cfg, draw_kernel<DT, VEC, SUB>, P);
  e = cudaLaunchKernelEx(&cfg, draw_sum_kernel<DT, VEC, SUB>, P);
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3((unsigned)P.B);
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, draw_finish_kernel<DT, VEC, SUB>, P);
}

cudaError_t prepare_device(int device) {
  if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  g_dev[device].ready = true;
  return cudaSuccess;
}

cudaError_t launch_all(Params P, bool aligned, cudaStream_t st, const Events& ev) {
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return e;
  e = prepare_device(device);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(P.ctrl, 0, P.ctrl_bytes, st);
  if (e != cudaSuccess) return e;
  // External records, so that the events become timing nodes when the stream
  // is being captured into a graph.
  if (ev.start) {
    e = cudaEventRecordWithFlags(ev.start, st, cudaEventRecordExternal);
    if (e != cudaSuccess) return e;
  }
  const bool big = P.sub_elems == 512;
  P.fused = take_fused(P.B, P.rows_per_seq, P.V, P.es, P.sampler != 0) ? 1 : 0;
  P.withhold = g_withhold.load();
  if (P.sampler) {
    if (P.dtype == 0)
      e = aligned ? (big ? launch_sampler<0, true, 512>(P, st) : launch_sampler<0, true, 256>(P, st))
                  : (big ? launch_sampler<0, false, 512>(P, st) : launch_sampler<0, false, 256>(P, st));
    else
      e = aligned ? (big ? launch_sampler<1, true, 512>(P, st) : launch_sampler<1, true, 256>(P, st))
                  : (big ? launch_sampler<1, false, 512>(P, st) : launch_sampler<1, false, 256>(P, st));
  } else if (P.fused) {
    if (P.dtype == 0)
      e = aligned ? (big ? launch_fused<0, true, 512>(P, st, ev) : launch_fused<0, true, 256>(P, st, ev))
                  : (big ? launch_fused<0, false, 512>(P, st, ev) : launch_fused<0, false, 256>(P, st, ev));
    else
      e = aligned ? (big ? launch_fused<1, true, 512>(P, st, ev) : launch_fused<1, true, 256>(P, st, ev))
                  : (big ? launch_fused<1, false, 512>(P, st, ev) : launch_fused<1, false, 256>(P, st, ev));
  } else if (P.dtype == 0) {
    e = aligned ? (big ? launch_pair<0, true, 512>(P, st, ev) : launch_pair<0, true, 256>(P, st, ev))
                : (big ? launch_pair<0, false, 512>(P, st, ev) : launch_pair<0, false, 256>(P, st, ev));
  } else {
    e = aligned ? (big ? launch_pair<1, true, 512>(P, st, ev) : launch_pair<1, true, 256>(P, st, ev))
                : (big ? launch_pair<1, false, 512>(P, st, ev) : launch_pair<1, false, 256>(P, st, ev));
  }
  if (e != cudaSuccess) return e;
  if (ev.end) e = cudaEventRecordWithFlags(ev.end, st, cudaEventRecordExternal);
  return e;
}

#endif  // SV_TU_HAS(1)

#if SV_TU_HAS(2)
template <int DT, bool VEC>
cudaError_t launch_select(const Params& P, unsigned rows, size_t smem, cudaStream_t st) {
  topk_select_kernel<DT, VEC><<<rows, kSelThreads, smem, st>>>(P);
  return cudaGetLastError();
}

cudaError_t launch_topk(const Params& P, bool aligned, cudaStream_t st) {
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return e;
  e = prepare_device(device);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(P.ctrl, 0, P.ctrl_bytes, st);
  if (e != cudaSuccess) return e;
  const unsigned rows = (unsigned)((long long)P.B * P.rows_per_seq);
  const size_t smem = sizeof(SelShared);
  if (P.dtype == 0)
    e = aligned ? launch_select<0, true>(P, rows, smem, st) : launch_select<0, false>(P, rows, smem, st);
  else
    e = aligned ? launch_select<1, true>(P, rows, smem, st) : launch_select<1, false>(P, rows, smem, st);
  if (e != cudaSuccess) return e;
  if (e != cudaSuccess) return e;
  topk_verify_kernel<<<(unsigned)P.B, kTvThreads, 0, st>>>(P);
  return cudaGetLastError();
}

#endif  // SV_TU_HAS(2)

#if SV_TU_HAS(3)
// The nucleus cut's cluster shape for rows of V elements of `es` bytes: CTAs
// per row and elements per CTA, with a slice budget of 64 KB (two CTAs per
// SM); nc = 0 for rows that would need more than kTcMaxCluster CTAs. (Longer
// rows measured faster on the one-CTA-per-row kernel, which re-reads them
// from L2 and memory: 4.06 ms against 7.16 ms with 16-CTA clusters for 2304
// rows of 256000 f32.)
static void topp_cluster_shape(long long V, int es, int* nc, int* slice_elems, size_t* smem) {
  constexpr long long kBudget = 64ll << 10;
  *nc = 0;
  const long long c = (V * es + kBudget - 1) / kBudget;
  if (c > kTcMaxCluster) return;
  const long long se = ((V + c - 1) / c + 7) / 8 * 8;
  *nc = (int)c;
  *slice_elems = (int)se;
  *smem = kTcSliceOffset + (size_t)((se * es + 127) / 128 * 128);
}

// Whether clusters of `nc` CTAs with `smem` bytes each can be resident (the
// answer cached per kernel and shape).
template <int DT, bool VEC>
static bool topp_cluster_ok(int nc, size_t smem, cudaLaunchConfig_t cfg) {
  static std::mutex mu;
  static std::map<std::pair<int, size_t>, bool> known;
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_pair(nc, smem);
  const auto it = known.find(key);
  if (it != known.end()) return it->second;
  bool ok = cudaFuncSetAttribute(topp_cluster_kernel<DT, VEC>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) == cudaSuccess;
  int clusters = 0;
  if (ok) ok = cudaOccupancyMaxActiveClusters(&clusters, topp_cluster_kernel<DT, VEC>, &cfg) ==
               cudaSuccess && clusters > 0;
  (void)cudaGetLastError();  // a refused shape leaves no sticky error behind
  known[key] = ok;
  return ok;
}

template <int DT, bool VEC>
static cudaError_t launch_topp_cut(const Params& P, cudaStream_t st) {
  const long long rows = (long long)P.B * P.rows_per_seq;
  int nc = 0, slice_elems = 0;
  size_t smem = 0;
  topp_cluster_shape(P.V, P.es, &nc, &slice_elems, &smem);
  if (nc > 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(rows * nc));
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)nc;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (topp_cluster_ok<DT, VEC>(nc, smem, cfg)) {
      cudaError_t e = cudaFuncSetAttribute(topp_cluster_kernel<DT, VEC>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      return cudaLaunchKernelEx(&cfg, topp_cluster_kernel<DT, VEC>, P, nc, slice_elems);
    }
  }
  const size_t tsmem = sizeof(TopPShared);
  cudaError_t e = cudaFuncSetAttribute(topp_cut_kernel<DT, VEC>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tsmem);
  if (e != cudaSuccess) return e;
  topp_cut_kernel<DT, VEC><<<(unsigned)rows, kTpThreads, tsmem, st>>>(P);
  return cudaGetLastError();
}

// The verification after the cut: one warp per sequence scans the kept-set
// statistics, then the draw (with the kept sets applied on load).
__global__ void __launch_bounds__(kStatsThreads) scan_kernel(Params P) {
  __shared__ WarpScan ws[kStatsWarps];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long b = (long long)blockIdx.x * kStatsWarps + warp;
  if (b < P.B) scan_warp(P, b, lane, ws[warp]);
}

template <int DT, bool VEC, int SUB>
static cudaError_t launch_masked_verify(const Params& P, cudaStream_t st) {
  scan_kernel<<<(unsigned)((P.B + kStatsWarps - 1) / kStatsWarps), kStatsThreads, 0, st>>>(P);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)((long long)P.B * P.np);
  if constexpr (SUB == 256) {
    draw_kernel<DT, VEC, SUB, true><<<grid, kThreads, 0, st>>>(P);
    return cudaGetLastError();
  }
  draw_sum_kernel<DT, VEC, SUB, true><<<grid, kThreads, 0, st>>>(P);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  draw_finish_kernel<DT, VEC, SUB, true><<<(unsigned)P.B, kThreads, 0, st>>>(P);
  return cudaGetLastError();
}

template <int DT, bool VEC>
static cudaError_t launch_topp_all(const Params& P, cudaStream_t st) {
  cudaError_t e = launch_topp_cut<DT, VEC>(P, st);
  if (e != cudaSuccess) return e;
  return P.sub_elems == 512 ? launch_masked_verify<DT, VEC, 512>(P, st)
                            : launch_masked_verify<DT, VEC, 256>(P, st);
}

cudaError_t launch_topp(Params P, bool aligned, cudaStream_t st) {
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return e;
  e = prepare_device(device);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(P.ctrl, 0, P.ctrl_bytes, st);
  if (e != cudaSuccess) return e;
  P.fused = 0;
  P.withhold = 0;
  if (P.dtype == 0)
    return aligned ? launch_topp_all<0, true>(P, st) : launch_topp_all<0, false>(P, st);
  return aligned ? launch_topp_all<1, true>(P, st) : launch_topp_all<1, false>(P, st);
}

#endif  // SV_TU_HAS(3)

#if SV_TU_HAS(2)
__global__ void fill_int_kernel(int* p, long long n, int v) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x)
    p[i] = v;
}

cudaError_t fill_int(int* p, long long n, int v, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  const long long blocks = (n + 255) / 256;
  fill_int_kernel<<<(unsigned)(blocks < 1024 ? blocks : 1024), 256, 0, st>>>(p, n, v);
  return cudaGetLastError();
}

cudaError_t launch_greedy(const Params& P, bool aligned, cudaStream_t st) {
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return e;
  e = prepare_device(device);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(P.ctrl, 0, P.ctrl_bytes, st);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)((P.n_units + kStatsWarps - 1) / kStatsWarps);
  if (P.dtype == 0) {
    if (aligned)
      greedy_kernel<0, true><<<grid, kStatsThreads, 0, st>>>(P);
    else
      greedy_kernel<0, false><<<grid, kStatsThreads, 0, st>>>(P);
  } else {
    if (aligned)
      greedy_kernel<1, true><<<grid, kStatsThreads, 0, st>>>(P);
    else
      greedy_kernel<1, false><<<grid, kStatsThreads, 0, st>>>(P);
  }
  return cudaGetLastError();
}

#endif  // SV_TU_HAS(2)

}  // namespace sv
