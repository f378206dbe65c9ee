// Device helpers of the verification kernels: streaming loads, bf16
// unpacking, float-float arithmetic, and a float-float exponential accurate
// to about 1e-12 relative.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "sv_exp_table.h"

#define SV_DEVINL __device__ __forceinline__

namespace sv {

SV_DEVINL float neg_inf() { return __int_as_float(0xff800000u); }

// ---------------------------------------------------------------- loads

// Streaming 16-byte global load that skips L1.
SV_DEVINL uint4 ld_global_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// ---------------------------------------------------------------- flags and bounded waits

SV_DEVINL uint32_t ld_acquire_u32(const unsigned* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

SV_DEVINL void st_release_u32(unsigned* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

SV_DEVINL uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Every wait in the kernels gives up after this much wall time.
constexpr uint64_t kWaitLimitNs = 200ull * 1000ull * 1000ull;

// ---------------------------------------------------------------- mbarriers and bulk copies

SV_DEVINL unsigned smem_u32(const void* p) {
  return static_cast<unsigned>(__cvta_generic_to_shared(p));
}

SV_DEVINL void mbar_init(unsigned bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// One arrival that also expects `bytes` of asynchronous copies.
SV_DEVINL void mbar_arrive_expect_tx(unsigned bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

SV_DEVINL bool mbar_test_parity(unsigned bar, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned)
// from global memory into this CTA's shared memory, counted on `bar`.
SV_DEVINL void bulk_copy_g2s(unsigned dst, const void* src, unsigned bytes, unsigned bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// ---------------------------------------------------------------- thread-block clusters

SV_DEVINL unsigned cluster_ctarank() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Every thread of every CTA of the cluster: shared-memory writes before it
// are visible to the cluster's loads after it.
SV_DEVINL void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// The two halves of cluster_sync, for a barrier whose wait comes later (the
// arrival orders nothing).
SV_DEVINL void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
SV_DEVINL void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }

// The shared::cluster address of this CTA's shared variable at `addr` in the
// CTA of rank `rank`.
SV_DEVINL unsigned dsmem_map(unsigned addr, unsigned rank) {
  unsigned r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
SV_DEVINL void dsmem_st_u64(unsigned a, unsigned long long v) {
  asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(a), "l"(v) : "memory");
}
SV_DEVINL void dsmem_st_f32(unsigned a, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(a), "f"(v) : "memory");
}
SV_DEVINL void dsmem_st_f32x2(unsigned a, float x, float y) {
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(a), "f"(x), "f"(y) : "memory");
}

// ---------------------------------------------------------------- bf16 and fast fp32 helpers

SV_DEVINL float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
SV_DEVINL float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Packed max of two bf16 pairs (a NaN operand yields the other operand).
SV_DEVINL uint32_t bf16x2_max(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Hardware 2^x (MUFU), flushes subnormal results to zero; 2^-inf = 0.
SV_DEVINL float ex2_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------- float-float arithmetic
// A float-float value is hi + lo with |lo| small against |hi|. The error-free
// transformations below use the _rn intrinsics so that the compiler neither
// contracts nor reassociates them.

struct ff {
  float hi, lo;
};

// s + e == a + b exactly (Knuth's TwoSum).
SV_DEVINL ff two_sum(float a, float b) {
  float s = __fadd_rn(a, b);
  float bb = __fsub_rn(s, a);
  float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
  return {s, e};
}

// s + e == a + b exactly, given |a| >= |b| (Dekker's FastTwoSum).
SV_DEVINL ff fast_two_sum(float a, float b) {
  float s = __fadd_rn(a, b);
  float e = __fsub_rn(b, __fsub_rn(s, a));
  return {s, e};
}

// p + e == a * b exactly (FMA-based).
SV_DEVINL ff two_prod(float a, float b) {
  float p = __fmul_rn(a, b);
  float e = __fmaf_rn(a, b, -p);
  return {p, e};
}

// acc += x, keeping the sum's low part unnormalised (normalise once at the end).
SV_DEVINL void ff_accumulate(ff& acc, ff x) {
  ff s = two_sum(acc.hi, x.hi);
  acc.hi = s.hi;
  acc.lo = __fadd_rn(acc.lo, __fadd_rn(s.lo, x.lo));
}

SV_DEVINL ff ff_normalize(ff a) { return fast_two_sum(a.hi, a.lo); }

// Accumulator for sums of terms in [0, 1]: it starts at 1 (ff_bias_start) so
// that its head is never smaller than a term, which makes Dekker's
// FastTwoSum exact for every addition; ff_bias_end removes the 1 exactly.
SV_DEVINL ff ff_bias_start() { return {1.0f, 0.0f}; }

SV_DEVINL void ff_accumulate_biased(ff& acc, ff x) {
  const float s = __fadd_rn(acc.hi, x.hi);
  const float e = __fsub_rn(x.hi, __fsub_rn(s, acc.hi));
  acc.hi = s;
  acc.lo = __fadd_rn(acc.lo, __fadd_rn(e, x.lo));
}

SV_DEVINL ff ff_bias_end(ff acc) { return fast_two_sum(__fsub_rn(acc.hi, 1.0f), acc.lo); }

SV_DEVINL ff ff_add(ff a, ff b) {
  ff s = two_sum(a.hi, b.hi);
  return fast_two_sum(s.hi, __fadd_rn(s.lo, __fadd_rn(a.lo, b.lo)));
}

SV_DEVINL double ff_to_double(ff a) { return (double)a.hi + (double)a.lo; }

SV_DEVINL ff ff_neg(ff a) { return {-a.hi, -a.lo}; }

SV_DEVINL ff ff_sub(ff a, ff b) { return ff_add(a, ff_neg(b)); }

// a * b for float-float operands (relative error about 2^-44).
SV_DEVINL ff ff_mul(ff a, ff b) {
  const ff p = two_prod(a.hi, b.hi);
  const float lo = __fmaf_rn(a.hi, b.lo, __fmaf_rn(a.lo, b.hi, p.lo));
  return fast_two_sum(p.hi, lo);
}

// a * b for a float-float and a float.
SV_DEVINL ff ff_mul_f(ff a, float b) {
  const ff p = two_prod(a.hi, b);
  return fast_two_sum(p.hi, __fmaf_rn(a.lo, b, p.lo));
}

// a > b for normalised float-float values.
SV_DEVINL bool ff_gt(ff a, ff b) { return a.hi > b.hi || (a.hi == b.hi && a.lo > b.lo); }

SV_DEVINL ff ff_shfl_up(ff a, int delta) {
  return {__shfl_up_sync(0xffffffffu, a.hi, delta), __shfl_up_sync(0xffffffffu, a.lo, delta)};
}

SV_DEVINL ff ff_shfl_xor(ff a, int lane_mask) {
  return {__shfl_xor_sync(0xffffffffu, a.hi, lane_mask),
          __shfl_xor_sync(0xffffffffu, a.lo, lane_mask)};
}

SV_DEVINL ff ff_warp_sum(ff a) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = ff_add(a, ff_shfl_xor(a, o));
  return a;
}

// ---------------------------------------------------------------- packed fp32 pairs
// f32x2 instructions: two independent fp32 operations per instruction, each
// lane rounded to nearest exactly as the scalar _rn operation would be, so a
// packed routine below gives bit for bit the results of its scalar
// counterpart on each lane.

SV_DEVINL float2 f2_add(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

// a + b rounded toward zero, on each lane.
SV_DEVINL float2 f2_add_rz(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "add.rz.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

SV_DEVINL float2 f2_sub(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "sub.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

SV_DEVINL float2 f2_mul(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

SV_DEVINL float2 f2_fma(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mov.b64 rc, {%6, %7};\n\tfma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

SV_DEVINL float2 f2(float v) { return make_float2(v, v); }

// Two float-float values side by side: lane x is (hi.x, lo.x), lane y is
// (hi.y, lo.y).
struct ff2 {
  float2 hi, lo;
};

// two_sum on each lane.
SV_DEVINL ff2 two_sum2(float2 a, float2 b) {
  const float2 s = f2_add(a, b);
  const float2 bb = f2_sub(s, a);
  const float2 e = f2_add(f2_sub(a, f2_sub(s, bb)), f2_sub(b, bb));
  return {s, e};
}

// ff_accumulate_biased on each lane.
SV_DEVINL void ff_accumulate_biased2(ff2& acc, const ff2& x) {
  const float2 s = f2_add(acc.hi, x.hi);
  const float2 e = f2_sub(x.hi, f2_sub(s, acc.hi));
  acc.hi = s;
  acc.lo = f2_add(acc.lo, f2_add(e, x.lo));
}

// ---------------------------------------------------------------- float-float exponential
//
// Adding 1.5 * 2^23 to a float y with |y| <= 2^22 rounds it to an integer
// (ties to even) in the low mantissa bits: (y + M) - M == rint(y), and the
// integer is bits(y + M) - bits(M).
constexpr float kRoundMagic = 12582912.0f;

// exp(xh + xl) for xh <= ~0 (|xl| at most an ulp of xh), after Tang's
// table-driven method: k = rint(x * 256/ln2), r = x - k*ln2/256 (two-constant
// reduction; the head product is exact because head(ln2/256) has its last bit
// at 2^-32 and |r| < 2^-9), exp(r) - 1 by its Taylor series to r^4 (|r| <=
// ln2/512, so the next term is below 4e-17), and 2^((k & 255)/256) from a
// head+tail table. Relative error about 1e-12 for x >= -30; exp(x) for x <
// -87 (below 2^-125) returns 0. `tab` points at the 256-entry table in
// shared memory.
SV_DEVINL ff exp_ff(float xh, float xl, const float2* tab) {
  // |x * 256/ln2| <= 2^22 wherever the result is not flushed to zero below.
  const float ym = __fadd_rn(__fmul_rn(xh, SV_EXP_INV_LN2_256), kRoundMagic);
  const float kf = __fsub_rn(ym, kRoundMagic);
  const float t = __fmaf_rn(-kf, SV_EXP_LN2_256_HI, xh);     // exact
  const float c = __fmaf_rn(-kf, SV_EXP_LN2_256_LO, xl);     // small correction, |c| < 1e-5
  const float t2 = __fmul_rn(t, t);
  const float poly = __fmaf_rn(__fmaf_rn(t, 1.0f / 24.0f, 1.0f / 6.0f), t, 0.5f);
  const float cc = __fmaf_rn(__fmul_rn(0.5f, c), c, c);       // c + c^2/2
  const float rest = __fmaf_rn(t2, poly, __fmaf_rn(cc, t, cc));  // expm1(t + c) - t
  const int k = __float_as_int(ym) - __float_as_int(kRoundMagic);
  const float2 T = tab[k & 255];
  const ff pr = two_prod(T.x, t);
  const ff s = fast_two_sum(T.x, pr.hi);
  const float lo =
      __fadd_rn(__fmaf_rn(T.x, rest, __fmaf_rn(T.y, t, T.y)), __fadd_rn(s.lo, pr.lo));
  const int q = k >> 8;  // floor(k / 256)
  const float scale = __int_as_float((q + 127) << 23);
  const bool under = xh < -87.0f;
  return {under ? 0.0f : __fmul_rn(s.hi, scale), under ? 0.0f : __fmul_rn(lo, scale)};
}

// d = l - m as a float-float (exact), then x = d / T via the float-float
// reciprocal (ih + il) of T. With `unit_t` the scaling is skipped (T == 1).
SV_DEVINL ff scaled_diff(float l, float m, float ih, float il, bool unit_t) {
  const ff d = two_sum(l, -m);
  if (unit_t) return d;
  const ff p = two_prod(d.hi, ih);
  const float lo = __fmaf_rn(d.hi, il, __fmaf_rn(d.lo, ih, p.lo));
  return {p.hi, lo};
}

// exp_ff on each lane of a pair: the same operations in the same order, with
// -k rounded from x * (-256/ln2), which gives exactly -rint(x * 256/ln2).
SV_DEVINL ff2 exp_ff2(float2 xh, float2 xl, const float2* tab) {
  const float2 ym = f2_add(f2_mul(xh, f2(-SV_EXP_INV_LN2_256)), f2(kRoundMagic));
  const float2 nkf = f2_sub(ym, f2(kRoundMagic));
  const float2 t = f2_fma(nkf, f2(SV_EXP_LN2_256_HI), xh);  // exact
  const float2 c = f2_fma(nkf, f2(SV_EXP_LN2_256_LO), xl);
  const float2 t2 = f2_mul(t, t);
  const float2 poly = f2_fma(f2_fma(t, f2(1.0f / 24.0f), f2(1.0f / 6.0f)), t, f2(0.5f));
  const float2 cc = f2_fma(f2_mul(f2(0.5f), c), c, c);
  const float2 rest = f2_fma(t2, poly, f2_fma(cc, t, cc));
  const int kx = __float_as_int(kRoundMagic) - __float_as_int(ym.x);
  const int ky = __float_as_int(kRoundMagic) - __float_as_int(ym.y);
  const float2 Tx = tab[kx & 255], Ty = tab[ky & 255];
  const float2 Th = make_float2(Tx.x, Ty.x), Tl = make_float2(Tx.y, Ty.y);
  const float2 ph = f2_mul(Th, t);
  const float2 pe = f2_fma(Th, t, f2_mul(ph, f2(-1.0f)));
  const float2 sh = f2_add(Th, ph);
  const float2 se = f2_sub(ph, f2_sub(sh, Th));
  const float2 lo = f2_add(f2_fma(Th, rest, f2_fma(Tl, t, Tl)), f2_add(se, pe));
  const float2 scale = make_float2(__int_as_float(((kx >> 8) + 127) << 23),
                                   __int_as_float(((ky >> 8) + 127) << 23));
  const float2 rh = f2_mul(sh, scale), rl = f2_mul(lo, scale);
  const bool ux = xh.x < -87.0f, uy = xh.y < -87.0f;
  return {make_float2(ux ? 0.0f : rh.x, uy ? 0.0f : rh.y),
          make_float2(ux ? 0.0f : rl.x, uy ? 0.0f : rl.y)};
}

// scaled_diff on each lane; `nm` holds -m of each lane.
SV_DEVINL ff2 scaled_diff2(float2 l, float2 nm, float ih, float il, bool unit_t) {
  const ff2 d = two_sum2(l, nm);
  if (unit_t) return d;
  const float2 ph = f2_mul(d.hi, f2(ih));
  const float2 pe = f2_fma(d.hi, f2(ih), f2_mul(ph, f2(-1.0f)));
  const float2 lo = f2_fma(d.hi, f2(il), f2_fma(d.lo, f2(ih), pe));
  return {ph, lo};
}

// ---------------------------------------------------------------- the draw's exponentials
//
// The draw needs w = exp(l/T) 2^-q0 for every element l of the one or two
// rows it reads, with q0 a per-row integer (above the row maximum's
// log2(e) m/T, so that every w is below 2). Elements scale by a power of two
// at most 2^0; a binary exponent field q + 127 <= 0 (the element more than
// 2^126 below the row maximum, or -inf) gives exactly 0. `qb` is 127 - q0.

// Constants of the fast reduction, per call: with C = T ln2/1024,
// ch = fp32(C), cli = fp32((C - ch)/T), inv = fp32(1024/(T ln2)), ih = fp32(1/T).
struct DrawConst {
  float inv, ch, cli, ih;
};

// The fast exponential of one element, used by the chunk pass (packed below,
// scalar here; both give the same bits). k = rint(l inv); r = l - k ch is
// exact (|r| < ch and the exact value spans at most 23 bits); s = r/T - k
// cli = (l - k C)/T, |s| <= ln2/2048 + 1e-5, rounded once (2.4e-11 of the
// value). exp(l/T) = 2^(k >> 10) (Th + Tl)(1 + u), 2^((k & 1023)/1024) = Th + Tl
// from the table, u = e^s - 1 = s + s^2/2 + s^3/6 (the next term is below 6e-16).
// The result is the unnormalised float-float (Th, fl(Th u + Tl)) scaled by
// 2^(q - q0): its low part is at most 3.6e-4 of its head and is rounded once,
// so the value carries a relative error of about 5e-11, of either sign.
// Valid for |l/T| <= 2048 (|k| < 2^22); callers clamp below and take the
// shifted path for rows whose maximum is beyond that.
SV_DEVINL ff exp_draw(float l, int qb, const DrawConst& dc, const float2* tab) {
  const float ym = __fmaf_rn(l, -dc.inv, kRoundMagic);   // 1.5 2^23 - k
  const float nkf = __fsub_rn(ym, kRoundMagic);           // -k
  const float r = __fmaf_rn(nkf, dc.ch, l);               // l - k ch, exact
  const float sv = __fmaf_rn(r, dc.ih, __fmul_rn(nkf, dc.cli));
  const float h = __fmul_rn(__fmaf_rn(sv, 1.0f / 6.0f, 0.5f), sv);
  const float u = __fmaf_rn(sv, h, sv);
  const int k = __float_as_int(kRoundMagic) - __float_as_int(ym);
  const float2 T = tab[k & 1023];
  const float lo = __fmaf_rn(T.x, u, T.y);
  const float scale = __int_as_float(max((k >> 10) + qb, 0) << 23);
  return {__fmul_rn(T.x, scale), __fmul_rn(lo, scale)};
}

// exp_draw on each lane of a pair (lane x with qb.x, lane y with qb.y).
SV_DEVINL ff2 exp_draw2(float2 l, int2 qb, const DrawConst& dc, const float2* tab) {
  const float2 ym = f2_fma(l, f2(-dc.inv), f2(kRoundMagic));
  const float2 nkf = f2_sub(ym, f2(kRoundMagic));
  const float2 r = f2_fma(nkf, f2(dc.ch), l);
  const float2 sv = f2_fma(r, f2(dc.ih), f2_mul(nkf, f2(dc.cli)));
  const float2 h = f2_mul(f2_fma(sv, f2(1.0f / 6.0f), f2(0.5f)), sv);
  const float2 u = f2_fma(sv, h, sv);
  const int kx = __float_as_int(kRoundMagic) - __float_as_int(ym.x);
  const int ky = __float_as_int(kRoundMagic) - __float_as_int(ym.y);
  const float2 Tx = tab[kx & 1023], Ty = tab[ky & 1023];
  const float2 Th = make_float2(Tx.x, Ty.x);
  const float2 lo = f2_fma(Th, u, make_float2(Tx.y, Ty.y));
  const float2 scale = make_float2(__int_as_float(max((kx >> 10) + qb.x, 0) << 23),
                                   __int_as_float(max((ky >> 10) + qb.y, 0) << 23));
  return {f2_mul(Th, scale), f2_mul(lo, scale)};
}

// The same quantity, exp(l/T) 2^-q0, to about 1e-12 (the finish's weights of
// its one sub-chunk): x = l/T as the float-float l (ih + il), then exp_ff's
// steps (Tang's method on the 256-entry table `tab`) with the result's binary
// exponent shifted by -q0. |x| <= 2048 keeps k within the rounding range
// and the reduction exact.
SV_DEVINL ff exp_precise(float l, int qb, float ih, float il, const float2* tab) {
  const float xh = __fmul_rn(l, ih);
  const float xl = __fmaf_rn(l, il, __fmaf_rn(l, ih, -xh));
  const float ym = __fadd_rn(__fmul_rn(xh, SV_EXP_INV_LN2_256), kRoundMagic);
  const float kf = __fsub_rn(ym, kRoundMagic);
  const float t = __fmaf_rn(-kf, SV_EXP_LN2_256_HI, xh);     // exact
  const float c = __fmaf_rn(-kf, SV_EXP_LN2_256_LO, xl);
  const float t2 = __fmul_rn(t, t);
  const float poly = __fmaf_rn(__fmaf_rn(t, 1.0f / 24.0f, 1.0f / 6.0f), t, 0.5f);
  const float cc = __fmaf_rn(__fmul_rn(0.5f, c), c, c);
  const float rest = __fmaf_rn(t2, poly, __fmaf_rn(cc, t, cc));
  const int k = __float_as_int(ym) - __float_as_int(kRoundMagic);
  const float2 T = tab[k & 255];
  const ff pr = two_prod(T.x, t);
  const ff s = fast_two_sum(T.x, pr.hi);
  const float lo =
      __fadd_rn(__fmaf_rn(T.x, rest, __fmaf_rn(T.y, t, T.y)), __fadd_rn(s.lo, pr.lo));
  const float scale = __int_as_float(max((k >> 8) + qb, 0) << 23);
  return {__fmul_rn(s.hi, scale), __fmul_rn(lo, scale)};
}

}  // namespace sv
