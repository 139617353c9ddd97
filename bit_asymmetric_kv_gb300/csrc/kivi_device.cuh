// kivi_device.cuh -- device helpers shared by the KIVI kernels (sm_103a).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace kivi {

constexpr int kD = 128;          // head dim
constexpr int kWordsPerRow = 8;  // 128 channels x 2 bits / 32
template <int BITS>
__host__ __device__ constexpr int words_per_row() { return kD * BITS / 32; }  // 8 (2-bit) or 16 (4-bit)

// ---- fp16 bit-pattern helpers ----------------------------------------------------
__device__ __forceinline__ float h2f(uint16_t b) { return __half2float(__ushort_as_half(b)); }
__device__ __forceinline__ uint16_t f2h(float x) { return __half_as_ushort(__float2half_rn(x)); }

// ---- the 2-bit quantizer ------------------------------------------------------------
// Per-group parameters.  The rounding rule
//     code = clamp(round_half_even(fl32(fl32(x - mn) / s)), 0, 3)
// is evaluated in its comparison form: with d = fl32(x - mn) and an fp16 scale s > 0,
//     code = [d > s/2] + [d >= 3s/2] + [d > 5s/2].
// Why the two agree: s has an 11-bit significand, so s/2, 3s/2 and 5s/2 are exact
// in fp32.  fl32(d/s) > 1/2 holds exactly when d/s > 1/2 + 2^-25 (above the midpoint
// to the next float; the midpoint itself rounds to the even 1/2), and s * 2^-25 is
// smaller than one ulp of s/2, so for an fp32 d this is d > s/2.  Likewise
// fl32(d/s) >= 3/2 iff d/s >= 3/2 - 2^-24 iff d >= 3s/2 (the gap s * 2^-24 is below
// one ulp of 3s/2), and fl32(d/s) > 5/2 iff d > 5s/2.  round_half_even then gives
// code >= 1, >= 2, >= 3 exactly at these three events, and d <= max - min keeps the
// code at most 3.  When the fp16 scale is 0 all codes are 0 (thresholds = +inf).
//
// The 4-bit width (15 levels) evaluates the rule as written: u = fl32(fl32(x - mn) / s)
// with an IEEE division, then round-half-even and a clamp to 15; fp32 operations of
// the same order as the definition, so the codes are the definition's.
struct QParams {
  float mn, t1, t2, t3;  // 2-bit thresholds
  float s;               // the fp16 scale in fp32 (0: every code is 0)
  uint32_t meta;         // fp16 s | fp16 z << 16
};

template <int BITS = 2>
__device__ __forceinline__ QParams make_qparams(float mn, float mx) {
  static_assert(BITS == 2 || BITS == 4, "2- or 4-bit codes");
  QParams p;
  float range = __fsub_rn(mx, mn);
  float s32 = __fdiv_rn(range, BITS == 2 ? 3.0f : 15.0f);
  uint16_t s16 = f2h(s32);
  float s = h2f(s16);
  uint16_t z16 = f2h(mn);  // exact: mn is an fp16 value
  if (z16 == 0x8000u) z16 = 0;  // -0 is stored as +0
  p.mn = mn;
  p.s = (s16 == 0) ? 0.f : s;
  if (s16 == 0) {
    p.t1 = p.t2 = p.t3 = __int_as_float(0x7f800000);  // +inf: every code is 0
  } else {
    p.t1 = __fmul_rn(0.5f, s);
    p.t2 = __fmul_rn(1.5f, s);
    p.t3 = __fmul_rn(2.5f, s);
  }
  p.meta = (uint32_t)s16 | ((uint32_t)z16 << 16);
  return p;
}

template <int BITS = 2>
__device__ __forceinline__ uint32_t quant_code(float x, const QParams &p) {
  float d = __fsub_rn(x, p.mn);
  if constexpr (BITS == 2) {
    return (uint32_t)(d > p.t1) + (uint32_t)(d >= p.t2) + (uint32_t)(d > p.t3);
  } else {
    if (p.s == 0.f) return 0u;
    const int c = __float2int_rn(__fdiv_rn(d, p.s));  // round half to even
    return (uint32_t)(c < 0 ? 0 : (c > 15 ? 15 : c));
  }
}

// Codes of the 8 channels held in one 16-byte chunk (4 half2), channel j of the
// chunk at bits [BITS*j, BITS*j + BITS - 1]: 16 bits for 2-bit codes, a whole
// word for 4-bit codes.
template <int BITS = 2>
__device__ __forceinline__ uint32_t quant_chunk8(const uint4 &c, const QParams &p) {
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
  uint32_t bits = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float lo = h2f((uint16_t)(w[k] & 0xffffu));
    float hi = h2f((uint16_t)(w[k] >> 16));
    bits |= quant_code<BITS>(lo, p) << (2 * BITS * k);
    bits |= quant_code<BITS>(hi, p) << (2 * BITS * k + BITS);
  }
  return bits;
}

// ---- packed half2 min / max of a 16-byte chunk ---------------------------------------
__device__ __forceinline__ __half2 u2h2(uint32_t u) { return *reinterpret_cast<const __half2 *>(&u); }
__device__ __forceinline__ uint32_t h22u(__half2 h) { return *reinterpret_cast<const uint32_t *>(&h); }

// ---- cp.async (16-byte global -> shared copies, completion tracked per thread) ----
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
  uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// ---- warp-level tensor-core MMA: D(16x8,f32) += A(16x16,f16) * B(16x8,f16) ---------
__device__ __forceinline__ void mma16816(float d[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ---- 2-bit code unpack into fp16 MMA operands ------------------------------------------
// A 32-bit word w holds 16 codes, code i at bits [2i, 2i+1].  Masking w with
// 0x00030003 << 2m (m = 0..3) leaves codes m and m+8 in the two 16-bit halves at
// bits [2m, 2m+1]; as fp16 bit patterns these are the subnormals
// code * 4^m * 2^-24, exact.  The same masks on w >> 8 give codes m+4 and m+12.
// Nine integer operations therefore give
//   r[k] = {code_k, code_{k+8}} * f_k * 2^-24,   f_k = 4^(k mod 4),   k = 0..7.
// f_k and 2^-24 are undone on the other MMA operand or after accumulation.
__device__ __forceinline__ void unpack16(uint32_t w, uint32_t r[8]) {
  const uint32_t x = w >> 8;
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    r[m] = w & (0x00030003u << (2 * m));
    r[m + 4] = x & (0x00030003u << (2 * m));
  }
}

// ---- 4-bit code unpack -------------------------------------------------------------------
// A word holds 8 codes, code i at bits [4i, 4i+3].  Masks 0x000F000F and 0x00F000F0 on
// w and on w >> 8 leave, in the two 16-bit halves, the fp16 subnormals
//   r[0] = {c0, c4} * 2^-24,  r[1] = {c1, c5} * 16 * 2^-24,
//   r[2] = {c2, c6} * 2^-24,  r[3] = {c3, c7} * 16 * 2^-24   (bits 0..7 are mantissa).
__device__ __forceinline__ void unpack8(uint32_t w, uint32_t r[4]) {
  const uint32_t x = w >> 8;
  r[0] = w & 0x000F000Fu;
  r[1] = w & 0x00F000F0u;
  r[2] = x & 0x000F000Fu;
  r[3] = x & 0x00F000F0u;
}

// ---- 2-bit codes by fp16 comparisons -------------------------------------------------
// The 2-bit code [d > t1] + [d >= t2] + [d > t3] of d = fl32(x - mn) never decreases as
// the fp16 input x grows (fp32 subtraction rounds monotonically), so each of its three
// terms is [x > X] for one fp16 threshold X: the largest fp16 x for which the term is
// 0.  fp16_threshold finds it from the estimate c = fp16 round-down of fl32(mn + t) and
// proves it with two evaluations of the term itself: X = c when the term is 0 at c and
// 1 at the next fp16 above c, X = the fp16 below c when the term is 1 at c and 0 there.
// Anything else clears `ok` and the caller takes the per-element fp32 path: that needs
// fp16 steps near mn + t finer than the fp32 rounding of d, i.e. mn + t close to zero
// next to a large t (a minimum far below zero).  With s = 0 every term is 0: X = +inf.

// Order-preserving key of fp16 bits (finite or infinite, not NaN): -0 and +0 share 0x8000.
__device__ __forceinline__ uint32_t h16_key(uint32_t b) {
  return (b & 0x8000u) ? 0x8000u - (b & 0x7fffu) : 0x8000u + b;
}
__device__ __forceinline__ uint32_t h16_from_key(uint32_t k) {
  return k >= 0x8000u ? k - 0x8000u : (0x8000u | (0x8000u - k));
}

// strict: the term is [d >= t] (X = the largest x with d < t); else [d > t].
__device__ __forceinline__ uint32_t fp16_threshold(float mn, float t, bool strict, bool &ok) {
  const uint32_t c = __half_as_ushort(__float2half_rd(__fadd_rn(mn, t)));
  const float dc = __fsub_rn(h2f((uint16_t)c), mn);
  const bool below_c = strict ? (dc < t) : (dc <= t);  // the term is 0 at c
  const uint32_t kc = h16_key(c);
  const uint32_t nb = h16_from_key(below_c ? kc + 1u : kc - 1u);  // the neighbour to test
  const float dn = __fsub_rn(h2f((uint16_t)nb), mn);
  const bool below_n = strict ? (dn < t) : (dn <= t);
  ok = below_c ? !below_n : below_n;
  return below_c ? c : nb;
}

// Thresholds (X1, X2, X3) of one set of 2-bit parameters; ok as above.
__device__ __forceinline__ void fp16_thresholds(const QParams &p, uint32_t &x1, uint32_t &x2, uint32_t &x3,
                                                bool &ok) {
  if (p.s == 0.f) {
    x1 = x2 = x3 = 0x7c00u;  // +inf: every code is 0
    ok = true;
    return;
  }
  bool o1, o2, o3;
  x1 = fp16_threshold(p.mn, p.t1, false, o1);
  x2 = fp16_threshold(p.mn, p.t2, true, o2);
  x3 = fp16_threshold(p.mn, p.t3, false, o3);
  ok = o1 && o2 && o3;
}

// 2-bit codes of the 8 channels of a 16-byte chunk from fp16 thresholds: pair j of the
// chunk (channels 2j, 2j+1) is compared with the half2 thresholds X1[j], X2[j], X3[j]
// (one threshold per channel).  The three masks are nested, so the code's low bit is
// their parity and its high bit the middle mask.  Channel i of the chunk lands at bits
// [2i, 2i+1] of the low 16 bits of the result (the high 16 bits are left over).
__device__ __forceinline__ uint32_t codes2_chunk8(const uint32_t x[4], const uint32_t X1[4], const uint32_t X2[4],
                                                  const uint32_t X3[4]) {
  uint32_t r = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const __half2 v = u2h2(x[j]);
    const uint32_t m1 = __hgt2_mask(v, u2h2(X1[j]));
    const uint32_t m2 = __hgt2_mask(v, u2h2(X2[j]));
    const uint32_t m3 = __hgt2_mask(v, u2h2(X3[j]));
    const uint32_t odd = m1 ^ m2 ^ m3;
    // channel 2j at bits 4j, 4j+1 (low half); channel 2j+1 at bits 16 + 4j+2, +3
    const uint32_t k0 = (1u << (4 * j)) | (1u << (18 + 4 * j));
    r |= (odd & k0) | (m2 & (k0 << 1));
  }
  return r | (r >> 16);
}

// ---- 4-bit codes without a division per element -------------------------------------
// The 4-bit code is clamp(rint(fl32(d / s)), 0, 15) with d = fl32(x - mn) >= 0 and the
// fp16 scale s > 0.  With rs = 1/s rounded to nearest, q = fl32(d * rs) lies within
// Q * 2^-23 of the quotient Q = d / s, and the correctly rounded quotient within
// Q * 2^-24 of Q; below 64 both are under 2^-16.  So when q is more than 2^-15 from
// every half-integer, the division rounds to the same integer as q; only there
// does the division itself run.  q >= 64 means Q > 63: the code is 15.
__device__ __forceinline__ uint32_t code4(float x, float mn, float s, float rs) {
  if (s == 0.f) return 0u;
  const float d = __fsub_rn(x, mn);
  const float q = __fmul_rn(d, rs);
  if (q >= 64.f) return 15u;
  float c = rintf(q);                                   // half to even, like the division's rounding
  if (fabsf(q - c) > 0.5f - 0x1p-15f) c = rintf(__fdiv_rn(d, s));  // q - c is exact
  const int ci = (int)c;
  return (uint32_t)(ci > 15 ? 15 : ci);
}

// Two 4-bit codes at once (channel pair or two elements of one row): x, mn, s and
// rs = 1/s (0 when s = 0: every code is then 0) per element.  d = fl(x - mn) and
// q = fl(d * rs) by paired fp32 operations, each element rounded to nearest like the
// scalar operations of code4.  rint(q) comes from adding and subtracting 1.5 * 2^23
// (round half to even for 0 <= q < 2^22; q stays below 32 here), its integer from the
// sum's bit pattern, and q - rint(q) is exact; within 2^-15 of a half-integer the
// division decides, as in code4.  Returns c0 | c1 << 4.
__device__ __forceinline__ uint32_t code4x2(float2 x, float2 mn, float2 s, float2 rs) {
  constexpr float kM = 12582912.f;  // 1.5 * 2^23
  const float2 d = __fadd2_rn(x, make_float2(-mn.x, -mn.y));
  const float2 q = __fmul2_rn(d, rs);
  const float2 t = __fadd2_rn(q, make_float2(kM, kM));
  const float2 r = __fadd2_rn(t, make_float2(-kM, -kM));
  const float2 e = __fadd2_rn(q, make_float2(-r.x, -r.y));
  int c0 = __float_as_int(t.x) - __float_as_int(kM), c1 = __float_as_int(t.y) - __float_as_int(kM);
  if (fabsf(e.x) > 0.5f - 0x1p-15f) c0 = (int)rintf(__fdiv_rn(d.x, s.x));
  if (fabsf(e.y) > 0.5f - 0x1p-15f) c1 = (int)rintf(__fdiv_rn(d.y, s.y));
  return (uint32_t)min(c0, 15) | ((uint32_t)min(c1, 15) << 4);
}

// One code of either width; rs = 1/s (used by 4-bit codes only).
template <int BITS>
__device__ __forceinline__ uint32_t qcode(float x, const QParams &p, float rs) {
  if constexpr (BITS == 2) {
    return quant_code<2>(x, p);
  } else {
    return code4(x, p.mn, p.s, rs);
  }
}

// Codes of the 8 channels of a 16-byte chunk under one set of parameters (channel j at
// bits [BITS*j, BITS*j + BITS - 1]).
template <int BITS>
__device__ __forceinline__ uint32_t qchunk8(const uint4 &c, const QParams &p) {
  if constexpr (BITS == 2) {
    return quant_chunk8<2>(c, p);
  } else {
    const float rs = p.s == 0.f ? 0.f : __frcp_rn(p.s);
    const float2 mn2 = make_float2(p.mn, p.mn), s2 = make_float2(p.s, p.s), rs2 = make_float2(rs, rs);
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
    uint32_t bits = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) bits |= code4x2(__half22float2(u2h2(w[k])), mn2, s2, rs2) << (8 * k);
    return bits;
  }
}

// Pieces of LPW lanes x LPW rows transposed across the lanes.  Before, lane j holds
// its piece of row i at bits [PB*i, PB*i + PB); after, lane j holds row j, with lane
// i's piece at bits [PB*i, PB*i + PB).  Stage d swaps the off-diagonal blocks of
// size d between lanes j and j ^ d (d = LPW/2 .. 1): log2(LPW) shuffles for LPW rows.
template <int LPW, int PB>
__device__ __forceinline__ uint32_t transpose_pieces(uint32_t A, int j) {
#pragma unroll
  for (int d = LPW / 2; d >= 1; d >>= 1) {
    uint32_t lo = 0;  // the pieces whose index has bit d clear
#pragma unroll
    for (int i = 0; i < 32 / PB; ++i)
      if (!(i & d)) lo |= ((1u << PB) - 1u) << (PB * i);
    const bool up = (j & d) != 0;
    const uint32_t send = up ? (A & lo) << (PB * d) : (A & ~lo) >> (PB * d);
    const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, d);
    A = (up ? (A & ~lo) : (A & lo)) | recv;
  }
  return A;
}

// Key codes of one channel pair over 32 token rows of one key group, held by one
// lane: x[r] = the fp16 pair (channels 2cp, 2cp+1) of row r, mn / mx their min and max
// over the whole group.  The lane derives both channels' parameters, writes their
// {s, z} words to meta_dst[0..1] when `write_meta`, codes its rows (2-bit: fp16
// comparisons with proven thresholds, the fp32 comparison form when a threshold of
// the warp is not proven; 4-bit: the reciprocal product), and the transpose above
// packs the LPW lanes of a code word: lane j of them stores word cp / LPW of row
// blk * LPW + j at codes_dst[(blk * LPW + j) * WPR], codes_dst pointing at that word
// of row 0.  Nothing is stored unless `whole` (a quantized group, not the residual).
// Every lane of the warp must call it (shuffles), the 32 lanes holding consecutive
// channel pairs.
template <int BITS>
__device__ __forceinline__ void key_pair_codes(const uint32_t (&x)[32], __half2 mn, __half2 mx, int lane, bool whole,
                                               bool write_meta, uint32_t *meta_dst, uint32_t *codes_dst) {
  constexpr int WPR = words_per_row<BITS>();
  constexpr int PB = 2 * BITS;   // bits of one lane's two codes
  constexpr int LPW = 32 / PB;   // lanes (channel pairs) per packed word
  const QParams p0 = make_qparams<BITS>(__low2float(mn), __low2float(mx));
  const QParams p1 = make_qparams<BITS>(__high2float(mn), __high2float(mx));
  if (whole && write_meta) *reinterpret_cast<uint2 *>(meta_dst) = make_uint2(p0.meta, p1.meta);
  uint32_t T1 = 0, T2 = 0, T3 = 0;
  bool fast = true;
  float rs0 = 0.f, rs1 = 0.f;
  if constexpr (BITS == 2) {
    uint32_t a1, a2, a3, b1, b2, b3;
    bool oa, ob;
    fp16_thresholds(p0, a1, a2, a3, oa);
    fp16_thresholds(p1, b1, b2, b3, ob);
    T1 = a1 | (b1 << 16);
    T2 = a2 | (b2 << 16);
    T3 = a3 | (b3 << 16);
    fast = __all_sync(0xffffffffu, oa && ob);
  } else {
    rs0 = p0.s == 0.f ? 0.f : __frcp_rn(p0.s);
    rs1 = p1.s == 0.f ? 0.f : __frcp_rn(p1.s);
  }
#pragma unroll
  for (int blk = 0; blk < 32 / LPW; ++blk) {
    uint32_t A = 0;
#pragma unroll
    for (int i = 0; i < LPW; ++i) {
      const uint32_t v = x[blk * LPW + i];
      uint32_t pc;
      if constexpr (BITS == 2) {
        if (fast) {
          const __half2 hv = u2h2(v);
          const uint32_t m1 = __hgt2_mask(hv, u2h2(T1)), m2 = __hgt2_mask(hv, u2h2(T2));
          const uint32_t m3 = __hgt2_mask(hv, u2h2(T3));
          // nested masks: the code's low bit is their parity, its high bit the middle one
          const uint32_t c = ((m1 ^ m2 ^ m3) & 0x00010001u) | (m2 & 0x00020002u);
          pc = (c | (c >> 14)) & 0xFu;
        } else {
          pc = quant_code<2>(h2f((uint16_t)(v & 0xffffu)), p0) | (quant_code<2>(h2f((uint16_t)(v >> 16)), p1) << 2);
        }
      } else {
        pc = code4x2(__half22float2(u2h2(v)), make_float2(p0.mn, p1.mn), make_float2(p0.s, p1.s),
                     make_float2(rs0, rs1));
      }
      A |= pc << (PB * i);
    }
    const int j = lane % LPW;
    const uint32_t word = transpose_pieces<LPW, PB>(A, j);
    if (whole) codes_dst[(blk * LPW + j) * WPR] = word;
  }
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) { return __byte_perm(a, b, sel); }

}  // namespace kivi
