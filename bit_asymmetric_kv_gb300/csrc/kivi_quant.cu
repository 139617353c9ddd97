// kivi_quant.cu -- quantize / pack kernels of the KIVI 2-bit KV cache and its 4-bit
// variant (sm_103a).
//
// KIVI page ("Makale Bulteni -- KIVI", cmlonder.com radar / paper-to-prod,
// 2026-11-01): headline paragraph (keys per channel, values per token, asymmetric
// 2-bit) and section "Iddia ve Gerceklik", paragraphs 2-3 (G-token key groups, a
// full-precision residual for the unfilled group).  The kernels here stream fp16
// inputs once from HBM and write 1/8 (2-bit) or 1/4 (4-bit) of that in codes; the
// per-element work is kept small (fp16 comparisons, a reciprocal product) so that
// the memory stream, not the arithmetic, sets their speed.
#include "kivi_device.cuh"
#include "kivi_internal.h"

namespace kivi {

// Row of token t of head bh in a paged pool (false: the block table gives no page
// of the pool for it, and the row is skipped).
__device__ __forceinline__ bool paged_row(const PageMap &pm, int64_t bh, int64_t t, int64_t *row) {
  const int64_t page = pm.bt[t >> pm.shift];
  if (page < 0 || page >= pm.num_pages) return false;
  *row = ((page * pm.Hkv + bh) << pm.shift) + (t & ((1 << pm.shift) - 1));
  return true;
}

// -------------------------------------------------------------------------------------
// Key groups: one CTA (4 warps) quantizes one G-token group of one (batch, KV head).
// Warp w owns channels 32w .. 32w+31.  Lane = 4 * t8 + c4: the lane loads the
// 16-byte chunk c4 (8 channels) of tokens t8, t8 + 8, ... so one warp instruction
// reads 8 token rows x 64 contiguous bytes.
// -------------------------------------------------------------------------------------
template <int G, bool PAGED, int BITS>
__global__ void __launch_bounds__(128) key_group_kernel(const uint16_t *__restrict__ in, int64_t in_head_stride,
                                                        int64_t groups_per_head, int64_t g0,
                                                        uint32_t *__restrict__ k_codes,
                                                        uint32_t *__restrict__ k_meta, int64_t max_tokens,
                                                        const PageMap pm) {
  // a decode launched as a programmatic dependent may start its independent work now
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  constexpr int TPL = G / 8;  // tokens per lane
  constexpr int WPR = words_per_row<BITS>();
  __shared__ __align__(16) uint32_t s_codes[G * WPR];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t8 = lane >> 2, c4 = lane & 3;
  // 32-bit division: the grid has fewer than 2^31 CTAs (a 64-bit one is a called routine)
  const int64_t bh = (int64_t)(blockIdx.x / (uint32_t)groups_per_head);
  const int64_t gi = (int64_t)(blockIdx.x % (uint32_t)groups_per_head);
  const int64_t g = g0 + gi;
  // destination: first token row of the group and its (group, channel) meta row
  int64_t row0, grp;
  if constexpr (PAGED) {
    if (!paged_row(pm, bh, g * G, &row0)) return;  // the whole CTA: one group, one page
    grp = row0 / G;  // pages hold whole groups, so row0 is a multiple of G
  } else {
    row0 = bh * max_tokens + g * G;
    grp = bh * (max_tokens / G) + g;
  }
  const uint16_t *src = in + bh * in_head_stride + gi * (int64_t)G * kD + 32 * warp + 8 * c4;

  // the lane's G/8 chunks as words (registers: every index below is a constant)
  uint32_t x[TPL][4];
#pragma unroll
  for (int k = 0; k < TPL; ++k) {
    const uint4 c = __ldg(reinterpret_cast<const uint4 *>(src + (int64_t)(t8 + 8 * k) * kD));
    x[k][0] = c.x;
    x[k][1] = c.y;
    x[k][2] = c.z;
    x[k][3] = c.w;
  }

  // per-channel min and max over the G tokens: local, then across the 8 token lanes
  __half2 mn[4], mx[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) mn[j] = mx[j] = u2h2(x[0][j]);
#pragma unroll
  for (int k = 1; k < TPL; ++k) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      mn[j] = __hmin2(mn[j], u2h2(x[k][j]));
      mx[j] = __hmax2(mx[j], u2h2(x[k][j]));
    }
  }
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      mn[j] = __hmin2(mn[j], u2h2(__shfl_xor_sync(0xffffffffu, h22u(mn[j]), off)));
      mx[j] = __hmax2(mx[j], u2h2(__shfl_xor_sync(0xffffffffu, h22u(mx[j]), off)));
    }
  }
  // lane (t8, c4) derives the parameters of channel t8 of its chunk, then they are
  // broadcast to the 8 lanes that hold the chunk
  uint32_t mn_bits = h22u(mn[0]), mx_bits = h22u(mx[0]);
#pragma unroll
  for (int j = 1; j < 4; ++j)
    if ((t8 >> 1) == j) {
      mn_bits = h22u(mn[j]);
      mx_bits = h22u(mx[j]);
    }
  const float my_mn = h2f((uint16_t)((t8 & 1) ? (mn_bits >> 16) : (mn_bits & 0xffffu)));
  const float my_mx = h2f((uint16_t)((t8 & 1) ? (mx_bits >> 16) : (mx_bits & 0xffffu)));
  const QParams mine = make_qparams<BITS>(my_mn, my_mx);
  k_meta[grp * kD + 32 * warp + 8 * c4 + t8] = mine.meta;

  // 2-bit codes by fp16 comparisons with the channels' thresholds (exact whenever every
  // threshold of the warp is proven; else the per-element fp32 form below)
  bool fast = false;
  if constexpr (BITS == 2) {
    uint32_t X1, X2, X3;
    bool ok;
    fp16_thresholds(mine, X1, X2, X3, ok);
    fast = __all_sync(0xffffffffu, ok);
    if (fast) {
      // half2 thresholds of channel pair (t8 & ~1, t8 | 1): the odd channel is lane ^ 4
      const uint32_t o1 = __shfl_xor_sync(0xffffffffu, X1, 4);
      const uint32_t o2 = __shfl_xor_sync(0xffffffffu, X2, 4);
      const uint32_t o3 = __shfl_xor_sync(0xffffffffu, X3, 4);
      const uint32_t sel = (t8 & 1) ? 0x1054u : 0x5410u;  // (even channel, odd channel)
      const uint32_t P1 = __byte_perm(X1, o1, sel), P2 = __byte_perm(X2, o2, sel), P3 = __byte_perm(X3, o3, sel);
      uint32_t T1[4], T2[4], T3[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int src_lane = 8 * j + c4;  // the lane of channel 2j of this chunk
        T1[j] = __shfl_sync(0xffffffffu, P1, src_lane);
        T2[j] = __shfl_sync(0xffffffffu, P2, src_lane);
        T3[j] = __shfl_sync(0xffffffffu, P3, src_lane);
      }
#pragma unroll
      for (int k = 0; k < TPL; ++k) {
        const uint32_t bits = codes2_chunk8(x[k], T1, T2, T3);
        // chunks 2m and 2m+1 form word 2*warp + m of the token row
        const uint32_t other = __shfl_xor_sync(0xffffffffu, bits, 1);
        if ((c4 & 1) == 0) s_codes[(t8 + 8 * k) * WPR + 2 * warp + (c4 >> 1)] = __byte_perm(bits, other, 0x5410);
      }
    }
  }
  if (!fast) {
    QParams p[8];
    float rs[8];  // 4-bit: 1/s, 0 where s = 0 (code4x2 then gives 0), one reciprocal per lane
    const float rs_mine = BITS == 4 && mine.s != 0.f ? __frcp_rn(mine.s) : 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int src_lane = 4 * j + c4;
      p[j].mn = __shfl_sync(0xffffffffu, mine.mn, src_lane);
      rs[j] = 0.f;
      if constexpr (BITS == 2) {
        p[j].t1 = __shfl_sync(0xffffffffu, mine.t1, src_lane);
        p[j].t2 = __shfl_sync(0xffffffffu, mine.t2, src_lane);
        p[j].t3 = __shfl_sync(0xffffffffu, mine.t3, src_lane);
      } else {
        p[j].s = __shfl_sync(0xffffffffu, mine.s, src_lane);
        rs[j] = __shfl_sync(0xffffffffu, rs_mine, src_lane);
      }
    }
#pragma unroll
    for (int k = 0; k < TPL; ++k) {
      uint32_t bits = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if constexpr (BITS == 4) {
          bits |= code4x2(__half22float2(u2h2(x[k][j])), make_float2(p[2 * j].mn, p[2 * j + 1].mn),
                          make_float2(p[2 * j].s, p[2 * j + 1].s), make_float2(rs[2 * j], rs[2 * j + 1]))
                  << (8 * j);
        } else {
          bits |= qcode<BITS>(h2f((uint16_t)(x[k][j] & 0xffffu)), p[2 * j], rs[2 * j]) << (2 * BITS * j);
          bits |= qcode<BITS>(h2f((uint16_t)(x[k][j] >> 16)), p[2 * j + 1], rs[2 * j + 1]) << (2 * BITS * j + BITS);
        }
      }
      if constexpr (BITS == 2) {
        // chunks 2m and 2m+1 form word 2*warp + m of the token row
        const uint32_t other = __shfl_xor_sync(0xffffffffu, bits, 1);
        if ((c4 & 1) == 0) s_codes[(t8 + 8 * k) * WPR + 2 * warp + (c4 >> 1)] = bits | (other << 16);
      } else {
        // chunk c4 of warp w is word 4w + c4 of the token row
        s_codes[(t8 + 8 * k) * WPR + 4 * warp + c4] = bits;
      }
    }
  }
  __syncthreads();
  // coalesced write of the G packed token rows
  uint4 *dst = reinterpret_cast<uint4 *>(k_codes + row0 * WPR);
  const uint4 *s4 = reinterpret_cast<const uint4 *>(s_codes);
  for (int i = threadIdx.x; i < G * WPR / 4; i += blockDim.x) dst[i] = s4[i];
}

// -------------------------------------------------------------------------------------
// Key groups of G = 32 tokens, two groups per CTA: warp w takes group w / 2 of
// the pair and channels 64 (w % 2) .. 64 (w % 2) + 63.  Lane = 8 * t4 + c8 loads the
// 16-byte chunk c8 (8 channels) of tokens t4, t4 + 4, .. t4 + 28, so that each lane
// holds 64 elements, as the G = 64 kernel's lanes do: the per-channel min/max then
// needs two shuffle rounds over the 4 token lanes, and lane (t4, c8) derives the
// parameters (and, for 2-bit codes, proves the thresholds) of channel pair t4 of its
// chunk.  4-bit codes: the chunk's parameters are broadcast to its lanes, and each
// token's chunk is one packed word, coded by pairs (code4x2).
// -------------------------------------------------------------------------------------
template <bool PAGED, int BITS>
__global__ void __launch_bounds__(128) key_pairs32_kernel(const uint16_t *__restrict__ in, int64_t in_head_stride,
                                                          int64_t groups_per_head, int64_t pairs_per_head,
                                                          int64_t g0, uint32_t *__restrict__ k_codes,
                                                          uint32_t *__restrict__ k_meta, int64_t max_tokens,
                                                          const PageMap pm) {
  // a decode launched as a programmatic dependent may start its independent work now
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  constexpr int G = 32, WPR = words_per_row<BITS>();
  __shared__ __align__(16) uint32_t s_codes[2 * G * WPR];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = warp >> 1, ch = warp & 1, t4 = lane >> 3, c8 = lane & 7;
  const int64_t bh = (int64_t)blockIdx.x / pairs_per_head;
  const int64_t gi0 = ((int64_t)blockIdx.x - bh * pairs_per_head) * 2;  // first group of the pair (source)
  const int ngrp = (int)min((int64_t)2, groups_per_head - gi0);          // 1 or 2
  const int64_t g = g0 + gi0;                                             // destination group
  int64_t row0, grp;
  if constexpr (PAGED) {
    if (!paged_row(pm, bh, g * G, &row0)) return;  // the whole CTA: both groups lie in one page
    grp = row0 / G;
  } else {
    row0 = bh * max_tokens + g * G;
    grp = bh * (max_tokens / G) + g;
  }
  if (gq < ngrp) {
    const uint16_t *src = in + bh * in_head_stride + (gi0 + gq) * (int64_t)G * kD + 64 * ch + 8 * c8;
    uint32_t x[8][4];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint4 c = __ldg(reinterpret_cast<const uint4 *>(src + (int64_t)(t4 + 4 * k) * kD));
      x[k][0] = c.x;
      x[k][1] = c.y;
      x[k][2] = c.z;
      x[k][3] = c.w;
    }
    __half2 mn[4], mx[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) mn[j] = mx[j] = u2h2(x[0][j]);
#pragma unroll
    for (int k = 1; k < 8; ++k)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        mn[j] = __hmin2(mn[j], u2h2(x[k][j]));
        mx[j] = __hmax2(mx[j], u2h2(x[k][j]));
      }
#pragma unroll
    for (int off = 8; off < 32; off <<= 1)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        mn[j] = __hmin2(mn[j], u2h2(__shfl_xor_sync(0xffffffffu, h22u(mn[j]), off)));
        mx[j] = __hmax2(mx[j], u2h2(__shfl_xor_sync(0xffffffffu, h22u(mx[j]), off)));
      }
    // this lane's channel pair: t4 of the chunk (channels 8 c8 + 2 t4, + 1)
    __half2 pmn = mn[0], pmx = mx[0];
#pragma unroll
    for (int j = 1; j < 4; ++j)
      if (t4 == j) {
        pmn = mn[j];
        pmx = mx[j];
      }
    const QParams p0 = make_qparams<BITS>(__low2float(pmn), __low2float(pmx));
    const QParams p1 = make_qparams<BITS>(__high2float(pmn), __high2float(pmx));
    *reinterpret_cast<uint2 *>(k_meta + (grp + gq) * kD + 64 * ch + 8 * c8 + 2 * t4) = make_uint2(p0.meta, p1.meta);
    if constexpr (BITS == 4) {
      // every channel of the chunk: pair j from lane 8 j + c8 (1/s, 0 where s = 0)
      const float rs0 = p0.s == 0.f ? 0.f : __frcp_rn(p0.s), rs1 = p1.s == 0.f ? 0.f : __frcp_rn(p1.s);
      float2 cmn[4], cs[4], crs[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int sl = 8 * j + c8;
        cmn[j] = make_float2(__shfl_sync(0xffffffffu, p0.mn, sl), __shfl_sync(0xffffffffu, p1.mn, sl));
        cs[j] = make_float2(__shfl_sync(0xffffffffu, p0.s, sl), __shfl_sync(0xffffffffu, p1.s, sl));
        crs[j] = make_float2(__shfl_sync(0xffffffffu, rs0, sl), __shfl_sync(0xffffffffu, rs1, sl));
      }
      // chunk c8 of channel half ch is word 8 ch + c8 of a token row
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        uint32_t word = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) word |= code4x2(__half22float2(u2h2(x[k][j])), cmn[j], cs[j], crs[j]) << (8 * j);
        s_codes[(gq * G + t4 + 4 * k) * WPR + 8 * ch + c8] = word;
      }
    } else {
    uint32_t a1, a2, a3, b1, b2, b3;
    bool oa, ob;
    fp16_thresholds(p0, a1, a2, a3, oa);
    fp16_thresholds(p1, b1, b2, b3, ob);
    uint32_t r[8];
    if (__all_sync(0xffffffffu, oa && ob)) {
      const uint32_t P1 = a1 | (b1 << 16), P2 = a2 | (b2 << 16), P3 = a3 | (b3 << 16);
      uint32_t T1[4], T2[4], T3[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {  // pair j of the chunk lives in lane 8 j + c8
        T1[j] = __shfl_sync(0xffffffffu, P1, 8 * j + c8);
        T2[j] = __shfl_sync(0xffffffffu, P2, 8 * j + c8);
        T3[j] = __shfl_sync(0xffffffffu, P3, 8 * j + c8);
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) r[k] = codes2_chunk8(x[k], T1, T2, T3);
    } else {
      // the fp32 comparison form with every channel's parameters of the chunk
      QParams q[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int sl = 8 * j + c8;
        q[2 * j].mn = __shfl_sync(0xffffffffu, p0.mn, sl);
        q[2 * j].t1 = __shfl_sync(0xffffffffu, p0.t1, sl);
        q[2 * j].t2 = __shfl_sync(0xffffffffu, p0.t2, sl);
        q[2 * j].t3 = __shfl_sync(0xffffffffu, p0.t3, sl);
        q[2 * j + 1].mn = __shfl_sync(0xffffffffu, p1.mn, sl);
        q[2 * j + 1].t1 = __shfl_sync(0xffffffffu, p1.t1, sl);
        q[2 * j + 1].t2 = __shfl_sync(0xffffffffu, p1.t2, sl);
        q[2 * j + 1].t3 = __shfl_sync(0xffffffffu, p1.t3, sl);
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        uint32_t bits = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          bits |= quant_code<2>(h2f((uint16_t)(x[k][j] & 0xffffu)), q[2 * j]) << (4 * j);
          bits |= quant_code<2>(h2f((uint16_t)(x[k][j] >> 16)), q[2 * j + 1]) << (4 * j + 2);
        }
        r[k] = bits;
      }
    }
    // chunks 2m and 2m+1 (lanes c8 and c8 ^ 1) form word 4 ch + m of a token row
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint32_t other = __shfl_xor_sync(0xffffffffu, r[k], 1);
      if ((c8 & 1) == 0)
        s_codes[(gq * G + t4 + 4 * k) * WPR + 4 * ch + (c8 >> 1)] = (r[k] & 0xffffu) | (other << 16);
    }
    }
  }
  __syncthreads();
  // coalesced write of the pair's packed token rows (contiguous: one page holds both)
  uint4 *dst = reinterpret_cast<uint4 *>(k_codes + row0 * WPR);
  const uint4 *s4 = reinterpret_cast<const uint4 *>(s_codes);
  for (int i = threadIdx.x; i < ngrp * G * WPR / 4; i += blockDim.x) dst[i] = s4[i];
}

// -------------------------------------------------------------------------------------
// Value tokens at append: 16 lanes per token row (one 16-byte chunk of 8 channels each).
// quantize_value_row works on one half-warp; `lane16` is the lane within it.
// -------------------------------------------------------------------------------------
// With value channel groups, lanes 8m/vg .. share group m: the min/max reduction runs
// over vg_lanes = vg / 8 lanes, and the group's first lane writes meta_out[group].
template <int BITS>
__device__ __forceinline__ void quantize_value_row(const uint4 x, int lane16, uint32_t half_mask,
                                                   uint32_t *codes_row, uint32_t *meta_out, int vg_lanes = 16) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
  __half2 mn = __hmin2(__hmin2(u2h2(w[0]), u2h2(w[1])), __hmin2(u2h2(w[2]), u2h2(w[3])));
  __half2 mx = __hmax2(__hmax2(u2h2(w[0]), u2h2(w[1])), __hmax2(u2h2(w[2]), u2h2(w[3])));
  // pack (min, -max) so one __hmin2 reduces both
  __half2 red = __halves2half2(__hmin(__low2half(mn), __high2half(mn)),
                               __hneg(__hmax(__low2half(mx), __high2half(mx))));
#pragma unroll
  for (int off = 1; off < 16; off <<= 1)
    if (off < vg_lanes) red = __hmin2(red, u2h2(__shfl_xor_sync(half_mask, h22u(red), off)));
  const float fmn = __low2float(red);
  const float fmx = -__high2float(red);
  const QParams p = make_qparams<BITS>(fmn, fmx);
  const uint32_t bits = qchunk8<BITS>(x, p);
  if constexpr (BITS == 2) {
    const uint32_t other = __shfl_xor_sync(half_mask, bits, 1);
    if ((lane16 & 1) == 0) codes_row[lane16 >> 1] = bits | (other << 16);
  } else {
    codes_row[lane16] = bits;  // chunk lane16 = channels 8*lane16 .. +7 = word lane16
  }
  if (lane16 % vg_lanes == 0) meta_out[lane16 / vg_lanes] = p.meta;
}

// Value rows, 4 lanes per row and 8 rows per warp: lane q of a row holds the 16-byte
// chunks q, q+4, q+8, q+12 (channels 8(q+4k) .. 8(q+4k)+7), so that every load
// instruction reads 64 contiguous bytes of each row.  The 4 lanes share the row's min
// and max and its parameters.  2-bit codes: lanes 0-2 each prove one fp16 threshold
// of the row and the codes are fp16 comparisons with them (the fp32 form when a
// threshold of the warp is not proven).  4-bit codes: the reciprocal product (code4);
// chunk c of a row is code word c.
// rows = heads * tokens_per_head; row r -> head r / tokens_per_head, token t0 + r % tokens_per_head,
// read from input row (head * in_rows_per_head + r % tokens_per_head)
// VG < 128 (value channel groups, dense 2-bit caches): lane q's chunk q + 4k lies in
// group k / (VG / 32); each group's min/max is reduced over the row's 4 lanes, and its
// codes take the fp32 comparison form; the row's meta holds 128 / VG {s, z} words.
template <bool PAGED, int BITS, int VG = kD>
__global__ void __launch_bounds__(256) value_rows2_kernel(const uint16_t *__restrict__ v, int64_t rows,
                                                          int64_t tokens_per_head, int64_t in_rows_per_head,
                                                          int64_t t0, uint32_t *__restrict__ v_codes,
                                                          uint32_t *__restrict__ v_meta, int64_t max_tokens,
                                                          const PageMap pm) {
  const int lane = threadIdx.x & 31, q = lane & 3;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t row0 = ((int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * 8; row0 < rows;
       row0 += warps * 8) {
    const int64_t row = row0 + (lane >> 2);
    bool ok_row = row < rows;
    int64_t bh = 0, i = 0, dst = 0;
    if (ok_row) {
      bh = row / tokens_per_head;
      i = row - bh * tokens_per_head;
      const int64_t t = t0 + i;
      dst = bh * max_tokens + t;
      if constexpr (PAGED) ok_row = paged_row(pm, bh, t, &dst);
    }
    const uint4 *src = reinterpret_cast<const uint4 *>(v + (bh * in_rows_per_head + i) * kD) + q;
    uint32_t x[4][4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint4 c = ok_row ? __ldg(src + 4 * k) : make_uint4(0u, 0u, 0u, 0u);
      x[k][0] = c.x;
      x[k][1] = c.y;
      x[k][2] = c.z;
      x[k][3] = c.w;
    }
    if constexpr (VG < kD) {
      static_assert(BITS == 2 && !PAGED, "value channel groups: dense 2-bit caches");
      constexpr int NV = kD / VG, KPG = VG / 32;  // groups per row, chunks of a lane per group
      QParams pg[NV];
#pragma unroll
      for (int m = 0; m < NV; ++m) {
        __half2 gmn = u2h2(x[m * KPG][0]), gmx = gmn;
#pragma unroll
        for (int k = m * KPG; k < (m + 1) * KPG; ++k)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            gmn = __hmin2(gmn, u2h2(x[k][j]));
            gmx = __hmax2(gmx, u2h2(x[k][j]));
          }
        __half2 gred = __halves2half2(__hmin(__low2half(gmn), __high2half(gmn)),
                                      __hneg(__hmax(__low2half(gmx), __high2half(gmx))));
        gred = __hmin2(gred, u2h2(__shfl_xor_sync(0xffffffffu, h22u(gred), 1)));
        gred = __hmin2(gred, u2h2(__shfl_xor_sync(0xffffffffu, h22u(gred), 2)));
        pg[m] = make_qparams<2>(__low2float(gred), -__high2float(gred));
      }
      uint32_t r[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) r[k] = quant_chunk8<2>(make_uint4(x[k][0], x[k][1], x[k][2], x[k][3]), pg[k / KPG]);
      const uint32_t A = __byte_perm(r[0], r[1], 0x5410), B = __byte_perm(r[2], r[3], 0x5410);
      const uint32_t recv = __shfl_xor_sync(0xffffffffu, (q & 1) ? A : B, 1);
      const uint32_t lo = (q & 1) ? recv : A, hi = (q & 1) ? B : recv;
      if (ok_row) {
        uint32_t *codes_row = v_codes + dst * 8;
        const int w = (q >> 1) + ((q & 1) ? 4 : 0);
        codes_row[w] = __byte_perm(lo, hi, 0x5410);
        codes_row[w + 2] = __byte_perm(lo, hi, 0x7632);
#pragma unroll
        for (int m = 0; m < NV; ++m)
          if (q == m) v_meta[dst * NV + m] = pg[m].meta;
      }
      continue;
    }
    __half2 mn = u2h2(x[0][0]), mx = mn;
#pragma unroll
    for (int k = 0; k < 4; ++k)
#pragma unroll
      for (int j = (k == 0 ? 1 : 0); j < 4; ++j) {
        mn = __hmin2(mn, u2h2(x[k][j]));
        mx = __hmax2(mx, u2h2(x[k][j]));
      }
    // (min, -max) so that one __hmin2 reduces both over the row's 4 lanes
    __half2 red = __halves2half2(__hmin(__low2half(mn), __high2half(mn)),
                                 __hneg(__hmax(__low2half(mx), __high2half(mx))));
    red = __hmin2(red, u2h2(__shfl_xor_sync(0xffffffffu, h22u(red), 1)));
    red = __hmin2(red, u2h2(__shfl_xor_sync(0xffffffffu, h22u(red), 2)));
    const QParams p = make_qparams<BITS>(__low2float(red), -__high2float(red));
    if constexpr (BITS == 4) {
      if (ok_row) {
        uint32_t *codes_row = v_codes + dst * 16;
#pragma unroll
        for (int k = 0; k < 4; ++k) codes_row[q + 4 * k] = qchunk8<4>(make_uint4(x[k][0], x[k][1], x[k][2], x[k][3]), p);
        if (q == 0) v_meta[dst] = p.meta;
      }
      continue;
    }
    // lane q < 3 proves threshold q + 1 (X2 is the strict one: d >= t2)
    bool ok = true;
    uint32_t xq = 0x7c00u;
    if (p.s != 0.f && q < 3) xq = fp16_threshold(p.mn, q == 0 ? p.t1 : (q == 1 ? p.t2 : p.t3), q == 1, ok);
    const int base = lane & ~3;
    const uint32_t x1 = __shfl_sync(0xffffffffu, xq, base), x2 = __shfl_sync(0xffffffffu, xq, base + 1),
                   x3 = __shfl_sync(0xffffffffu, xq, base + 2);
    uint32_t r[4];
    if (__all_sync(0xffffffffu, ok)) {
      const uint32_t p1 = x1 | (x1 << 16), p2 = x2 | (x2 << 16), p3 = x3 | (x3 << 16);
      const uint32_t X1[4] = {p1, p1, p1, p1}, X2[4] = {p2, p2, p2, p2}, X3[4] = {p3, p3, p3, p3};
#pragma unroll
      for (int k = 0; k < 4; ++k) r[k] = codes2_chunk8(x[k], X1, X2, X3);
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k) r[k] = quant_chunk8<2>(make_uint4(x[k][0], x[k][1], x[k][2], x[k][3]), p);
    }
    // word w of the row = chunk 2w (low 16 bits) | chunk 2w+1 (high 16 bits): lanes q and
    // q^1 hold the two halves of words q/2 + 2k; the even lane stores k = 0, 1, the odd k = 2, 3
    const uint32_t A = __byte_perm(r[0], r[1], 0x5410), B = __byte_perm(r[2], r[3], 0x5410);
    const uint32_t recv = __shfl_xor_sync(0xffffffffu, (q & 1) ? A : B, 1);
    const uint32_t lo = (q & 1) ? recv : A, hi = (q & 1) ? B : recv;
    if (ok_row) {
      uint32_t *codes_row = v_codes + dst * 8;
      const int w = (q >> 1) + ((q & 1) ? 4 : 0);
      codes_row[w] = __byte_perm(lo, hi, 0x5410);
      codes_row[w + 2] = __byte_perm(lo, hi, 0x7632);
      if (q == 0) v_meta[dst] = p.meta;
    }
  }
}


// Append: one warp per (batch, KV head).  Lanes 0-15 quantize the new value row (or,
// with a value residual, copy it into residual slot r); lanes 16-31 copy the new
// key (256 bytes) into residual slot r.
template <int BITS>
__global__ void __launch_bounds__(128) append_kernel(const uint16_t *__restrict__ k_new,
                                                     const uint16_t *__restrict__ v_new, int64_t heads,
                                                     int64_t n, int G, uint16_t *__restrict__ k_res,
                                                     uint32_t *__restrict__ v_codes,
                                                     uint32_t *__restrict__ v_meta, int64_t max_tokens,
                                                     uint16_t *__restrict__ v_res, int vg) {
  // a decode launched as a programmatic dependent may start its independent work now
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  const int64_t bh = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (bh >= heads) return;
  const int lane = threadIdx.x & 31;
  const int lane16 = lane & 15;
  if (lane < 16) {
    const uint4 x = __ldg(reinterpret_cast<const uint4 *>(v_new + bh * kD) + lane16);
    if (v_res)
      reinterpret_cast<uint4 *>(v_res + (bh * G + n % G) * kD)[lane16] = x;
    else
      quantize_value_row<BITS>(x, lane16, 0x0000ffffu, v_codes + (bh * max_tokens + n) * words_per_row<BITS>(),
                               v_meta + (bh * max_tokens + n) * (kD / vg), vg / 8);
  } else {
    const int64_t r = n % G;
    const uint4 x = __ldg(reinterpret_cast<const uint4 *>(k_new + bh * kD) + lane16);
    reinterpret_cast<uint4 *>(k_res + (bh * G + r) * kD)[lane16] = x;
  }
}

// Paged append: one warp per (sequence b, KV head), the token at position
// len = seq_lens[b] of sequence b.  Lanes 0-15 quantize the value row into the page
// that holds position len (with a value residual: copy it into residual slot
// len mod G, and the group's G values are quantized row by row at the flush);
// lanes 16-31 copy the key into residual slot len mod G.
// When that slot is the group's last one, the warp quantizes the group at once
// (sequences of a batch fill their groups on different steps): lane l takes channels
// 4l .. 4l+3 of the G keys (slots 0 .. G-2 from the residual, the new key from the
// input), finds their min and max, then packs each token row.  A full sequence
// (len at the block table's capacity) or a page id outside the pool drops the token.
template <int G, int BITS>
__global__ void __launch_bounds__(128) paged_append_kernel(const PagedAppendArgs a) {
  constexpr int WPR = words_per_row<BITS>();
  // a decode launched as a programmatic dependent may start its independent work now
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  const int64_t bh = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (bh >= (int64_t)a.B * a.Hkv) return;
  const int lane = threadIdx.x & 31, lane16 = lane & 15;
  const int b = (int)(bh / a.Hkv), kvh = (int)(bh - (int64_t)b * a.Hkv);
  const int32_t len = a.seq_lens[b];
  if (len < 0 || len >= (a.max_pages << a.shift)) return;
  const int64_t page = a.bt[(int64_t)b * a.max_pages + (len >> a.shift)];
  if (page < 0 || page >= a.num_pages) return;
  const int64_t P = 1 << a.shift;
  const int64_t ph = page * a.Hkv + kvh;
  const int64_t off = len & (P - 1);
  const int r = len % G;
  if (lane < 16) {
    const uint4 x = __ldg(reinterpret_cast<const uint4 *>(a.v_new + bh * kD) + lane16);
    if (a.v_res)
      reinterpret_cast<uint4 *>(a.v_res + (bh * G + r) * kD)[lane16] = x;
    else
      quantize_value_row<BITS>(x, lane16, 0x0000ffffu, a.v_codes + (ph * P + off) * WPR, a.v_meta + ph * P + off);
  } else {
    const uint4 x = __ldg(reinterpret_cast<const uint4 *>(a.k_new + bh * kD) + lane16);
    reinterpret_cast<uint4 *>(a.k_res + (bh * G + r) * kD)[lane16] = x;
  }
  if (r != G - 1) return;
  // ---- flush: the group's G tokens are positions len-G+1 .. len, rows of one page
  const uint16_t *res = a.k_res + bh * G * kD + 4 * lane;  // slots 0 .. G-2 (earlier launches)
  const uint2 last = *reinterpret_cast<const uint2 *>(a.k_new + bh * kD + 4 * lane);
  auto key = [&](int t) -> uint2 { return t == G - 1 ? last : *reinterpret_cast<const uint2 *>(res + t * kD); };
  __half2 mn0 = u2h2(last.x), mx0 = mn0, mn1 = u2h2(last.y), mx1 = mn1;
#pragma unroll 8
  for (int t = 0; t < G - 1; ++t) {
    const uint2 x = key(t);
    mn0 = __hmin2(mn0, u2h2(x.x));
    mx0 = __hmax2(mx0, u2h2(x.x));
    mn1 = __hmin2(mn1, u2h2(x.y));
    mx1 = __hmax2(mx1, u2h2(x.y));
  }
  const QParams p0 = make_qparams<BITS>(__low2float(mn0), __low2float(mx0));
  const QParams p1 = make_qparams<BITS>(__high2float(mn0), __high2float(mx0));
  const QParams p2 = make_qparams<BITS>(__low2float(mn1), __low2float(mx1));
  const QParams p3 = make_qparams<BITS>(__high2float(mn1), __high2float(mx1));
  const float rs0 = BITS == 4 ? __frcp_rn(p0.s) : 0.f, rs1 = BITS == 4 ? __frcp_rn(p1.s) : 0.f;
  const float rs2 = BITS == 4 ? __frcp_rn(p2.s) : 0.f, rs3 = BITS == 4 ? __frcp_rn(p3.s) : 0.f;
  const int64_t row0 = ph * P + off - (G - 1);
  reinterpret_cast<uint4 *>(a.k_meta + (row0 / G) * kD)[lane] = make_uint4(p0.meta, p1.meta, p2.meta, p3.meta);
  // 2-bit: channel 4l + j sits in word l / 4 at bits 8 (l mod 4) + 2j;
  // 4-bit: in word l / 2 at bits 16 (l mod 2) + 4j
  constexpr int LPW = 32 / (4 * BITS);  // lanes per word: 4 or 2
  const int shift = 4 * BITS * (lane & (LPW - 1));
  uint32_t *dst = a.k_codes + row0 * WPR + lane / LPW;
#pragma unroll 8
  for (int t = 0; t < G; ++t) {
    const uint2 x = key(t);
    uint32_t bits = qcode<BITS>(h2f((uint16_t)(x.x & 0xffffu)), p0, rs0) |
                    (qcode<BITS>(h2f((uint16_t)(x.x >> 16)), p1, rs1) << BITS) |
                    (qcode<BITS>(h2f((uint16_t)(x.y & 0xffffu)), p2, rs2) << (2 * BITS)) |
                    (qcode<BITS>(h2f((uint16_t)(x.y >> 16)), p3, rs3) << (3 * BITS));
    bits <<= shift;
    bits |= __shfl_xor_sync(0xffffffffu, bits, 1);
    if constexpr (LPW == 4) bits |= __shfl_xor_sync(0xffffffffu, bits, 2);
    if ((lane & (LPW - 1)) == 0) dst[t * WPR] = bits;
  }
  if (a.v_res) {
    // the group's values, one token row per half-warp (slots 0 .. G-2 from the
    // residual, the new value from the input)
    const int half = lane >> 4;
    const uint32_t half_mask = half ? 0xffff0000u : 0x0000ffffu;
    for (int t = half; t < G; t += 2) {
      const uint16_t *src = (t == G - 1) ? a.v_new + bh * kD : a.v_res + (bh * G + t) * kD;
      const uint4 x = reinterpret_cast<const uint4 *>(src)[lane16];
      quantize_value_row<BITS>(x, lane16, half_mask, a.v_codes + (row0 + t) * WPR, a.v_meta + row0 + t);
    }
  }
}

__global__ void set_len_kernel(int32_t *seq_lens, int32_t seq, int32_t n) { seq_lens[seq] = n; }

__global__ void __launch_bounds__(128) advance_lens_kernel(int32_t *seq_lens, int B, int32_t cap) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < B) {
    const int32_t len = seq_lens[b];
    if (len >= 0) seq_lens[b] = len < cap ? len + 1 : cap;
  }
}

// Residual copy at prefill: tokens nq .. n-1 of every head into slots 0 .. r-1.
__global__ void __launch_bounds__(128) residual_copy_kernel(const uint16_t *__restrict__ k, int64_t n, int64_t nq,
                                                            int G, uint16_t *__restrict__ k_res) {
  const int64_t bh = blockIdx.x;
  const int64_t chunks = (n - nq) * (kD / 8);
  const uint4 *src = reinterpret_cast<const uint4 *>(k + (bh * n + nq) * kD);
  uint4 *dst = reinterpret_cast<uint4 *>(k_res + bh * G * kD);
  for (int64_t i = threadIdx.x; i < chunks; i += blockDim.x) dst[i] = __ldg(src + i);
}

// Dequantize (test aid): thread per (head, token, 8-channel chunk).
template <int BITS>
__global__ void __launch_bounds__(256) dequant_kernel(const uint32_t *__restrict__ k_codes,
                                                      const uint32_t *__restrict__ k_meta,
                                                      const uint16_t *__restrict__ k_res,
                                                      const uint32_t *__restrict__ v_codes,
                                                      const uint32_t *__restrict__ v_meta, int64_t heads, int64_t n,
                                                      int G, int64_t max_tokens, float *__restrict__ k_out,
                                                      float *__restrict__ v_out,
                                                      const uint16_t *__restrict__ v_res, int vg) {
  const int64_t total = heads * n * (kD / 8);
  const int64_t nq = (n / G) * G;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int chunk = (int)(i % (kD / 8));
    const int64_t t = (i / (kD / 8)) % n;
    const int64_t bh = i / ((kD / 8) * n);
    const int c0 = chunk * 8;
    float *ko = k_out + (bh * n + t) * kD + c0;
    float *vo = v_out + (bh * n + t) * kD + c0;
    if (t < nq) {
      // the chunk's 8 codes: BITS * 8 bits starting at bit BITS * c0 of the row
      const uint32_t word = k_codes[(bh * max_tokens + t) * words_per_row<BITS>() + (c0 * BITS) / 32] >>
                            ((c0 * BITS) % 32);
      const uint32_t *meta = k_meta + (bh * (max_tokens / G) + t / G) * kD + c0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float s = h2f((uint16_t)(meta[j] & 0xffffu)), z = h2f((uint16_t)(meta[j] >> 16));
        ko[j] = __fadd_rn(z, __fmul_rn((float)((word >> (BITS * j)) & ((1u << BITS) - 1u)), s));
      }
    } else {
      const uint16_t *res = k_res + (bh * G + (t - nq)) * kD + c0;
#pragma unroll
      for (int j = 0; j < 8; ++j) ko[j] = h2f(res[j]);
    }
    if (v_res && t >= nq) {
      const uint16_t *res = v_res + (bh * G + (t - nq)) * kD + c0;
#pragma unroll
      for (int j = 0; j < 8; ++j) vo[j] = h2f(res[j]);
      continue;
    }
    const uint32_t vm = v_meta[(bh * max_tokens + t) * (kD / vg) + c0 / vg];  // the chunk's value group
    const float s = h2f((uint16_t)(vm & 0xffffu)), z = h2f((uint16_t)(vm >> 16));
    const uint32_t word = v_codes[(bh * max_tokens + t) * words_per_row<BITS>() + (c0 * BITS) / 32] >>
                          ((c0 * BITS) % 32);
#pragma unroll
    for (int j = 0; j < 8; ++j) vo[j] = __fadd_rn(z, __fmul_rn((float)((word >> (BITS * j)) & ((1u << BITS) - 1u)), s));
  }
}

// ------------------------------------------------------------------ host launchers
static int grid_cap(int64_t want) {
  const int64_t cap = 152LL * 32;
  return (int)(want < 1 ? 1 : (want > cap ? cap : want));
}

template <bool PAGED, int BITS>
void key_groups(const uint16_t *in, int64_t in_head_stride, int64_t blocks, int64_t groups_per_head, int64_t g0,
                int G, uint32_t *k_codes, uint32_t *k_meta, int64_t max_tokens, const PageMap &pm, cudaStream_t st) {
  if (G == 32) {  // two groups per CTA
    const int64_t heads = blocks / groups_per_head, pairs = (groups_per_head + 1) / 2;
    key_pairs32_kernel<PAGED, BITS><<<(unsigned)(heads * pairs), 128, 0, st>>>(
        in, in_head_stride, groups_per_head, pairs, g0, k_codes, k_meta, max_tokens, pm);
  } else
    key_group_kernel<64, PAGED, BITS><<<(unsigned)blocks, 128, 0, st>>>(in, in_head_stride, groups_per_head, g0,
                                                                        k_codes, k_meta, max_tokens, pm);
}

cudaError_t launch_key_groups(const uint16_t *in, int64_t in_head_stride, int64_t heads, int64_t groups_per_head,
                              int64_t g0, int G, int bits, uint32_t *k_codes, uint32_t *k_meta, int64_t max_tokens,
                              cudaStream_t st) {
  const int64_t blocks = heads * groups_per_head;
  if (blocks == 0) return cudaSuccess;
  if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;  // one CTA per key group
  const PageMap none = {};
  if (bits == 2)
    key_groups<false, 2>(in, in_head_stride, blocks, groups_per_head, g0, G, k_codes, k_meta, max_tokens, none, st);
  else
    key_groups<false, 4>(in, in_head_stride, blocks, groups_per_head, g0, G, k_codes, k_meta, max_tokens, none, st);
  return cudaGetLastError();
}

cudaError_t launch_key_groups_paged(const uint16_t *in, int64_t in_head_stride, int64_t heads,
                                    int64_t groups_per_head, int G, int bits, const PageMap &pm, uint32_t *k_codes,
                                    uint32_t *k_meta, cudaStream_t st) {
  const int64_t blocks = heads * groups_per_head;
  if (blocks == 0) return cudaSuccess;
  if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;  // one CTA per key group
  if (bits == 2)
    key_groups<true, 2>(in, in_head_stride, blocks, groups_per_head, 0, G, k_codes, k_meta, 0, pm, st);
  else
    key_groups<true, 4>(in, in_head_stride, blocks, groups_per_head, 0, G, k_codes, k_meta, 0, pm, st);
  return cudaGetLastError();
}

cudaError_t launch_value_rows(const uint16_t *v, int64_t heads, int64_t tokens_per_head, int64_t in_rows_per_head,
                              int64_t t0, int bits, uint32_t *v_codes, uint32_t *v_meta, int64_t max_tokens,
                              cudaStream_t st, int vg) {
  const int64_t rows = heads * tokens_per_head;
  if (rows == 0) return cudaSuccess;
  const int grid = grid_cap((rows + 63) / 64);  // 64 rows per CTA and pass
  if (vg == 32)
    value_rows2_kernel<false, 2, 32><<<grid, 256, 0, st>>>(v, rows, tokens_per_head, in_rows_per_head, t0, v_codes,
                                                            v_meta, max_tokens, PageMap{});
  else if (vg == 64)
    value_rows2_kernel<false, 2, 64><<<grid, 256, 0, st>>>(v, rows, tokens_per_head, in_rows_per_head, t0, v_codes,
                                                            v_meta, max_tokens, PageMap{});
  else if (bits == 2)
    value_rows2_kernel<false, 2><<<grid, 256, 0, st>>>(v, rows, tokens_per_head, in_rows_per_head, t0, v_codes,
                                                        v_meta, max_tokens, PageMap{});
  else
    value_rows2_kernel<false, 4><<<grid, 256, 0, st>>>(v, rows, tokens_per_head, in_rows_per_head, t0, v_codes,
                                                        v_meta, max_tokens, PageMap{});
  return cudaGetLastError();
}

cudaError_t launch_value_rows_paged(const uint16_t *v, int64_t heads, int64_t tokens_per_head,
                                    int64_t in_rows_per_head, int bits, const PageMap &pm, uint32_t *v_codes,
                                    uint32_t *v_meta, cudaStream_t st) {
  const int64_t rows = heads * tokens_per_head;
  if (rows == 0) return cudaSuccess;
  const int grid = grid_cap((rows + 63) / 64);  // 64 rows per CTA and pass
  if (bits == 2)
    value_rows2_kernel<true, 2><<<grid, 256, 0, st>>>(v, rows, tokens_per_head, in_rows_per_head, 0, v_codes, v_meta,
                                                       0, pm);
  else
    value_rows2_kernel<true, 4><<<grid, 256, 0, st>>>(v, rows, tokens_per_head, in_rows_per_head, 0, v_codes, v_meta,
                                                       0, pm);
  return cudaGetLastError();
}

cudaError_t launch_append(const uint16_t *k_new, const uint16_t *v_new, int64_t heads, int64_t n, int G, int bits,
                          uint16_t *k_res, uint32_t *v_codes, uint32_t *v_meta, int64_t max_tokens, uint16_t *v_res,
                          cudaStream_t st, int vg) {
  const unsigned grid = (unsigned)((heads + 3) / 4);
  if (bits == 2)
    append_kernel<2><<<grid, 128, 0, st>>>(k_new, v_new, heads, n, G, k_res, v_codes, v_meta, max_tokens, v_res, vg);
  else
    append_kernel<4><<<grid, 128, 0, st>>>(k_new, v_new, heads, n, G, k_res, v_codes, v_meta, max_tokens, v_res, vg);
  return cudaGetLastError();
}

cudaError_t launch_paged_append(const PagedAppendArgs &a, cudaStream_t st) {
  const int64_t heads = (int64_t)a.B * a.Hkv;
  const unsigned blocks = (unsigned)((heads + 3) / 4);
  if (a.G == 32)
    (a.bits == 2 ? paged_append_kernel<32, 2> : paged_append_kernel<32, 4>)<<<blocks, 128, 0, st>>>(a);
  else
    (a.bits == 2 ? paged_append_kernel<64, 2> : paged_append_kernel<64, 4>)<<<blocks, 128, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_set_len(int32_t *seq_lens, int32_t seq, int32_t n, cudaStream_t st) {
  set_len_kernel<<<1, 1, 0, st>>>(seq_lens, seq, n);
  return cudaGetLastError();
}

cudaError_t launch_advance_lens(int32_t *seq_lens, int B, int32_t cap, cudaStream_t st) {
  advance_lens_kernel<<<(unsigned)((B + 127) / 128), 128, 0, st>>>(seq_lens, B, cap);
  return cudaGetLastError();
}

cudaError_t launch_residual_copy(const uint16_t *k, int64_t heads, int64_t n, int64_t nq, int G, uint16_t *k_res,
                                 cudaStream_t st) {
  if (n == nq) return cudaSuccess;
  residual_copy_kernel<<<(unsigned)heads, 128, 0, st>>>(k, n, nq, G, k_res);
  return cudaGetLastError();
}

cudaError_t launch_dequant(const uint32_t *k_codes, const uint32_t *k_meta, const uint16_t *k_res,
                           const uint32_t *v_codes, const uint32_t *v_meta, const uint16_t *v_res, int64_t heads,
                           int64_t n, int G, int bits, int64_t max_tokens, float *k_out, float *v_out,
                           cudaStream_t st, int vg) {
  const int64_t total = heads * n * (kD / 8);
  if (total == 0) return cudaSuccess;
  const int grid = grid_cap((total + 255) / 256);
  if (bits == 2)
    dequant_kernel<2><<<grid, 256, 0, st>>>(k_codes, k_meta, k_res, v_codes, v_meta, heads, n, G, max_tokens, k_out,
                                            v_out, v_res, vg);
  else
    dequant_kernel<4><<<grid, 256, 0, st>>>(k_codes, k_meta, k_res, v_codes, v_meta, heads, n, G, max_tokens, k_out,
                                            v_out, v_res, vg);
  return cudaGetLastError();
}

}  // namespace kivi
