// kivi_decode.cu -- fused decode attention over the 2-bit KIVI cache (sm_103a).
//
// KIVI page ("Makale Bulteni -- KIVI", cmlonder.com radar / paper-to-prod,
// 2026-11-01), section "Iddia ve Gerceklik": the attention output is a weighted sum
// of per-token-quantized values (paragraph 2); keys are per-channel quantized in
// G-token groups plus an fp16 residual, and the 2-bit codes are unpacked with shifts
// and masks for 16-bit tensor cores (paragraph 3).
//
// For one (batch, KV head) and the R = Hq/Hkv query heads that read it:
//   score_t = sigma * sum_c q_c (code_tc s_gc + z_gc) = sigma * (sum_c qs_gc code_tc + beta_g)
//       with qs_g = q (.) s_g and beta_g = q . z_g, once per key group g;
//   out_c   = sum_t p_t (code_tc s_t + z_t) = sum_t (p_t s_t) code_tc + sum_t p_t z_t.
// Both contractions run on the tensor cores (mma.sync m16n8k16, fp32 accumulate):
//   * the codes enter as fp16 subnormals (exact, see unpack16);
//   * the fp32 factors qs and p*s enter as an fp16 pair hi + lo (hi = fp16(x),
//     lo = fp16(x - hi)), one per MMA column, which keeps ~22 significant bits;
//     qs is first scaled by a power of two chosen per group so that its largest
//     entry sits just below 2^14 (no fp16 overflow, full precision for any range).
// Tokens are tiled by 16 (the MMA M dimension for q.K, the K dimension for P.V).
// The 4 column pairs of an MMA carry (tile slot, query head): a softmax step covers
// T = 4/R tiles at once, so that for every R each lane owns the scores of one
// (tile, head) pair: lane (g, tig) holds tokens g and g+8 of tile slot tig/R for
// head tig%R.  For q.K the per-head factors are replicated over the slots and each
// tile accumulates separately; for P.V each tile's weights sit in its own column
// pairs and all tiles accumulate together (the slots are summed at the end).
//
// Work decomposition (persistent, balanced): a "unit" is 64 tokens of one (batch, KV
// head) -- one or two key groups -- plus one unit for the fp16 residual keys when
// n mod G > 0.  The grid holds exactly as many warps as fit on the GPU at once; warp
// w takes the contiguous unit range [w*W/NW, (w+1)*W/NW), staging each unit (codes,
// scales, zeros) in its shared memory with cp.async two units ahead, and runs an
// online softmax over it.  At every head boundary the warp writes a partial (max,
// sum, unnormalised output) to the workspace; the combine kernel merges a head's
// partials (flash-decoding) and is launched as a programmatic dependent.
#include <math.h>

#include <type_traits>

#include "kivi_device.cuh"
#include "kivi_internal.h"

// Resident CTAs per SM the register allocation is sized for (3: up to 168 registers).
#ifndef KIVI_DECODE_MIN_CTAS
#define KIVI_DECODE_MIN_CTAS 3
#endif

namespace kivi {

namespace {

constexpr int kWarps = kDecodeWarps;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 3;
// Units staged ahead of the one being computed (at most kStages - 1).
#ifndef KIVI_DECODE_AHEAD
#define KIVI_DECODE_AHEAD 2
#endif
constexpr int kAhead = KIVI_DECODE_AHEAD;
static_assert(kAhead >= 1 && kAhead < kStages, "the ring must hold the computed unit and the staged ones");
constexpr int kUnit = kDecodeUnit;                   // tokens per unit
constexpr int kFragRowWords = 20;                    // 16 B-fragment words + 4 pad (bank spread)
constexpr float kLog2e = 1.4426950408889634f;

// Shared-memory layout of one warp's ring for BITS-bit codes.  4-bit rows are twice
// as long, so their ring has two stages (one unit staged ahead) to keep two CTAs
// per SM; 2-bit rows keep three.
template <int R, int G, int BITS = 2>
struct Layout {
  static constexpr int kRowBytes = 16 * BITS;                 // packed codes of one token row
  static constexpr int kRowChunks = kRowBytes / 16;           // 16-byte copies per row
  static constexpr int kStages = BITS == 2 ? 3 : 2;
  static constexpr int kAheadUnits = BITS == 2 ? kAhead : 1;  // units staged ahead of the computed one
  static constexpr int kGroups = kUnit / G;                   // key groups per unit
  static constexpr int kKCodes = 0;                           // 64 rows
  static constexpr int kVCodes = kUnit * kRowBytes;           // 64 rows
  static constexpr int kVMeta = 2 * kUnit * kRowBytes;        // 64 x 4 B
  static constexpr int kKMeta = kVMeta + kUnit * 4;           // kGroups x 128 x 4 B
  static constexpr int kStageBytes = kKMeta + kGroups * kD * 4;
  static constexpr int kFragGroupBytes = 8 * R * kFragRowWords * 4;  // rows 4*(2h+p)+tig
  static constexpr int kWarpBytes = kStages * kStageBytes + kGroups * kFragGroupBytes;
  static constexpr int kSmem = kWarps * kWarpBytes;
  static_assert(kAheadUnits >= 1 && kAheadUnits < kStages, "the ring holds the computed unit and the staged ones");
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float pow2i(int e) { return __int_as_float((e + 127) << 23); }  // e in [-126, 127]

__device__ __forceinline__ uint2 lds64(const unsigned char *p) { return *reinterpret_cast<const uint2 *>(p); }
__device__ __forceinline__ uint32_t lds32(const unsigned char *p) { return *reinterpret_cast<const uint32_t *>(p); }

__device__ __forceinline__ void load_frag(const unsigned char *row, uint32_t bf[16]) {
  const uint4 *p = reinterpret_cast<const uint4 *>(row);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint4 u = p[k];
    bf[4 * k] = u.x;
    bf[4 * k + 1] = u.y;
    bf[4 * k + 2] = u.z;
    bf[4 * k + 3] = u.w;
  }
}

// q.K of one 16-token tile: A from the unpacked codes (or fp16 keys) of token g
// (ra*) and g+8 (rb*), words 2tig (..0) and 2tig+1 (..1); accumulates into sc.
__device__ __forceinline__ void qk_tile(const uint32_t ra0[8], const uint32_t ra1[8], const uint32_t rb0[8],
                                        const uint32_t rb1[8], const uint32_t bf[16], float sc[4]) {
  float s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    mma16816(sc, ra0[2 * j], rb0[2 * j], ra0[2 * j + 1], rb0[2 * j + 1], bf[2 * j], bf[2 * j + 1]);
    mma16816(s1, ra1[2 * j], rb1[2 * j], ra1[2 * j + 1], rb1[2 * j + 1], bf[8 + 2 * j], bf[8 + 2 * j + 1]);
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) sc[k] += s1[k];
}

// P.V of one 16-token tile: A = value codes of word g of tokens tig, tig+4, tig+8,
// tig+12 (v[0..3]), B = (bw0, bw1).
__device__ __forceinline__ void pv_tile(float acc[8][4], const uint32_t v[4], uint32_t bw0, uint32_t bw1) {
  uint32_t x01[8], y01[8], x23[8], y23[8];
  unpack16(prmt(v[0], v[1], 0x5410u), x01);
  unpack16(prmt(v[0], v[1], 0x7632u), y01);
  unpack16(prmt(v[2], v[3], 0x5410u), x23);
  unpack16(prmt(v[2], v[3], 0x7632u), y23);
#pragma unroll
  for (int j = 0; j < 8; ++j) mma16816(acc[j], x01[j], y01[j], x23[j], y23[j], bw0, bw1);
}

// P.V of one 16-token tile from 4-bit value codes: v[k] = words 2g and 2g+1 of
// token tig + 4k (channels 16g .. 16g+15).  One prmt pairs two tokens' halves of a
// word, unpack8 splits them into channel registers; MMA j takes channel 16g + j
// (row g) and 16g + 8 + j (row g+8), with code factor 16^(j mod 2).
__device__ __forceinline__ void pv_tile4(float acc[8][4], const uint2 v[4], uint32_t bw0, uint32_t bw1) {
  uint32_t a01[2][8], a23[2][8];  // [word 2g + p][channel within the word], tokens (tig, tig+4) / (tig+8, tig+12)
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    const uint32_t w0 = p ? v[0].y : v[0].x, w1 = p ? v[1].y : v[1].x;
    const uint32_t w2 = p ? v[2].y : v[2].x, w3 = p ? v[3].y : v[3].x;
    unpack8(prmt(w0, w1, 0x5410u), a01[p]);
    unpack8(prmt(w0, w1, 0x7632u), a01[p] + 4);
    unpack8(prmt(w2, w3, 0x5410u), a23[p]);
    unpack8(prmt(w2, w3, 0x7632u), a23[p] + 4);
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) mma16816(acc[j], a01[0][j], a01[1][j], a23[0][j], a23[1][j], bw0, bw1);
}

// 32 fp16 keys (channels 32tig .. 32tig+31) of one residual token, paired (m, m+8)
// like the unpacked codes.
__device__ __forceinline__ void residual_pairs(const uint16_t *row, bool valid, int tig, uint32_t r0[8],
                                               uint32_t r1[8]) {
  uint32_t p[16];
  if (valid) {
    const uint4 *src = reinterpret_cast<const uint4 *>(row + 32 * tig);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint4 uu = __ldg(src + k);
      p[4 * k] = uu.x;
      p[4 * k + 1] = uu.y;
      p[4 * k + 2] = uu.z;
      p[4 * k + 3] = uu.w;
    }
  } else {
#pragma unroll
    for (int k = 0; k < 16; ++k) p[k] = 0u;
  }
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    const uint32_t sel = (m & 1) ? 0x7632u : 0x5410u;
    r0[m] = prmt(p[m >> 1], p[(m >> 1) + 4], sel);
    r1[m] = prmt(p[8 + (m >> 1)], p[8 + (m >> 1) + 4], sel);
  }
}

// Index of the first warp whose unit range contains unit u.
__device__ __forceinline__ int64_t owner_warp(int64_t u, int64_t W, int64_t NW) { return ((u + 1) * NW - 1) / W; }

// Per-lane constants of the fragment bookkeeping.
struct LaneInfo {
  int g, tig, slot_mine, pv_slot, src_a, src_b;
  uint32_t pv_sel;
};

// Softmax state of the q.K side: running max (log2 domain, per head) and this
// lane's shares of sum_t p_t and sum_t p_t z_t.
struct SoftState {
  float m, l, zs;
};

// Max over the lanes that share this lane's query head.
template <int R>
__device__ __forceinline__ float head_max(float x) {
  if constexpr (R == 1) {
    // one head per warp: an order-preserving integer key and one warp reduction
    const int k = __float_as_int(x);
    const int key = k ^ ((k >> 31) & 0x7fffffff);
    const int mk = __reduce_max_sync(0xffffffffu, key);
    return __int_as_float(mk ^ ((mk >> 31) & 0x7fffffff));
  } else {
#pragma unroll
    for (int off = R; off < 32; off <<= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, off));
    return x;
  }
}

// q.K side of one softmax step over T = 4/R tiles of 16 tokens.
//   kfill(i, sc)  accumulates tile slot i's q.K MMA into sc[4];
//   cq, beta      this lane's score scale and offset (log2 domain);
//   n_valid       tokens of the step that exist (FULL: all 16*T);
//   vmeta(tok)    {s, z} of step token tok.
// Returns the P.V B operand of this lane (bw0, bw1) and the rescale factor alpha
// that the P.V accumulators need before this step's contribution is added.
template <int R, bool FULL, class KF, class VM>
__device__ __forceinline__ void qk_step(SoftState &st, const LaneInfo &li, KF &&kfill, float cq, float beta,
                                        int n_valid, VM &&vmeta, uint32_t &bw0, uint32_t &bw1, float &alpha) {
  constexpr int T = 4 / R;
  float S[T][4];
#pragma unroll
  for (int i = 0; i < T; ++i) {
#pragma unroll
    for (int k = 0; k < 4; ++k) S[i][k] = 0.f;
    if (FULL || 16 * i < n_valid) kfill(i, S[i]);
  }
  float d[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) d[k] = S[0][k];
#pragma unroll
  for (int i = 1; i < T; ++i)
#pragma unroll
    for (int k = 0; k < 4; ++k) d[k] = (li.slot_mine == i) ? S[i][k] : d[k];
  const int ta = 16 * li.slot_mine + li.g, tb = ta + 8;  // this lane's tokens in the step
  const bool va = FULL || ta < n_valid, vb = FULL || tb < n_valid;
  const float sa = va ? fmaf(cq, d[0] + d[1], beta) : -INFINITY;
  const float sb = vb ? fmaf(cq, d[2] + d[3], beta) : -INFINITY;
  const float m_new = fmaxf(st.m, head_max<R>(fmaxf(sa, sb)));
  alpha = ex2(st.m - m_new);  // st.m = -inf at the start of a head: alpha = 0
  st.m = m_new;
  const uint32_t vma = vmeta(va ? ta : 0), vmb = vmeta(vb ? tb : 0);
  const float pa = va ? ex2(sa - m_new) : 0.f;
  const float pb = vb ? ex2(sb - m_new) : 0.f;
  const float2 fa = __half22float2(u2h2(vma)), fb = __half22float2(u2h2(vmb));  // {s, z}
  const float sva = va ? fa.x : 0.f, zva = va ? fa.y : 0.f;
  const float svb = vb ? fb.x : 0.f, zvb = vb ? fb.y : 0.f;
  st.l = fmaf(st.l, alpha, pa + pb);
  st.zs = fmaf(st.zs, alpha, fmaf(pa, zva, pb * zvb));
  const float wa = pa * sva, wb = pb * svb;
  // hi/lo split of the two weights: q1 = {hi_a, lo_a}, q2 = {hi_b, lo_b}
  const __half2 hab = __floats2half2_rn(wa, wb);
  const float2 fab = __half22float2(hab);
  const __half2 lab = __floats2half2_rn(wa - fab.x, wb - fab.y);
  const uint32_t q1 = prmt(h22u(hab), h22u(lab), 0x5410u);
  const uint32_t q2 = prmt(h22u(hab), h22u(lab), 0x7632u);
  // B of P.V for tile slot pv_slot, column g = (slot, head, part): K slots
  // 2tig, 2tig+1, 2tig+8, 2tig+9 hold tokens tig, tig+4, tig+8, tig+12; token u's
  // weight lives in lane 4*(u%8) + (g>>1) (first token if u < 8, else second)
  const uint32_t a1 = __shfl_sync(0xffffffffu, q1, li.src_a);
  const uint32_t b1 = __shfl_sync(0xffffffffu, q1, li.src_b);
  const uint32_t a2 = __shfl_sync(0xffffffffu, q2, li.src_a);
  const uint32_t b2 = __shfl_sync(0xffffffffu, q2, li.src_b);
  bw0 = prmt(a1, b1, li.pv_sel);
  bw1 = prmt(a2, b2, li.pv_sel);
}

// P.V side of one step: rescale the accumulators, then add the T tiles.
//   vword(i, k)   word g of the value row of token tig + 4k of tile slot i.
template <int R, int BITS, class VW>
__device__ __forceinline__ void pv_step(float acc[8][4], const LaneInfo &li, int n_valid, uint32_t bw0, uint32_t bw1,
                                        float alpha, VW &&vword) {
  constexpr int T = 4 / R;
  if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[j][k] *= alpha;
  }
#pragma unroll
  for (int i = 0; i < T; ++i) {
    if (16 * i < n_valid) {
      const bool mine = li.pv_slot == i;
      if constexpr (BITS == 2) {
        uint32_t v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) v[k] = vword(i, k);
        pv_tile(acc, v, mine ? bw0 : 0u, mine ? bw1 : 0u);
      } else {
        uint2 v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) v[k] = vword(i, k);
        pv_tile4(acc, v, mine ? bw0 : 0u, mine ? bw1 : 0u);
      }
    }
  }
}

// Position of a warp's cursor: head h = b * Hkv + kvh, unit uu of the head, and the
// head's geometry (units U, full key groups NG, residual keys r, code units ncu).
// Dense caches share one geometry; paged ones take it from the sequence's length.
struct Cursor {
  int64_t h;
  int b, kvh, uu;
  int U, NG, r, ncu;
};

template <int G>
__device__ __forceinline__ void set_geometry(Cursor &c, int64_t len) {
  constexpr int NGU = kUnit / G;
  c.NG = (int)(len / G);
  c.r = (int)(len - (int64_t)c.NG * G);
  c.ncu = (c.NG + NGU - 1) / NGU;
  c.U = c.ncu + (c.r > 0 ? 1 : 0);
}

// Paged layout: per-sequence lengths (clamped to the block table's capacity) and the
// exclusive prefix sum of the sequences' unit counts, in shared memory.  All threads
// of the CTA take part; B <= 4 * kThreads.
template <int G>
__device__ void paged_prefix(const DecodeArgs &a, int *s_len, int *s_cum) {
  constexpr int NGU = kUnit / G;
  int *s_tot = s_cum + a.B + 1;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  int u[4], loc = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int b = 4 * t + j;
    u[j] = 0;
    if (b < a.B) {
      int len = a.seq_lens[b] + a.len_offset;
      len = len < 0 ? 0 : (len > a.cap_tokens ? a.cap_tokens : len);
      s_len[b] = len;
      const int ng = len / G;
      u[j] = (ng + NGU - 1) / NGU + (len - ng * G > 0 ? 1 : 0);
    }
    loc += u[j];
  }
  int inc = loc;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, inc, off);
    if (lane >= off) inc += y;
  }
  if (lane == 31) s_tot[warp] = inc;
  __syncthreads();
  int ex = inc - loc;
  for (int w = 0; w < warp; ++w) ex += s_tot[w];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int b = 4 * t + j;
    if (b < a.B) s_cum[b] = ex;
    ex += u[j];
  }
  if (t == kThreads - 1) s_cum[a.B] = ex;  // the total
  __syncthreads();
}

// P.V of one step over fp16 values (the value residual): the same tile and column
// layout as pv_step, with A built from the values of tokens tig, tig+4, tig+8,
// tig+12 of each tile (channels 16g + j and 16g + 8 + j for MMA j) instead of
// unpacked codes.  `rows` points at the step's first token row; tokens at or beyond
// n_valid read as zero.  The accumulators must hold output units (no code factors).
template <int R>
__device__ __forceinline__ void pv_step_f16(float acc[8][4], const LaneInfo &li, int n_valid, uint32_t bw0,
                                            uint32_t bw1, float alpha, const uint16_t *rows) {
  constexpr int T = 4 / R;
  if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[j][k] *= alpha;
  }
#pragma unroll
  for (int i = 0; i < T; ++i) {
    if (16 * i < n_valid) {
      uint32_t w[4][8];  // token tig + 4k: channels 16g .. 16g+15 as 8 half2 words
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int tok = 16 * i + li.tig + 4 * k;
        uint4 lo = make_uint4(0u, 0u, 0u, 0u), hi = lo;
        if (tok < n_valid) {
          const uint4 *src = reinterpret_cast<const uint4 *>(rows + tok * kD + 16 * li.g);
          lo = __ldg(src);
          hi = __ldg(src + 1);
        }
        w[k][0] = lo.x; w[k][1] = lo.y; w[k][2] = lo.z; w[k][3] = lo.w;
        w[k][4] = hi.x; w[k][5] = hi.y; w[k][6] = hi.z; w[k][7] = hi.w;
      }
      const bool mine = li.pv_slot == i;
      const uint32_t b0 = mine ? bw0 : 0u, b1 = mine ? bw1 : 0u;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t sel = (j & 1) ? 0x7632u : 0x5410u;
        const int x = j >> 1, y = 4 + (j >> 1);  // words of channels 16g + j and 16g + 8 + j
        mma16816(acc[j], prmt(w[0][x], w[1][x], sel), prmt(w[0][y], w[1][y], sel), prmt(w[2][x], w[3][x], sel),
                 prmt(w[2][y], w[3][y], sel), b0, b1);
      }
    }
  }
}

template <int R, int G, bool PAGED, int BITS>
__global__ void __launch_bounds__(kThreads, KIVI_DECODE_MIN_CTAS) decode_kernel(const DecodeArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  using L = Layout<R, G, BITS>;
  constexpr int WPR = words_per_row<BITS>();
  constexpr int kStages = L::kStages;
  constexpr int kAhead = L::kAheadUnits;
  constexpr int T = 4 / R;           // tile slots per softmax step
  constexpr int TPG = G / 16;        // tiles per key group
  constexpr int NGU = L::kGroups;    // key groups per unit
  // the combine grid may launch now; it waits for this grid's completion
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t gw = (int64_t)blockIdx.x * kWarps + warp;
  int64_t NW = a.n_warps;
  int64_t W;
  int *s_len = nullptr, *s_cum = nullptr;
  int2 *hdr = nullptr;
  float *part = a.ws;
  const int P = 1 << a.page_shift;
  if constexpr (PAGED) {
    s_len = reinterpret_cast<int *>(smem + L::kSmem);
    s_cum = s_len + a.B;
    paged_prefix<G>(a, s_len, s_cum);
    W = (int64_t)a.Hkv * s_cum[a.B];
    hdr = reinterpret_cast<int2 *>(a.ws);
    part = a.ws + 2 * (int64_t)a.B * a.Hkv;
    // sequences without tokens get an empty header (their output is zero)
    if (blockIdx.x == 0)
      for (int b = threadIdx.x; b < a.B; b += kThreads)
        if (s_cum[b + 1] == s_cum[b])
          for (int kvh = 0; kvh < a.Hkv; ++kvh) hdr[(int64_t)b * a.Hkv + kvh] = make_int2(0, 0);
    // fewer units than warps: use one warp per unit, so that no warp between a
    // head's first and last owner is left without units (every partial is written)
    if (W < NW) NW = W;
  } else {
    W = a.total_units;
  }
  if (gw >= NW) return;
  const int64_t u0 = gw * W / NW, u1 = (gw + 1) * W / NW;
  if (u0 >= u1) return;
  const int n_my = (int)(u1 - u0);

  unsigned char *wbase = smem + warp * L::kWarpBytes;
  unsigned char *frag = wbase + kStages * L::kStageBytes;
  const float c0 = a.softmax_scale * kLog2e;

  LaneInfo li;
  li.g = lane >> 2;
  li.tig = lane & 3;
  li.slot_mine = li.tig / R;
  li.pv_slot = (li.g >> 1) / R;
  li.src_a = 4 * li.tig + (li.g >> 1);
  li.src_b = li.src_a + 16;
  li.pv_sel = (li.g & 1) ? 0x7632u : 0x5410u;
  const int g = li.g, tig = li.tig;
  const int head_mine = tig % R;
  const int frag_row = 4 * (2 * ((g >> 1) % R) + (g & 1)) + tig;
  // prep: channel c = lane + 32k lands in row 4*(2h+p) + k, half-word wh of the row
  // (the same position for the channels lane + 32k of every k: the row differs).
  // wh_pairs is the order of the fp16 residual keys (residual_pairs), which is also
  // the order of the unpacked 2-bit codes: B half-word 2i + d of lane tig holds
  // channel 32tig + 16(i >= 8) + (i mod 8) + 8d.
  int wh_pairs;
  {
    const int i = lane & 15, i8 = i & 7;
    const int j = 4 * (lane >> 4) + (i8 >> 1);
    wh_pairs = (2 * j + (i8 & 1)) * 2 + (i >= 8 ? 1 : 0);
  }
  int wh;
  float mult;
  if constexpr (BITS == 2) {
    wh = wh_pairs;
    // codes of channel index i (mod 16) are unpacked with factor 4^(i mod 4);
    // 4^(3 - i mod 4) brings every q.K product to code * qs * 64
    mult = (float)(64 >> (2 * (lane & 3)));
  } else {
    // B half-word 2i + d holds channel 32tig + 16(i >= 8) + 8q + t + 4d, i = 8(i >= 8) + 4q + t
    const int t = lane & 3, d = (lane >> 2) & 1, q = (lane >> 3) & 1, s16 = lane >> 4;
    wh = 2 * (8 * s16 + 4 * q + t) + d;
    // channel position t is unpacked with factor 16^(t mod 2); 16^(1 - t mod 2) brings
    // every q.K product to code * qs * 16
    mult = (t & 1) ? 1.f : 16.f;
  }

  // ---- cursors: ic stages unit u0 + kk (one ahead), cc computes it
  Cursor ic;
  if constexpr (PAGED) {
    // the sequence holding unit u0: the last b with Hkv * cum[b] <= u0 (it has units)
    int lo = 0, hi = a.B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if ((int64_t)a.Hkv * s_cum[mid] <= u0) lo = mid; else hi = mid - 1;
    }
    ic.b = lo;
    set_geometry<G>(ic, s_len[lo]);
    const int64_t rel = u0 - (int64_t)a.Hkv * s_cum[lo];
    ic.kvh = (int)(rel / ic.U);
    ic.uu = (int)(rel - (int64_t)ic.kvh * ic.U);
    ic.h = (int64_t)ic.b * a.Hkv + ic.kvh;
  } else {
    set_geometry<G>(ic, a.n);
    ic.h = u0 / ic.U;
    ic.uu = (int)(u0 - ic.h * ic.U);
    ic.b = ic.kvh = 0;
  }
  Cursor cc = ic;
  auto advance = [&](Cursor &c) {
    if (++c.uu == c.U) {
      c.uu = 0;
      if constexpr (PAGED) {
        if (++c.kvh == a.Hkv) {
          c.kvh = 0;
          do {
            ++c.b;
          } while (c.b < a.B && s_cum[c.b + 1] == s_cum[c.b]);
          if (c.b < a.B) set_geometry<G>(c, s_len[c.b]);
        }
        c.h = (int64_t)c.b * a.Hkv + c.kvh;
      } else {
        ++c.h;
      }
    }
  };
  // page of token tok of sequence b (ids outside the pool are clamped into it: the
  // caller's block table is trusted for values, never for addresses)
  auto page_of = [&](int b, int tok) -> int64_t {
    int64_t pg = __ldg(a.block_table + (int64_t)b * a.max_pages + (tok >> a.page_shift));
    return pg < 0 ? 0 : (pg >= a.num_pages ? a.num_pages - 1 : pg);
  };
  int64_t pg_next = 0;  // page of ic's unit, loaded one unit ahead of its use
  if constexpr (PAGED) {
    if (ic.uu < ic.ncu) pg_next = page_of(ic.b, ic.uu * kUnit);
  }

  bool waited = false;
  auto issue = [&](int kk) {
    // the last unit of a head holds the token a preceding append just wrote: when
    // this grid was launched as a programmatic dependent of that append, wait for it
    if (a.wait_tail && !waited && kk < n_my && ic.uu == ic.U - 1) {
      asm volatile("griddepcontrol.wait;\n" ::: "memory");
      waited = true;
    }
    if (kk < n_my && ic.uu < ic.ncu) {
      const int g0 = ic.uu * NGU;
      const int ngr = min(NGU, ic.NG - g0);  // 1 or 2 groups (G = 32)
      const int rows = ngr * G;
      unsigned char *stg = wbase + (kk % kStages) * L::kStageBytes;
      int64_t row0, grp0;
      if constexpr (PAGED) {
        const int64_t ph = pg_next * a.Hkv + ic.kvh;
        const int off = (g0 * G) & (P - 1);
        row0 = ph * P + off;
        grp0 = ph * (P / G) + off / G;
      } else {
        row0 = ic.h * a.max_tokens + (int64_t)g0 * G;
        grp0 = ic.h * (a.max_tokens / G) + g0;
      }
      const unsigned char *kc = reinterpret_cast<const unsigned char *>(a.k_codes + row0 * WPR);
      const unsigned char *vc = reinterpret_cast<const unsigned char *>(a.v_codes + row0 * WPR);
      const unsigned char *vm = reinterpret_cast<const unsigned char *>(a.v_meta + row0);
      const unsigned char *km = reinterpret_cast<const unsigned char *>(a.k_meta + grp0 * kD);
      if (rows == kUnit) {
#pragma unroll
        for (int c = lane; c < kUnit * L::kRowChunks; c += 32) {
          cp_async16(stg + L::kKCodes + c * 16, kc + c * 16);
          cp_async16(stg + L::kVCodes + c * 16, vc + c * 16);
        }
        if (lane < kUnit / 4) cp_async16(stg + L::kVMeta + lane * 16, vm + lane * 16);
#pragma unroll
        for (int c = lane; c < NGU * 32; c += 32) cp_async16(stg + L::kKMeta + c * 16, km + c * 16);
      } else {
        for (int c = lane; c < rows * L::kRowChunks; c += 32) {
          cp_async16(stg + L::kKCodes + c * 16, kc + c * 16);
          cp_async16(stg + L::kVCodes + c * 16, vc + c * 16);
        }
        if (lane < rows / 4) cp_async16(stg + L::kVMeta + lane * 16, vm + lane * 16);
        for (int c = lane; c < ngr * 32; c += 32) cp_async16(stg + L::kKMeta + c * 16, km + c * 16);
      }
    }
    cp_async_commit();
    advance(ic);
    if constexpr (PAGED) {
      if (kk + 1 < n_my && ic.uu < ic.ncu) pg_next = page_of(ic.b, ic.uu * kUnit);
    }
  };

  SoftState ss = {-INFINITY, 0.f, 0.f};
  float acc[8][4];
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[j][k] = 0.f;
  float qv[R][4];

  // Write the partial of head h (this warp's share of it) from the P.V accumulators
  // and the softmax state (m, l, zs) that belongs to them.  acc_true: the
  // accumulators already hold output units (a value residual was added to them).
  bool acc_true = false;
  auto emit = [&](int64_t h, const SoftState &fin) {
    float l = fin.l, zs = fin.zs;
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l += __shfl_xor_sync(0xffffffffu, l, off);
      zs += __shfl_xor_sync(0xffffffffu, zs, off);
    }
    float o[16];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      o[j] = acc[j][0] + acc[j][1];
      o[8 + j] = acc[j][2] + acc[j][3];
    }
    // sum the tile slots of the same head (tig bits above the head bits)
#pragma unroll
    for (int off = R; off < 4; off <<= 1) {
      l += __shfl_xor_sync(0xffffffffu, l, off);
      zs += __shfl_xor_sync(0xffffffffu, zs, off);
#pragma unroll
      for (int j = 0; j < 16; ++j) o[j] += __shfl_xor_sync(0xffffffffu, o[j], off);
    }
    if (li.slot_mine == 0) {
      float *dst;
      if constexpr (PAGED) {
        // pair index gw + h grows strictly along the unit order: unique per (warp, head)
        dst = part + ((gw + h) * R + head_mine) * (kD + 2);
      } else {
        const int64_t b = h / a.Hkv, kvh = h - b * a.Hkv;
        const int64_t slot = gw - owner_warp(h * a.units_per_head, W, NW);
        dst = a.ws + ((b * a.Hq + kvh * R + head_mine) * a.pmax + slot) * (kD + 2);
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        // undo the code factor 4^(j mod 4) and the 2^-24 of the subnormal codes
        const float un = acc_true ? 1.f : pow2i(BITS == 2 ? 24 - 2 * (j & 3) : 24 - 4 * (j & 1));
        dst[16 * g + j] = fmaf(o[j], un, zs);
        dst[16 * g + 8 + j] = fmaf(o[8 + j], un, zs);
      }
      if (g == 0) {
        dst[kD] = fin.m;
        dst[kD + 1] = l;
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[j][k] = 0.f;
    acc_true = false;
  };
  auto load_q = [&](const Cursor &c) {
    int64_t b, kvh;
    if constexpr (PAGED) {
      b = c.b;
      kvh = c.kvh;
    } else {
      b = c.h / a.Hkv;
      kvh = c.h - b * a.Hkv;
    }
    const uint16_t *qh = a.q + (b * a.Hq + kvh * R) * kD + lane;
#pragma unroll
    for (int hh = 0; hh < R; ++hh)
#pragma unroll
      for (int k = 0; k < 4; ++k) qv[hh][k] = h2f(qh[hh * kD + 32 * k]);
  };

  load_q(cc);
#pragma unroll
  for (int kk = 0; kk < kAhead; ++kk) issue(kk);

  for (int kk = 0; kk < n_my; ++kk) {
    issue(kk + kAhead);
    if constexpr (PAGED) {
      // the warp that takes a head's first unit publishes where its partials go
      if (cc.uu == 0 && lane == 0) {
        const int64_t start = (int64_t)a.Hkv * s_cum[cc.b] + (int64_t)cc.kvh * cc.U;
        const int64_t last = owner_warp(start + cc.U - 1, W, NW);
        hdr[cc.h] = make_int2((int)(gw + cc.h), (int)(last - gw + 1));
      }
    }
    cp_async_wait<kAhead>();
    __syncwarp();
    const int stage = kk % kStages;
    uint32_t nw0[R], nw1[R];
    float nalpha[R];
#pragma unroll
    for (int j = 0; j < R; ++j) {
      nw0[j] = nw1[j] = 0u;
      nalpha[j] = 1.f;
    }
    int n_kind, n_ntok;
    int64_t n_res_row = 0;

    if (cc.uu < cc.ncu) {
      const unsigned char *stg = wbase + stage * L::kStageBytes;
      const int ngr = min(NGU, cc.NG - cc.uu * NGU);
      // ---- per group: qs = q * s scaled by 2^E * mult, split hi/lo into the
      //      group's B fragment; this lane's score scale and beta = q . z
      float cq_g[NGU], beta_g[NGU];
#pragma unroll
      for (int gi = 0; gi < NGU; ++gi) {
        cq_g[gi] = 0.f;
        beta_g[gi] = 0.f;
        if (gi < ngr) {
          uint16_t *fb = reinterpret_cast<uint16_t *>(frag + gi * L::kFragGroupBytes);
          float x[R][4], beta[R];
#pragma unroll
          for (int hh = 0; hh < R; ++hh) beta[hh] = 0.f;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t mt = lds32(stg + L::kKMeta + (gi * kD + lane + 32 * k) * 4);
            const float2 sz = __half22float2(u2h2(mt));
#pragma unroll
            for (int hh = 0; hh < R; ++hh) {
              x[hh][k] = qv[hh][k] * sz.x;
              beta[hh] = fmaf(qv[hh][k], sz.y, beta[hh]);
            }
          }
#pragma unroll
          for (int hh = 0; hh < R; ++hh) {
            const float mabs =
                fmaxf(fmaxf(fabsf(x[hh][0]), fabsf(x[hh][1])), fmaxf(fabsf(x[hh][2]), fabsf(x[hh][3])));
            const uint32_t mbits = __reduce_max_sync(0xffffffffu, __float_as_uint(mabs));
            // largest |qs| in [2^e, 2^(e+1)): scale by 2^E, E = 7 - e, so |B| < 2^14
            const int E = min(100, max(-100, 134 - (int)(mbits >> 23)));
            const float sc = pow2i(E) * mult;
#pragma unroll
            for (int k = 0; k < 4; k += 2) {
              const float y0 = x[hh][k] * sc, y1 = x[hh][k + 1] * sc;
              const __half2 hi = __floats2half2_rn(y0, y1);
              const float2 fh = __half22float2(hi);
              const __half2 lo = __floats2half2_rn(y0 - fh.x, y1 - fh.y);
              fb[(k + 8 * hh) * (kFragRowWords * 2) + wh] = __half_as_ushort(__low2half(hi));
              fb[(k + 1 + 8 * hh) * (kFragRowWords * 2) + wh] = __half_as_ushort(__high2half(hi));
              fb[(k + 8 * hh + 4) * (kFragRowWords * 2) + wh] = __half_as_ushort(__low2half(lo));
              fb[(k + 1 + 8 * hh + 4) * (kFragRowWords * 2) + wh] = __half_as_ushort(__high2half(lo));
            }
            float bsum = beta[hh];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) bsum += __shfl_xor_sync(0xffffffffu, bsum, off);
            if (head_mine == hh) {
              // products are code * qs * 2^(E - 18) (2-bit) or 2^(E - 20) (4-bit)
              cq_g[gi] = c0 * pow2i((BITS == 2 ? 18 : 20) - E);
              beta_g[gi] = c0 * bsum;
            }
          }
        }
      }
      __syncwarp();
      // ---- R steps of T tiles cover the unit (a trailing single group: 32 tokens)
      auto run = [&](auto full_tag, int n_tok) {
        constexpr bool FULL = decltype(full_tag)::value;
#pragma unroll
        for (int s = 0; s < R; ++s) {
          if (!FULL && 16 * T * s >= n_tok) break;
          const int my_grp = (s * T + li.slot_mine) / TPG;
          float cq = cq_g[0], beta = beta_g[0];
          if (NGU > 1 && my_grp == 1) {
            cq = cq_g[NGU - 1];
            beta = beta_g[NGU - 1];
          }
          uint32_t bf[16];
          auto kfill = [&](int i, float sc[4]) {
            const int t = s * T + i;
            // (re)load the B fragment at the first tile of each group in the step
            if (i == 0 || t % TPG == 0)
              load_frag(frag + (t / TPG) * L::kFragGroupBytes + frag_row * kFragRowWords * 4, bf);
            uint32_t ra0[8], ra1[8], rb0[8], rb1[8];
            if constexpr (BITS == 2) {
              // words 2tig, 2tig+1 of tokens g and g+8: channels 32tig .. 32tig+31
              const uint2 ka = lds64(stg + L::kKCodes + (16 * t + g) * 32 + tig * 8);
              const uint2 kb = lds64(stg + L::kKCodes + (16 * t + g + 8) * 32 + tig * 8);
              unpack16(ka.x, ra0);
              unpack16(ka.y, ra1);
              unpack16(kb.x, rb0);
              unpack16(kb.y, rb1);
            } else {
              // words 4tig .. 4tig+3 of tokens g and g+8: channels 32tig .. 32tig+31
              const uint4 ka = *reinterpret_cast<const uint4 *>(stg + L::kKCodes + (16 * t + g) * 64 + tig * 16);
              const uint4 kb = *reinterpret_cast<const uint4 *>(stg + L::kKCodes + (16 * t + g + 8) * 64 + tig * 16);
              unpack8(ka.x, ra0);
              unpack8(ka.y, ra0 + 4);
              unpack8(ka.z, ra1);
              unpack8(ka.w, ra1 + 4);
              unpack8(kb.x, rb0);
              unpack8(kb.y, rb0 + 4);
              unpack8(kb.z, rb1);
              unpack8(kb.w, rb1 + 4);
            }
            qk_tile(ra0, ra1, rb0, rb1, bf, sc);
          };
          auto vmeta = [&](int tok) -> uint32_t { return lds32(stg + L::kVMeta + (16 * T * s + tok) * 4); };
          qk_step<R, FULL>(ss, li, kfill, cq, beta, FULL ? 16 * T : n_tok - 16 * T * s, vmeta, nw0[s], nw1[s],
                           nalpha[s]);
        }
      };
      if (ngr == NGU)
        run(std::true_type{}, kUnit);
      else
        run(std::false_type{}, ngr * G);
      n_kind = 1;
      n_ntok = ngr * G;
    } else {
      // ---- fp16 residual keys of the head: B = q itself (hi part, lo = 0), A = keys
      uint16_t *fb = reinterpret_cast<uint16_t *>(frag);
#pragma unroll
      for (int k = 0; k < 4; ++k)
#pragma unroll
        for (int hh = 0; hh < R; ++hh) {
          fb[(k + 8 * hh) * (kFragRowWords * 2) + wh_pairs] = f2h(qv[hh][k]);
          fb[(k + 8 * hh + 4) * (kFragRowWords * 2) + wh_pairs] = 0;
        }
      __syncwarp();
      uint32_t bf[16];
      load_frag(frag + frag_row * kFragRowWords * 4, bf);
      const int r = cc.r;
      const int64_t nq = (int64_t)cc.NG * G;
      const uint16_t *res_head = a.k_res + cc.h * G * kD;
      // value rows of the residual tokens nq .. nq + r - 1 (one page: pages hold whole groups)
      if constexpr (PAGED) {
        const int64_t ph = page_of(cc.b, (int)nq) * a.Hkv + cc.kvh;
        n_res_row = ph * P + (nq & (P - 1));
      } else {
        n_res_row = cc.h * a.max_tokens + nq;
      }
      const uint32_t *vm_head = a.v_meta + n_res_row;
#pragma unroll
      for (int s = 0; s < R; ++s) {
        const int base = 16 * T * s;
        if (base >= r) break;
        auto kfill = [&](int i, float sc[4]) {
          const int sa_slot = base + 16 * i + g, sb_slot = sa_slot + 8;
          uint32_t ra0[8], ra1[8], rb0[8], rb1[8];
          residual_pairs(res_head + sa_slot * kD, sa_slot < r, tig, ra0, ra1);
          residual_pairs(res_head + sb_slot * kD, sb_slot < r, tig, rb0, rb1);
          qk_tile(ra0, ra1, rb0, rb1, bf, sc);
        };
        // residual values are quantized ({s, z} of their row) or, with a value
        // residual, fp16 themselves: weight p with s = 1, z = 0
        auto vmeta = [&](int tok) -> uint32_t { return a.v_res ? 0x00003C00u : vm_head[base + tok]; };
        qk_step<R, false>(ss, li, kfill, c0, 0.f, min(16 * T, r - base), vmeta, nw0[s], nw1[s], nalpha[s]);
      }
      n_kind = 2;
      n_ntok = r;
    }

    // ---- P.V of this unit: value codes from the stage, or (residual unit) from HBM
    if (n_kind == 1) {
      const unsigned char *stg = wbase + stage * L::kStageBytes;
#pragma unroll
      for (int s = 0; s < R; ++s) {
        const int nv = min(16 * T, n_ntok - 16 * T * s);
        if (nv <= 0) break;
        if constexpr (BITS == 2) {
          pv_step<R, 2>(acc, li, nv, nw0[s], nw1[s], nalpha[s], [&](int i, int k) -> uint32_t {
            return lds32(stg + L::kVCodes + (16 * (s * T + i) + tig + 4 * k) * 32 + g * 4);
          });
        } else {
          pv_step<R, 4>(acc, li, nv, nw0[s], nw1[s], nalpha[s], [&](int i, int k) -> uint2 {
            return lds64(stg + L::kVCodes + (16 * (s * T + i) + tig + 4 * k) * 64 + g * 8);
          });
        }
      }
    } else if (a.v_res) {
      // fp16 residual values: this is the head's last unit, so the accumulators move
      // to output units here and the head's partial is written without code factors
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float un = pow2i(BITS == 2 ? 24 - 2 * (j & 3) : 24 - 4 * (j & 1));
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[j][k] *= un;
      }
      acc_true = true;
      const uint16_t *vres_head = a.v_res + cc.h * G * kD;
#pragma unroll
      for (int s = 0; s < R; ++s) {
        const int nv = min(16 * T, n_ntok - 16 * T * s);
        if (nv <= 0) break;
        pv_step_f16<R>(acc, li, nv, nw0[s], nw1[s], nalpha[s], vres_head + 16 * T * s * kD);
      }
    } else {
      const uint32_t *vc_head = a.v_codes + n_res_row * WPR;
#pragma unroll
      for (int s = 0; s < R; ++s) {
        const int nv = min(16 * T, n_ntok - 16 * T * s);
        if (nv <= 0) break;
        if constexpr (BITS == 2) {
          pv_step<R, 2>(acc, li, nv, nw0[s], nw1[s], nalpha[s], [&](int i, int k) -> uint32_t {
            const int slot = 16 * (s * T + i) + tig + 4 * k;
            return vc_head[(slot < n_ntok ? slot : 0) * WPR + g];
          });
        } else {
          pv_step<R, 4>(acc, li, nv, nw0[s], nw1[s], nalpha[s], [&](int i, int k) -> uint2 {
            const int slot = 16 * (s * T + i) + tig + 4 * k;
            return *reinterpret_cast<const uint2 *>(vc_head + (slot < n_ntok ? slot : 0) * WPR + 2 * g);
          });
        }
      }
    }
    __syncwarp();  // this unit's stage may be refilled from now on
    if (kk + 1 < n_my) {
      if (cc.uu + 1 == cc.U) {  // the next unit starts a new head
        emit(cc.h, ss);
        ss.m = -INFINITY;
        ss.l = 0.f;
        ss.zs = 0.f;
        advance(cc);
        load_q(cc);
      } else {
        advance(cc);
      }
    }
  }
  emit(cc.h, ss);
  cp_async_wait<0>();
}

// Merge np partials (max, sum, unnormalised output; `stride` floats apart) of one
// (batch, query head) into out_row with one warp: lane l owns channels 2l, 2l+1,
// 64+2l, 64+2l+1.  Every partial's loads are issued before any is used (the
// partials sit in L2), then an online max-rescaled sum merges them.  np == 0 (no
// tokens) writes zeros.  Partial rows are 8-byte aligned (stride 130 floats).
__device__ __forceinline__ void combine_row(const float *__restrict__ p, int np, int64_t stride,
                                            uint16_t *__restrict__ out_row, int lane) {
  constexpr int kBatch = 16;
  float M = -INFINITY, L = 0.f, o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;
  for (int j0 = 0; j0 < np; j0 += kBatch) {
    float2 ml[kBatch], lo[kBatch], hi[kBatch];
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      if (j0 + k < np) {
        const float *r = p + (int64_t)(j0 + k) * stride;
        ml[k] = __ldcg(reinterpret_cast<const float2 *>(r + kD));
        lo[k] = __ldcg(reinterpret_cast<const float2 *>(r + 2 * lane));
        hi[k] = __ldcg(reinterpret_cast<const float2 *>(r + 64 + 2 * lane));
      }
    }
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      if (j0 + k < np && ml[k].x != -INFINITY) {
        const float m = fmaxf(M, ml[k].x);
        const float a = ex2(M - m);  // M = -inf on the first partial: a = 0
        const float w = ex2(ml[k].x - m);
        L = fmaf(L, a, w * ml[k].y);
        o0 = fmaf(o0, a, w * lo[k].x);
        o1 = fmaf(o1, a, w * lo[k].y);
        o2 = fmaf(o2, a, w * hi[k].x);
        o3 = fmaf(o3, a, w * hi[k].y);
        M = m;
      }
    }
  }
  const float inv = np > 0 ? 1.f / L : 0.f;
  uint32_t *dst = reinterpret_cast<uint32_t *>(out_row);
  dst[lane] = h22u(__floats2half2_rn(o0 * inv, o1 * inv));
  dst[32 + lane] = h22u(__floats2half2_rn(o2 * inv, o3 * inv));
}

// Dense layout: the partials of (batch, query head) `row` sit at slots 0 .. np-1 of
// the row's pmax slots; np follows from the unit split.
__global__ void __launch_bounds__(32 * kCombineRows) combine_kernel(const float *__restrict__ ws, int64_t pmax,
                                                                    int64_t W, int64_t NW, int64_t U, int Hkv,
                                                                    int Hq, int64_t rows,
                                                                    uint16_t *__restrict__ out) {
  asm volatile("griddepcontrol.wait;\n" ::: "memory");  // the decode grid has completed
  const int64_t row = (int64_t)blockIdx.x * kCombineRows + (threadIdx.x >> 5);  // b * Hq + h
  if (row >= rows) return;
  const int64_t b = row / Hq, hq = row - b * Hq;
  const int64_t head = b * Hkv + hq / (Hq / Hkv);
  const int64_t first = owner_warp(head * U, W, NW), last = owner_warp(head * U + U - 1, W, NW);
  combine_row(ws + row * pmax * (kD + 2), (int)(last - first + 1), kD + 2, out + row * kD, threadIdx.x & 31);
}

// Paged layout: the decode grid wrote, per (batch, KV head), the index of its first
// partial pair and their count; pair i holds the R query heads' partials.  With
// `advance`, the grid then moves every sequence's length past the token the step
// appended (the decode grid, and so the append before it, has completed).
__global__ void __launch_bounds__(32 * kCombineRows) paged_combine_kernel(const float *__restrict__ ws, int Hkv,
                                                                          int Hq, int B, int32_t *advance,
                                                                          int32_t cap, uint16_t *__restrict__ out) {
  asm volatile("griddepcontrol.wait;\n" ::: "memory");  // the decode grid has completed
  const int64_t row = (int64_t)blockIdx.x * kCombineRows + (threadIdx.x >> 5);  // b * Hq + h
  if (row >= (int64_t)B * Hq) return;
  const int lane = threadIdx.x & 31;
  const int64_t b = row / Hq, hq = row - b * Hq;
  const int R = Hq / Hkv;
  const int64_t head = b * Hkv + hq / R;
  const int2 hd = __ldcg(reinterpret_cast<const int2 *>(ws) + head);
  const float *part = ws + 2 * (int64_t)B * Hkv;
  combine_row(part + ((int64_t)hd.x * R + hq % R) * (kD + 2), hd.y, (int64_t)R * (kD + 2), out + row * kD, lane);
  if (advance && hq == 0 && lane == 0) {
    const int32_t len = advance[b];
    advance[b] = len < cap ? len + 1 : cap;
  }
}

template <int R, int G, bool PAGED, int BITS>
const void *kernel_ptr() {
  return reinterpret_cast<const void *>(&decode_kernel<R, G, PAGED, BITS>);
}

template <bool PAGED, int BITS>
const void *select_kernel(int R, int G) {
  if (G == 32)
    return R == 1   ? kernel_ptr<1, 32, PAGED, BITS>()
           : R == 2 ? kernel_ptr<2, 32, PAGED, BITS>()
                    : kernel_ptr<4, 32, PAGED, BITS>();
  return R == 1 ? kernel_ptr<1, 64, PAGED, BITS>() : R == 2 ? kernel_ptr<2, 64, PAGED, BITS>() : kernel_ptr<4, 64, PAGED, BITS>();
}

template <int BITS>
int smem_bytes(int R, int G) {
  if (G == 32)
    return R == 1 ? Layout<1, 32, BITS>::kSmem : R == 2 ? Layout<2, 32, BITS>::kSmem : Layout<4, 32, BITS>::kSmem;
  return R == 1 ? Layout<1, 64, BITS>::kSmem : R == 2 ? Layout<2, 64, BITS>::kSmem : Layout<4, 64, BITS>::kSmem;
}

// Paged kernels append the lengths, the unit prefix and 4 warp totals: 2B + 5 ints.
constexpr int paged_extra(int B) { return (4 * (2 * B + 5) + 15) & ~15; }

}  // namespace

DecodeKernels decode_kernels(int R, int G, int bits, bool paged, int B) {
  DecodeKernels k;
  const int base = bits == 2 ? smem_bytes<2>(R, G) : smem_bytes<4>(R, G);
  if (paged) {
    k.decode = bits == 2 ? select_kernel<true, 2>(R, G) : select_kernel<true, 4>(R, G);
    k.smem = base + paged_extra(B);
    k.smem_limit = base + paged_extra(kPagedMaxBatch);
    k.combine = reinterpret_cast<const void *>(&paged_combine_kernel);
  } else {
    k.decode = bits == 2 ? select_kernel<false, 2>(R, G) : select_kernel<false, 4>(R, G);
    k.smem = k.smem_limit = base;
    k.combine = reinterpret_cast<const void *>(&combine_kernel);
  }
  return k;
}

}  // namespace kivi
