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
//     qs is scaled by a power of two per (head, group) chosen from a bound on its
//     entries (the largest |q| of the head times the largest scale of the group), so
//     that every entry stays below 2^15 (no fp16 overflow) and the large entries keep
//     their lo parts out of the fp16 subnormals (full precision for any range).
// Tokens are tiled by 16 (the MMA M dimension for q.K, the K dimension for P.V).
// The 4 column pairs of an MMA carry (tile slot, query head): a round covers
// T = 4/R tiles at once, so that for every R each lane owns the scores of one
// (tile, head) pair: lane (g, tig) holds tokens g and g+8 of tile slot tig/R for
// head tig%R.  For q.K the per-head factors are replicated over the slots and each
// tile accumulates separately; for P.V each tile's weights sit in its own column
// pairs and all tiles accumulate together (the slots are summed at the end).
//
// Work decomposition (persistent, balanced): a "unit" is 64 tokens of one (batch, KV
// head) -- one or two key groups -- plus one unit for the fp16 residual keys when
// n mod G > 0.  The grid holds exactly as many warps as fit on the GPU at once; warp
// w takes the contiguous unit range [w*W/NW, (w+1)*W/NW).  At every head boundary
// the warp writes a partial (max, sum, unnormalised output) to the workspace; the
// combine kernel merges a head's partials (flash-decoding) and is launched as a
// programmatic dependent.
//
// Staging: each warp owns a ring of stages in shared memory, filled one or two units
// ahead of the one it computes.  One lane stages a unit with four linear bulk copies
// (cp.async.bulk, executed by the TMA engine): key codes, value codes, value
// {scale, zero} words and key-group {scale, zero} words, whose completion is counted
// on the stage's mbarrier.  Every wait on an mbarrier is bounded: a warp whose copy
// never completes records the fault, waits (bounded again) for its other copies and
// stops; the combine then writes NaN outputs.
//
// One softmax update per unit for all R heads: the q.K MMAs of the unit's four
// 16-token tiles come first (R rounds of T tiles), then the running maximum, the
// probabilities and the P.V operand of every round, then the P.V MMAs.
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

// Set when a decode warp's wait for a staged unit ran out; the combine kernels then
// write NaN outputs.  It stays set for the life of the process.
__device__ int g_decode_fault = 0;

constexpr int kWarps = kDecodeWarps;
constexpr int kThreads = kWarps * 32;
constexpr int kUnit = kDecodeUnit;  // tokens per unit
constexpr float kLog2e = 1.4426950408889634f;
constexpr unsigned kFull = 0xffffffffu;
// Polls of a stage's mbarrier before a warp gives up on it.  Each poll may suspend
// the warp for a short, hardware-chosen time, so this bound is far beyond the latency
// of any copy.
constexpr int kWaitPolls = 1 << 22;

// Shared-memory layout of one warp: the ring of stages for BITS-bit codes, the q.K
// B fragment of one key group, and one mbarrier per stage.  4-bit rows are twice as
// long, so their ring has two stages (one unit staged ahead) to keep two CTAs per SM;
// 2-bit rows keep three (two ahead).  VG < 128: each value token carries 128 / VG
// {s, z} words (value channel groups of VG channels).
template <int R, int G, int BITS = 2, int VG = kD>
struct Layout {
  static constexpr int kNV = kD / VG;                         // {s, z} words per value token
  static constexpr int kRowBytes = 16 * BITS;                 // packed codes of one token row
  static constexpr int kStages = BITS == 2 ? 3 : 2;
  static constexpr int kAhead = kStages - 1;                  // units staged ahead of the computed one
  static constexpr int kGroups = kUnit / G;                   // key groups per unit
  static constexpr int kKCodes = 0;                           // 64 rows
  static constexpr int kVCodes = kUnit * kRowBytes;           // 64 rows
  static constexpr int kVMeta = 2 * kUnit * kRowBytes;        // 64 x kNV x 4 B
  static constexpr int kKMeta = kVMeta + kUnit * kNV * 4;     // kGroups x 128 x 4 B
  static constexpr int kStageBytes = kKMeta + kGroups * kD * 4;
  // B fragment rows (2h + part) * 4 + tig of 16 words.  With fewer than four heads
  // four lanes read each row, so rows are padded to 20 words to spread them over the
  // shared-memory banks; with four heads every lane reads its own row.
  static constexpr int kFragRowWords = R == 4 ? 16 : 20;
  static constexpr int kFrag = kStages * kStageBytes;
  static constexpr int kBars = kFrag + 8 * R * kFragRowWords * 4;
  static constexpr int kWarpBytes = kBars + 32;               // kStages mbarriers of 8 bytes
  static constexpr int kSmem = kWarps * kWarpBytes;
  static_assert(kStages * 8 <= 32, "the barrier block holds every stage's mbarrier");
  static_assert(kStageBytes % 16 == 0 && kFrag % 16 == 0 && kBars % 16 == 0, "16-byte aligned regions");
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float pow2i(int e) { return __int_as_float((e + 127) << 23); }  // e in [-126, 127]

__device__ __forceinline__ uint2 lds64(const unsigned char *p) { return *reinterpret_cast<const uint2 *>(p); }
__device__ __forceinline__ uint32_t lds32(const unsigned char *p) { return *reinterpret_cast<const uint32_t *>(p); }

// ---- mbarriers and bulk copies (TMA engine), all on this CTA's shared memory ----------
__device__ __forceinline__ uint32_t smem_addr(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t bar) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(bar) : "memory");
}

// This thread's arrival on `bar`, with `bytes` more bytes expected in the phase.
__device__ __forceinline__ void mbar_arm(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes) : "memory");
}

// Linear global -> shared copy of `bytes` (a multiple of 16, both ends 16-byte
// aligned); its completion is counted on `bar`.
__device__ __forceinline__ void bulk_copy(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// Wait until the phase of parity `parity` of `bar` has completed; false if it did not
// within kWaitPolls polls.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  for (int i = 0; i < kWaitPolls; ++i) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

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
// (ra*) and g+8 (rb*), words 2tig (..0) and 2tig+1 (..1); accumulates into sc.  The
// two words accumulate in separate chains of four MMAs (shorter dependences).
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

// P.V of one 16-token tile over fp16 values (the value residual): A is built from
// the fp16 values of tokens tig, tig+4, tig+8, tig+12 of the tile (channels 16g + j
// and 16g + 8 + j for MMA j) instead of unpacked codes.  `rows` points at the tile's
// first token row; tokens at or beyond n_valid read as zero.
__device__ __forceinline__ void pv_tile_f16(float acc[8][4], const uint16_t *rows, int n_valid, int g, int tig,
                                            uint32_t b0, uint32_t b1) {
  uint32_t w[4][8];  // token tig + 4k: channels 16g .. 16g+15 as 8 half2 words
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int tok = tig + 4 * k;
    uint4 lo = make_uint4(0u, 0u, 0u, 0u), hi = lo;
    if (tok < n_valid) {
      const uint4 *src = reinterpret_cast<const uint4 *>(rows + tok * kD + 16 * g);
      lo = __ldg(src);
      hi = __ldg(src + 1);
    }
    w[k][0] = lo.x; w[k][1] = lo.y; w[k][2] = lo.z; w[k][3] = lo.w;
    w[k][4] = hi.x; w[k][5] = hi.y; w[k][6] = hi.z; w[k][7] = hi.w;
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t sel = (j & 1) ? 0x7632u : 0x5410u;
    const int x = j >> 1, y = 4 + (j >> 1);  // words of channels 16g + j and 16g + 8 + j
    mma16816(acc[j], prmt(w[0][x], w[1][x], sel), prmt(w[0][y], w[1][y], sel), prmt(w[2][x], w[3][x], sel),
             prmt(w[2][y], w[3][y], sel), b0, b1);
  }
}

// Index of the first warp whose unit range contains unit u.
__device__ __forceinline__ int64_t owner_warp(int64_t u, int64_t W, int64_t NW) { return ((u + 1) * NW - 1) / W; }

// Softmax state of a head: running max (log2 domain) and this lane's shares of
// sum_t p_t and sum_t p_t z_t.
// Running softmax state of a head: max m and sum l of the weights (log2 domain), and
// zs[m] = sum of weight * z over the tokens, one per value channel group.
template <int NV>
struct SoftState {
  float m, l, zs[NV];
};

// Max over the lanes that share this lane's query head.
template <int R>
__device__ __forceinline__ float head_max(float x) {
  if constexpr (R == 1) {
    // one head per warp: an order-preserving integer key and one warp reduction
    const int k = __float_as_int(x);
    const int key = k ^ ((k >> 31) & 0x7fffffff);
    const int mk = __reduce_max_sync(kFull, key);
    return __int_as_float(mk ^ ((mk >> 31) & 0x7fffffff));
  } else {
#pragma unroll
    for (int off = R; off < 32; off <<= 1) x = fmaxf(x, __shfl_xor_sync(kFull, x, off));
    return x;
  }
}

// Warp sums of the q . z partials v[gi][h] (gi < NG key groups, h < R heads),
// delivered where they are used: afterwards v[gi][0] holds, for every group, the sum
// for this lane's head h = tig % R.  The heads are first scattered over lane bits
// 0 .. log2(R) - 1 (each exchange sends the half of the heads that the partner keeps),
// then the other lane bits are summed by a butterfly.  With one head and two groups
// the group is scattered over lane bit 1 instead (lane tig reads tile slot tig, whose
// group is tig >> 1), and v[0][0] = v[1][0] holds the lane's group's sum.
template <int R, int NG>
__device__ __forceinline__ void beta_reduce_heads(float (&v)[NG][R], int lane);

template <int R, int NG>
__device__ __forceinline__ void beta_reduce(float (&v)[NG][R], int lane) {
  if constexpr (R == 1 && NG == 2) {
    const bool up = (lane >> 1) & 1;
    const float keep = up ? v[1][0] : v[0][0], send = up ? v[0][0] : v[1][0];
    float s = keep + __shfl_xor_sync(kFull, send, 2);
    s += __shfl_xor_sync(kFull, s, 1);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) s += __shfl_xor_sync(kFull, s, off);
    v[0][0] = v[1][0] = s;
  } else {
    beta_reduce_heads<R, NG>(v, lane);
  }
}

template <int R, int NG>
__device__ __forceinline__ void beta_reduce_heads(float (&v)[NG][R], int lane) {
  if constexpr (R >= 2) {
    const bool up = lane & 1;
#pragma unroll
    for (int gi = 0; gi < NG; ++gi)
#pragma unroll
      for (int i = 0; i < R / 2; ++i) {
        const float keep = up ? v[gi][2 * i + 1] : v[gi][2 * i];
        const float send = up ? v[gi][2 * i] : v[gi][2 * i + 1];
        v[gi][i] = keep + __shfl_xor_sync(kFull, send, 1);
      }
  }
  if constexpr (R == 4) {
    const bool up = (lane >> 1) & 1;
#pragma unroll
    for (int gi = 0; gi < NG; ++gi) {
      const float keep = up ? v[gi][1] : v[gi][0], send = up ? v[gi][0] : v[gi][1];
      v[gi][0] = keep + __shfl_xor_sync(kFull, send, 2);
    }
  }
#pragma unroll
  for (int off = R; off < 32; off <<= 1)
#pragma unroll
    for (int gi = 0; gi < NG; ++gi) v[gi][0] += __shfl_xor_sync(kFull, v[gi][0], off);
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
    const int y = __shfl_up_sync(kFull, inc, off);
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

// Merge np partials (max, sum, unnormalised output; `stride` floats apart) of one
// (batch, query head) into out_row with one warp: lane l owns channels 2l, 2l+1,
// 64+2l, 64+2l+1.  Every partial's loads are issued before any is used (the
// partials sit in L2, or in shared memory with SHARED), then an online max-rescaled
// sum merges them.  np == 0 (no
// tokens) writes zeros; after a decode fault (g_decode_fault) the row is NaN.
// Partial rows are 8-byte aligned (stride 130 floats).
// Partial j starts at row(j).
template <bool SHARED, typename RowFn>
__device__ __forceinline__ void combine_rows(RowFn row, int np, uint16_t *__restrict__ out_row, int lane) {
  constexpr int kBatch = 16;
  float M = -INFINITY, L = 0.f, o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;
  for (int j0 = 0; j0 < np; j0 += kBatch) {
    float2 ml[kBatch], lo[kBatch], hi[kBatch];
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      if (j0 + k < np) {
        const float *r = row(j0 + k);
        if constexpr (SHARED) {
          ml[k] = *reinterpret_cast<const float2 *>(r + kD);
          lo[k] = *reinterpret_cast<const float2 *>(r + 2 * lane);
          hi[k] = *reinterpret_cast<const float2 *>(r + 64 + 2 * lane);
        } else {
          ml[k] = __ldcg(reinterpret_cast<const float2 *>(r + kD));
          lo[k] = __ldcg(reinterpret_cast<const float2 *>(r + 2 * lane));
          hi[k] = __ldcg(reinterpret_cast<const float2 *>(r + 64 + 2 * lane));
        }
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
  float inv = np > 0 ? 1.f / L : 0.f;
  // a decode warp that gave up on a staged copy left partials unwritten: say so
  if (*reinterpret_cast<volatile int *>(&g_decode_fault)) inv = __int_as_float(0x7fc00000);
  uint32_t *dst = reinterpret_cast<uint32_t *>(out_row);
  dst[lane] = h22u(__floats2half2_rn(o0 * inv, o1 * inv));
  dst[32 + lane] = h22u(__floats2half2_rn(o2 * inv, o3 * inv));
}

// Partial j at p + j * stride.
template <bool SHARED>
__device__ __forceinline__ void combine_row(const float *__restrict__ p, int np, int64_t stride,
                                            uint16_t *__restrict__ out_row, int lane) {
  combine_rows<SHARED>([&](int j) { return p + (int64_t)j * stride; }, np, out_row, lane);
}


// Thread-block cluster barrier halves and the shared-memory window of a cluster peer.
// Threads that have exited count as arrived, and no kernel here waits on a cluster
// barrier inside a loop, so every wait ends once each CTA of the cluster gets there.
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release;\n" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire;\n" ::: "memory"); }
__device__ __forceinline__ int cluster_rank() {
  int r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
  return r;
}
// Generic address of `p` (this CTA's shared memory) in the shared memory of cluster CTA `rank`.
__device__ __forceinline__ const float *cluster_peer(const float *p, int rank) {
  const float *q;
  asm volatile("mapa.u64 %0, %1, %2;\n" : "=l"(q) : "l"(p), "r"(rank));
  return q;
}

// The small path's merge: once every warp of the CTA (CL = 1), or of every CTA of the
// cluster (CL > 1), has written its partials into its own CTA's shared memory, warp r
// of the first CTA merges query head r's partials of the (batch, KV head) into the
// output.  A cluster's first CTA reads the other CTAs' partials in their shared memory
// (coalesced 8-byte loads; scattered 4-byte stores into its own memory from the other
// CTAs were slower), and they stay resident until it has.
template <int R, int CL, int NWARPS>
__device__ __forceinline__ void small_merge(const DecodeArgs &a, const float *s_part, int64_t NW, int warp,
                                            int lane) {
  const int64_t h = blockIdx.x / CL, b = h / a.Hkv, kvh = h - b * a.Hkv;
  uint16_t *out_row = a.out + (b * a.Hq + kvh * R + warp) * kD;
  if constexpr (CL == 1) {
    __syncthreads();
    if (warp < R) combine_row<true>(s_part + warp * (kD + 2), (int)NW, (int64_t)R * (kD + 2), out_row, lane);
  } else {
    cluster_arrive();  // release: this CTA's partials
    cluster_wait();    // acquire: every CTA's
    if (warp < R && cluster_rank() == 0) {
      // partial j: warp j mod NWARPS of cluster CTA j / NWARPS
      const float *mine = s_part + warp * (kD + 2);
      combine_rows<true>(
          [&](int j) { return cluster_peer(mine + (j % NWARPS) * R * (kD + 2), j / NWARPS); }, (int)NW, out_row,
          lane);
    }
    cluster_arrive();  // the first CTA has read every partial
    cluster_wait();
  }
}

// Launch modes of the decode body: the persistent grid over a dense or a paged cache,
// and the small-context path (one CTA of kSmallWarps warps per (batch, KV head) of a
// dense cache, its warps' partials merged in shared memory: no workspace round trip
// and no combine launch).  With CL > 1 the small path runs on a cluster of CL CTAs
// per (batch, KV head), whose first CTA merges the partials of all of them.
constexpr int kModeDense = 0, kModePaged = 1, kModeSmall = 2;
constexpr int kSmallWarps = kDecodeSmallWarps;

// Partials of the small path: [warp][R] rows of kD + 2 floats after the warps' rings
// (each CTA of a cluster holds its own warps').
template <int R, int NW = kSmallWarps>
__host__ __device__ constexpr int small_part_bytes() { return NW * R * (kD + 2) * 4; }

template <int R, int G, int MODE, int BITS, int NWARPS, int VG = kD, int CL = 1>
__device__ __forceinline__ void decode_body(const DecodeArgs &a) {
  constexpr bool PAGED = MODE == kModePaged;
  constexpr bool SMALL = MODE == kModeSmall;
  static_assert(CL == 1 || SMALL, "clusters: the small path only");
  extern __shared__ __align__(16) unsigned char smem[];
  using L = Layout<R, G, BITS, VG>;
  // value channel groups (VG < 128): NV {s, z} words per value token, group m over
  // channels VG*m .. VG*m + VG - 1, i.e. code words WG*m .. WG*m + WG - 1 of a row
  constexpr int NV = L::kNV;
  constexpr int WG = VG / 16;
  static_assert(NV == 1 || (BITS == 2 && MODE == kModeDense), "value groups: dense 2-bit caches");
  constexpr int WPR = words_per_row<BITS>();
  constexpr int S = L::kStages;
  constexpr int AH = L::kAhead;
  constexpr int T = 4 / R;                 // tile slots per round
  constexpr int TPG = G / 16;              // tiles per key group
  constexpr int NGU = L::kGroups;          // key groups per unit
  constexpr int FRW = L::kFragRowWords;
  constexpr int SH = BITS == 2 ? 18 : 20;  // a q.K MMA product is code * qs * 2^(E - SH) for B scaled by 2^E
  constexpr int PD = BITS == 2 ? 8 : 4;    // channel distance of the two codes of an unpacked register
  // the combine grid may launch now; it waits for this grid's completion
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = CL > 1 ? cluster_rank() : 0;
  const int64_t gw = SMALL ? (int64_t)rank * NWARPS + warp : (int64_t)blockIdx.x * NWARPS + warp;
  int64_t NW = a.n_warps;
  int64_t W;
  float *s_part = reinterpret_cast<float *>(smem + NWARPS * L::kWarpBytes);  // small path only
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
  } else if constexpr (SMALL) {
    W = a.units_per_head;  // the units of head blockIdx.x / CL
    NW = W < CL * NWARPS ? W : CL * NWARPS;
  } else {
    W = a.total_units;
  }
  int64_t u0 = 0, u1 = 0;
  if (gw < NW) {
    u0 = gw * W / NW;
    u1 = (gw + 1) * W / NW;
  }
  if constexpr (SMALL) {
    u0 += (int64_t)(blockIdx.x / CL) * W;
    u1 += (int64_t)(blockIdx.x / CL) * W;
  }
  if (u0 >= u1) {
    if constexpr (SMALL) small_merge<R, CL, NWARPS>(a, s_part, NW, warp, lane);
    return;
  }
  const int n_my = (int)(u1 - u0);

  unsigned char *wbase = smem + warp * L::kWarpBytes;
  unsigned char *frag = wbase + L::kFrag;
  const uint32_t bar0 = smem_addr(wbase + L::kBars);
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < S; ++s) mbar_init(bar0 + 8 * s);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncwarp();
  const float c0 = a.softmax_scale * kLog2e;

  // ---- lane roles in the MMAs
  const int g = lane >> 2, tig = lane & 3;
  const int head_mine = tig % R, slot_mine = tig / R;
  const int pv_slot = (g >> 1) / R;
  const int src_a = 4 * tig + (g >> 1), src_b = src_a + 16;
  const uint32_t pv_sel = (g & 1) ? 0x7632u : 0x5410u;
  const int frag_row = 4 * (2 * ((g >> 1) % R) + (g & 1)) + tig;
  // ---- lane roles in the factor preparation: B registers 8w + 2j and 8w + 2j + 1 of
  // fragment row tig' (tig' = lane >> 3, w = bit 2, j = bits 0-1).  Like the unpacked
  // codes they meet, register 8w + 2j pairs channels pc and pc + PD, register
  // 8w + 2j + 1 channels pc + 1 and pc + PD + 1; fa and fb are the powers of two that
  // bring each register's products to code * qs * 2^-SH (the codes' own factors are
  // 4^(i mod 4) for 2-bit register i, 16^(i mod 2) for 4-bit register i).
  const int pt = lane >> 3, pw = (lane >> 2) & 1, pj = lane & 3;
  const int pc = BITS == 2 ? 32 * pt + 16 * pw + 2 * pj : 32 * pt + 16 * pw + 8 * (pj >> 1) + 2 * (pj & 1);
  const int pword = 8 * pw + 2 * pj;
  const float fa = BITS == 2 ? ((pj & 1) ? 4.f : 64.f) : 16.f;
  const float fb = BITS == 2 ? ((pj & 1) ? 1.f : 16.f) : 1.f;
  const float ifa = 1.f / fa, ifb = 1.f / fb;

  // ---- the query heads of the current KV head: q of this lane's preparation
  // channels (pc, pc + PD, pc + 1, pc + PD + 1) times fa / fb and 2^A_h, where A_h puts
  // the head's largest |q * f| below 2^14; with every scale of a group below
  // 2^(es + 1) and scaled by 2^-es, each B entry stays below 2^15
  float qa[R][4];
  // 1.5 * 2^23 * u_h: adding and subtracting it times f rounds an entry x to the grid
  // u_h * f of the hi parts (see write_frag); u_h = 2^(E_h - 8), E_h = floor(log2 of the
  // head's largest |q| * 2^A), so that every |x| / (u_h * f) stays below 2^10
  float gu[R];
  float cqh = 0.f, cbh = 0.f;  // c0 * 2^(SH - A) and c0 * 2^-A of this lane's head
  auto q_row = [&](int64_t b, int64_t kvh) { return a.q + (b * a.Hq + kvh * R) * kD; };
  auto load_q = [&](const uint16_t *qh) {
#pragma unroll
    for (int hh = 0; hh < R; ++hh) {
      const uint32_t w01 = __ldg(reinterpret_cast<const unsigned int *>(qh + hh * kD + pc));
      const uint32_t wd = __ldg(reinterpret_cast<const unsigned int *>(qh + hh * kD + pc + PD));
      float x[4];
      x[0] = h2f((uint16_t)(w01 & 0xffffu)) * fa;
      x[1] = h2f((uint16_t)(wd & 0xffffu)) * fa;
      x[2] = h2f((uint16_t)(w01 >> 16)) * fb;
      x[3] = h2f((uint16_t)(wd >> 16)) * fb;
      const float mx = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
      const float my = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])) * ifa, fmaxf(fabsf(x[2]), fabsf(x[3])) * ifb);
      const uint32_t mb = __reduce_max_sync(kFull, __float_as_uint(mx));
      const uint32_t yb = __reduce_max_sync(kFull, __float_as_uint(my));
      const int A = min(100, max(-100, 13 - ((int)(mb >> 23) - 127)));
      const float sc = pow2i(A);
#pragma unroll
      for (int k = 0; k < 4; ++k) qa[hh][k] = x[k] * sc;
      gu[hh] = 1.5f * pow2i(min(100, max(-100, (int)(yb >> 23) - 127 + A + 15)));
      if (hh == head_mine) {
        cqh = c0 * pow2i(SH - A);
        cbh = c0 * pow2i(-A);
      }
    }
  };
  // head of a dense cursor
  auto head_bk = [&](int64_t h, int64_t &b, int64_t &kvh) {
    b = h / a.Hkv;
    kvh = h - b * a.Hkv;
  };

  // ---- cursors: ic stages unit u0 + kk (ahead), cc computes it
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
  auto cursor_q = [&](const Cursor &c) {
    int64_t b, kvh;
    if constexpr (PAGED) {
      b = c.b;
      kvh = c.kvh;
    } else {
      head_bk(c.h, b, kvh);
    }
    return q_row(b, kvh);
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
  uint32_t armed = 0;  // stages with copies in flight (the same in every lane)
  auto issue = [&](int kk) {
    if (kk >= n_my) return;
    // the last unit of a head holds the token a preceding append just wrote: when
    // this grid was launched as a programmatic dependent of that append, wait for it
    if (a.wait_tail && !waited && ic.uu == ic.U - 1) {
      asm volatile("griddepcontrol.wait;\n" ::: "memory");
      asm volatile("fence.proxy.async;\n" ::: "memory");  // its writes, for the bulk copies too
      waited = true;
    }
    if (ic.uu < ic.ncu) {
      const int g0 = ic.uu * NGU;
      const int ngr = min(NGU, ic.NG - g0);  // 1 or 2 groups (G = 32)
      const int rows = ngr * G;
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
      const int st = kk % S;
      if (lane == 0) {
        const uint32_t bar = bar0 + 8 * st;
        const uint32_t dst = smem_addr(wbase + st * L::kStageBytes);
        const uint32_t cb = (uint32_t)rows * L::kRowBytes;
        asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
        mbar_arm(bar, 2 * cb + (uint32_t)rows * NV * 4 + (uint32_t)ngr * kD * 4);
        bulk_copy(dst + L::kKCodes, a.k_codes + row0 * WPR, cb, bar);
        bulk_copy(dst + L::kVCodes, a.v_codes + row0 * WPR, cb, bar);
        bulk_copy(dst + L::kVMeta, a.v_meta + row0 * NV, (uint32_t)rows * NV * 4, bar);
        bulk_copy(dst + L::kKMeta, a.k_meta + grp0 * kD, (uint32_t)ngr * kD * 4, bar);
      }
      armed |= 1u << st;
    }
    advance(ic);
    if constexpr (PAGED) {
      if (kk + 1 < n_my && ic.uu < ic.ncu) pg_next = page_of(ic.b, ic.uu * kUnit);
    }
  };

  SoftState<NV> ss;
  auto reset_state = [&]() {
    ss.m = -INFINITY;
    ss.l = 0.f;
#pragma unroll
    for (int m = 0; m < NV; ++m) ss.zs[m] = 0.f;
  };
  reset_state();
  float acc[8][4];
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[j][k] = 0.f;

  // Write the partial of head h (this warp's share of it) from the P.V accumulators
  // and the softmax state (m, l, zs) that belongs to them.  acc_true: the
  // accumulators already hold output units (a value residual was added to them).
  bool acc_true = false;
  auto emit = [&](int64_t h, const SoftState<NV> &fin) {
    float l = fin.l, zs[NV];
#pragma unroll
    for (int m = 0; m < NV; ++m) zs[m] = fin.zs[m];
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l += __shfl_xor_sync(kFull, l, off);
#pragma unroll
      for (int m = 0; m < NV; ++m) zs[m] += __shfl_xor_sync(kFull, zs[m], off);
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
      l += __shfl_xor_sync(kFull, l, off);
#pragma unroll
      for (int m = 0; m < NV; ++m) zs[m] += __shfl_xor_sync(kFull, zs[m], off);
#pragma unroll
      for (int j = 0; j < 16; ++j) o[j] += __shfl_xor_sync(kFull, o[j], off);
    }
    if (slot_mine == 0) {
      float *dst;
      if constexpr (SMALL) {
        dst = s_part + (warp * R + head_mine) * (kD + 2);
      } else if constexpr (PAGED) {
        // pair index gw + h grows strictly along the unit order: unique per (warp, head)
        dst = part + ((gw + h) * R + head_mine) * (kD + 2);
      } else {
        const int64_t b = h / a.Hkv, kvh = h - b * a.Hkv;
        const int64_t slot = gw - owner_warp(h * a.units_per_head, W, NW);
        dst = a.ws + ((b * a.Hq + kvh * R + head_mine) * a.pmax + slot) * (kD + 2);
      }
      if constexpr (NV == 1) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          // undo the code factor 4^(j mod 4) (16^(j mod 2)) and the 2^-24 of the subnormal codes
          const float un = acc_true ? 1.f : pow2i(BITS == 2 ? 24 - 2 * (j & 3) : 24 - 4 * (j & 1));
          dst[16 * g + j] = fmaf(o[j], un, zs[0]);
          dst[16 * g + 8 + j] = fmaf(o[8 + j], un, zs[0]);
        }
      } else {
        // accumulator w holds channels 16w + g and 16w + 8 + g (code word w), both with
        // the code factor 4^(g mod 4); word w lies in value group w / WG
        const float un = pow2i(24 - 2 * (g & 3));
#pragma unroll
        for (int w = 0; w < 8; ++w) {
          dst[16 * w + g] = fmaf(o[w], un, zs[w / WG]);
          dst[16 * w + 8 + g] = fmaf(o[8 + w], un, zs[w / WG]);
        }
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

  // The P.V B operand of one round from the weights wa, wb of this lane's two tokens
  // (tokens g and g + 8 of its tile slot): each weight split hi/lo and moved to the
  // lanes whose B registers hold it.
  auto to_b = [&](float wa, float wb, uint32_t &b0, uint32_t &b1) {
    // hi/lo split of the two weights: q1 = {hi_a, lo_a}, q2 = {hi_b, lo_b}
    const __half2 hab = __floats2half2_rn(wa, wb);
    const float2 fab = __half22float2(hab);
    const float2 lo = __fadd2_rn(make_float2(wa, wb), make_float2(-fab.x, -fab.y));
    const __half2 lab = __floats2half2_rn(lo.x, lo.y);
    const uint32_t q1 = prmt(h22u(hab), h22u(lab), 0x5410u);
    const uint32_t q2 = prmt(h22u(hab), h22u(lab), 0x7632u);
    // B of P.V, column g = (slot, head, part): K slots 2tig, 2tig+1, 2tig+8, 2tig+9
    // hold tokens tig, tig+4, tig+8, tig+12; token u's weight lives in lane
    // 4*(u%8) + (g>>1) (first token if u < 8, else second)
    const uint32_t a1 = __shfl_sync(kFull, q1, src_a), b1v = __shfl_sync(kFull, q1, src_b);
    const uint32_t a2 = __shfl_sync(kFull, q2, src_a), b2v = __shfl_sync(kFull, q2, src_b);
    b0 = prmt(a1, b1v, pv_sel);
    b1 = prmt(a2, b2v, pv_sel);
  };

  // One softmax update for a unit: sc[rho] holds the q.K accumulators of this lane's
  // tile slot in round rho (tile rho*T + slot_mine, tokens g and g + 8, hi and lo
  // columns); cq_of(rho), be_of(rho) are that tile's score scale and offset (log2
  // domain), ntok the unit's valid tokens, vmeta(tok, m) the {s, z} word of value
  // group m of its token tok.  With one value group it builds the P.V B operand of
  // every round (bw0, bw1); with several it keeps the weights (pp) for the per-group
  // operands.  Returns the factor alpha that the P.V accumulators need before this
  // unit's contribution is added.
  auto update = [&](auto full_tag, const float (&sc)[R][4], auto &&cq_of, auto &&be_of, int ntok, auto &&vmeta,
                    uint32_t (&bw0)[R], uint32_t (&bw1)[R], float (&pp)[R][2]) -> float {
    constexpr bool FULL = decltype(full_tag)::value;
    float sv[R][2];
    float mloc = -INFINITY;
#pragma unroll
    for (int rho = 0; rho < R; ++rho) {
      const int ta = 16 * (rho * T + slot_mine) + g;
      const bool va = FULL || ta < ntok, vb = FULL || ta + 8 < ntok;
      const float cqv = cq_of(rho), bev = be_of(rho);
      const float2 t = __fadd2_rn(make_float2(sc[rho][0], sc[rho][2]), make_float2(sc[rho][1], sc[rho][3]));
      const float2 sab = __ffma2_rn(make_float2(cqv, cqv), t, make_float2(bev, bev));
      sv[rho][0] = va ? sab.x : -INFINITY;
      sv[rho][1] = vb ? sab.y : -INFINITY;
      mloc = fmaxf(mloc, fmaxf(sv[rho][0], sv[rho][1]));
    }
    const float m_new = fmaxf(ss.m, head_max<R>(mloc));
    const float alpha = ex2(ss.m - m_new);  // ss.m = -inf at the start of a head: alpha = 0
    ss.m = m_new;
    float lsum = 0.f, zsum[NV];
#pragma unroll
    for (int m = 0; m < NV; ++m) zsum[m] = 0.f;
#pragma unroll
    for (int rho = 0; rho < R; ++rho) {
      const int ta = 16 * (rho * T + slot_mine) + g;
      const bool va = FULL || ta < ntok, vb = FULL || ta + 8 < ntok;
      const float pa = ex2(sv[rho][0] - m_new), pb = ex2(sv[rho][1] - m_new);
      lsum += pa + pb;
      if constexpr (NV == 1) {
        const float2 fva = __half22float2(u2h2(vmeta(va ? ta : 0, 0)));
        const float2 fvb = __half22float2(u2h2(vmeta(vb ? ta + 8 : 0, 0)));
        const float sva = va ? fva.x : 0.f, zva = va ? fva.y : 0.f;
        const float svb = vb ? fvb.x : 0.f, zvb = vb ? fvb.y : 0.f;
        zsum[0] = fmaf(pa, zva, fmaf(pb, zvb, zsum[0]));
        const float2 w = __fmul2_rn(make_float2(pa, pb), make_float2(sva, svb));
        to_b(w.x, w.y, bw0[rho], bw1[rho]);
      } else {
        pp[rho][0] = va ? pa : 0.f;
        pp[rho][1] = vb ? pb : 0.f;
#pragma unroll
        for (int m = 0; m < NV; ++m) {
          const float zva = va ? __high2float(u2h2(vmeta(ta, m))) : 0.f;
          const float zvb = vb ? __high2float(u2h2(vmeta(ta + 8, m))) : 0.f;
          zsum[m] = fmaf(pp[rho][0], zva, fmaf(pp[rho][1], zvb, zsum[m]));
        }
      }
    }
    ss.l = fmaf(ss.l, alpha, lsum);
#pragma unroll
    for (int m = 0; m < NV; ++m) ss.zs[m] = fmaf(ss.zs[m], alpha, zsum[m]);
    return alpha;
  };
  // P.V of a unit with value channel groups: the MMA of code word w takes channels
  // 16w + g (row g, the low half of the word) and 16w + 8 + g (row g + 8, the high
  // half) of the lane's four tokens; so one MMA stays inside one value group, and its
  // B operand is p * s of that group.  One prmt pairs two tokens' halves; for g >= 4
  // it takes the upper byte of each half, so that the code lands at bits
  // [2(g mod 4), 2(g mod 4) + 1] of each fp16 half (bits 8 and up are the exponent
  // and sign), and the mask leaves the subnormal code * 4^(g mod 4) * 2^-24.
  // word(tok, w) loads code word w of the unit's token tok, vmeta(tok, m) the {s, z}
  // word of group m.
  auto pv_groups = [&](auto full_tag, int ntok, auto &&word, auto &&vmeta, const float (&pp)[R][2]) {
    constexpr bool FULL = decltype(full_tag)::value;
    const uint32_t M = 0x00030003u << (2 * (g & 3));
    const uint32_t sel_lo = (g & 4) ? 0x5511u : 0x5410u, sel_hi = (g & 4) ? 0x7733u : 0x7632u;
#pragma unroll
    for (int rho = 0; rho < R; ++rho) {
      const int ta = 16 * (rho * T + slot_mine) + g;
      const bool va = FULL || ta < ntok, vb = FULL || ta + 8 < ntok;
#pragma unroll
      for (int m = 0; m < NV; ++m) {
        const float sa = va ? __low2float(u2h2(vmeta(ta, m))) : 0.f;
        const float sb = vb ? __low2float(u2h2(vmeta(ta + 8, m))) : 0.f;
        uint32_t bm0, bm1;
        to_b(pp[rho][0] * sa, pp[rho][1] * sb, bm0, bm1);
#pragma unroll
        for (int i = 0; i < T; ++i) {
          const int t = rho * T + i;
          if (FULL || 16 * t < ntok) {
            const bool mine = pv_slot == i;
            const uint32_t b0 = mine ? bm0 : 0u, b1 = mine ? bm1 : 0u;
#pragma unroll
            for (int ww = 0; ww < WG; ++ww) {
              const int w = WG * m + ww;
              uint32_t v[4];
#pragma unroll
              for (int k = 0; k < 4; ++k) v[k] = word(16 * t + tig + 4 * k, w);
              mma16816(acc[w], prmt(v[0], v[1], sel_lo) & M, prmt(v[0], v[1], sel_hi) & M,
                       prmt(v[2], v[3], sel_lo) & M, prmt(v[2], v[3], sel_hi) & M, b0, b1);
            }
          }
        }
      }
    }
  };
  auto rescale = [&](float alpha) {
    if (__any_sync(kFull, alpha != 1.f)) {
#pragma unroll
      for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[j][k] *= alpha;
    }
  };
  // keep tile slot i's q.K accumulators in out if it is this lane's slot (slot 0
  // initialises out)
  auto keep_slot = [&](int i, const float (&s4)[4], float (&out)[4]) {
#pragma unroll
    for (int k = 0; k < 4; ++k) out[k] = (i == 0 || slot_mine == i) ? s4[k] : out[k];
  };

  // ---- a unit of quantized keys: ntok = 64 tokens, or 32 for a trailing single group
  auto code_unit = [&](auto full_tag, const unsigned char *stg, int ntok) {
    constexpr bool FULL = decltype(full_tag)::value;
    const int ngr = FULL ? NGU : ntok / G;
    // key codes, 2-bit: words 2tig, 2tig+1 of tokens g and g+8 (channels 32tig ..
    // 32tig+31).  With one head all four tiles are in the first round; their codes are
    // loaded before the factor preparation, so that the loads' latency overlaps it.
    auto kcodes = [&](int t, uint2 (&kw)[2]) {
      kw[0] = lds64(stg + L::kKCodes + (16 * t + g) * 32 + tig * 8);
      kw[1] = lds64(stg + L::kKCodes + (16 * t + g + 8) * 32 + tig * 8);
    };
    uint2 kw0[T][2];
    (void)kw0;
    if constexpr (BITS == 2 && R == 1) {
#pragma unroll
      for (int i = 0; i < T; ++i)
        if (FULL || 16 * i < ntok) kcodes(i, kw0[i]);
    }
    // per key group: this lane's scales scaled by 2^-es (every scale of the group lies
    // below 2^(es + 1)), the q . z partials of every head, and the score scale
    float sp[NGU][4], bv[NGU][R], cq[NGU];
#pragma unroll
    for (int gi = 0; gi < NGU; ++gi) {
      if (FULL || gi < ngr) {
        const unsigned char *km = stg + L::kKMeta + gi * kD * 4;
        const uint2 m01 = lds64(km + pc * 4), md = lds64(km + (pc + PD) * 4);
        // non-negative fp16 scales order like their bit patterns
        uint32_t smx = max(max(m01.x & 0xffffu, m01.y & 0xffffu), max(md.x & 0xffffu, md.y & 0xffffu));
        smx = __reduce_max_sync(kFull, smx);
        const int es = (int)(smx >> 10) - 15;
        const float ps = pow2i(-es);
        const float2 v0 = __half22float2(u2h2(m01.x)), v1 = __half22float2(u2h2(md.x));
        const float2 v2 = __half22float2(u2h2(m01.y)), v3 = __half22float2(u2h2(md.y));
        const float2 s01 = __fmul2_rn(make_float2(v0.x, v1.x), make_float2(ps, ps));
        const float2 s23 = __fmul2_rn(make_float2(v2.x, v3.x), make_float2(ps, ps));
        sp[gi][0] = s01.x;
        sp[gi][1] = s01.y;
        sp[gi][2] = s23.x;
        sp[gi][3] = s23.y;
        const float2 z01 = __fmul2_rn(make_float2(v0.y, v1.y), make_float2(ifa, ifa));
        const float2 z23 = __fmul2_rn(make_float2(v2.y, v3.y), make_float2(ifb, ifb));
        const float z0 = z01.x, z1 = z01.y, z2 = z23.x, z3 = z23.y;
#pragma unroll
        for (int hh = 0; hh < R; ++hh)
          bv[gi][hh] = fmaf(qa[hh][3], z3, fmaf(qa[hh][2], z2, fmaf(qa[hh][1], z1, qa[hh][0] * z0)));
        cq[gi] = cqh * pow2i(es);
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) sp[gi][k] = 0.f;
#pragma unroll
        for (int hh = 0; hh < R; ++hh) bv[gi][hh] = 0.f;
        cq[gi] = 0.f;
      }
    }
    beta_reduce<R, NGU>(bv, lane);
    // B fragment of group gi: hi and lo rows of every head
    // The hi parts lie on a grid: the tensor cores add the 16 products of an MMA
    // k-step keeping only about 15 bits below the largest of them, so hi is rounded
    // to a multiple of u_h * f.  Every scaled scale of a group is below 2, so every
    // |x| / f is below 2^(E_h + 2) = 2^10 u_h, every hi product is code * 64 * 2^-24 *
    // (a multiple of u_h) of at most 3 * 2^10 units, and the MMA adds them exactly;
    // lo = x - hi (at most u_h * f / 2) carries the rest in fp16, and its own sums lose
    // at most about 2^-23 of the head's largest entry.
    auto write_frag = [&](int gi) {
      uint32_t *fw = reinterpret_cast<uint32_t *>(frag);
#pragma unroll
      for (int hh = 0; hh < R; ++hh) {
        // paired fp32 operations (each element rounded to nearest, like the scalar ones)
        const float2 xa = __fmul2_rn(make_float2(qa[hh][0], qa[hh][1]), make_float2(sp[gi][0], sp[gi][1]));
        const float2 xb = __fmul2_rn(make_float2(qa[hh][2], qa[hh][3]), make_float2(sp[gi][2], sp[gi][3]));
        // fp32 round to nearest even onto the grid: |x| / (u_h f) < 2^10, far inside
        // the 2^22 that adding and subtracting 1.5 * 2^23 * u_h * f needs
        const float2 m = __fmul2_rn(make_float2(gu[hh], gu[hh]), make_float2(fa, fb));
        const float2 ma = make_float2(m.x, m.x), mb = make_float2(m.y, m.y);
        const float2 ha = __fadd2_rn(__fadd2_rn(xa, ma), make_float2(-ma.x, -ma.y));
        const float2 hb = __fadd2_rn(__fadd2_rn(xb, mb), make_float2(-mb.x, -mb.y));
        const float2 la = __fadd2_rn(xa, make_float2(-ha.x, -ha.y)), lb = __fadd2_rn(xb, make_float2(-hb.x, -hb.y));
        const __half2 hA = __floats2half2_rn(ha.x, ha.y), hB = __floats2half2_rn(hb.x, hb.y);
        const __half2 lA = __floats2half2_rn(la.x, la.y), lB = __floats2half2_rn(lb.x, lb.y);
        *reinterpret_cast<uint2 *>(fw + ((2 * hh) * 4 + pt) * FRW + pword) = make_uint2(h22u(hA), h22u(hB));
        *reinterpret_cast<uint2 *>(fw + ((2 * hh + 1) * 4 + pt) * FRW + pword) = make_uint2(h22u(lA), h22u(lB));
      }
    };
    write_frag(0);
    __syncwarp();
    uint32_t bf[16];
    load_frag(frag + frag_row * FRW * 4, bf);
    // ---- q.K: R rounds of T tiles, tiles in increasing order (group 1 from tile TPG on)
    float sc[R][4];
#pragma unroll
    for (int rho = 0; rho < R; ++rho) {
#pragma unroll
      for (int i = 0; i < T; ++i) {
        const int t = rho * T + i;
        float s4[4] = {0.f, 0.f, 0.f, 0.f};
        if (FULL || 16 * t < ntok) {
          if (NGU == 2 && t == TPG) {
            __syncwarp();  // every lane has its copy of the first group's fragment
            write_frag(1);
            __syncwarp();
            load_frag(frag + frag_row * FRW * 4, bf);
          }
          uint32_t ra0[8], ra1[8], rb0[8], rb1[8];
          if constexpr (BITS == 2) {
            uint2 kw[2];
            if (R == 1) {
              kw[0] = kw0[i][0];
              kw[1] = kw0[i][1];
            } else {
              kcodes(t, kw);
            }
            unpack16(kw[0].x, ra0);
            unpack16(kw[0].y, ra1);
            unpack16(kw[1].x, rb0);
            unpack16(kw[1].y, rb1);
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
          qk_tile(ra0, ra1, rb0, rb1, bf, s4);
        }
        keep_slot(i, s4, sc[rho]);
      }
    }
    // ---- softmax update of the unit
    float be[NGU];
#pragma unroll
    for (int gi = 0; gi < NGU; ++gi) be[gi] = bv[gi][0] * cbh;
    auto grp = [&](int rho) { return NGU == 1 ? 0 : (rho * T + slot_mine) / TPG; };
    uint32_t bw0[R], bw1[R];
    float pp[R][2];
    auto vmeta = [&](int tok, int m) -> uint32_t { return lds32(stg + L::kVMeta + (tok * NV + m) * 4); };
    const float alpha = update(
        full_tag, sc, [&](int rho) { return grp(rho) ? cq[NGU - 1] : cq[0]; },
        [&](int rho) { return grp(rho) ? be[NGU - 1] : be[0]; }, ntok, vmeta, bw0, bw1, pp);
    // ---- P.V of the unit's tiles from the staged value codes
    rescale(alpha);
    if constexpr (NV > 1) {
      pv_groups(full_tag, ntok, [&](int tok, int w) { return lds32(stg + L::kVCodes + tok * 32 + w * 4); }, vmeta,
                pp);
    } else {
#pragma unroll
      for (int rho = 0; rho < R; ++rho)
#pragma unroll
        for (int i = 0; i < T; ++i) {
          const int t = rho * T + i;
          if (FULL || 16 * t < ntok) {
            const bool mine = pv_slot == i;
            const uint32_t b0 = mine ? bw0[rho] : 0u, b1 = mine ? bw1[rho] : 0u;
            if constexpr (BITS == 2) {
              uint32_t v[4];
#pragma unroll
              for (int k = 0; k < 4; ++k) v[k] = lds32(stg + L::kVCodes + (16 * t + tig + 4 * k) * 32 + g * 4);
              pv_tile(acc, v, b0, b1);
            } else {
              uint2 v[4];
#pragma unroll
              for (int k = 0; k < 4; ++k) v[k] = lds64(stg + L::kVCodes + (16 * t + tig + 4 * k) * 64 + g * 8);
              pv_tile4(acc, v, b0, b1);
            }
          }
        }
    }
  };

  // ---- the residual unit of a head: its r fp16 keys (read from the residual buffer)
  // and their values (quantized rows nq .. nq + r - 1, or the fp16 value residual)
  auto residual_unit = [&]() {
    const int r = cc.r;
    const int64_t nq = (int64_t)cc.NG * G;
    const uint16_t *res_head = a.k_res + cc.h * G * kD;
    int64_t vrow;  // value row of token nq (one page: pages hold whole groups)
    if constexpr (PAGED) {
      const int64_t ph = page_of(cc.b, (int)nq) * a.Hkv + cc.kvh;
      vrow = ph * P + (nq & (P - 1));
    } else {
      vrow = cc.h * a.max_tokens + nq;
    }
    // q.K of the fp16 residual keys on the CUDA cores in fp32 (full products and
    // fp32 sums; the tensor cores' narrow addition window would cost precision on keys
    // with outlier channels): lane (g, tig) scores tokens 16t + g and 16t + g + 8 of
    // its tile slot t of every round, for its head.  The hi/lo column pair of the MMA
    // layout becomes (score, 0).
    const uint4 *qp = reinterpret_cast<const uint4 *>(cursor_q(cc) + head_mine * kD);
    float sc[R][4];
#pragma unroll
    for (int rho = 0; rho < R; ++rho) {
      const int sa = 16 * (rho * T + slot_mine) + g, sb = sa + 8;
      const bool va = sa < r, vb = sb < r;
      const uint4 *ka = reinterpret_cast<const uint4 *>(res_head + (va ? sa : 0) * kD);
      const uint4 *kb = reinterpret_cast<const uint4 *>(res_head + (vb ? sb : 0) * kD);
      float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
      if (va || vb) {  // the two keys of the lane share each query load
#pragma unroll 4
        for (int c = 0; c < kD / 8; ++c) {
          const uint4 qq = __ldg(qp + c), xa = __ldg(ka + c), xb = __ldg(kb + c);
          const uint32_t qw[4] = {qq.x, qq.y, qq.z, qq.w}, wa[4] = {xa.x, xa.y, xa.z, xa.w};
          const uint32_t wb[4] = {xb.x, xb.y, xb.z, xb.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 fq = __half22float2(u2h2(qw[i]));
            const float2 fa2 = __half22float2(u2h2(wa[i])), fb2 = __half22float2(u2h2(wb[i]));
            a0 = fmaf(fq.x, fa2.x, a0);
            a1 = fmaf(fq.y, fa2.y, a1);
            b0 = fmaf(fq.x, fb2.x, b0);
            b1 = fmaf(fq.y, fb2.y, b1);
          }
        }
      }
      sc[rho][0] = va ? a0 + a1 : 0.f;
      sc[rho][1] = 0.f;
      sc[rho][2] = vb ? b0 + b1 : 0.f;
      sc[rho][3] = 0.f;
    }
    // residual values are quantized ({s, z} of their row) or, with a value residual,
    // fp16 themselves: weight p with s = 1, z = 0
    const uint32_t *vm_head = a.v_meta + vrow * NV;
    uint32_t bw0[R], bw1[R];
    float pp[R][2];
    auto vmeta = [&](int tok, int m) -> uint32_t { return a.v_res ? 0x00003C00u : __ldg(vm_head + tok * NV + m); };
    const float alpha = update(
        std::false_type{}, sc, [&](int) { return c0; }, [&](int) { return 0.f; }, r, vmeta, bw0, bw1, pp);
    if constexpr (NV > 1) {
      // (value channel groups come without a value residual)
      rescale(alpha);
      const uint32_t *vc_head = a.v_codes + vrow * WPR;
      pv_groups(std::false_type{}, r, [&](int tok, int w) { return __ldg(vc_head + (tok < r ? tok : 0) * WPR + w); },
                vmeta, pp);
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
      rescale(alpha);
      const uint16_t *vres_head = a.v_res + cc.h * G * kD;
#pragma unroll
      for (int rho = 0; rho < R; ++rho)
#pragma unroll
        for (int i = 0; i < T; ++i) {
          const int t = rho * T + i;
          if (16 * t < r) {
            const bool mine = pv_slot == i;
            pv_tile_f16(acc, vres_head + 16 * t * kD, r - 16 * t, g, tig, mine ? bw0[rho] : 0u,
                        mine ? bw1[rho] : 0u);
          }
        }
    } else {
      rescale(alpha);
      const uint32_t *vc_head = a.v_codes + vrow * WPR;
#pragma unroll
      for (int rho = 0; rho < R; ++rho)
#pragma unroll
        for (int i = 0; i < T; ++i) {
          const int t = rho * T + i;
          if (16 * t < r) {
            const bool mine = pv_slot == i;
            const uint32_t b0 = mine ? bw0[rho] : 0u, b1 = mine ? bw1[rho] : 0u;
            if constexpr (BITS == 2) {
              uint32_t v[4];
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const int slot = 16 * t + tig + 4 * k;
                v[k] = vc_head[(slot < r ? slot : 0) * WPR + g];
              }
              pv_tile(acc, v, b0, b1);
            } else {
              uint2 v[4];
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const int slot = 16 * t + tig + 4 * k;
                v[k] = *reinterpret_cast<const uint2 *>(vc_head + (slot < r ? slot : 0) * WPR + 2 * g);
              }
              pv_tile4(acc, v, b0, b1);
            }
          }
        }
    }
  };

  // ---- the warp's units (the first copies go out before the query is loaded, so
  // that the two latencies overlap)
#pragma unroll
  for (int kk = 0; kk < AH; ++kk) issue(kk);
  load_q(cursor_q(cc));
  uint32_t phase = 0;  // parity of each stage's next phase
  bool fault = false;
  for (int kk = 0; kk < n_my; ++kk) {
    issue(kk + AH);  // into the stage of unit kk - 1, which every lane has finished reading
    if constexpr (PAGED) {
      // the warp that takes a head's first unit publishes where its partials go
      if (cc.uu == 0 && lane == 0) {
        const int64_t start = (int64_t)a.Hkv * s_cum[cc.b] + (int64_t)cc.kvh * cc.U;
        const int64_t last = owner_warp(start + cc.U - 1, W, NW);
        hdr[cc.h] = make_int2((int)(gw + cc.h), (int)(last - gw + 1));
      }
    }
    if (cc.uu < cc.ncu) {
      const int st = kk % S;
      if (!mbar_wait(bar0 + 8 * st, (phase >> st) & 1u)) {
        fault = true;
        break;
      }
      phase ^= 1u << st;
      armed &= ~(1u << st);
      const unsigned char *stg = wbase + st * L::kStageBytes;
      if constexpr (NGU == 1) {
        code_unit(std::true_type{}, stg, kUnit);
      } else {
        const int ngr = min(NGU, cc.NG - cc.uu * NGU);  // a trailing single group: 32 tokens
        if (ngr == NGU)
          code_unit(std::true_type{}, stg, kUnit);
        else
          code_unit(std::false_type{}, stg, ngr * G);
      }
    } else {
      residual_unit();
    }
    __syncwarp();  // this unit's stage and the fragment may be rewritten from now on
    if (kk + 1 < n_my) {
      if (cc.uu + 1 == cc.U) {  // the next unit starts a new head
        emit(cc.h, ss);
        reset_state();
        advance(cc);
        load_q(cursor_q(cc));
      } else {
        advance(cc);
      }
    }
  }
  if (fault) {
    // a staged copy never completed: record it, wait (bounded) for this warp's other
    // copies in flight, and stop without writing partials
    if (lane == 0) atomicExch(&g_decode_fault, 1);
#pragma unroll
    for (int s = 0; s < S; ++s)
      if ((armed >> s) & 1u) mbar_wait(bar0 + 8 * s, (phase >> s) & 1u);
  } else {
    emit(cc.h, ss);
  }
  if constexpr (SMALL) small_merge<R, CL, NWARPS>(a, s_part, NW, warp, lane);
}

template <int R, int G, bool PAGED, int BITS, int VG = kD>
__global__ void __launch_bounds__(kThreads, KIVI_DECODE_MIN_CTAS) decode_kernel(const DecodeArgs a) {
  decode_body<R, G, PAGED ? kModePaged : kModeDense, BITS, kWarps, VG>(a);
}

template <int R, int G, int BITS>
__global__ void __launch_bounds__(kSmallWarps * 32, 1) decode_small_kernel(const DecodeArgs a) {
  decode_body<R, G, kModeSmall, BITS, kSmallWarps>(a);
}

// The small path on clusters: CTAs CL * h .. CL * h + CL - 1 of NW warps each form the
// cluster of (batch, KV head) h.
template <int R, int G, int BITS, int CL, int NW>
__global__ void __cluster_dims__(CL, 1, 1) __launch_bounds__(NW * 32, 1) decode_cluster_kernel(const DecodeArgs a) {
  decode_body<R, G, kModeSmall, BITS, NW, kD, CL>(a);
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
  combine_row<false>(ws + row * pmax * (kD + 2), (int)(last - first + 1), kD + 2, out + row * kD, threadIdx.x & 31);
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
  combine_row<false>(part + ((int64_t)hd.x * R + hq % R) * (kD + 2), hd.y, (int64_t)R * (kD + 2), out + row * kD, lane);
  if (advance && hq == 0 && lane == 0) {
    const int32_t len = advance[b];
    advance[b] = len < cap ? len + 1 : cap;
  }
}

template <int R, int G, bool PAGED, int BITS>
const void *kernel_ptr() {
  return reinterpret_cast<const void *>(&decode_kernel<R, G, PAGED, BITS>);
}

// Dense 2-bit kernels with value channel groups of VG channels (persistent grid only).
template <int VG>
const void *select_vg_kernel(int R, int G) {
  if (G == 32)
    return R == 1   ? reinterpret_cast<const void *>(&decode_kernel<1, 32, false, 2, VG>)
           : R == 2 ? reinterpret_cast<const void *>(&decode_kernel<2, 32, false, 2, VG>)
                    : reinterpret_cast<const void *>(&decode_kernel<4, 32, false, 2, VG>);
  return R == 1   ? reinterpret_cast<const void *>(&decode_kernel<1, 64, false, 2, VG>)
         : R == 2 ? reinterpret_cast<const void *>(&decode_kernel<2, 64, false, 2, VG>)
                  : reinterpret_cast<const void *>(&decode_kernel<4, 64, false, 2, VG>);
}

template <int VG>
int vg_smem_bytes(int R, int G) {
  if (G == 32)
    return R == 1 ? Layout<1, 32, 2, VG>::kSmem : R == 2 ? Layout<2, 32, 2, VG>::kSmem : Layout<4, 32, 2, VG>::kSmem;
  return R == 1 ? Layout<1, 64, 2, VG>::kSmem : R == 2 ? Layout<2, 64, 2, VG>::kSmem : Layout<4, 64, 2, VG>::kSmem;
}

template <bool PAGED, int BITS>
const void *select_kernel(int R, int G) {
  if (G == 32)
    return R == 1   ? kernel_ptr<1, 32, PAGED, BITS>()
           : R == 2 ? kernel_ptr<2, 32, PAGED, BITS>()
                    : kernel_ptr<4, 32, PAGED, BITS>();
  return R == 1 ? kernel_ptr<1, 64, PAGED, BITS>() : R == 2 ? kernel_ptr<2, 64, PAGED, BITS>() : kernel_ptr<4, 64, PAGED, BITS>();
}

template <int R, int G, int BITS>
const void *small_ptr() {
  return reinterpret_cast<const void *>(&decode_small_kernel<R, G, BITS>);
}

template <int BITS>
const void *select_small(int R, int G) {
  if (G == 32) return R == 1 ? small_ptr<1, 32, BITS>() : R == 2 ? small_ptr<2, 32, BITS>() : small_ptr<4, 32, BITS>();
  return R == 1 ? small_ptr<1, 64, BITS>() : R == 2 ? small_ptr<2, 64, BITS>() : small_ptr<4, 64, BITS>();
}

template <int R, int G, int BITS, int CL, int NW>
const void *cluster_ptr() {
  return reinterpret_cast<const void *>(&decode_cluster_kernel<R, G, BITS, CL, NW>);
}

template <int BITS, int CL, int NW>
const void *select_cluster(int R, int G) {
  if (G == 32)
    return R == 1   ? cluster_ptr<1, 32, BITS, CL, NW>()
           : R == 2 ? cluster_ptr<2, 32, BITS, CL, NW>()
                    : cluster_ptr<4, 32, BITS, CL, NW>();
  return R == 1 ? cluster_ptr<1, 64, BITS, CL, NW>() : R == 2 ? cluster_ptr<2, 64, BITS, CL, NW>() : cluster_ptr<4, 64, BITS, CL, NW>();
}

// Shared memory of a cluster kernel's CTA: its warps' rings and partials.  A CTA of
// fewer than 8 warps claims more than half of an SM's 228 KB, so that every CTA of a
// cluster has an SM to itself (8 warps of two CTAs on one SM take each unit's compute
// longer).
constexpr int kOwnSmSmem = 116 * 1024;
template <int R, int G, int BITS, int CL, int NW>
constexpr int cluster_smem() {
  constexpr int b = NW * Layout<R, G, BITS>::kWarpBytes + small_part_bytes<R, NW>();
  return NW < 8 && b < kOwnSmSmem ? kOwnSmSmem : b;
}

template <int BITS, int CL, int NW>
int cluster_smem_bytes(int R, int G) {
  if (G == 32)
    return R == 1   ? cluster_smem<1, 32, BITS, CL, NW>()
           : R == 2 ? cluster_smem<2, 32, BITS, CL, NW>()
                    : cluster_smem<4, 32, BITS, CL, NW>();
  return R == 1 ? cluster_smem<1, 64, BITS, CL, NW>() : R == 2 ? cluster_smem<2, 64, BITS, CL, NW>() : cluster_smem<4, 64, BITS, CL, NW>();
}

template <int BITS>
int small_smem_bytes(int R, int G) {
  if (G == 32)
    return R == 1   ? kSmallWarps * Layout<1, 32, BITS>::kWarpBytes + small_part_bytes<1>()
           : R == 2 ? kSmallWarps * Layout<2, 32, BITS>::kWarpBytes + small_part_bytes<2>()
                    : kSmallWarps * Layout<4, 32, BITS>::kWarpBytes + small_part_bytes<4>();
  return R == 1   ? kSmallWarps * Layout<1, 64, BITS>::kWarpBytes + small_part_bytes<1>()
         : R == 2 ? kSmallWarps * Layout<2, 64, BITS>::kWarpBytes + small_part_bytes<2>()
                  : kSmallWarps * Layout<4, 64, BITS>::kWarpBytes + small_part_bytes<4>();
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

DecodeKernels decode_kernels(int R, int G, int bits, bool paged, int B, int vg) {
  DecodeKernels k;
  if (vg != kD) {  // value channel groups: dense 2-bit caches, persistent grid
    k.decode = vg == 64 ? select_vg_kernel<64>(R, G) : select_vg_kernel<32>(R, G);
    k.smem = k.smem_limit = vg == 64 ? vg_smem_bytes<64>(R, G) : vg_smem_bytes<32>(R, G);
    k.combine = reinterpret_cast<const void *>(&combine_kernel);
    k.small = k.pair = k.quad = nullptr;
    k.small_smem = k.pair_smem = k.quad_smem = 0;
    return k;
  }
  const int base = bits == 2 ? smem_bytes<2>(R, G) : smem_bytes<4>(R, G);
  if (paged) {
    k.decode = bits == 2 ? select_kernel<true, 2>(R, G) : select_kernel<true, 4>(R, G);
    k.smem = base + paged_extra(B);
    k.smem_limit = base + paged_extra(kPagedMaxBatch);
    k.combine = reinterpret_cast<const void *>(&paged_combine_kernel);
    k.small = k.pair = k.quad = nullptr;
    k.small_smem = k.pair_smem = k.quad_smem = 0;
  } else {
    k.decode = bits == 2 ? select_kernel<false, 2>(R, G) : select_kernel<false, 4>(R, G);
    k.smem = k.smem_limit = base;
    k.combine = reinterpret_cast<const void *>(&combine_kernel);
    k.small = bits == 2 ? select_small<2>(R, G) : select_small<4>(R, G);
    k.small_smem = bits == 2 ? small_smem_bytes<2>(R, G) : small_smem_bytes<4>(R, G);
    constexpr int PC = kDecodePairCtas, PW = kDecodePairWarps, QC = kDecodeQuadCtas, QW = kDecodeQuadWarps;
    k.pair = bits == 2 ? select_cluster<2, PC, PW>(R, G) : select_cluster<4, PC, PW>(R, G);
    k.pair_smem = bits == 2 ? cluster_smem_bytes<2, PC, PW>(R, G) : cluster_smem_bytes<4, PC, PW>(R, G);
    k.quad = bits == 2 ? select_cluster<2, QC, QW>(R, G) : select_cluster<4, QC, QW>(R, G);
    k.quad_smem = bits == 2 ? cluster_smem_bytes<2, QC, QW>(R, G) : cluster_smem_bytes<4, QC, QW>(R, G);
  }
  return k;
}

}  // namespace kivi
