// kivi_prefill.cu -- fused prefill: causal attention over the fp16 prompt, with the
// KIVI cache quantized from the same key and value tiles while they are on chip
// (sm_103a).
//
// KIVI page ("Makale Bulteni -- KIVI", cmlonder.com radar / paper-to-prod,
// 2026-11-01), section "Kod ve Entegrasyon Haritasi": FlashAttention runs the prompt
// (prefill) attention over the full-precision keys and values, and KIVI quantizes
// the cache that the decode steps read afterwards (keys per channel in G-token
// groups plus an fp16 residual, values per token; headline paragraph and section
// "Iddia ve Gerceklik", paragraphs 2-3).
//
// For every batch b, query head h (reading KV head h / (Hq/Hkv)) and prompt position i:
//   out_i = sum_{j <= i} softmax_j(sigma * q_i . k_j) v_j.
// One CTA of 4 warps takes 64 consecutive query rows of one (b, h), 16 per warp, and
// walks the key/value tiles of 64 tokens up to and including its diagonal tile,
// double-buffered in shared memory by cp.async (rows past the prompt read as zero).
// q.K and P.V run on mma.sync m16n8k16 with fp32 accumulation: q and k are exact fp16
// operands; the probabilities enter P.V as an fp16 pair hi + lo (two MMAs), which
// keeps ~22 significant bits.  The online softmax runs in the log2 domain.
//
// Quantization: the cache of KV head (b, kvh) is written by the CTAs of query head
// kvh * (Hq/Hkv): CTA (qt, b, h) quantizes key/value tile qt, its own diagonal tile
// and the last one it loads, after its attention.  Key groups of G tokens per channel
// (a 64-token tile holds 64/G whole groups), value rows per token, the last n mod G
// keys (and values, with a value residual) copied to the residual buffers.  The
// rounding rule is the library's (kivi_device.cuh: make_qparams, the proven fp16
// thresholds of 2-bit codes with the fp32 comparison form as the fallback, the
// reciprocal product of 4-bit codes), so the cache is bit for bit the one
// kivi_quantize_prefill writes.
#include <math.h>

#include "kivi_device.cuh"
#include "kivi_internal.h"

namespace kivi {

namespace {

constexpr int kPWarps = 4;
constexpr int kPThreads = 32 * kPWarps;
constexpr int kPTile = 64;                    // query rows per CTA, tokens per key/value tile
constexpr int kPRow = 272;                    // padded row: 256 B of fp16 + 16 B (conflict-free ldmatrix)
constexpr int kPTileBytes = kPTile * kPRow;   // one 64-row tile of K or V
constexpr int kPStage = 2 * kPTileBytes;      // K and V
constexpr int kPSmem = 2 * kPStage;           // two stages
constexpr float kPLog2e = 1.4426950408889634f;

__device__ __forceinline__ float pex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void pldsm_x4(const unsigned char *p, uint32_t r[4]) {
  const uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(a));
}

__device__ __forceinline__ void pldsm_x4_t(const unsigned char *p, uint32_t r[4]) {
  const uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(a));
}

// 16-byte copy that writes zeros (and reads nothing) when `valid` is false.
__device__ __forceinline__ void pcp_async16(void *smem, const void *gmem, bool valid) {
  const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
  const int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(n) : "memory");
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) { return h22u(__floats2half2_rn(lo, hi)); }

// Quantize key/value tile t0 / 64 of one (batch, KV head), staged in shared memory as
// 64 rows of kPRow bytes (rows past the prompt hold zeros and are not written).  All
// threads of the CTA take part; `scratch` holds 1 KB.
// Keys: thread (rh, cp) = (tid / 64, tid % 64) holds channels 2cp, 2cp+1 of rows
// 32rh .. 32rh+31 in registers (one whole group for G = 32; with G = 64 the two row
// halves merge their min/max through `scratch`), derives both channels' parameters
// and codes each row, two codes per lane; a transpose across the LPW lanes of a word
// then gives each lane one packed word of one row.  Values: 4 lanes per row, lane
// (q, r8) = (lane / 8, lane % 8) holding channels 32q .. 32q+31 of row r8 of its
// 8-row step, so that the 8 lanes of a shared-memory phase read 8 different rows; a
// value channel group of 32 (64) channels is one lane's (two lanes') channels.
// 2-bit codes come from fp16 thresholds (the per-element fp32 form when a warp holds
// a threshold that is not proven), 4-bit codes from the reciprocal product: the rule
// and its fast forms are those of the standalone quantizers, bit for bit.
template <int BITS>
__device__ void quantize_tile(const PrefillArgs &a, int64_t bh, int64_t t0, const unsigned char *ks,
                              const unsigned char *vs, unsigned char *scratch) {
  constexpr int WPR = words_per_row<BITS>();
  constexpr int LPW = 16 / BITS;  // channel pairs per packed word
  const int G = a.G;
  const int64_t n = a.n, nq = (n / G) * G;
  const int64_t t_end = min(n, t0 + kPTile);
  const int tid = threadIdx.x, lane = tid & 31;

  // ---- key groups
  const int cp = tid & 63, rh = tid >> 6;
  uint32_t x[32];
#pragma unroll
  for (int r = 0; r < 32; ++r) x[r] = *reinterpret_cast<const uint32_t *>(ks + (32 * rh + r) * kPRow + 4 * cp);
  __half2 mn = u2h2(x[0]), mx = mn;
#pragma unroll
  for (int r = 1; r < 32; ++r) {
    mn = __hmin2(mn, u2h2(x[r]));
    mx = __hmax2(mx, u2h2(x[r]));
  }
  if (G == 64) {  // uniform over the CTA
    uint2 *s_mm = reinterpret_cast<uint2 *>(scratch);
    s_mm[tid] = make_uint2(h22u(mn), h22u(mx));
    __syncthreads();
    const uint2 o = s_mm[tid ^ 64];
    mn = __hmin2(mn, u2h2(o.x));
    mx = __hmax2(mx, u2h2(o.y));
  }
  const int64_t g0 = G == 32 ? t0 + 32 * rh : t0;  // first token of this thread's group
  const bool whole = g0 + G <= nq;                  // a quantized group (not the residual)
  key_pair_codes<BITS>(x, mn, mx, lane, whole, (G == 32 || rh == 0),
                       a.k_meta + (bh * (a.max_tokens / G) + g0 / G) * kD + 2 * cp,
                       a.k_codes + (bh * a.max_tokens + t0 + 32 * rh) * WPR + cp / LPW);
  // the residual keys (and values): positions nq .. n - 1 that lie in this tile
  for (int it = tid; it < kPTile * (kD / 8); it += kPThreads) {
    const int r = it / (kD / 8), ch = it - r * (kD / 8);
    const int64_t t = t0 + r;
    if (t < nq || t >= t_end) continue;
    const uint4 xk = *reinterpret_cast<const uint4 *>(ks + r * kPRow + 16 * ch);
    *reinterpret_cast<uint4 *>(a.k_res + (bh * G + (t - nq)) * kD + 8 * ch) = xk;
    if (a.v_res) {
      const uint4 y = *reinterpret_cast<const uint4 *>(vs + r * kPRow + 16 * ch);
      *reinterpret_cast<uint4 *>(a.v_res + (bh * G + (t - nq)) * kD + 8 * ch) = y;
    }
  }
  // ---- value rows
  const int64_t nv = a.v_res ? nq : n;  // values quantized per token
  const int vg = a.vg;                  // channels per value {s, z}: 128, 64 or 32 (2-bit codes)
  const int vq = lane >> 3, vr = lane & 7, warp = tid >> 5;
  for (int r0 = 8 * warp; r0 < kPTile; r0 += 8 * kPWarps) {
    const int r = r0 + vr;
    const int64_t t = t0 + r;
    const bool ok_row = t < nv;
    uint32_t xv[4][4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint4 c = *reinterpret_cast<const uint4 *>(vs + r * kPRow + 16 * (4 * vq + k));
      xv[k][0] = c.x;
      xv[k][1] = c.y;
      xv[k][2] = c.z;
      xv[k][3] = c.w;
    }
    __half2 mn2 = u2h2(xv[0][0]), mx2 = mn2;
#pragma unroll
    for (int k = 0; k < 4; ++k)
#pragma unroll
      for (int e = (k == 0 ? 1 : 0); e < 4; ++e) {
        mn2 = __hmin2(mn2, u2h2(xv[k][e]));
        mx2 = __hmax2(mx2, u2h2(xv[k][e]));
      }
    // (min, -max) so that one __hmin2 reduces both over the row's 4 lanes
    __half2 red = __halves2half2(__hmin(__low2half(mn2), __high2half(mn2)),
                                 __hneg(__hmax(__low2half(mx2), __high2half(mx2))));
    // over the lanes of the row's value group: all 4 lanes (vg = 128), lanes q and
    // q ^ 1 (vg = 64), this lane alone (vg = 32)
    if (vg >= 64) red = __hmin2(red, u2h2(__shfl_xor_sync(0xffffffffu, h22u(red), 8)));
    if (vg == kD) red = __hmin2(red, u2h2(__shfl_xor_sync(0xffffffffu, h22u(red), 16)));
    const QParams p = make_qparams<BITS>(__low2float(red), -__high2float(red));
    uint32_t *row = a.v_codes + (bh * a.max_tokens + t) * WPR;
    if constexpr (BITS == 2) {
      // one set of parameters per row: lane q < 3 of the row proves threshold q + 1 (X2
      // is the strict one: d >= t2); per value group: each lane proves its group's three
      bool ok = true;
      uint32_t x1, x2, x3;
      if (vg == kD) {
        uint32_t xq = 0x7c00u;
        if (p.s != 0.f && vq < 3) xq = fp16_threshold(p.mn, vq == 0 ? p.t1 : (vq == 1 ? p.t2 : p.t3), vq == 1, ok);
        x1 = __shfl_sync(0xffffffffu, xq, vr);
        x2 = __shfl_sync(0xffffffffu, xq, vr + 8);
        x3 = __shfl_sync(0xffffffffu, xq, vr + 16);
      } else {
        fp16_thresholds(p, x1, x2, x3, ok);
      }
      uint32_t c[4];
      if (__all_sync(0xffffffffu, ok)) {
        const uint32_t p1 = x1 | (x1 << 16), p2 = x2 | (x2 << 16), p3 = x3 | (x3 << 16);
        const uint32_t X1[4] = {p1, p1, p1, p1}, X2[4] = {p2, p2, p2, p2}, X3[4] = {p3, p3, p3, p3};
#pragma unroll
        for (int k = 0; k < 4; ++k) c[k] = codes2_chunk8(xv[k], X1, X2, X3);
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) c[k] = quant_chunk8<2>(make_uint4(xv[k][0], xv[k][1], xv[k][2], xv[k][3]), p);
      }
      // chunks 4q .. 4q+3 are words 2q (chunks 4q, 4q+1) and 2q+1
      if (ok_row)
        *reinterpret_cast<uint2 *>(row + 2 * vq) =
            make_uint2((c[0] & 0xffffu) | (c[1] << 16), (c[2] & 0xffffu) | (c[3] << 16));
    } else {
      uint32_t c[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) c[k] = qchunk8<4>(make_uint4(xv[k][0], xv[k][1], xv[k][2], xv[k][3]), p);
      if (ok_row) *reinterpret_cast<uint4 *>(row + 4 * vq) = make_uint4(c[0], c[1], c[2], c[3]);
    }
    if (ok_row && vq % (vg / 32) == 0) a.v_meta[(bh * a.max_tokens + t) * (kD / vg) + vq / (vg / 32)] = p.meta;
  }
}

// Three CTAs (12 warps) per SM: 168 registers, a few spilled in the 2-bit kernels, are
// 1.7% faster on the Llama-2 prompt than 177 registers at two CTAs per SM (measured).
template <int R, int BITS>
__global__ void __launch_bounds__(kPThreads, 3) prefill_kernel(const PrefillArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, tig = lane & 3;
  const int64_t n = a.n;
  const int64_t n_tiles = (n + kPTile - 1) / kPTile;
  const int64_t qt = n_tiles - 1 - blockIdx.x;  // the longest rows first
  const int64_t bq = blockIdx.y;                // b * Hq + h
  const int64_t b = bq / a.Hq, h = bq - b * a.Hq;
  const int64_t bh = b * a.Hkv + h / R;
  const uint16_t *qh = a.q + bq * n * kD;
  const uint16_t *kh = a.k + bh * n * kD;
  const uint16_t *vh = a.v + bh * n * kD;
  const float c0 = a.softmax_scale * kPLog2e;

  // ---- this warp's 16 query rows as A fragments (zero past the prompt)
  const int64_t row_a = qt * kPTile + 16 * warp + g, row_b = row_a + 8;
  uint32_t qa[8][4];
  {
    const uint32_t *qa32 = reinterpret_cast<const uint32_t *>(qh + (row_a < n ? row_a : 0) * kD);
    const uint32_t *qb32 = reinterpret_cast<const uint32_t *>(qh + (row_b < n ? row_b : 0) * kD);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      qa[j][0] = row_a < n ? __ldg(qa32 + 8 * j + tig) : 0u;
      qa[j][1] = row_b < n ? __ldg(qb32 + 8 * j + tig) : 0u;
      qa[j][2] = row_a < n ? __ldg(qa32 + 8 * j + 4 + tig) : 0u;
      qa[j][3] = row_b < n ? __ldg(qb32 + 8 * j + 4 + tig) : 0u;
    }
  }

  auto issue = [&](int64_t kt) {
    unsigned char *ks = smem + (kt & 1) * kPStage;
    unsigned char *vs = ks + kPTileBytes;
    for (int c = threadIdx.x; c < kPTile * 16; c += kPThreads) {
      const int row = c >> 4, ch = c & 15;
      const int64_t tok = kt * kPTile + row;
      const bool ok = tok < n;
      const int64_t src = (ok ? tok : 0) * kD + ch * 8;
      pcp_async16(ks + row * kPRow + ch * 16, kh + src, ok);
      pcp_async16(vs + row * kPRow + ch * 16, vh + src, ok);
    }
    cp_async_commit();
  };

  float o[16][4];
#pragma unroll
  for (int j = 0; j < 16; ++j)
#pragma unroll
    for (int k = 0; k < 4; ++k) o[j][k] = 0.f;
  float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;
  // ldmatrix row addresses: lane (mi = lane/8, r = lane%8)
  const int mi = lane >> 3, rr = lane & 7;

  issue(0);
  for (int64_t kt = 0; kt <= qt; ++kt) {
    if (kt + 1 <= qt) {
      issue(kt + 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const unsigned char *ks = smem + (kt & 1) * kPStage;
    const unsigned char *vs = ks + kPTileBytes;
    // ---- S = q . K over the tile's 64 keys: 8 n-tiles of 8 keys
    float s[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int k = 0; k < 4; ++k) s[nt][k] = 0.f;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {  // two d-steps of 16 per ldmatrix.x4
        uint32_t bk[4];
        pldsm_x4(ks + (8 * nt + rr) * kPRow + (32 * kk + 8 * mi) * 2, bk);
        mma16816(s[nt], qa[2 * kk][0], qa[2 * kk][1], qa[2 * kk][2], qa[2 * kk][3], bk[0], bk[1]);
        mma16816(s[nt], qa[2 * kk + 1][0], qa[2 * kk + 1][1], qa[2 * kk + 1][2], qa[2 * kk + 1][3], bk[2], bk[3]);
      }
    }
    // ---- scale, causal mask on the diagonal tile, online softmax (rows a = g, b = g+8)
    const bool diag = kt == qt;
    float mx_a = -INFINITY, mx_b = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const int64_t key = kt * kPTile + 8 * nt + 2 * tig;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        s[nt][e] = (diag && key + e > row_a) ? -INFINITY : c0 * s[nt][e];
        s[nt][2 + e] = (diag && key + e > row_b) ? -INFINITY : c0 * s[nt][2 + e];
        mx_a = fmaxf(mx_a, s[nt][e]);
        mx_b = fmaxf(mx_b, s[nt][2 + e]);
      }
    }
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
      mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, off));
      mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, off));
    }
    const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
    const float al_a = pex2(m_a - mn_a), al_b = pex2(m_b - mn_b);  // 0 on the first tile
    m_a = mn_a;
    m_b = mn_b;
    l_a *= al_a;
    l_b *= al_b;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      o[j][0] *= al_a;
      o[j][1] *= al_a;
      o[j][2] *= al_b;
      o[j][3] *= al_b;
    }
    // P as A fragments, hi and lo parts: k-step kk (keys 16kk .. 16kk+15) from n-tiles 2kk, 2kk+1
    uint32_t ph[4][4], pl[4][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const float p0 = pex2(s[nt][0] - m_a), p1 = pex2(s[nt][1] - m_a);
      const float p2 = pex2(s[nt][2] - m_b), p3 = pex2(s[nt][3] - m_b);
      l_a += p0 + p1;
      l_b += p2 + p3;
      const __half2 hA = __floats2half2_rn(p0, p1), hB = __floats2half2_rn(p2, p3);
      const float2 fA = __half22float2(hA), fB = __half22float2(hB);
      const int kk = nt >> 1, half = (nt & 1) * 2;
      ph[kk][half] = h22u(hA);
      ph[kk][half + 1] = h22u(hB);
      pl[kk][half] = pack_h2(p0 - fA.x, p1 - fA.y);
      pl[kk][half + 1] = pack_h2(p2 - fB.x, p3 - fB.y);
    }
    // ---- O += P . V: k-step kk (16 keys), 16 d-tiles of 8 channels (two per ldmatrix.x4)
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
      for (int dt = 0; dt < 8; ++dt) {
        uint32_t bv[4];
        pldsm_x4_t(vs + (16 * kk + (mi & 1) * 8 + rr) * kPRow + (16 * dt + (mi >> 1) * 8) * 2, bv);
        // A = P: rows g / g+8, k-slots: {ph[kk][0], ph[kk][1], ph[kk][2], ph[kk][3]}
        mma16816(o[2 * dt], ph[kk][0], ph[kk][1], ph[kk][2], ph[kk][3], bv[0], bv[1]);
        mma16816(o[2 * dt], pl[kk][0], pl[kk][1], pl[kk][2], pl[kk][3], bv[0], bv[1]);
        mma16816(o[2 * dt + 1], ph[kk][0], ph[kk][1], ph[kk][2], ph[kk][3], bv[2], bv[3]);
        mma16816(o[2 * dt + 1], pl[kk][0], pl[kk][1], pl[kk][2], pl[kk][3], bv[2], bv[3]);
      }
    }
    __syncthreads();  // the stage may be refilled from now on
  }
  // ---- normalise and write the rows of this warp
#pragma unroll
  for (int off = 1; off < 4; off <<= 1) {
    l_a += __shfl_xor_sync(0xffffffffu, l_a, off);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, off);
  }
  const float ia = 1.f / l_a, ib = 1.f / l_b;
  if (row_a < n) {
    uint32_t *dst = reinterpret_cast<uint32_t *>(a.out + (bq * n + row_a) * kD);
#pragma unroll
    for (int j = 0; j < 16; ++j) dst[4 * j + tig] = pack_h2(o[j][0] * ia, o[j][1] * ia);
  }
  if (row_b < n) {
    uint32_t *dst = reinterpret_cast<uint32_t *>(a.out + (bq * n + row_b) * kD);
#pragma unroll
    for (int j = 0; j < 16; ++j) dst[4 * j + tig] = pack_h2(o[j][2] * ib, o[j][3] * ib);
  }
  // ---- the cache: the first query head of a KV head quantizes its diagonal tile,
  // still staged in shared memory (the last tile it loaded)
  if (a.k_codes && h % R == 0) {
    const unsigned char *ks = smem + (qt & 1) * kPStage;
    unsigned char *scratch = smem + ((qt + 1) & 1) * kPStage;
    quantize_tile<BITS>(a, bh, qt * kPTile, ks, ks + kPTileBytes, scratch);
  }
}

template <int BITS>
cudaError_t launch_bits(const PrefillArgs &a, cudaStream_t st) {
  const int R = a.Hq / a.Hkv;
  const void *fn = R == 1   ? reinterpret_cast<const void *>(&prefill_kernel<1, BITS>)
                   : R == 2 ? reinterpret_cast<const void *>(&prefill_kernel<2, BITS>)
                            : reinterpret_cast<const void *>(&prefill_kernel<4, BITS>);
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kPSmem);
  if (e != cudaSuccess) return e;
  const int64_t n_tiles = (a.n + kPTile - 1) / kPTile;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)n_tiles, (unsigned)((int64_t)a.B * a.Hq));
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = kPSmem;
  cfg.stream = st;
  void *args[] = {const_cast<PrefillArgs *>(&a)};
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace

cudaError_t launch_prefill_attention(const PrefillArgs &a, cudaStream_t st) {
  return a.bits == 4 ? launch_bits<4>(a, st) : launch_bits<2>(a, st);
}

}  // namespace kivi
