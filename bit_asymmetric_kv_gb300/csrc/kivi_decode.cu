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
//   * the 8 MMA columns are (query head r, hi/lo part) = 2r + part.
// Tokens are tiled by 16 (the MMA M dimension for q.K, the K dimension for P.V).
// Each CTA covers one context split of one (batch, KV head); its 4 warps take the
// split's key groups round-robin, staging each group (codes, scales, zeros) into
// shared memory with cp.async three groups ahead.  The last split also covers the
// fp16 residual keys.  Partial (max, sum, output) per split go to the workspace and
// a combine kernel merges the splits (flash-decoding).
#include <math.h>

#include "kivi_device.cuh"
#include "kivi_internal.h"

namespace kivi {

namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 3;
constexpr int kFragRowWords = 20;                    // 16 B-fragment words + 4 pad (bank spread)
constexpr int kFragBytes = 32 * kFragRowWords * 4;   // per warp
constexpr float kLog2e = 1.4426950408889634f;

template <int G>
struct Stage {
  static constexpr int kKCodes = 0;                  // G rows x 32 B
  static constexpr int kVCodes = G * 32;             // G rows x 32 B
  static constexpr int kVMeta = 2 * G * 32;          // G x 4 B
  static constexpr int kKMeta = 2 * G * 32 + G * 4;  // 128 x 4 B
  static constexpr int kBytes = kKMeta + kD * 4;
  static constexpr int kWarpBytes = kStages * kBytes + kFragBytes;
  static constexpr int kSmem = kWarps * kWarpBytes;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint2 lds64(const unsigned char *p) { return *reinterpret_cast<const uint2 *>(p); }
__device__ __forceinline__ uint32_t lds32(const unsigned char *p) { return *reinterpret_cast<const uint32_t *>(p); }

// Per-warp running softmax state and P.V accumulators.  Lane (g, tig) owns query
// head tig: acc[j] = O[channel 16g+j | 16g+8+j][head tig, hi | lo].
struct WarpState {
  float acc[8][4];
  float m;     // running max, log2 domain
  float l;     // this lane's share of sum_t p_t
  float zs;    // this lane's share of sum_t p_t z_t
};

// Online softmax over one 16-token tile, then P.V on the tensor cores.
//   sa, sb   : log2-domain scores of tokens g and g+8 for head tig (-inf if masked)
//   vma, vmb : {s, z} words of those tokens (ignored where masked)
//   v[4]     : word g of the value rows of tokens tig, tig+4, tig+8, tig+12
__device__ __forceinline__ void softmax_pv(WarpState &st, float sa, float sb, bool va, bool vb, uint32_t vma,
                                           uint32_t vmb, const uint32_t v[4], int lane) {
  const int g = lane >> 2, tig = lane & 3;
  float tmax = fmaxf(sa, sb);
  tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 4));
  tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 8));
  tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 16));
  const float m_new = fmaxf(st.m, tmax);
  if (__any_sync(0xffffffffu, m_new > st.m)) {
    const float alpha = ex2(st.m - m_new);  // st.m = -inf at the start: alpha = 0
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int k = 0; k < 4; ++k) st.acc[j][k] *= alpha;
    st.l *= alpha;
    st.zs *= alpha;
    st.m = m_new;
  }
  const float pa = va ? ex2(sa - st.m) : 0.f;
  const float pb = vb ? ex2(sb - st.m) : 0.f;
  const float sva = va ? h2f((uint16_t)(vma & 0xffffu)) : 0.f, zva = va ? h2f((uint16_t)(vma >> 16)) : 0.f;
  const float svb = vb ? h2f((uint16_t)(vmb & 0xffffu)) : 0.f, zvb = vb ? h2f((uint16_t)(vmb >> 16)) : 0.f;
  st.l += pa + pb;
  st.zs = fmaf(pa, zva, fmaf(pb, zvb, st.zs));
  const float wa = pa * sva, wb = pb * svb;
  const uint16_t ha = f2h(wa), hb = f2h(wb);
  const uint16_t la = f2h(wa - h2f(ha)), lb = f2h(wb - h2f(hb));
  const uint32_t q1 = (uint32_t)ha | ((uint32_t)la << 16);
  const uint32_t q2 = (uint32_t)hb | ((uint32_t)lb << 16);
  // B operand of P.V: column g = (head g/2, part g%2); K slots 2tig, 2tig+1,
  // 2tig+8, 2tig+9 hold tokens tig, tig+4, tig+8, tig+12.  Token u's weight for
  // head h lives in lane 4*(u%8) + h (first token if u < 8, second otherwise).
  const int src_a = 4 * tig + (g >> 1);
  const int src_b = src_a + 16;
  const uint32_t a1 = __shfl_sync(0xffffffffu, q1, src_a);
  const uint32_t b1 = __shfl_sync(0xffffffffu, q1, src_b);
  const uint32_t a2 = __shfl_sync(0xffffffffu, q2, src_a);
  const uint32_t b2 = __shfl_sync(0xffffffffu, q2, src_b);
  const uint32_t sel = (g & 1) ? 0x7632u : 0x5410u;
  const uint32_t bw0 = prmt(a1, b1, sel), bw1 = prmt(a2, b2, sel);
  // A operand of P.V: rows = channels 16g + j (from the low 16 bits of word g) and
  // 16g + 8 + j (high 16 bits), columns = the four tokens paired as above.
  uint32_t x01[8], y01[8], x23[8], y23[8];
  unpack16(prmt(v[0], v[1], 0x5410u), x01);
  unpack16(prmt(v[0], v[1], 0x7632u), y01);
  unpack16(prmt(v[2], v[3], 0x5410u), x23);
  unpack16(prmt(v[2], v[3], 0x7632u), y23);
#pragma unroll
  for (int j = 0; j < 8; ++j) mma16816(st.acc[j], x01[j], y01[j], x23[j], y23[j], bw0, bw1);
}

// q.K of one 16-token tile from unpacked A registers: ra* for token g, rb* for
// token g+8, words 2tig (…0) and 2tig+1 (…1).  Returns the 4 accumulator values.
__device__ __forceinline__ void qk_tile(const uint32_t ra0[8], const uint32_t ra1[8], const uint32_t rb0[8],
                                        const uint32_t rb1[8], const uint32_t bf[16], float sc[4]) {
  float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    mma16816(s0, ra0[2 * j], rb0[2 * j], ra0[2 * j + 1], rb0[2 * j + 1], bf[2 * j], bf[2 * j + 1]);
    mma16816(s1, ra1[2 * j], rb1[2 * j], ra1[2 * j + 1], rb1[2 * j + 1], bf[8 + 2 * j], bf[8 + 2 * j + 1]);
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) sc[k] = s0[k] + s1[k];
}

// Channel c's place in the q.K B fragment: lane row 4*col + tig, word 2j + (c odd),
// half (c mod 16 >= 8).  Word w of a token row feeds MMA steps 4*(w&1) .. +3 of the
// lanes with tig = w >> 1.
__device__ __forceinline__ int frag_half_index(int c, int col) {
  const int W = c >> 4, i = c & 15, i8 = i & 7;
  const int tig = W >> 1;
  const int j = 4 * (W & 1) + (i8 >> 1);
  const int word = 2 * j + (i8 & 1);
  return (4 * col + tig) * (kFragRowWords * 2) + word * 2 + (i >= 8 ? 1 : 0);
}

template <int R>
__device__ __forceinline__ void load_frag(const unsigned char *frag, int lane, uint32_t bf[16]) {
  const int g = lane >> 2;
  if (g < 2 * R) {
    const uint4 *p = reinterpret_cast<const uint4 *>(frag + lane * kFragRowWords * 4);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint4 u = p[k];
      bf[4 * k] = u.x;
      bf[4 * k + 1] = u.y;
      bf[4 * k + 2] = u.z;
      bf[4 * k + 3] = u.w;
    }
  } else {
#pragma unroll
    for (int k = 0; k < 16; ++k) bf[k] = 0u;
  }
}

template <int R, int G>
__global__ void __launch_bounds__(kThreads) decode_kernel(const DecodeArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  using S = Stage<G>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, tig = lane & 3;
  const int split = blockIdx.x;
  const int64_t bh = blockIdx.y;
  const int b = (int)(bh / a.Hkv), kvh = (int)(bh % a.Hkv);
  const int64_t n_groups = a.n / G;
  const int64_t nq = n_groups * G;
  const int r = (int)(a.n - nq);
  const int64_t gb = (int64_t)split * a.groups_per_split;
  const int64_t ge = min(n_groups, gb + a.groups_per_split);
  const bool last = split == a.splits - 1;

  unsigned char *wbase = smem + warp * S::kWarpBytes;
  unsigned char *frag = wbase + kStages * S::kBytes;
  uint16_t *frag16 = reinterpret_cast<uint16_t *>(frag);

  // this lane's query values for channels lane + 32k, heads r < R (fp32, exact)
  float qv[R][4];
#pragma unroll
  for (int h = 0; h < R; ++h)
#pragma unroll
    for (int k = 0; k < 4; ++k) qv[h][k] = h2f(a.q[((int64_t)b * a.Hq + kvh * R + h) * kD + lane + 32 * k]);
  // even channels meet codes unpacked with factor 1, odd channels with factor 4;
  // both carry 2^-24.  B = qs * (4 | 1) makes every product code * qs * 2^-22.
  const float fac = (lane & 1) ? 1.f : 4.f;
  const float c_q = a.softmax_scale * kLog2e * 4194304.f;  // 2^22
  const float c_b = a.softmax_scale * kLog2e;

  WarpState st;
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int k = 0; k < 4; ++k) st.acc[j][k] = 0.f;
  st.m = -INFINITY;
  st.l = 0.f;
  st.zs = 0.f;

  const int64_t first = gb + warp;
  const int n_my = (first < ge) ? (int)((ge - first + kWarps - 1) / kWarps) : 0;
  const uint32_t *kc_head = a.k_codes + bh * a.max_tokens * kWordsPerRow;
  const uint32_t *vc_head = a.v_codes + bh * a.max_tokens * kWordsPerRow;
  const uint32_t *vm_head = a.v_meta + bh * a.max_tokens;
  const uint32_t *km_head = a.k_meta + bh * (a.max_tokens / G) * kD;

  auto issue = [&](int kk) {
    if (kk < n_my) {
      const int64_t grp = first + (int64_t)kk * kWarps;
      unsigned char *stg = wbase + (kk % kStages) * S::kBytes;
      const unsigned char *kc = reinterpret_cast<const unsigned char *>(kc_head + grp * G * kWordsPerRow);
      const unsigned char *vc = reinterpret_cast<const unsigned char *>(vc_head + grp * G * kWordsPerRow);
      const unsigned char *vm = reinterpret_cast<const unsigned char *>(vm_head + grp * G);
      const unsigned char *km = reinterpret_cast<const unsigned char *>(km_head + grp * kD);
#pragma unroll
      for (int c = lane; c < G * 2; c += 32) {
        cp_async16(stg + S::kKCodes + c * 16, kc + c * 16);
        cp_async16(stg + S::kVCodes + c * 16, vc + c * 16);
      }
      if (lane < G / 4) cp_async16(stg + S::kVMeta + lane * 16, vm + lane * 16);
      cp_async16(stg + S::kKMeta + lane * 16, km + lane * 16);
    }
    cp_async_commit();
  };

#pragma unroll
  for (int kk = 0; kk < kStages - 1; ++kk) issue(kk);

  for (int kk = 0; kk < n_my; ++kk) {
    issue(kk + kStages - 1);
    cp_async_wait<kStages - 1>();
    __syncwarp();
    const unsigned char *stg = wbase + (kk % kStages) * S::kBytes;

    // ---- per-group B fragment: qs * fac split into hi/lo, and beta = q . z
    float beta[R];
#pragma unroll
    for (int h = 0; h < R; ++h) beta[h] = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int c = lane + 32 * k;
      const uint32_t mt = lds32(stg + S::kKMeta + c * 4);
      const float s = h2f((uint16_t)(mt & 0xffffu)), z = h2f((uint16_t)(mt >> 16));
#pragma unroll
      for (int h = 0; h < R; ++h) {
        const float x = qv[h][k] * s * fac;
        const uint16_t hi = f2h(x);
        const uint16_t lo = f2h(x - h2f(hi));
        frag16[frag_half_index(c, 2 * h)] = hi;
        frag16[frag_half_index(c, 2 * h + 1)] = lo;
        beta[h] = fmaf(qv[h][k], z, beta[h]);
      }
    }
    float beta_mine = 0.f;
#pragma unroll
    for (int h = 0; h < R; ++h) {
      float v = beta[h];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      if (tig == h) beta_mine = v;
    }
    const float beta2 = c_b * beta_mine;
    __syncwarp();
    uint32_t bf[16];
    load_frag<R>(frag, lane, bf);

#pragma unroll
    for (int i = 0; i < G / 16; ++i) {
      const uint2 ka = lds64(stg + S::kKCodes + (16 * i + g) * 32 + tig * 8);
      const uint2 kb = lds64(stg + S::kKCodes + (16 * i + g + 8) * 32 + tig * 8);
      uint32_t ra0[8], ra1[8], rb0[8], rb1[8];
      unpack16(ka.x, ra0);
      unpack16(ka.y, ra1);
      unpack16(kb.x, rb0);
      unpack16(kb.y, rb1);
      float sc[4];
      qk_tile(ra0, ra1, rb0, rb1, bf, sc);
      const float sa = fmaf(c_q, sc[0] + sc[1], beta2);
      const float sb = fmaf(c_q, sc[2] + sc[3], beta2);
      const uint32_t vma = lds32(stg + S::kVMeta + (16 * i + g) * 4);
      const uint32_t vmb = lds32(stg + S::kVMeta + (16 * i + g + 8) * 4);
      uint32_t v[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) v[k] = lds32(stg + S::kVCodes + (16 * i + tig + 4 * k) * 32 + g * 4);
      softmax_pv(st, sa, sb, true, true, vma, vmb, v, lane);
    }
    __syncwarp();
  }
  cp_async_wait<0>();

  // ---- fp16 residual keys (last split only): B = q itself (hi part, lo = 0)
  if (last && r > 0) {
    const int n_tiles = (r + 15) / 16;
    if (warp < n_tiles) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int c = lane + 32 * k;
#pragma unroll
        for (int h = 0; h < R; ++h) {
          frag16[frag_half_index(c, 2 * h)] = f2h(qv[h][k]);
          frag16[frag_half_index(c, 2 * h + 1)] = 0;
        }
      }
      __syncwarp();
      uint32_t bf[16];
      load_frag<R>(frag, lane, bf);
      const float c_r = a.softmax_scale * kLog2e;
      const uint16_t *res_head = a.k_res + bh * G * kD;
      for (int i = warp; i < n_tiles; i += kWarps) {
        const int sa_slot = 16 * i + g, sb_slot = 16 * i + g + 8;
        const bool va = sa_slot < r, vb = sb_slot < r;
        uint32_t ra0[8], ra1[8], rb0[8], rb1[8];
        // 32 fp16 keys (channels 32tig .. 32tig+31) of each token, paired (m, m+8)
        auto load_pairs = [&](int slot, bool valid, uint32_t r0[8], uint32_t r1[8]) {
          uint32_t p[16];
          if (valid) {
            const uint4 *src = reinterpret_cast<const uint4 *>(res_head + (int64_t)slot * kD + 32 * tig);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint4 u = __ldg(src + k);
              p[4 * k] = u.x;
              p[4 * k + 1] = u.y;
              p[4 * k + 2] = u.z;
              p[4 * k + 3] = u.w;
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
        };
        load_pairs(sa_slot, va, ra0, ra1);
        load_pairs(sb_slot, vb, rb0, rb1);
        float sc[4];
        qk_tile(ra0, ra1, rb0, rb1, bf, sc);
        const float sa = va ? c_r * (sc[0] + sc[1]) : -INFINITY;
        const float sb = vb ? c_r * (sc[2] + sc[3]) : -INFINITY;
        const int64_t t_a = nq + (va ? sa_slot : 0), t_b = nq + (vb ? sb_slot : 0);
        const uint32_t vma = vm_head[t_a], vmb = vm_head[t_b];
        uint32_t v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int slot = 16 * i + tig + 4 * k;
          const int64_t t = nq + (slot < r ? slot : 0);
          v[k] = vc_head[t * kWordsPerRow + g];
        }
        softmax_pv(st, sa, sb, va, vb, vma, vmb, v, lane);
      }
    }
  }

  // ---- per-warp totals, then merge the 4 warps in shared memory
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    st.l += __shfl_xor_sync(0xffffffffu, st.l, off);
    st.zs += __shfl_xor_sync(0xffffffffu, st.zs, off);
  }
  __syncthreads();  // every warp is done with its stages: reuse them for the merge
  float *mrg = reinterpret_cast<float *>(smem);  // [warp][R][kD + 2]
  if (tig < R) {
    float *row = mrg + (warp * R + tig) * (kD + 2);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      // undo the code factor (4 for odd j) and the 2^-24 of the subnormal codes
      const float un = (j & 1) ? 4194304.f : 16777216.f;
      row[16 * g + j] = fmaf(st.acc[j][0] + st.acc[j][1], un, st.zs);
      row[16 * g + 8 + j] = fmaf(st.acc[j][2] + st.acc[j][3], un, st.zs);
    }
    if (g == 0) {
      row[kD] = st.m;
      row[kD + 1] = st.l;
    }
  }
  __syncthreads();
  const int c = threadIdx.x;  // one output channel per thread
#pragma unroll
  for (int h = 0; h < R; ++h) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, mrg[(w * R + h) * (kD + 2) + kD]);
    float L = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float *row = mrg + (w * R + h) * (kD + 2);
      const float sc = (row[kD] == -INFINITY) ? 0.f : ex2(row[kD] - M);
      L = fmaf(sc, row[kD + 1], L);
      O = fmaf(sc, row[c], O);
    }
    float *dst = a.ws + (((int64_t)b * a.Hq + kvh * R + h) * a.splits + split) * (kD + 2);
    dst[c] = O;
    if (c == 0) {
      dst[kD] = M;
      dst[kD + 1] = L;
    }
  }
}

// Merge the per-split partials of one (batch, query head): one thread per channel.
__global__ void __launch_bounds__(128) combine_kernel(const float *__restrict__ ws, int splits,
                                                      uint16_t *__restrict__ out) {
  const int64_t row = blockIdx.x;  // b * Hq + h
  const int c = threadIdx.x;
  const float *p = ws + row * splits * (kD + 2);
  float M = -INFINITY;
  for (int s = 0; s < splits; ++s) M = fmaxf(M, p[s * (kD + 2) + kD]);
  float L = 0.f, O = 0.f;
  for (int s = 0; s < splits; ++s) {
    const float m = p[s * (kD + 2) + kD];
    const float sc = (m == -INFINITY) ? 0.f : ex2(m - M);
    L = fmaf(sc, p[s * (kD + 2) + kD + 1], L);
    O = fmaf(sc, p[s * (kD + 2) + c], O);
  }
  out[row * kD + c] = f2h(O / L);
}

template <int R, int G>
cudaError_t launch_rg(const DecodeArgs &a, cudaStream_t st) {
  const int smem = Stage<G>::kSmem;
  cudaError_t e = cudaFuncSetAttribute(decode_kernel<R, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)a.splits, (unsigned)(a.B * a.Hkv));
  decode_kernel<R, G><<<grid, kThreads, smem, st>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  combine_kernel<<<(unsigned)(a.B * a.Hq), 128, 0, st>>>(a.ws, a.splits, a.out);
  return cudaGetLastError();
}

}  // namespace

void decode_plan(int B, int Hkv, int G, int64_t n, int num_sms, int *splits, int *groups_per_split) {
  const int64_t n_groups = n / G;
  if (n_groups == 0) {
    *splits = 1;
    *groups_per_split = 1;
    return;
  }
  const int64_t heads = (int64_t)B * Hkv;
  const int64_t target_ctas = (int64_t)num_sms * 8;
  int64_t s = (target_ctas + heads - 1) / heads;
  const int64_t s_max = (n_groups + kWarps - 1) / kWarps;  // at least ~one group per warp
  if (s > s_max) s = s_max;
  if (s < 1) s = 1;
  int64_t gps = (n_groups + s - 1) / s;
  gps = (gps + kWarps - 1) / kWarps * kWarps;
  s = (n_groups + gps - 1) / gps;
  *splits = (int)s;
  *groups_per_split = (int)gps;
}

cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t st) {
  const int R = a.Hq / a.Hkv;
  if (a.G == 32) {
    if (R == 1) return launch_rg<1, 32>(a, st);
    if (R == 2) return launch_rg<2, 32>(a, st);
    return launch_rg<4, 32>(a, st);
  }
  if (R == 1) return launch_rg<1, 64>(a, st);
  if (R == 2) return launch_rg<2, 64>(a, st);
  return launch_rg<4, 64>(a, st);
}

}  // namespace kivi
