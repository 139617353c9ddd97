// kivi_fp16.cu -- decode attention over an unquantized fp16 KV cache (sm_103a).
//
// The comparison point for the 2-bit cache: the same decode step (score = sigma *
// q.K, online softmax, out = sum p V, split-K with a final merge) over fp16 keys and
// values [B][Hkv][n][128], as in the long-context fp16-KV decode that the KIVI page
// ("Makale Bulteni -- KIVI", section "Makale Bulteni") measures its memory savings
// against.  It reads 512 bytes per token per KV head, 6-7x the 2-bit cache.
//
// Layout of the work: one CTA per (context split, batch x KV head); its 4 warps take
// the split's 16-token tiles round-robin, each staging its tiles (16 key rows + 16
// value rows, padded to 272 bytes so ldmatrix is conflict-free) in a 3-deep cp.async
// ring.  q.K and P.V run on mma.sync m16n8k16 with ldmatrix fragments (ldmatrix
// .trans for the P.V operand V^T).  The B operand of q.K is q itself (exact fp16);
// the P.V weights enter as hi/lo fp16 pairs in two columns per query head.
#include <math.h>

#include "kivi_device.cuh"
#include "kivi_internal.h"

namespace kivi {

namespace {

constexpr int kWarps16 = 4;
constexpr int kStages16 = 3;
constexpr int kRow = 272;                    // padded row: 256 B of fp16 + 16 B
constexpr int kStage16 = 2 * 16 * kRow;      // 16 key rows + 16 value rows
constexpr int kSmem16 = kWarps16 * kStages16 * kStage16;
constexpr float kLog2e16 = 1.4426950408889634f;

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void ldsm_x4(const unsigned char *p, uint32_t r[4]) {
  const uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(a));
}

__device__ __forceinline__ void ldsm_x4_t(const unsigned char *p, uint32_t r[4]) {
  const uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(a));
}

// 16-byte copy that writes zeros (and reads nothing) when `valid` is false.
__device__ __forceinline__ void cp_async16_zfill(void *smem, const void *gmem, bool valid) {
  const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
  const int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(n) : "memory");
}

template <int R>
__global__ void __launch_bounds__(kWarps16 * 32) fp16_decode_kernel(const Fp16Args a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, tig = lane & 3;
  const int split = blockIdx.x;
  const int64_t bh = blockIdx.y;
  const int64_t b = bh / a.Hkv, kvh = bh - b * a.Hkv;
  const int64_t n = a.n;
  const int64_t n_tiles = (n + 15) / 16;
  const int64_t t_begin = (int64_t)split * a.tiles_per_split;
  const int64_t t_end = min(n_tiles, t_begin + a.tiles_per_split);
  const int64_t first = t_begin + warp;
  const int n_my = first < t_end ? (int)((t_end - first + kWarps16 - 1) / kWarps16) : 0;
  const uint16_t *kh = a.k + bh * n * kD;
  const uint16_t *vh = a.v + bh * n * kD;
  unsigned char *wbase = smem + warp * kStages16 * kStage16;
  const float c0 = a.softmax_scale * kLog2e16;

  // B of q.K: column g = (head g/2, part g%2); part 1 (lo) is zero since q is exact
  uint32_t bq[16];
  {
    const int h = g >> 1;
    const bool use = (g & 1) == 0 && h < R;
    const uint32_t *q32 = reinterpret_cast<const uint32_t *>(a.q + ((b * a.Hq) + kvh * R + (use ? h : 0)) * kD);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      bq[2 * j] = use ? q32[8 * j + tig] : 0u;
      bq[2 * j + 1] = use ? q32[8 * j + 4 + tig] : 0u;
    }
  }
  const int src_a = 8 * tig + (g >> 1), src_b = src_a + 4;
  const uint32_t pv_sel = (g & 1) ? 0x7632u : 0x5410u;
  // ldmatrix row addresses: lane (mi = lane/8, r = lane%8)
  const int mi = lane >> 3, rr = lane & 7;
  const int k_row = (mi & 1) * 8 + rr, k_col = (mi >> 1) * 8;  // K: rows = tokens
  const int v_row = (mi >> 1) * 8 + rr, v_col = (mi & 1) * 8;  // V^T via .trans

  auto issue = [&](int kk) {
    if (kk < n_my) {
      const int64_t t = first + (int64_t)kk * kWarps16;
      unsigned char *stg = wbase + (kk % kStages16) * kStage16;
#pragma unroll
      for (int c = lane; c < 16 * 16; c += 32) {
        const int row = c >> 4, ch = c & 15;
        const int64_t tok = t * 16 + row;
        const bool ok = tok < n;
        const int64_t src = (ok ? tok : 0) * kD + ch * 8;
        cp_async16_zfill(stg + row * kRow + ch * 16, kh + src, ok);
        cp_async16_zfill(stg + 16 * kRow + row * kRow + ch * 16, vh + src, ok);
      }
    }
    cp_async_commit();
  };

  float acc[8][4];
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[j][k] = 0.f;
  float m_run = -INFINITY, l_run = 0.f;

#pragma unroll
  for (int kk = 0; kk < kStages16 - 1; ++kk) issue(kk);
  for (int kk = 0; kk < n_my; ++kk) {
    issue(kk + kStages16 - 1);
    cp_async_wait<kStages16 - 1>();
    __syncwarp();
    const unsigned char *ks = wbase + (kk % kStages16) * kStage16;
    const unsigned char *vs = ks + 16 * kRow;
    const int64_t tok0 = (first + (int64_t)kk * kWarps16) * 16;
    float S[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      uint32_t ak[4];
      ldsm_x4(ks + k_row * kRow + (16 * j + k_col) * 2, ak);
      mma16816(S, ak[0], ak[1], ak[2], ak[3], bq[2 * j], bq[2 * j + 1]);
    }
    const bool va = tok0 + g < n, vb = tok0 + g + 8 < n;
    const float sa = va ? c0 * (S[0] + S[1]) : -INFINITY;
    const float sb = vb ? c0 * (S[2] + S[3]) : -INFINITY;
    float tmax = fmaxf(sa, sb);
    tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 4));
    tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 8));
    tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 16));
    const float m_new = fmaxf(m_run, tmax);
    if (__any_sync(0xffffffffu, m_new > m_run)) {
      const float alpha = ex2f(m_run - m_new);
#pragma unroll
      for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[j][k] *= alpha;
      l_run *= alpha;
      m_run = m_new;
    }
    const float pa = va ? ex2f(sa - m_run) : 0.f, pb = vb ? ex2f(sb - m_run) : 0.f;
    l_run += pa + pb;
    const __half2 hab = __floats2half2_rn(pa, pb);
    const float2 fab = __half22float2(hab);
    const __half2 lab = __floats2half2_rn(pa - fab.x, pb - fab.y);
    const uint32_t q1 = prmt(h22u(hab), h22u(lab), 0x5410u);
    const uint32_t q2 = prmt(h22u(hab), h22u(lab), 0x7632u);
    // B of P.V, column g = (head g/2, part g%2), K slots = tokens 2tig, 2tig+1,
    // 2tig+8, 2tig+9; token u's weights live in lane 4*(u%8) + head
    const uint32_t bw0 = prmt(__shfl_sync(0xffffffffu, q1, src_a), __shfl_sync(0xffffffffu, q1, src_b), pv_sel);
    const uint32_t bw1 = prmt(__shfl_sync(0xffffffffu, q2, src_a), __shfl_sync(0xffffffffu, q2, src_b), pv_sel);
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) {
      uint32_t av[4];
      ldsm_x4_t(vs + v_row * kRow + (16 * jj + v_col) * 2, av);
      mma16816(acc[jj], av[0], av[1], av[2], av[3], bw0, bw1);
    }
    __syncwarp();
  }
  cp_async_wait<0>();

  // ---- merge the 4 warps (lane (g, tig) owns head tig, channels 16jj+g, 16jj+8+g)
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) l_run += __shfl_xor_sync(0xffffffffu, l_run, off);
  __syncthreads();
  float *mrg = reinterpret_cast<float *>(smem);  // [warp][R][kD + 2]
  if (tig < R) {
    float *row = mrg + (warp * R + tig) * (kD + 2);
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) {
      row[16 * jj + g] = acc[jj][0] + acc[jj][1];
      row[16 * jj + 8 + g] = acc[jj][2] + acc[jj][3];
    }
    if (g == 0) {
      row[kD] = m_run;
      row[kD + 1] = l_run;
    }
  }
  __syncthreads();
  const int c = threadIdx.x;
#pragma unroll
  for (int h = 0; h < R; ++h) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps16; ++w) M = fmaxf(M, mrg[(w * R + h) * (kD + 2) + kD]);
    float L = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps16; ++w) {
      const float *row = mrg + (w * R + h) * (kD + 2);
      const float sc = (row[kD] == -INFINITY) ? 0.f : ex2f(row[kD] - M);
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

// Merge the splits of one (batch, query head): one thread per channel.
__global__ void __launch_bounds__(128) fp16_combine_kernel(const float *__restrict__ ws, int splits,
                                                           uint16_t *__restrict__ out) {
  const int64_t row = blockIdx.x;
  const int c = threadIdx.x;
  const float *p = ws + row * splits * (kD + 2);
  float M = -INFINITY;
  for (int s = 0; s < splits; ++s) M = fmaxf(M, __ldcg(p + s * (kD + 2) + kD));
  float L = 0.f, O = 0.f;
#pragma unroll 4
  for (int s = 0; s < splits; ++s) {
    const float m = __ldcg(p + s * (kD + 2) + kD);
    const float sc = (m == -INFINITY) ? 0.f : ex2f(m - M);
    L = fmaf(sc, __ldcg(p + s * (kD + 2) + kD + 1), L);
    O = fmaf(sc, __ldcg(p + s * (kD + 2) + c), O);
  }
  out[row * kD + c] = f2h(O / L);
}

template <int R>
cudaError_t launch_r(const Fp16Args &a, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(fp16_decode_kernel<R>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem16);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)a.splits, (unsigned)(a.B * a.Hkv));
  fp16_decode_kernel<R><<<grid, kWarps16 * 32, kSmem16, st>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  fp16_combine_kernel<<<(unsigned)(a.B * a.Hq), 128, 0, st>>>(a.ws, a.splits, a.out);
  return cudaGetLastError();
}

}  // namespace

void fp16_plan(int B, int Hkv, int64_t n, int num_sms, int *splits, int64_t *tiles_per_split) {
  const int64_t heads = (int64_t)B * Hkv;
  const int64_t tiles = (n + 15) / 16;
  int64_t s = ((int64_t)num_sms * 8 + heads - 1) / heads;  // ~4 waves of 2 resident CTAs per SM
  const int64_t s_max = (tiles + 7) / 8;                      // at least 8 tiles (2 per warp) per split
  if (s > s_max) s = s_max;
  if (s < 1) s = 1;
  const int64_t tps = (tiles + s - 1) / s;
  *tiles_per_split = tps;
  *splits = (int)((tiles + tps - 1) / tps);
}

cudaError_t launch_fp16(const Fp16Args &a, cudaStream_t st) {
  const int R = a.Hq / a.Hkv;
  if (R == 1) return launch_r<1>(a, st);
  if (R == 2) return launch_r<2>(a, st);
  return launch_r<4>(a, st);
}

}  // namespace kivi
