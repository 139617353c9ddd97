// kivi_decode_host.cu -- grid sizing and launches of the decode kernels in
// kivi_decode.cu (host code only, so that the kernels' source is one file).
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "kivi_internal.h"

namespace kivi {

namespace {

constexpr int kD = 128;

// Warps of `fn` resident at once on the current device with `smem` bytes of dynamic
// shared memory.  The first query per (device, kernel, size) raises the kernel's
// dynamic shared-memory limit to `smem_limit` (the most any launch of it uses, so
// that an entry for one size never lowers the limit another size needs) and asks
// the occupancy calculator; later calls read a table, so that decode calls make no
// CUDA runtime query but cudaGetDevice (and can be captured in a CUDA graph once a
// first call has run).
struct WarpsEntry {
  int dev;
  const void *fn;
  int smem;
  int n_warps;
  int sms;
  int pair_clusters;  // clusters of the pair kernel resident at once (0 without one)
  int quad_clusters;  // the same for the quad kernel
};
constexpr int kWarpsCache = 256;
WarpsEntry g_warps[kWarpsCache];
int g_warps_used = 0;
std::mutex g_warps_lock;

// Clusters of `fn` (CTAs of `warps` warps with `smem` bytes; its cluster shape is fixed
// at compile time) resident at once on the current device, of `sms` SMs.
cudaError_t clusters_on_device(const void *fn, int ctas, int warps, int smem, int sms, int *n) {
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(ctas * sms));
  cfg.blockDim = dim3(32 * warps);
  cfg.dynamicSmemBytes = (size_t)smem;
  return cudaOccupancyMaxActiveClusters(n, fn, &cfg);
}

cudaError_t warps_on_device(const DecodeKernels &k, int *n_warps, int *n_sms = nullptr, int *n_pairs = nullptr,
                            int *n_quads = nullptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  {
    std::lock_guard<std::mutex> guard(g_warps_lock);
    for (int i = 0; i < g_warps_used; ++i)
      if (g_warps[i].dev == dev && g_warps[i].fn == k.decode && g_warps[i].smem == k.smem) {
        *n_warps = g_warps[i].n_warps;
        if (n_sms) *n_sms = g_warps[i].sms;
        if (n_pairs) *n_pairs = g_warps[i].pair_clusters;
        if (n_quads) *n_quads = g_warps[i].quad_clusters;
        return cudaSuccess;
      }
  }
  e = cudaFuncSetAttribute(k.decode, cudaFuncAttributeMaxDynamicSharedMemorySize, k.smem_limit);
  if (e != cudaSuccess) return e;
  if (k.small) {  // the small-context kernel of the same shapes: one CTA per SM at most
    e = cudaFuncSetAttribute(k.small, cudaFuncAttributeMaxDynamicSharedMemorySize, k.small_smem);
    if (e != cudaSuccess) return e;
  }
  int sms = 0, per_sm = 0, pairs = 0, quads = 0;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k.decode, 32 * kDecodeWarps, k.smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  // the small path's clusters: how many fit at once (SMs of a GPC left over from whole
  // clusters stay unused)
  if (k.pair && (e = clusters_on_device(k.pair, kDecodePairCtas, kDecodePairWarps, k.pair_smem, sms, &pairs)) != cudaSuccess)
    return e;
  if (k.quad && (e = clusters_on_device(k.quad, kDecodeQuadCtas, kDecodeQuadWarps, k.quad_smem, sms, &quads)) != cudaSuccess)
    return e;
  *n_warps = sms * per_sm * kDecodeWarps;
  if (n_sms) *n_sms = sms;
  if (n_pairs) *n_pairs = pairs;
  if (n_quads) *n_quads = quads;
  std::lock_guard<std::mutex> guard(g_warps_lock);
  if (g_warps_used < kWarpsCache)
    g_warps[g_warps_used++] = WarpsEntry{dev, k.decode, k.smem, *n_warps, sms, pairs, quads};
  return cudaSuccess;
}

// Launch the decode grid (a programmatic dependent of the preceding kernel when
// `dependent`), then the combine as a programmatic dependent of the decode grid.
cudaError_t launch_with_combine(const DecodeKernels &k, const DecodeArgs &a, void **combine_args, cudaStream_t st) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t dcfg = {};
  dcfg.gridDim = dim3((unsigned)a.grid);
  dcfg.blockDim = dim3(32 * kDecodeWarps);
  dcfg.dynamicSmemBytes = (size_t)k.smem;
  dcfg.stream = st;
  dcfg.attrs = attr;
  dcfg.numAttrs = a.wait_tail ? 1 : 0;  // overlap a preceding append only when asked
  void *args[] = {const_cast<DecodeArgs *>(&a)};
  cudaError_t e = cudaLaunchKernelExC(&dcfg, k.decode, args);
  if (e != cudaSuccess) return e;
  const int64_t rows = (int64_t)a.B * a.Hq;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((rows + kCombineRows - 1) / kCombineRows));
  cfg.blockDim = dim3(32 * kCombineRows);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, k.combine, combine_args);
}

}  // namespace

cudaError_t decode_geometry(int B, int Hkv, int Hq, int G, int bits, int64_t n, DecodeGeom *out, int vg) {
  const int R = Hq / Hkv;
  int nw = 0, sms = 0, pairs = 0, quads = 0;
  cudaError_t e = warps_on_device(decode_kernels(R, G, bits, false, B, vg), &nw, &sms, &pairs, &quads);
  if (e != cudaSuccess) return e;
  const int64_t heads = (int64_t)B * Hkv;
  const int64_t ng = n / G;
  const int64_t U = (ng * G + kDecodeUnit - 1) / kDecodeUnit + ((n % G) ? 1 : 0);
  const int64_t W = heads * U;
  int64_t NW = nw;
  if (NW > W) NW = W;
  const int64_t q = W / NW;  // every warp holds at least q units
  out->units_per_head = U;
  out->total_units = W;
  out->n_warps = (int)NW;
  out->grid = (int)((NW + kDecodeWarps - 1) / kDecodeWarps);
  out->pmax = (int)((U + q - 1) / q + 1);
  // small contexts: one CTA, or one cluster, per (batch, KV head), all resident at
  // once, and at most one unit per warp.  There the persistent grid's fixed cost (the
  // workspace round trip and the combine launch) outweighs its wider split; with two
  // units per warp the second unit's compute, serial in each warp, costs more than
  // the combine saves (measured), so 9 to 16 units take a cluster: 4 CTAs of 4 warps,
  // one CTA per SM, while they fit (one unit's compute is faster with 4 warps on an SM
  // than with 8), else 2 CTAs of 8 warps.
  static_assert(kDecodeQuadCtas * kDecodeQuadWarps == 16 && kDecodePairCtas * kDecodePairWarps == 16, "16 units");
  out->small = 0;
  if (vg == kD && U <= kDecodeSmallWarps && heads <= sms) out->small = 1;
  else if (vg == kD && U <= 16 && heads <= quads) out->small = kDecodeQuadCtas;
  else if (vg == kD && U <= 16 && heads <= pairs) out->small = kDecodePairCtas;
  return cudaSuccess;
}

cudaError_t paged_decode_geometry(int B, int Hkv, int Hq, int G, int bits, PagedGeom *out) {
  const int R = Hq / Hkv;
  int nw = 0;
  cudaError_t e = warps_on_device(decode_kernels(R, G, bits, true, B), &nw);
  if (e != cudaSuccess) return e;
  const size_t heads = (size_t)B * Hkv;
  out->n_warps = nw;
  out->grid = nw / kDecodeWarps;
  // header int2 per head; pair indices warp + head < n_warps + heads
  out->ws_bytes = heads * 8 + ((size_t)nw + heads) * R * (kD + 2) * sizeof(float);
  return cudaSuccess;
}

cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t st) {
  const DecodeKernels k = decode_kernels(a.Hq / a.Hkv, a.G, a.bits, false, a.B, a.vg ? a.vg : kD);
  if (a.small) {
    // one CTA (a.small = 1) or a cluster of a.small CTAs per (batch, KV head); a
    // programmatic dependent of a preceding append when asked (the same tail wait as
    // the persistent grid)
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    const bool quad = a.small == kDecodeQuadCtas, pair = a.small == kDecodePairCtas;
    cfg.gridDim = dim3((unsigned)((int64_t)a.B * a.Hkv * a.small));
    cfg.blockDim = dim3(32 * (quad ? kDecodeQuadWarps : pair ? kDecodePairWarps : kDecodeSmallWarps));
    cfg.dynamicSmemBytes = (size_t)(quad ? k.quad_smem : pair ? k.pair_smem : k.small_smem);
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = a.wait_tail ? 1 : 0;
    void *args[] = {const_cast<DecodeArgs *>(&a)};
    return cudaLaunchKernelExC(&cfg, quad ? k.quad : pair ? k.pair : k.small, args);
  }
  const float *ws = a.ws;
  int64_t pmax = a.pmax, W = a.total_units, NW = a.n_warps, U = a.units_per_head;
  int Hkv = a.Hkv, Hq = a.Hq;
  int64_t rows = (int64_t)a.B * a.Hq;
  uint16_t *out = a.out;
  void *cargs[] = {&ws, &pmax, &W, &NW, &U, &Hkv, &Hq, &rows, &out};
  return launch_with_combine(k, a, cargs, st);
}

cudaError_t launch_paged_decode(const DecodeArgs &a, cudaStream_t st) {
  const DecodeKernels k = decode_kernels(a.Hq / a.Hkv, a.G, a.bits, true, a.B);
  const float *ws = a.ws;
  int Hkv = a.Hkv, Hq = a.Hq, B = a.B;
  int32_t *advance = a.advance_lens;
  int32_t cap = a.cap_tokens;
  uint16_t *out = a.out;
  void *cargs[] = {&ws, &Hkv, &Hq, &B, &advance, &cap, &out};
  return launch_with_combine(k, a, cargs, st);
}

}  // namespace kivi
