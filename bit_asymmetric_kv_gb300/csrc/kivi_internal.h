// kivi_internal.h -- launchers shared between the kernel files and the C ABI layer.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace kivi {

// `bits` is the code width, 2 or 4.
cudaError_t launch_key_groups(const uint16_t *in, int64_t in_head_stride, int64_t heads, int64_t groups_per_head,
                              int64_t g0, int G, int bits, uint32_t *k_codes, uint32_t *k_meta, int64_t max_tokens,
                              cudaStream_t st);
// vg: channels per value {s, z} (128: one per token; 64 or 32: value channel groups,
// 2-bit codes, v_meta rows of 128 / vg words).
cudaError_t launch_value_rows(const uint16_t *v, int64_t heads, int64_t tokens_per_head, int64_t in_rows_per_head,
                              int64_t t0, int bits, uint32_t *v_codes, uint32_t *v_meta, int64_t max_tokens,
                              cudaStream_t st, int vg = 128);
cudaError_t launch_append(const uint16_t *k_new, const uint16_t *v_new, int64_t heads, int64_t n, int G, int bits,
                          uint16_t *k_res, uint32_t *v_codes, uint32_t *v_meta, int64_t max_tokens, uint16_t *v_res,
                          cudaStream_t st, int vg = 128);
cudaError_t launch_residual_copy(const uint16_t *k, int64_t heads, int64_t n, int64_t nq, int G, uint16_t *k_res,
                                 cudaStream_t st);
// Paged destinations of a prefill: the block-table row of one sequence.
struct PageMap {
  const int32_t *bt;   // [max_pages] page ids of the sequence
  int64_t num_pages;   // pages in the pool (ids outside [0, num_pages) are skipped)
  int shift;           // log2(tokens per page)
  int Hkv;
};
cudaError_t launch_key_groups_paged(const uint16_t *in, int64_t in_head_stride, int64_t heads,
                                    int64_t groups_per_head, int G, int bits, const PageMap &pm, uint32_t *k_codes,
                                    uint32_t *k_meta, cudaStream_t st);
cudaError_t launch_value_rows_paged(const uint16_t *v, int64_t heads, int64_t tokens_per_head,
                                    int64_t in_rows_per_head, int bits, const PageMap &pm, uint32_t *v_codes,
                                    uint32_t *v_meta, cudaStream_t st);
cudaError_t launch_set_len(int32_t *seq_lens, int32_t seq, int32_t n, cudaStream_t st);

// Paged append of one token per (sequence, KV head) at position seq_lens[b], with the
// residual flush done in the same kernel.  seq_lens is read, never written: the
// lengths are advanced afterwards (launch_advance_lens, or the paged combine).
struct PagedAppendArgs {
  const uint16_t *k_new, *v_new;  // [B][Hkv][128]
  const int32_t *bt;              // [B][max_pages]
  int32_t *seq_lens;              // [B]
  uint16_t *k_res;                // [B][Hkv][G][128]
  uint16_t *v_res;                // [B][Hkv][G][128] with a value residual, else null
  uint32_t *k_codes, *k_meta, *v_codes, *v_meta;
  int64_t num_pages;
  int B, Hkv, G, bits, shift, max_pages;
};
cudaError_t launch_paged_append(const PagedAppendArgs &a, cudaStream_t st);
cudaError_t launch_advance_lens(int32_t *seq_lens, int B, int32_t cap, cudaStream_t st);

cudaError_t launch_dequant(const uint32_t *k_codes, const uint32_t *k_meta, const uint16_t *k_res,
                           const uint32_t *v_codes, const uint32_t *v_meta, const uint16_t *v_res, int64_t heads,
                           int64_t n, int G, int bits, int64_t max_tokens, float *k_out, float *v_out,
                           cudaStream_t st, int vg = 128);

struct DecodeArgs {
  const uint32_t *k_codes;
  const uint32_t *k_meta;
  const uint16_t *k_res;
  const uint32_t *v_codes;
  const uint32_t *v_meta;
  const uint16_t *v_res;   // fp16 residual values [B][Hkv][G][128], or null (values all quantized)
  const uint16_t *q;
  uint16_t *out;
  float *ws;
  int64_t max_tokens;
  int64_t n;
  int B, Hkv, Hq, G;
  int bits;                // code width: 2 or 4
  int64_t units_per_head;  // full key groups + 1 if there are residual keys
  int64_t total_units;     // B * Hkv * units_per_head
  int n_warps;             // warps of the persistent grid (each takes a contiguous unit range)
  int grid;                // CTAs (4 warps each)
  int pmax;                // partial slots per query head in the workspace
  int wait_tail;           // launched as a dependent of an append: wait before each head's last unit
  int small;               // dense: CTAs per (batch, KV head) of the small-context path, 0 for the
                           // persistent grid (decode_geometry's choice)
  int vg;                  // channels per value {s, z}: 128 (per token), 64 or 32 (value channel groups)
  float softmax_scale;
  // paged layout only: per-sequence lengths on the device, rows found through the
  // block table; the partials are addressed by (warp + head) and a per-head header
  const int32_t *block_table;  // [B][max_pages]
  const int32_t *seq_lens;     // [B]
  int32_t *advance_lens;       // non-null: the combine sets seq_lens[b] = min(len + 1, cap) afterwards
  int64_t num_pages;
  int page_shift;              // log2(tokens per page)
  int max_pages;
  int len_offset;              // tokens appended just before (0 or 1): the context is seq_lens[b] + len_offset
  int32_t cap_tokens;          // max_pages << page_shift
};

// Decode kernels (kivi_decode.cu) and their launch shape.  The host side
// (kivi_decode_host.cu) sizes the grid from the occupancy of `decode` with `smem`
// bytes of dynamic shared memory; `smem_limit` is the most any launch of it uses.
constexpr int kDecodeWarps = 4;   // warps per decode CTA
constexpr int kDecodeSmallWarps = 8;  // warps per CTA of the small-context path
// Its clusters for 9 to 16 units: 4 CTAs of 4 warps while that many clusters fit at
// once, else 2 CTAs of 8 warps.
constexpr int kDecodeQuadCtas = 4, kDecodeQuadWarps = 4;
constexpr int kDecodePairCtas = 2, kDecodePairWarps = 8;
constexpr int kDecodeUnit = 64;   // tokens per unit of work
constexpr int kCombineRows = 4;   // (batch, query head) rows per combine CTA, one warp each
struct DecodeKernels {
  const void *decode;
  int smem;
  int smem_limit;
  const void *combine;  // dense: (ws, pmax, W, NW, U, Hkv, Hq, rows, out);
                        // paged: (ws, Hkv, Hq, B, advance, cap, out)
  const void *small;    // dense only: one CTA of kDecodeSmallWarps warps per (batch, KV head)
  int small_smem;
  const void *pair;     // dense only: a cluster of kDecodePairCtas CTAs per (batch, KV head)
  int pair_smem;
  const void *quad;     // dense only: a cluster of kDecodeQuadCtas CTAs per (batch, KV head)
  int quad_smem;
};
// vg: channels per value scale (128, or 64 / 32 for value channel groups: dense
// 2-bit caches only, no small-context kernel).
DecodeKernels decode_kernels(int R, int G, int bits, bool paged, int B, int vg = 128);

// Geometry of one decode call on the current device (deterministic for given sizes).
struct DecodeGeom {
  int64_t units_per_head;
  int64_t total_units;
  int n_warps;
  int grid;
  int pmax;
  int small;  // the small-context path, no workspace and no combine: CTAs per (batch, KV
              // head), 1, kDecodePairCtas or kDecodeQuadCtas; 0 for the persistent grid
};
cudaError_t decode_geometry(int B, int Hkv, int Hq, int G, int bits, int64_t n, DecodeGeom *out, int vg = 128);
cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t st);

// Paged decode: the grid fills the GPU whatever the lengths; n_warps and grid come
// from here, the rest is found on the device.  Workspace: a header of B*Hkv int2
// {first partial, count}, then (n_warps + B*Hkv) * R partials of 130 floats.
struct PagedGeom {
  int n_warps;
  int grid;
  size_t ws_bytes;
};
constexpr int kPagedMaxBatch = 512;
cudaError_t paged_decode_geometry(int B, int Hkv, int Hq, int G, int bits, PagedGeom *out);
cudaError_t launch_paged_decode(const DecodeArgs &a, cudaStream_t st);

// Fused prefill (kivi_prefill.cu): causal attention over the fp16 prompt and, when
// k_codes is not null, the cache quantized from the same tiles.
struct PrefillArgs {
  const uint16_t *q;  // [B][Hq][n][128]
  const uint16_t *k;  // [B][Hkv][n][128]
  const uint16_t *v;
  uint16_t *out;      // [B][Hq][n][128]
  uint32_t *k_codes, *k_meta, *v_codes, *v_meta;  // the cache (null: attention only)
  uint16_t *k_res, *v_res;                        // v_res null without a value residual
  int64_t n, max_tokens;
  int B, Hkv, Hq, G, bits;
  int vg;             // channels per value {s, z}: 128, 64 or 32
  float softmax_scale;
};
cudaError_t launch_prefill_attention(const PrefillArgs &a, cudaStream_t st);

// Decode attention over an unquantized fp16 cache (the comparison kernel).
struct Fp16Args {
  const uint16_t *k;  // [B][Hkv][n][128]
  const uint16_t *v;
  const uint16_t *q;  // [B][Hq][128]
  uint16_t *out;
  float *ws;
  int64_t n;
  int B, Hkv, Hq;
  int splits;
  int64_t tiles_per_split;
  float softmax_scale;
};
void fp16_plan(int B, int Hkv, int64_t n, int num_sms, int *splits, int64_t *tiles_per_split);
cudaError_t launch_fp16(const Fp16Args &a, cudaStream_t st);

}  // namespace kivi
