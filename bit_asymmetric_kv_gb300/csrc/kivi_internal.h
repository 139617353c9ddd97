// kivi_internal.h -- launchers shared between the kernel files and the C ABI layer.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace kivi {

cudaError_t launch_key_groups(const uint16_t *in, int64_t in_head_stride, int64_t heads, int64_t groups_per_head,
                              int64_t g0, int G, uint32_t *k_codes, uint32_t *k_meta, int64_t max_tokens,
                              cudaStream_t st);
cudaError_t launch_value_rows(const uint16_t *v, int64_t heads, int64_t tokens_per_head, int64_t t0,
                              uint32_t *v_codes, uint32_t *v_meta, int64_t max_tokens, cudaStream_t st);
cudaError_t launch_append(const uint16_t *k_new, const uint16_t *v_new, int64_t heads, int64_t n, int G,
                          uint16_t *k_res, uint32_t *v_codes, uint32_t *v_meta, int64_t max_tokens, cudaStream_t st);
cudaError_t launch_residual_copy(const uint16_t *k, int64_t heads, int64_t n, int64_t nq, int G, uint16_t *k_res,
                                 cudaStream_t st);
cudaError_t launch_dequant(const uint32_t *k_codes, const uint32_t *k_meta, const uint16_t *k_res,
                           const uint32_t *v_codes, const uint32_t *v_meta, int64_t heads, int64_t n, int G,
                           int64_t max_tokens, float *k_out, float *v_out, cudaStream_t st);

struct DecodeArgs {
  const uint32_t *k_codes;
  const uint32_t *k_meta;
  const uint16_t *k_res;
  const uint32_t *v_codes;
  const uint32_t *v_meta;
  const uint16_t *q;
  uint16_t *out;
  float *ws;
  int64_t max_tokens;
  int64_t n;
  int B, Hkv, Hq, G;
  int64_t units_per_head;  // full key groups + 1 if there are residual keys
  int64_t total_units;     // B * Hkv * units_per_head
  int n_warps;             // warps of the persistent grid (each takes a contiguous unit range)
  int grid;                // CTAs (4 warps each)
  int pmax;                // partial slots per query head in the workspace
  int wait_tail;           // launched as a dependent of an append: wait before each head's last unit
  float softmax_scale;
};

// Geometry of one decode call on the current device (deterministic for given sizes).
struct DecodeGeom {
  int64_t units_per_head;
  int64_t total_units;
  int n_warps;
  int grid;
  int pmax;
};
cudaError_t decode_geometry(int B, int Hkv, int Hq, int G, int64_t n, DecodeGeom *out);
cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t st);

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
