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
  int splits;
  int groups_per_split;
  float softmax_scale;
};

// Split of the context for one decode call (host heuristic, deterministic).
void decode_plan(int B, int Hkv, int G, int64_t n, int num_sms, int *splits, int *groups_per_split);
cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t st);

}  // namespace kivi
