/*
 * kivi.h -- C ABI of the GB300 (sm_103a) KIVI asymmetric 2-bit KV-cache library.
 *
 * The method is KIVI ("KIVI: A Tuning-Free Asymmetric 2bit Quantization for KV
 * Cache", ICML 2024) as summarised on the page "Makale Bulteni -- KIVI"
 * (cmlonder.com, radar / paper-to-prod, 2026-11-01):
 *   - headline paragraph: keys are quantized per channel and values per token, in
 *     an asymmetric 2-bit format;
 *   - section "Iddia ve Gerceklik", paragraph 2: key outlier channels stay fixed
 *     over the sequence (so keys are grouped along the channel axis); values are
 *     kept per token because the attention output is a weighted sum of values;
 *   - same section, paragraph 3: keys are split into groups of G = 32 or 64 tokens;
 *     the tokens of a group that has not filled yet stay in a full-precision
 *     residual buffer; unpacking 2-bit codes for 16-bit tensor cores is done with
 *     bit shifts and masks on the GPU.
 * The page gives no formulas, so these readings apply throughout:
 *   - zero = min, scale = (max - min) / 3, both stored as fp16;
 *   - code = clamp(round_half_even(fp32((x - min) / scale)), 0, 3), all fp32
 *     operations IEEE round-to-nearest-even, computed with the stored fp16 scale;
 *     a group whose fp16 scale is 0 gets all-zero codes; a zero of -0 is stored +0;
 *   - one (scale, zero) pair per value token per KV head over all D channels;
 *   - variant (value_group = vg < D): a value token is quantized in D / vg groups of
 *     vg consecutive channels (group g = channels g*vg .. g*vg + vg - 1), each by the
 *     rule above, its D / vg {s, z} words stored in group order;
 *   - only keys have a residual; a key group is quantized ("flushed") as soon as it
 *     holds G tokens, so the residual holds n mod G tokens;
 *   - variant (value_residual = 1): the values keep the same residual as the keys,
 *     in fp16, and the G values of a group are quantized token by token when the
 *     key group flushes;
 *   - query head h reads KV head h / (Hq / Hkv) (grouped-query attention).
 *
 * Supported shapes: D = 128, bits in {2, 4} (the code width; 4 is a variant, see
 * kivi_dims.bits), G in {32, 64}, Hq / Hkv in {1, 2, 4}.
 * Inputs must be finite; codes for non-finite inputs are unspecified.
 *
 * Memory: every buffer is device memory owned by the caller (nothing is allocated
 * inside the library, nothing is freed), 16-byte aligned, in these layouts:
 *   k_codes  uint32 [B][Hkv][max_tokens][D/16]  token rows of packed key codes
 *   k_meta   uint32 [B][Hkv][max_tokens/G][D]   per (group, channel) {s, z}
 *   k_res    fp16   [B][Hkv][G][D]              residual keys, slot j = token nq + j
 *   v_codes  uint32 [B][Hkv][max_tokens][D/16]  token rows of packed value codes
 *   v_meta   uint32 [B][Hkv][max_tokens][D/vg]  per token {s, z} of each value channel
 *                                               group (vg = dims.value_group, D when 0:
 *                                               one word per token)
 *   v_res    fp16   [B][Hkv][G][D]              residual values (value_residual = 1
 *                                               only; NULL otherwise)
 * A {s, z} word holds the fp16 scale in bits 0-15 and the fp16 zero in bits 16-31.
 * Packing: word w of a token row holds channels 16w .. 16w+15; channel 16w+i sits
 * in bits [2i, 2i+1].  fp16 buffers are IEEE binary16 bit patterns (uint16_t).
 * nq = floor(n / G) * G tokens are quantized keys; rows at or beyond nq of k_codes,
 * groups at or beyond n / G of k_meta, residual slots at or beyond n mod G and
 * value rows at or beyond n (at or beyond nq with a value residual) are not read.
 *
 * Streams and state: every compute call is asynchronous on the given stream and
 * never synchronises with the host.  The cache state is the caller's kivi_cache;
 * its n_tokens field is host memory, updated by the library when a call succeeds
 * and left unchanged when it fails.  Concurrent calls on the same cache race.
 * No call throws across the ABI; every call returns a kivi_status.
 *
 * Process-wide tables: the decode calls size their grids from the occupancy of
 * their kernels on the current device.  The first decode call for a given (device,
 * kernel, shared-memory size) asks the CUDA runtime (it raises the kernels'
 * dynamic shared-memory limits and queries the occupancy calculator, for CTAs and
 * for the small-context path's thread-block clusters) and records the
 * answer in a table inside the library, guarded by a mutex; later calls only read
 * it, so they make no runtime query but cudaGetDevice and can be captured in a CUDA
 * graph.  Make a first decode call (or a kivi_decode_workspace_bytes /
 * kivi_paged_decode_workspace_bytes query) on each device before capturing.  The
 * table holds no cache data and never changes a result.  The allocation-free entry
 * point keeps a second table (see kivi_decode_attention_noalloc).
 *
 * Device dependence: the split of the context between the GPU's warps, and with it
 * kivi_decode_splits, kivi_decode_workspace_bytes and
 * kivi_paged_decode_workspace_bytes, depend on the current device (its SM count
 * and the kernels' occupancy on it).  Query them with the device current that the
 * calls will run on, and re-query after switching devices.
 */
#ifndef KIVI_H
#define KIVI_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define KIVI_API __attribute__((visibility("default")))
#else
#define KIVI_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KIVI_OK = 0,
  KIVI_ERR_ARG = 1,          /* null pointer, non-positive size, n > max_tokens ... */
  KIVI_ERR_ALIGN = 2,        /* a buffer is not 16-byte aligned */
  KIVI_ERR_UNSUPPORTED = 3,  /* D != 128, bits not 2 or 4, G not in {32, 64}, Hq/Hkv not in {1,2,4},
                                value_group not in {0, 32, 64, 128}, or below 128 with 4-bit
                                codes or a value residual; sizes beyond the supported range */
  KIVI_ERR_CAPACITY = 4,     /* append on a full cache, prefill longer than max_tokens */
  KIVI_ERR_WORKSPACE = 5,    /* workspace missing or smaller than required */
  KIVI_ERR_CUDA = 6          /* a CUDA runtime call or launch failed */
} kivi_status;

/* Cache geometry.  max_tokens must be a positive multiple of G, and B * Hkv *
 * max_tokens at most 2^40 token rows (KIVI_ERR_UNSUPPORTED beyond). */
typedef struct {
  int32_t B;         /* batch */
  int32_t Hkv;       /* KV heads */
  int32_t D;         /* head dim, 128 */
  int32_t G;         /* key group size, 32 or 64 */
  int32_t bits;      /* code width, 2 or 4 */
  int32_t value_residual; /* 1: values keep an fp16 residual beside the keys'; 0: none */
  int32_t value_group;    /* channels per value {s, z}: 0 or D (one per token), or the
                             variant 32 / 64 (value channel groups; 2-bit codes without a
                             value residual only, else KIVI_ERR_UNSUPPORTED) */
  int64_t max_tokens;
} kivi_dims;

/* Caller-owned device buffers (layouts above) plus the host-side token count. */
typedef struct {
  uint32_t *k_codes;
  uint32_t *k_meta;
  uint16_t *k_res;
  uint32_t *v_codes;
  uint32_t *v_meta;
  uint16_t *v_res;   /* value_residual = 1 only; may be NULL otherwise */
  int64_t n_tokens;
} kivi_cache;

/* Bytes of the cache buffers, in the order k_codes, k_meta, k_res, v_codes, v_meta,
 * v_res (0 without a value residual).  Pure host arithmetic. */
KIVI_API int kivi_buffer_bytes(const kivi_dims *dims, size_t out_bytes[6]);

/*
 * Quantize a prompt of n tokens into an empty cache (headline paragraph; section
 * "Iddia ve Gerceklik", paragraphs 2-3).  k, v: fp16 [B][Hkv][n][D] device.
 * Keys of the floor(n/G) full groups are quantized per channel; the last n mod G
 * keys are copied to k_res; all n values are quantized per token (with a value
 * residual: the first floor(n/G)*G, the last n mod G go to v_res).  Sets
 * cache->n_tokens = n.  n == 0 launches nothing.  n > max_tokens: KIVI_ERR_CAPACITY.
 */
KIVI_API int kivi_quantize_prefill(const kivi_dims *dims, kivi_cache *cache, const uint16_t *k,
                          const uint16_t *v, int64_t n, cudaStream_t stream);

/*
 * Append one token per (batch, KV head) (section "Iddia ve Gerceklik", paragraph 3).
 * k_new, v_new: fp16 [B][Hkv][D] device.  The key goes to residual slot
 * n_tokens mod G; the value is quantized at once (with a value residual: it goes
 * to the same slot of v_res); when the residual fills, its G keys are quantized as
 * one group in the same call (with a value residual, its G values too, token by
 * token).  Increments cache->n_tokens.  A full cache returns KIVI_ERR_CAPACITY.
 */
KIVI_API int kivi_append_token(const kivi_dims *dims, kivi_cache *cache, const uint16_t *k_new,
                      const uint16_t *v_new, cudaStream_t stream);

/* kivi_decode_attention splits the context of every (batch, KV head) between the
 * GPU's warps and merges the pieces (flash-decoding).  This is the largest number
 * of pieces one query head can have for these sizes on the current device (>= 1;
 * 0 on bad arguments or without a device). */
KIVI_API int kivi_decode_splits(const kivi_dims *dims, int32_t Hq, int64_t n_tokens);

/* Workspace bytes kivi_decode_attention needs for these sizes on the current
 * device: B * Hq * kivi_decode_splits() * (D + 2) floats.  0 on bad arguments. */
KIVI_API size_t kivi_decode_workspace_bytes(const kivi_dims *dims, int32_t Hq, int64_t n_tokens);

/*
 * One decode step of attention over the quantized cache (section "Iddia ve
 * Gerceklik", paragraphs 2-3): for every batch b and query head h,
 *   score_t = softmax_scale * q[b][h] . K'_t  over the cache's n_tokens tokens,
 *   out[b][h] = sum_t softmax(score)_t V'_t,
 * where K'_t = z + code * s for quantized keys, the fp16 residual key itself for
 * the last n mod G tokens, and V'_t = z_t + code * s_t.  q, out: fp16 [B][Hq][D]
 * device.  ws: device workspace of at least kivi_decode_workspace_bytes() bytes,
 * caller-owned, contents overwritten.  n_tokens == 0 returns KIVI_ERR_ARG.
 * Small contexts (a unit being 64 quantized tokens or the residual) leave ws
 * unused: at most 8 units per (batch, KV head), with no more (batch, KV head) pairs
 * than SMs, run on one CTA per pair; 9 to 16 units, with no more pairs than
 * two-CTA clusters fit on the device at once, on a cluster of two CTAs per pair.
 * Device faults: every wait of the kernel for its own staged copies is bounded; a
 * wait that runs out (a copy that never completes) makes every later output of the
 * decode attention calls in this process NaN instead of hanging the GPU.
 */
KIVI_API int kivi_decode_attention(const kivi_dims *dims, const kivi_cache *cache, const uint16_t *q,
                          int32_t Hq, float softmax_scale, uint16_t *out, void *ws,
                          size_t ws_bytes, cudaStream_t stream);

/*
 * One whole decode step: kivi_append_token(k_new, v_new) followed by
 * kivi_decode_attention(q) over the n_tokens + 1 tokens (section "Iddia ve
 * Gerceklik", paragraphs 2-3).  Same arguments, layouts and statuses as those two
 * calls; ws must hold kivi_decode_workspace_bytes(dims, Hq, n_tokens + 1) bytes.
 * The attention kernel is launched as a programmatic dependent of the append, so it
 * starts on the cached tokens while the append runs and waits for it only before
 * the block of each head that holds the new token.  Increments cache->n_tokens on
 * success; every argument is checked before anything is launched.  If a launch
 * fails (KIVI_ERR_CUDA) after the append was queued, n_tokens is left unchanged
 * although the append may have written token n_tokens (its residual slot, its value
 * row and, on a flush, its key group); calling kivi_decode_step again with the same
 * k_new and v_new rewrites that token with the same bits, so a retry is safe.
 */
KIVI_API int kivi_decode_step(const kivi_dims *dims, kivi_cache *cache, const uint16_t *k_new,
                              const uint16_t *v_new, const uint16_t *q, int32_t Hq, float softmax_scale,
                              uint16_t *out, void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Fused prefill: the prompt's causal attention over its full-precision keys and
 * values, with the cache quantized from the same key and value tiles while they are
 * on chip (section "Kod ve Entegrasyon Haritasi": FlashAttention runs the prefill,
 * KIVI quantizes the cache; headline paragraph and section "Iddia ve Gerceklik",
 * paragraphs 2-3, for the cache).  For every batch b, query head h and prompt
 * position i:
 *   out[b][h][i] = sum_{j <= i} softmax_j(softmax_scale * q[b][h][i] . k[b][h / (Hq/Hkv)][j])
 *                  v[b][h / (Hq/Hkv)][j].
 * q, out: fp16 [B][Hq][n][D]; k, v: fp16 [B][Hkv][n][D]; all device, 16-byte aligned.
 * With a cache, it is written exactly as kivi_quantize_prefill(k, v, n) writes it
 * (codes, scales and zeros bit for bit; the residual; n_tokens = n); cache == NULL
 * computes the attention alone.  The probabilities enter the P.V contraction as an
 * fp16 pair hi + lo.  n <= 0: KIVI_ERR_ARG; with a cache, n > max_tokens:
 * KIVI_ERR_CAPACITY; B * Hq > 65535: KIVI_ERR_UNSUPPORTED.  Nothing is allocated.
 */
KIVI_API int kivi_prefill_attention(const kivi_dims *dims, kivi_cache *cache, const uint16_t *q, int32_t Hq,
                                    const uint16_t *k, const uint16_t *v, int64_t n, float softmax_scale,
                                    uint16_t *out, cudaStream_t stream);

/*
 * Test aid: write the dequantized cache as fp32 [B][Hkv][n_tokens][D] to k_out and
 * v_out (device, caller-owned).  Quantized entries are fp32(z) + code * fp32(s)
 * (exact product, one rounding); residual keys are copied exactly.
 */
KIVI_API int kivi_dequantize_debug(const kivi_dims *dims, const kivi_cache *cache, float *k_out,
                          float *v_out, cudaStream_t stream);

/*
 * Decode attention over an unquantized fp16 cache of the same shapes, the point of
 * comparison for the 2-bit cache (the page's "Makale Bulteni" section states KIVI's
 * savings against an FP16 KV cache).  k, v: fp16 [B][Hkv][n][D] device, read-only;
 * q, out: fp16 [B][Hq][D]; ws: device workspace of at least
 * kivi_decode_fp16_workspace_bytes() bytes, contents overwritten.  Same score,
 * softmax and GQA conventions as kivi_decode_attention; D = 128, Hq/Hkv in
 * {1, 2, 4}.  kivi_decode_fp16_workspace_bytes returns 0 on bad arguments.
 */
KIVI_API size_t kivi_decode_fp16_workspace_bytes(int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int64_t n);
KIVI_API int kivi_decode_attention_fp16(int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int64_t n,
                                        const uint16_t *k, const uint16_t *v, const uint16_t *q,
                                        float softmax_scale, uint16_t *out, void *ws, size_t ws_bytes,
                                        cudaStream_t stream);

/*
 * kivi_decode_attention for callers that cannot allocate device memory (for
 * instance a serving loop that must not call cudaMalloc between steps, or a process
 * whose device memory is reserved up front).  The method's page has no counterpart:
 * this is a deployment aid.  Same arguments, results and statuses as
 * kivi_decode_attention, without the workspace: the workspace is taken from an
 * 8 MiB array compiled into the library, which occupies device memory on every GPU
 * that loads the library until the process exits.  Sizes whose workspace
 * (kivi_decode_workspace_bytes) exceeds kivi_decode_attention_noalloc_max_workspace()
 * return KIVI_ERR_WORKSPACE and launch nothing; every other argument is checked
 * first, in the order and with the statuses of kivi_decode_attention.  The first
 * call on a device looks up the array's device address (a runtime query, done once
 * per device), so make it before any stream capture.  The address is kept for the
 * life of the process: after a cudaDeviceReset of a device, do not call this entry
 * point on that device again.  Calls share the array: calls whose kernels overlap
 * on the GPU race.  No call allocates or frees memory.
 */
KIVI_API size_t kivi_decode_attention_noalloc_max_workspace(void);
KIVI_API int kivi_decode_attention_noalloc(const kivi_dims *dims, const kivi_cache *cache,
                                           const uint16_t *q, int32_t Hq, float softmax_scale,
                                           uint16_t *out, cudaStream_t stream);

/*
 * ---- Paged cache -------------------------------------------------------------------
 * The same 2-bit cache, with token storage split into fixed-size pages drawn from one
 * pool and found through a per-sequence block table, as serving engines keep KV
 * caches; sequences of a batch may have different lengths.  The page notes that
 * KIVI's grouped residual and layout do not fit a paged block manager as they are,
 * and that serving engines need paged 2-bit kernels for it (section "Kod ve
 * Entegrasyon Haritasi", paragraph 3).  The method itself is unchanged: per-channel
 * key groups of G tokens with an fp16 residual, per-token values, the same codes,
 * scales and packing as above.
 *
 * A page holds P consecutive token positions of one sequence for all Hkv KV heads.
 * P (page_tokens) is a power of two and a multiple of 64, so a page holds whole key
 * groups.  Device buffers (caller-owned, 16-byte aligned):
 *   k_codes      uint32 [num_pages][Hkv][P][D/16]   token rows of packed key codes
 *   k_meta       uint32 [num_pages][Hkv][P/G][D]    per (group, channel) {s, z}
 *   v_codes      uint32 [num_pages][Hkv][P][D/16]   token rows of packed value codes
 *   v_meta       uint32 [num_pages][Hkv][P]         per token {s, z}
 *   k_res        fp16   [B][Hkv][G][D]              residual keys of sequence b
 *   v_res        fp16   [B][Hkv][G][D]              residual values (value_residual = 1)
 *   block_table  int32  [B][max_pages_per_seq]      page of positions j*P .. j*P+P-1
 *   seq_lens     int32  [B]                         tokens held by sequence b
 * Position t of sequence b is row t mod P of page block_table[b][t / P].  The block
 * table and the lengths live on the device and are the caller's: the caller assigns
 * pages before a call needs them (a sequence at length n needs pages for positions
 * 0 .. n, the next token included) and reads seq_lens back only when it needs them.
 * The host sees neither, so the kernels guard them instead of the host: a length is
 * clamped to [0, max_pages_per_seq * P]; a token appended to a full sequence, or to
 * a position whose page id lies outside [0, num_pages), is dropped; a page id outside
 * the pool that attention reads is clamped into it (results undefined, no access
 * outside the buffers).  A sequence of length 0 attends to nothing: its output rows
 * are zero.  B <= 512.
 */
typedef struct {
  int32_t B;                  /* sequences (rows of the block table) */
  int32_t Hkv;                /* KV heads */
  int32_t D;                  /* head dim, 128 */
  int32_t G;                  /* key group size, 32 or 64 */
  int32_t bits;               /* code width, 2 or 4 */
  int32_t value_residual;     /* as kivi_dims.value_residual */
  int32_t page_tokens;        /* P: a power of two, >= 64 */
  int32_t max_pages_per_seq;  /* columns of the block table */
  int64_t num_pages;          /* pages in the pool; num_pages * Hkv * P at most 2^40 */
} kivi_paged_dims;

typedef struct {
  uint32_t *k_codes;
  uint32_t *k_meta;
  uint32_t *v_codes;
  uint32_t *v_meta;
  uint16_t *k_res;
  uint16_t *v_res;            /* [B][Hkv][G][D] fp16, value_residual = 1 only */
  const int32_t *block_table;
  int32_t *seq_lens;
} kivi_paged_cache;

/* Bytes of the pool and per-sequence buffers, in the order k_codes, k_meta, v_codes,
 * v_meta, k_res, block_table, seq_lens, v_res (0 without a value residual).  Pure
 * host arithmetic. */
KIVI_API int kivi_paged_buffer_bytes(const kivi_paged_dims *dims, size_t out_bytes[8]);

/*
 * Quantize the prompt of sequence `seq` (0 <= seq < B) into its pages, as
 * kivi_quantize_prefill does for one batch row: k, v fp16 [Hkv][n][D] device; the
 * keys of floor(n/G) groups are quantized per channel, the last n mod G keys go to
 * the sequence's residual, all n values are quantized per token.  Then sets
 * seq_lens[seq] = n on the device (stream-ordered).  n > max_pages_per_seq * P:
 * KIVI_ERR_CAPACITY.  Other sequences are not touched.
 */
KIVI_API int kivi_paged_prefill(const kivi_paged_dims *dims, const kivi_paged_cache *cache, int32_t seq,
                                const uint16_t *k, const uint16_t *v, int64_t n, cudaStream_t stream);

/*
 * Append one token to every sequence, at position seq_lens[b] (section "Iddia ve
 * Gerceklik", paragraph 3): k_new, v_new fp16 [B][Hkv][D] device.  The value is
 * quantized at once; the key goes to residual slot seq_lens[b] mod G, and a
 * sequence whose residual fills has its group quantized in the same kernel.  Then
 * seq_lens[b] += 1 on the device (capped at the capacity).
 */
KIVI_API int kivi_paged_append_token(const kivi_paged_dims *dims, const kivi_paged_cache *cache,
                                     const uint16_t *k_new, const uint16_t *v_new, cudaStream_t stream);

/* Workspace bytes of the paged decode calls for these sizes on the current device
 * (independent of the lengths).  0 on bad arguments. */
KIVI_API size_t kivi_paged_decode_workspace_bytes(const kivi_paged_dims *dims, int32_t Hq);

/*
 * kivi_decode_attention over the paged cache, each sequence over its own
 * seq_lens[b] tokens: q, out fp16 [B][Hq][D] device; ws of at least
 * kivi_paged_decode_workspace_bytes() bytes, contents overwritten.  The context of
 * all sequences is split evenly between the GPU's warps on the device (the host
 * does not know the lengths).
 */
KIVI_API int kivi_paged_decode_attention(const kivi_paged_dims *dims, const kivi_paged_cache *cache,
                                         const uint16_t *q, int32_t Hq, float softmax_scale, uint16_t *out,
                                         void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * One whole paged decode step: append k_new, v_new at position seq_lens[b] of every
 * sequence, attend with q over the seq_lens[b] + 1 tokens, then seq_lens[b] += 1
 * (capped at the capacity).  The attention overlaps the append as in
 * kivi_decode_step.  Arguments as kivi_paged_append_token and
 * kivi_paged_decode_attention.
 */
KIVI_API int kivi_paged_decode_step(const kivi_paged_dims *dims, const kivi_paged_cache *cache,
                                    const uint16_t *k_new, const uint16_t *v_new, const uint16_t *q, int32_t Hq,
                                    float softmax_scale, uint16_t *out, void *ws, size_t ws_bytes,
                                    cudaStream_t stream);

/* Human-readable name of a kivi_status. */
KIVI_API const char *kivi_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* KIVI_H */
