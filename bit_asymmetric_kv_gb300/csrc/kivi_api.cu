// kivi_api.cu -- the C ABI (include/kivi.h): argument checks, then kernel launches.
// Nothing here allocates device memory, synchronises with the host or keeps state.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kivi.h"
#include "kivi_internal.h"

namespace {

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// Most token rows (B * Hkv * max_tokens, or pool pages * Hkv * page tokens) a cache may
// have: 2^40, far beyond any device memory and far inside int64 row arithmetic.
constexpr uint64_t kMaxRows = 1ull << 40;

int check_dims(const kivi_dims *d) {
  if (!d) return KIVI_ERR_ARG;
  if (d->B <= 0 || d->Hkv <= 0 || d->max_tokens <= 0) return KIVI_ERR_ARG;
  if (d->D != 128 || (d->bits != 2 && d->bits != 4) || (d->G != 32 && d->G != 64)) return KIVI_ERR_UNSUPPORTED;
  if (d->max_tokens % d->G != 0) return KIVI_ERR_ARG;
  if (d->value_residual != 0 && d->value_residual != 1) return KIVI_ERR_ARG;
  if (d->value_group < 0) return KIVI_ERR_ARG;
  if (d->value_group != 0 && d->value_group != 32 && d->value_group != 64 && d->value_group != 128)
    return KIVI_ERR_UNSUPPORTED;
  // value channel groups: built for 2-bit codes without a value residual
  if (d->value_group != 0 && d->value_group != 128 && (d->bits != 2 || d->value_residual)) return KIVI_ERR_UNSUPPORTED;
  // token rows are indexed with int64 and buffer sizes in size_t: keep far from both
  const uint64_t heads = (uint64_t)d->B * (uint64_t)d->Hkv;  // below 2^62
  if (heads > kMaxRows || (uint64_t)d->max_tokens > kMaxRows / heads) return KIVI_ERR_UNSUPPORTED;
  return KIVI_OK;
}

int check_cache(const kivi_dims *d, const kivi_cache *c) {
  if (!c || !c->k_codes || !c->k_meta || !c->k_res || !c->v_codes || !c->v_meta) return KIVI_ERR_ARG;
  if (d->value_residual && !c->v_res) return KIVI_ERR_ARG;
  if (!aligned16(c->k_codes) || !aligned16(c->k_meta) || !aligned16(c->k_res) || !aligned16(c->v_codes) ||
      !aligned16(c->v_meta) || (d->value_residual && !aligned16(c->v_res)))
    return KIVI_ERR_ALIGN;
  return KIVI_OK;
}

// The value residual buffer the kernels use: null without the variant.
uint16_t *vres(const kivi_dims *d, const kivi_cache *c) { return d->value_residual ? c->v_res : nullptr; }

// Channels per value {s, z}: D (one per token) unless value channel groups are set.
int vgroup(const kivi_dims *d) { return d->value_group ? d->value_group : d->D; }

// Append token n of every (batch, KV head); when that fills the residual, quantize
// it as group n / G (keys per channel; with a value residual, values per token).
cudaError_t append_and_flush(const kivi_dims *d, const kivi_cache *c, const uint16_t *k_new,
                             const uint16_t *v_new, int64_t n, cudaStream_t st) {
  const int64_t heads = (int64_t)d->B * d->Hkv;
  cudaError_t e = kivi::launch_append(k_new, v_new, heads, n, d->G, d->bits, c->k_res, c->v_codes, c->v_meta,
                                      d->max_tokens, vres(d, c), st, vgroup(d));
  if (e == cudaSuccess && (n % d->G) + 1 == d->G) {
    e = kivi::launch_key_groups(c->k_res, (int64_t)d->G * 128, heads, 1, n / d->G, d->G, d->bits, c->k_codes,
                                c->k_meta, d->max_tokens, st);
    if (e == cudaSuccess && d->value_residual)
      e = kivi::launch_value_rows(c->v_res, heads, d->G, d->G, (n / d->G) * d->G, d->bits, c->v_codes, c->v_meta,
                                  d->max_tokens, st);
  }
  return e;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? KIVI_OK : KIVI_ERR_CUDA; }

int check_heads(const kivi_dims *d, int32_t Hq) {
  if (Hq <= 0) return KIVI_ERR_ARG;
  if (Hq % d->Hkv != 0) return KIVI_ERR_UNSUPPORTED;
  const int R = Hq / d->Hkv;
  if (R != 1 && R != 2 && R != 4) return KIVI_ERR_UNSUPPORTED;
  return KIVI_OK;
}

// ---- paged layout
bool aligned4(const void *p) { return ((uintptr_t)p & 3u) == 0; }

int page_shift_of(int32_t P) {
  int s = 0;
  while ((1 << s) < P && s < 30) ++s;
  return (1 << s) == P ? s : -1;
}

int check_paged_dims(const kivi_paged_dims *d) {
  if (!d) return KIVI_ERR_ARG;
  if (d->B <= 0 || d->Hkv <= 0 || d->page_tokens <= 0 || d->max_pages_per_seq <= 0 || d->num_pages <= 0)
    return KIVI_ERR_ARG;
  if (d->value_residual != 0 && d->value_residual != 1) return KIVI_ERR_ARG;
  if (d->D != 128 || (d->bits != 2 && d->bits != 4) || (d->G != 32 && d->G != 64)) return KIVI_ERR_UNSUPPORTED;
  if (d->B > kivi::kPagedMaxBatch) return KIVI_ERR_UNSUPPORTED;
  const int sh = page_shift_of(d->page_tokens);
  if (sh < 6 || sh > 24) return KIVI_ERR_UNSUPPORTED;  // a power of two, 64 .. 2^24 tokens
  // positions and the device-side unit counts are int32
  const int64_t cap = (int64_t)d->max_pages_per_seq << sh;
  if (cap > INT32_MAX) return KIVI_ERR_UNSUPPORTED;
  if ((int64_t)d->B * (cap / 64 + 1) > INT32_MAX) return KIVI_ERR_UNSUPPORTED;
  if ((int64_t)d->B * d->Hkv > INT32_MAX / 2) return KIVI_ERR_UNSUPPORTED;
  const uint64_t rows_per_page = (uint64_t)d->Hkv << sh;  // below 2^55
  if ((uint64_t)d->num_pages > kMaxRows / rows_per_page) return KIVI_ERR_UNSUPPORTED;
  return KIVI_OK;
}

int check_paged_cache(const kivi_paged_dims *d, const kivi_paged_cache *c) {
  if (!c || !c->k_codes || !c->k_meta || !c->v_codes || !c->v_meta || !c->k_res || !c->block_table ||
      !c->seq_lens)
    return KIVI_ERR_ARG;
  if (d->value_residual && !c->v_res) return KIVI_ERR_ARG;
  if (!aligned16(c->k_codes) || !aligned16(c->k_meta) || !aligned16(c->v_codes) || !aligned16(c->v_meta) ||
      !aligned16(c->k_res) || !aligned4(c->block_table) || !aligned4(c->seq_lens) ||
      (d->value_residual && !aligned16(c->v_res)))
    return KIVI_ERR_ALIGN;
  return KIVI_OK;
}

uint16_t *paged_vres(const kivi_paged_dims *d, const kivi_paged_cache *c) {
  return d->value_residual ? c->v_res : nullptr;
}

int check_paged_heads(const kivi_paged_dims *d, int32_t Hq) {
  if (Hq <= 0) return KIVI_ERR_ARG;
  if (Hq % d->Hkv != 0) return KIVI_ERR_UNSUPPORTED;
  const int R = Hq / d->Hkv;
  if (R != 1 && R != 2 && R != 4) return KIVI_ERR_UNSUPPORTED;
  return KIVI_OK;
}

int32_t paged_cap(const kivi_paged_dims *d) { return d->max_pages_per_seq << page_shift_of(d->page_tokens); }

kivi::PagedAppendArgs paged_append_args(const kivi_paged_dims *d, const kivi_paged_cache *c, const uint16_t *k_new,
                                        const uint16_t *v_new) {
  kivi::PagedAppendArgs a = {};
  a.k_new = k_new;
  a.v_new = v_new;
  a.bt = c->block_table;
  a.seq_lens = c->seq_lens;
  a.k_res = c->k_res;
  a.v_res = paged_vres(d, c);
  a.k_codes = c->k_codes;
  a.k_meta = c->k_meta;
  a.v_codes = c->v_codes;
  a.v_meta = c->v_meta;
  a.num_pages = d->num_pages;
  a.B = d->B;
  a.Hkv = d->Hkv;
  a.G = d->G;
  a.bits = d->bits;
  a.shift = page_shift_of(d->page_tokens);
  a.max_pages = d->max_pages_per_seq;
  return a;
}

kivi::DecodeArgs paged_decode_args(const kivi_paged_dims *d, const kivi_paged_cache *c, const uint16_t *q,
                                   int32_t Hq, float softmax_scale, uint16_t *out, void *ws,
                                   const kivi::PagedGeom &g) {
  kivi::DecodeArgs a = {};
  a.k_codes = c->k_codes;
  a.k_meta = c->k_meta;
  a.k_res = c->k_res;
  a.v_codes = c->v_codes;
  a.v_meta = c->v_meta;
  a.v_res = paged_vres(d, c);
  a.q = q;
  a.out = out;
  a.ws = static_cast<float *>(ws);
  a.B = d->B;
  a.Hkv = d->Hkv;
  a.Hq = Hq;
  a.G = d->G;
  a.bits = d->bits;
  a.n_warps = g.n_warps;
  a.grid = g.grid;
  a.softmax_scale = softmax_scale;
  a.block_table = c->block_table;
  a.seq_lens = c->seq_lens;
  a.num_pages = d->num_pages;
  a.page_shift = page_shift_of(d->page_tokens);
  a.max_pages = d->max_pages_per_seq;
  a.cap_tokens = paged_cap(d);
  return a;
}

}  // namespace

extern "C" {

const char *kivi_status_string(int s) {
  switch (s) {
    case KIVI_OK: return "KIVI_OK";
    case KIVI_ERR_ARG: return "KIVI_ERR_ARG";
    case KIVI_ERR_ALIGN: return "KIVI_ERR_ALIGN";
    case KIVI_ERR_UNSUPPORTED: return "KIVI_ERR_UNSUPPORTED";
    case KIVI_ERR_CAPACITY: return "KIVI_ERR_CAPACITY";
    case KIVI_ERR_WORKSPACE: return "KIVI_ERR_WORKSPACE";
    case KIVI_ERR_CUDA: return "KIVI_ERR_CUDA";
    default: return "KIVI_ERR_UNKNOWN";
  }
}

int kivi_buffer_bytes(const kivi_dims *d, size_t out[6]) {
  int s = check_dims(d);
  if (s != KIVI_OK) return s;
  if (!out) return KIVI_ERR_ARG;
  const size_t heads = (size_t)d->B * (size_t)d->Hkv;
  const size_t T = (size_t)d->max_tokens;
  const size_t wpr = (size_t)d->D * d->bits / 32;  // words of a packed token row
  out[0] = heads * T * wpr * sizeof(uint32_t);
  out[1] = heads * (T / d->G) * d->D * sizeof(uint32_t);
  out[2] = heads * (size_t)d->G * d->D * sizeof(uint16_t);
  out[3] = heads * T * wpr * sizeof(uint32_t);
  out[4] = heads * T * (size_t)(d->D / vgroup(d)) * sizeof(uint32_t);
  out[5] = d->value_residual ? out[2] : 0;
  return KIVI_OK;
}

int kivi_quantize_prefill(const kivi_dims *d, kivi_cache *c, const uint16_t *k, const uint16_t *v, int64_t n,
                          cudaStream_t st) {
  int s = check_dims(d);
  if (s != KIVI_OK) return s;
  if ((s = check_cache(d, c)) != KIVI_OK) return s;
  if (n < 0) return KIVI_ERR_ARG;
  if (n > d->max_tokens) return KIVI_ERR_CAPACITY;
  if (n > 0) {
    if (!k || !v) return KIVI_ERR_ARG;
    if (!aligned16(k) || !aligned16(v)) return KIVI_ERR_ALIGN;
    const int64_t heads = (int64_t)d->B * d->Hkv;
    const int64_t groups = n / d->G, nq = groups * d->G;
    cudaError_t e = kivi::launch_key_groups(k, n * 128, heads, groups, 0, d->G, d->bits, c->k_codes, c->k_meta,
                                            d->max_tokens, st);
    if (e == cudaSuccess) e = kivi::launch_residual_copy(k, heads, n, nq, d->G, c->k_res, st);
    // values: all n quantized, or with a value residual the first nq and the rest kept
    const int64_t nv = d->value_residual ? nq : n;
    if (e == cudaSuccess)
      e = kivi::launch_value_rows(v, heads, nv, n, 0, d->bits, c->v_codes, c->v_meta, d->max_tokens, st, vgroup(d));
    if (e == cudaSuccess && d->value_residual) e = kivi::launch_residual_copy(v, heads, n, nq, d->G, c->v_res, st);
    if ((s = cuda_status(e)) != KIVI_OK) return s;
  }
  c->n_tokens = n;
  return KIVI_OK;
}

int kivi_append_token(const kivi_dims *d, kivi_cache *c, const uint16_t *k_new, const uint16_t *v_new,
                      cudaStream_t st) {
  int s = check_dims(d);
  if (s != KIVI_OK) return s;
  if ((s = check_cache(d, c)) != KIVI_OK) return s;
  if (!k_new || !v_new) return KIVI_ERR_ARG;
  if (!aligned16(k_new) || !aligned16(v_new)) return KIVI_ERR_ALIGN;
  const int64_t n = c->n_tokens;
  if (n < 0) return KIVI_ERR_ARG;
  if (n >= d->max_tokens) return KIVI_ERR_CAPACITY;
  if ((s = cuda_status(append_and_flush(d, c, k_new, v_new, n, st))) != KIVI_OK) return s;
  c->n_tokens = n + 1;
  return KIVI_OK;
}

int kivi_decode_splits(const kivi_dims *d, int32_t Hq, int64_t n) {
  if (check_dims(d) != KIVI_OK || check_heads(d, Hq) != KIVI_OK || n <= 0) return 0;
  kivi::DecodeGeom g;
  if (kivi::decode_geometry(d->B, d->Hkv, Hq, d->G, d->bits, n, &g, vgroup(d)) != cudaSuccess) return 0;
  return g.pmax;
}

size_t kivi_decode_workspace_bytes(const kivi_dims *d, int32_t Hq, int64_t n) {
  const int slots = kivi_decode_splits(d, Hq, n);
  if (slots <= 0) return 0;
  return (size_t)d->B * (size_t)Hq * (size_t)slots * (size_t)(d->D + 2) * sizeof(float);
}

int kivi_decode_attention(const kivi_dims *d, const kivi_cache *c, const uint16_t *q, int32_t Hq,
                          float softmax_scale, uint16_t *out, void *ws, size_t ws_bytes, cudaStream_t st) {
  int s = check_dims(d);
  if (s != KIVI_OK) return s;
  if ((s = check_cache(d, c)) != KIVI_OK) return s;
  if ((s = check_heads(d, Hq)) != KIVI_OK) return s;
  if (!q || !out) return KIVI_ERR_ARG;
  if (!aligned16(q) || !aligned16(out)) return KIVI_ERR_ALIGN;
  if (c->n_tokens <= 0 || c->n_tokens > d->max_tokens) return KIVI_ERR_ARG;
  kivi::DecodeGeom g;
  if (kivi::decode_geometry(d->B, d->Hkv, Hq, d->G, d->bits, c->n_tokens, &g, vgroup(d)) != cudaSuccess)
    return KIVI_ERR_CUDA;
  const size_t need = (size_t)d->B * (size_t)Hq * (size_t)g.pmax * (size_t)(d->D + 2) * sizeof(float);
  if (!ws || ws_bytes < need) return KIVI_ERR_WORKSPACE;
  if (!aligned16(ws)) return KIVI_ERR_ALIGN;
  kivi::DecodeArgs a = {};
  a.k_codes = c->k_codes;
  a.k_meta = c->k_meta;
  a.k_res = c->k_res;
  a.v_codes = c->v_codes;
  a.v_meta = c->v_meta;
  a.v_res = vres(d, c);
  a.q = q;
  a.out = out;
  a.ws = static_cast<float *>(ws);
  a.max_tokens = d->max_tokens;
  a.n = c->n_tokens;
  a.B = d->B;
  a.Hkv = d->Hkv;
  a.Hq = Hq;
  a.G = d->G;
  a.bits = d->bits;
  a.units_per_head = g.units_per_head;
  a.total_units = g.total_units;
  a.n_warps = g.n_warps;
  a.grid = g.grid;
  a.pmax = g.pmax;
  a.small = g.small;
  a.vg = vgroup(d);
  a.wait_tail = 0;
  a.softmax_scale = softmax_scale;
  return cuda_status(kivi::launch_decode(a, st));
}

int kivi_decode_step(const kivi_dims *d, kivi_cache *c, const uint16_t *k_new, const uint16_t *v_new,
                     const uint16_t *q, int32_t Hq, float softmax_scale, uint16_t *out, void *ws, size_t ws_bytes,
                     cudaStream_t st) {
  int s = check_dims(d);
  if (s != KIVI_OK) return s;
  if ((s = check_cache(d, c)) != KIVI_OK) return s;
  if ((s = check_heads(d, Hq)) != KIVI_OK) return s;
  if (!k_new || !v_new || !q || !out) return KIVI_ERR_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(q) || !aligned16(out)) return KIVI_ERR_ALIGN;
  const int64_t n = c->n_tokens;
  if (n < 0) return KIVI_ERR_ARG;
  if (n >= d->max_tokens) return KIVI_ERR_CAPACITY;
  kivi::DecodeGeom g;
  if (kivi::decode_geometry(d->B, d->Hkv, Hq, d->G, d->bits, n + 1, &g, vgroup(d)) != cudaSuccess) return KIVI_ERR_CUDA;
  const size_t need = (size_t)d->B * (size_t)Hq * (size_t)g.pmax * (size_t)(d->D + 2) * sizeof(float);
  if (!ws || ws_bytes < need) return KIVI_ERR_WORKSPACE;
  if (!aligned16(ws)) return KIVI_ERR_ALIGN;
  // 1. append (and flush a full residual group)
  if ((s = cuda_status(append_and_flush(d, c, k_new, v_new, n, st))) != KIVI_OK) return s;
  // 2. decode attention over n + 1 tokens, overlapping the append: only the last
  //    unit of each head (the one holding the new token) waits for it
  kivi::DecodeArgs a = {};
  a.k_codes = c->k_codes;
  a.k_meta = c->k_meta;
  a.k_res = c->k_res;
  a.v_codes = c->v_codes;
  a.v_meta = c->v_meta;
  a.v_res = vres(d, c);
  a.q = q;
  a.out = out;
  a.ws = static_cast<float *>(ws);
  a.max_tokens = d->max_tokens;
  a.n = n + 1;
  a.B = d->B;
  a.Hkv = d->Hkv;
  a.Hq = Hq;
  a.G = d->G;
  a.bits = d->bits;
  a.units_per_head = g.units_per_head;
  a.total_units = g.total_units;
  a.n_warps = g.n_warps;
  a.grid = g.grid;
  a.pmax = g.pmax;
  a.small = g.small;
  a.vg = vgroup(d);
  a.wait_tail = 1;
  a.softmax_scale = softmax_scale;
  if ((s = cuda_status(kivi::launch_decode(a, st))) != KIVI_OK) return s;
  c->n_tokens = n + 1;
  return KIVI_OK;
}

int kivi_dequantize_debug(const kivi_dims *d, const kivi_cache *c, float *k_out, float *v_out, cudaStream_t st) {
  int s = check_dims(d);
  if (s != KIVI_OK) return s;
  if ((s = check_cache(d, c)) != KIVI_OK) return s;
  if (!k_out || !v_out) return KIVI_ERR_ARG;
  if (!aligned16(k_out) || !aligned16(v_out)) return KIVI_ERR_ALIGN;
  if (c->n_tokens < 0 || c->n_tokens > d->max_tokens) return KIVI_ERR_ARG;
  return cuda_status(kivi::launch_dequant(c->k_codes, c->k_meta, c->k_res, c->v_codes, c->v_meta, vres(d, c),
                                          (int64_t)d->B * d->Hkv, c->n_tokens, d->G, d->bits, d->max_tokens, k_out, v_out,
                                          st, vgroup(d)));
}

int kivi_prefill_attention(const kivi_dims *d, kivi_cache *c, const uint16_t *q, int32_t Hq, const uint16_t *k,
                           const uint16_t *v, int64_t n, float softmax_scale, uint16_t *out, cudaStream_t st) {
  int s = check_dims(d);
  if (s != KIVI_OK) return s;
  if (c && (s = check_cache(d, c)) != KIVI_OK) return s;
  if ((s = check_heads(d, Hq)) != KIVI_OK) return s;
  if (n <= 0 || !q || !k || !v || !out) return KIVI_ERR_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return KIVI_ERR_ALIGN;
  if ((int64_t)d->B * Hq > 65535) return KIVI_ERR_UNSUPPORTED;  // grid.y of the launch
  if (c && n > d->max_tokens) return KIVI_ERR_CAPACITY;
  kivi::PrefillArgs a = {};
  a.q = q;
  a.k = k;
  a.v = v;
  a.out = out;
  if (c) {
    a.k_codes = c->k_codes;
    a.k_meta = c->k_meta;
    a.v_codes = c->v_codes;
    a.v_meta = c->v_meta;
    a.k_res = c->k_res;
    a.v_res = vres(d, c);
  }
  a.n = n;
  a.max_tokens = d->max_tokens;
  a.B = d->B;
  a.Hkv = d->Hkv;
  a.Hq = Hq;
  a.G = d->G;
  a.bits = d->bits;
  a.vg = vgroup(d);
  a.softmax_scale = softmax_scale;
  if ((s = cuda_status(kivi::launch_prefill_attention(a, st))) != KIVI_OK) return s;
  if (c) c->n_tokens = n;
  return KIVI_OK;
}

static int fp16_sizes(int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int64_t n, int *splits, int64_t *tps) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || n <= 0) return KIVI_ERR_ARG;
  if (D != 128 || Hq % Hkv != 0) return KIVI_ERR_UNSUPPORTED;
  const int R = Hq / Hkv;
  if (R != 1 && R != 2 && R != 4) return KIVI_ERR_UNSUPPORTED;
  if ((int64_t)B * Hkv > 65535) return KIVI_ERR_UNSUPPORTED;  // grid.y of the launch
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KIVI_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return KIVI_ERR_CUDA;
  kivi::fp16_plan(B, Hkv, n, sms, splits, tps);
  return KIVI_OK;
}

size_t kivi_decode_fp16_workspace_bytes(int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int64_t n) {
  int splits = 0;
  int64_t tps = 0;
  if (fp16_sizes(B, Hq, Hkv, D, n, &splits, &tps) != KIVI_OK) return 0;
  return (size_t)B * (size_t)Hq * (size_t)splits * (size_t)(D + 2) * sizeof(float);
}

int kivi_decode_attention_fp16(int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int64_t n, const uint16_t *k,
                               const uint16_t *v, const uint16_t *q, float softmax_scale, uint16_t *out, void *ws,
                               size_t ws_bytes, cudaStream_t st) {
  if (!k || !v || !q || !out) return KIVI_ERR_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(q) || !aligned16(out)) return KIVI_ERR_ALIGN;
  int splits = 0;
  int64_t tps = 0;
  int s = fp16_sizes(B, Hq, Hkv, D, n, &splits, &tps);
  if (s != KIVI_OK) return s;
  const size_t need = (size_t)B * (size_t)Hq * (size_t)splits * (size_t)(D + 2) * sizeof(float);
  if (!ws || ws_bytes < need) return KIVI_ERR_WORKSPACE;
  if (!aligned16(ws)) return KIVI_ERR_ALIGN;
  kivi::Fp16Args a;
  a.k = k;
  a.v = v;
  a.q = q;
  a.out = out;
  a.ws = static_cast<float *>(ws);
  a.n = n;
  a.B = B;
  a.Hkv = Hkv;
  a.Hq = Hq;
  a.splits = splits;
  a.tiles_per_split = tps;
  a.softmax_scale = softmax_scale;
  return cuda_status(kivi::launch_fp16(a, st));
}

// ---------------------------------------------------------------------- paged cache
int kivi_paged_buffer_bytes(const kivi_paged_dims *d, size_t out[8]) {
  int s = check_paged_dims(d);
  if (s != KIVI_OK) return s;
  if (!out) return KIVI_ERR_ARG;
  const size_t rows = (size_t)d->num_pages * (size_t)d->Hkv * (size_t)d->page_tokens;
  const size_t wpr = (size_t)d->D * d->bits / 32;  // words of a packed token row
  out[0] = rows * wpr * sizeof(uint32_t);
  out[1] = rows / d->G * d->D * sizeof(uint32_t);
  out[2] = rows * wpr * sizeof(uint32_t);
  out[3] = rows * sizeof(uint32_t);
  out[4] = (size_t)d->B * d->Hkv * d->G * d->D * sizeof(uint16_t);
  out[5] = (size_t)d->B * d->max_pages_per_seq * sizeof(int32_t);
  out[6] = (size_t)d->B * sizeof(int32_t);
  out[7] = d->value_residual ? out[4] : 0;
  return KIVI_OK;
}

int kivi_paged_prefill(const kivi_paged_dims *d, const kivi_paged_cache *c, int32_t seq, const uint16_t *k,
                       const uint16_t *v, int64_t n, cudaStream_t st) {
  int s = check_paged_dims(d);
  if (s != KIVI_OK) return s;
  if ((s = check_paged_cache(d, c)) != KIVI_OK) return s;
  if (seq < 0 || seq >= d->B || n < 0) return KIVI_ERR_ARG;
  if (n > paged_cap(d)) return KIVI_ERR_CAPACITY;
  cudaError_t e = cudaSuccess;
  if (n > 0) {
    if (!k || !v) return KIVI_ERR_ARG;
    if (!aligned16(k) || !aligned16(v)) return KIVI_ERR_ALIGN;
    kivi::PageMap pm;
    pm.bt = c->block_table + (int64_t)seq * d->max_pages_per_seq;
    pm.num_pages = d->num_pages;
    pm.shift = page_shift_of(d->page_tokens);
    pm.Hkv = d->Hkv;
    const int64_t groups = n / d->G, nq = groups * d->G;
    e = kivi::launch_key_groups_paged(k, n * 128, d->Hkv, groups, d->G, d->bits, pm, c->k_codes, c->k_meta, st);
    if (e == cudaSuccess)
      e = kivi::launch_residual_copy(k, d->Hkv, n, nq, d->G, c->k_res + (int64_t)seq * d->Hkv * d->G * 128, st);
    const int64_t nv = d->value_residual ? nq : n;
    if (e == cudaSuccess)
      e = kivi::launch_value_rows_paged(v, d->Hkv, nv, n, d->bits, pm, c->v_codes, c->v_meta, st);
    if (e == cudaSuccess && d->value_residual)
      e = kivi::launch_residual_copy(v, d->Hkv, n, nq, d->G, c->v_res + (int64_t)seq * d->Hkv * d->G * 128, st);
  }
  if (e == cudaSuccess) e = kivi::launch_set_len(c->seq_lens, seq, (int32_t)n, st);
  return cuda_status(e);
}

int kivi_paged_append_token(const kivi_paged_dims *d, const kivi_paged_cache *c, const uint16_t *k_new,
                            const uint16_t *v_new, cudaStream_t st) {
  int s = check_paged_dims(d);
  if (s != KIVI_OK) return s;
  if ((s = check_paged_cache(d, c)) != KIVI_OK) return s;
  if (!k_new || !v_new) return KIVI_ERR_ARG;
  if (!aligned16(k_new) || !aligned16(v_new)) return KIVI_ERR_ALIGN;
  cudaError_t e = kivi::launch_paged_append(paged_append_args(d, c, k_new, v_new), st);
  if (e == cudaSuccess) e = kivi::launch_advance_lens(c->seq_lens, d->B, paged_cap(d), st);
  return cuda_status(e);
}

size_t kivi_paged_decode_workspace_bytes(const kivi_paged_dims *d, int32_t Hq) {
  if (check_paged_dims(d) != KIVI_OK || check_paged_heads(d, Hq) != KIVI_OK) return 0;
  kivi::PagedGeom g;
  if (kivi::paged_decode_geometry(d->B, d->Hkv, Hq, d->G, d->bits, &g) != cudaSuccess) return 0;
  return g.ws_bytes;
}

int kivi_paged_decode_attention(const kivi_paged_dims *d, const kivi_paged_cache *c, const uint16_t *q, int32_t Hq,
                                float softmax_scale, uint16_t *out, void *ws, size_t ws_bytes, cudaStream_t st) {
  int s = check_paged_dims(d);
  if (s != KIVI_OK) return s;
  if ((s = check_paged_cache(d, c)) != KIVI_OK) return s;
  if ((s = check_paged_heads(d, Hq)) != KIVI_OK) return s;
  if (!q || !out) return KIVI_ERR_ARG;
  if (!aligned16(q) || !aligned16(out)) return KIVI_ERR_ALIGN;
  kivi::PagedGeom g;
  if (kivi::paged_decode_geometry(d->B, d->Hkv, Hq, d->G, d->bits, &g) != cudaSuccess) return KIVI_ERR_CUDA;
  if (!ws || ws_bytes < g.ws_bytes) return KIVI_ERR_WORKSPACE;
  if (!aligned16(ws)) return KIVI_ERR_ALIGN;
  const kivi::DecodeArgs a = paged_decode_args(d, c, q, Hq, softmax_scale, out, ws, g);
  return cuda_status(kivi::launch_paged_decode(a, st));
}

int kivi_paged_decode_step(const kivi_paged_dims *d, const kivi_paged_cache *c, const uint16_t *k_new,
                           const uint16_t *v_new, const uint16_t *q, int32_t Hq, float softmax_scale, uint16_t *out,
                           void *ws, size_t ws_bytes, cudaStream_t st) {
  int s = check_paged_dims(d);
  if (s != KIVI_OK) return s;
  if ((s = check_paged_cache(d, c)) != KIVI_OK) return s;
  if ((s = check_paged_heads(d, Hq)) != KIVI_OK) return s;
  if (!k_new || !v_new || !q || !out) return KIVI_ERR_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(q) || !aligned16(out)) return KIVI_ERR_ALIGN;
  kivi::PagedGeom g;
  if (kivi::paged_decode_geometry(d->B, d->Hkv, Hq, d->G, d->bits, &g) != cudaSuccess) return KIVI_ERR_CUDA;
  if (!ws || ws_bytes < g.ws_bytes) return KIVI_ERR_WORKSPACE;
  if (!aligned16(ws)) return KIVI_ERR_ALIGN;
  // 1. append (flushing the groups that fill), lengths unchanged
  cudaError_t e = kivi::launch_paged_append(paged_append_args(d, c, k_new, v_new), st);
  if ((s = cuda_status(e)) != KIVI_OK) return s;
  // 2. attention over seq_lens + 1 tokens, overlapping the append; its combine
  //    advances the lengths once everything before it has completed
  kivi::DecodeArgs a = paged_decode_args(d, c, q, Hq, softmax_scale, out, ws, g);
  a.wait_tail = 1;
  a.len_offset = 1;
  a.advance_lens = c->seq_lens;
  return cuda_status(kivi::launch_paged_decode(a, st));
}

}  // extern "C"
