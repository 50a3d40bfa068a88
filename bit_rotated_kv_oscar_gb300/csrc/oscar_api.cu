// C ABI of liboscar: context, validation, workspace and kernel launches.
// The statement of every entry point is in include/oscar.h.
#include <math.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <new>
#include <string>
#include <vector>

#include "oscar_internal.cuh"

using namespace oscar;

struct oscar_ctx {
  oscar_config cfg{};
  int device = 0;
  int num_sms = 0;
  // bound cache
  uint8_t* pool = nullptr;
  int64_t num_pages = 0;
  __nv_bfloat16* window = nullptr;
  // owned device memory
  float* R_K = nullptr;
  float* R_V = nullptr;
  float* R_VT = nullptr;
  float* clip_K = nullptr;
  float* clip_V = nullptr;
  float* pv_scale = nullptr;
  uint8_t* images = nullptr;    // per KV head: R_K hi/lo, R_V hi/lo as swizzled bf16 tensor-core operands
  uint32_t* qrec = nullptr;
  float* part = nullptr;
  uint32_t* flags = nullptr;    // [0] error flags, [1] append ticket counter
  int max_splits = 0;
  bool loaded = false;
  std::string last_error;
};

namespace {

const char* kNullCtxMsg = "null context";

int fail(oscar_ctx* ctx, int status, const std::string& msg) {
  if (ctx) ctx->last_error = msg;
  return status;
}

int cuda_fail(oscar_ctx* ctx, cudaError_t e, const char* what) {
  std::string m = std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
  return fail(ctx, OSCAR_ERR_CUDA, m);
}

int check_config_msg(const oscar_config* c, std::string* msg) {
  if (!c) {
    *msg = "null config";
    return OSCAR_ERR_INVALID_ARG;
  }
  if (c->num_q_heads < 1 || c->num_kv_heads < 1 || c->num_q_heads % c->num_kv_heads) {
    *msg = "num_q_heads must be a positive multiple of num_kv_heads";
    return OSCAR_ERR_INVALID_ARG;
  }
  if (c->sink < 0 || c->recent < 1 || c->max_batch < 1 || c->max_pages_per_seq < 1 ||
      c->num_splits < 0 || !(c->softmax_scale >= 0.f) || isinf(c->softmax_scale)) {
    *msg = "sink >= 0, recent >= 1, max_batch >= 1, max_pages_per_seq >= 1, num_splits >= 0, "
           "finite softmax_scale >= 0 required";
    return OSCAR_ERR_INVALID_ARG;
  }
  if (c->head_dim != kHeadDim || c->page_size != kPage || (c->group_size != 32 && c->group_size != 64)) {
    *msg = "only head_dim 128, page_size 16, group_size 32 or 64 are built";
    return OSCAR_ERR_UNSUPPORTED;
  }
  const int g = c->num_q_heads / c->num_kv_heads;
  if (g != 1 && g != 2 && g != 4 && g != 8) {
    *msg = "query group size must be 1, 2, 4 or 8";
    return OSCAR_ERR_UNSUPPORTED;
  }
  if (c->num_splits > 256) {
    *msg = "num_splits must not exceed 256";
    return OSCAR_ERR_UNSUPPORTED;
  }
  if (c->sink + c->recent > 1024) {
    *msg = "sink + recent must not exceed 1024";
    return OSCAR_ERR_UNSUPPORTED;
  }
  if ((int64_t)c->max_pages_per_seq * kPage > INT32_MAX) {
    *msg = "max_pages_per_seq too large for int32 positions";
    return OSCAR_ERR_INVALID_ARG;
  }
  return OSCAR_OK;
}

// device address of page-locked host memory, nullptr for other memory
void* mapped_host(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

// window CTAs per (request, KV head): at most this many (the short chunks)
int win_slots(const oscar_config* c) { return window_slots(c->sink + c->recent, kWindowChunkSmall); }
int win_chunk_for(const oscar_ctx* ctx, int batch) {
  return window_chunk(ctx->cfg.sink + ctx->cfg.recent, (int64_t)batch * ctx->cfg.num_kv_heads, ctx->num_sms);
}

// extra: CTAs per (request, KV head) besides the window and the splits (a
// decode step's append CTA)
int auto_splits(const oscar_ctx* ctx, int batch, int extra = 0) {
  if (ctx->cfg.num_splits > 0) return ctx->cfg.num_splits;
  const int64_t units = (int64_t)batch * ctx->cfg.num_kv_heads;
  const int64_t pages = ctx->cfg.max_pages_per_seq;
  // fill one wave of decode CTAs together with the BF16-window CTAs; at most
  // kSplitPages pages per CTA
  const int64_t wins = units * (window_slots(ctx->cfg.sink + ctx->cfg.recent, win_chunk_for(ctx, batch)) + extra);
  int64_t by_wave = (kDecodeCtasPerSm * (int64_t)ctx->num_sms - wins) / units;
  int64_t by_pages = (pages + kSplitPages - 1) / kSplitPages;
  int64_t s = by_wave > by_pages ? by_wave : by_pages;
  const int64_t cap = (pages + 7) / 8;  // keep >= 8 pages per split
  if (s > cap) s = cap;
  if (s > 256) s = 256;
  if (s < 1) s = 1;
  return (int)s;
}

// bf16 bits of a finite float, round to nearest even
uint16_t bf16_bits(float x) {
  uint32_t u;
  memcpy(&u, &x, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}
float bf16_value(uint16_t b) {
  const uint32_t u = (uint32_t)b << 16;
  float x;
  memcpy(&x, &u, 4);
  return x;
}

// Tensor-core operand images of one 128 x 128 rotation R: B[n][k] = R[k][n]
// (K-major, output channel n per row), split R = hi + lo in bf16, laid out in
// 128-byte-swizzle atoms of 64 columns: element (n, k) at atom k / 64, row n,
// 16-byte chunk ((k % 64) / 8) ^ (n % 8), position k % 8.
void rotation_images(const float* R, bool identity, uint16_t* hi, uint16_t* lo) {
  for (int k = 0; k < kHeadDim; ++k)
    for (int n = 0; n < kHeadDim; ++n) {
      const float r = identity ? (k == n ? 1.f : 0.f) : R[k * kHeadDim + n];
      const uint16_t bh = bf16_bits(r);
      const uint16_t bl = bf16_bits(r - bf16_value(bh));
      const int atom = k >> 6, cc = (k & 63) >> 3;
      const size_t off = (size_t)atom * 8192 + (size_t)n * 64 + (size_t)((cc ^ (n & 7)) * 8) + (k & 7);
      hi[off] = bh;
      lo[off] = bl;
    }
}

template <class T>
cudaError_t dalloc(T** p, size_t bytes) {
  return cudaMalloc(reinterpret_cast<void**>(p), bytes);
}

}  // namespace

extern "C" {

int oscar_version(void) { return OSCAR_ABI_VERSION; }

const char* oscar_status_string(int status) {
  switch (status) {
    case OSCAR_OK: return "ok";
    case OSCAR_ERR_INVALID_ARG: return "invalid argument";
    case OSCAR_ERR_NOT_LOADED: return "rotations not loaded";
    case OSCAR_ERR_OUT_OF_RANGE: return "out of range";
    case OSCAR_ERR_CUDA: return "CUDA error";
    case OSCAR_ERR_UNSUPPORTED: return "unsupported shape";
    case OSCAR_ERR_NOT_BOUND: return "cache not bound";
    default: return "unknown status";
  }
}

int oscar_check_config(const oscar_config* cfg) {
  std::string msg;
  return check_config_msg(cfg, &msg);
}

int oscar_cache_bytes(const oscar_config* cfg, int64_t num_pages, size_t* pool_bytes,
                      size_t* window_bytes) {
  std::string msg;
  int st = check_config_msg(cfg, &msg);
  if (st) return st;
  if (num_pages < 0 || !pool_bytes || !window_bytes) return OSCAR_ERR_INVALID_ARG;
  *pool_bytes = (size_t)num_pages * cfg->num_kv_heads * block_bytes(kHeadDim / cfg->group_size);
  *window_bytes = (size_t)cfg->max_batch * cfg->num_kv_heads * 2 * (cfg->sink + cfg->recent) *
                  kHeadDim * sizeof(__nv_bfloat16);
  return OSCAR_OK;
}

void oscar_destroy(oscar_ctx* ctx) {
  if (!ctx) return;
  cudaFree(ctx->R_K);
  cudaFree(ctx->R_V);
  cudaFree(ctx->R_VT);
  cudaFree(ctx->clip_K);
  cudaFree(ctx->clip_V);
  cudaFree(ctx->pv_scale);
  cudaFree(ctx->images);
  cudaFree(ctx->qrec);
  cudaFree(ctx->part);
  cudaFree(ctx->flags);
  delete ctx;
}

int oscar_create(const oscar_config* cfg, oscar_ctx** out) {
  if (!out) return OSCAR_ERR_INVALID_ARG;
  *out = nullptr;
  std::string msg;
  int st = check_config_msg(cfg, &msg);
  if (st) return st;
  oscar_ctx* ctx = new (std::nothrow) oscar_ctx();
  if (!ctx) return OSCAR_ERR_CUDA;
  ctx->cfg = *cfg;
  if (ctx->cfg.softmax_scale == 0.f) ctx->cfg.softmax_scale = 1.f / sqrtf((float)kHeadDim);
  cudaError_t e = cudaGetDevice(&ctx->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&ctx->num_sms, cudaDevAttrMultiProcessorCount, ctx->device);
  const int hkv = cfg->num_kv_heads, g = cfg->num_q_heads / cfg->num_kv_heads;
  const size_t rbytes = (size_t)hkv * kHeadDim * kHeadDim * sizeof(float);
  if (e == cudaSuccess) e = dalloc(&ctx->R_K, rbytes);
  if (e == cudaSuccess) e = dalloc(&ctx->R_V, rbytes);
  if (e == cudaSuccess) e = dalloc(&ctx->R_VT, rbytes);
  if (e == cudaSuccess) e = dalloc(&ctx->clip_K, hkv * sizeof(float));
  if (e == cudaSuccess) e = dalloc(&ctx->clip_V, hkv * sizeof(float));
  if (e == cudaSuccess) e = dalloc(&ctx->pv_scale, hkv * sizeof(float));
  if (e == cudaSuccess) e = dalloc(&ctx->images, (size_t)hkv * prefill_image_bytes());
  if (e == cudaSuccess) {
    ctx->max_splits = auto_splits(ctx, cfg->max_batch);
    for (int b = 1; b < cfg->max_batch; ++b) {
      int s = auto_splits(ctx, b);
      if (s > ctx->max_splits) ctx->max_splits = s;
    }
    e = dalloc(&ctx->qrec, (size_t)cfg->max_batch * hkv * kQrecWords * sizeof(uint32_t));
  }
  if (e == cudaSuccess)
    e = dalloc(&ctx->part, (size_t)cfg->max_batch * hkv * (2 * ctx->max_splits + win_slots(cfg)) * g *
                               kPartFloats * sizeof(float));  // shared-prefix calls: two sets of splits
  if (e == cudaSuccess) e = dalloc(&ctx->flags, 2 * sizeof(uint32_t));
  if (e == cudaSuccess) e = cudaMemset(ctx->flags, 0, 2 * sizeof(uint32_t));
  if (e != cudaSuccess) {
    oscar_destroy(ctx);
    return OSCAR_ERR_CUDA;
  }
  *out = ctx;
  return OSCAR_OK;
}

int oscar_bind_cache(oscar_ctx* ctx, void* int2_pool, int64_t num_pages, void* window) {
  if (!ctx) return OSCAR_ERR_INVALID_ARG;
  if (!int2_pool || !window || num_pages < 1)
    return fail(ctx, OSCAR_ERR_INVALID_ARG, "bind_cache: null buffer or num_pages < 1");
  if (((uintptr_t)int2_pool & 15) || ((uintptr_t)window & 15))
    return fail(ctx, OSCAR_ERR_INVALID_ARG, "bind_cache: pool and window must be 16-byte aligned");
  if (num_pages > INT32_MAX) return fail(ctx, OSCAR_ERR_INVALID_ARG, "bind_cache: page ids are int32");
  ctx->pool = static_cast<uint8_t*>(int2_pool);
  ctx->num_pages = num_pages;
  ctx->window = static_cast<__nv_bfloat16*>(window);
  return OSCAR_OK;
}

int oscar_load_rotations(oscar_ctx* ctx, const float* R_K, const float* R_V, const float* clip_K,
                         const float* clip_V) {
  if (!ctx) return OSCAR_ERR_INVALID_ARG;
  if (!R_K || !R_V || !clip_K || !clip_V)
    return fail(ctx, OSCAR_ERR_INVALID_ARG, "load_rotations: null pointer");
  const int hkv = ctx->cfg.num_kv_heads;
  const size_t n = (size_t)hkv * kHeadDim * kHeadDim;
  std::vector<float> rvt(n), ps(hkv);
  for (int h = 0; h < hkv; ++h) {
    if (!(clip_K[h] > 0.f) || !(clip_V[h] > 0.f) || isinf(clip_K[h]) || isinf(clip_V[h]))
      return fail(ctx, OSCAR_ERR_INVALID_ARG, "load_rotations: clip values must be finite and > 0");
    for (int i = 0; i < kHeadDim; ++i)
      for (int j = 0; j < kHeadDim; ++j) {
        const float a = R_K[((size_t)h * kHeadDim + i) * kHeadDim + j];
        const float bv = R_V[((size_t)h * kHeadDim + i) * kHeadDim + j];
        if (!isfinite(a) || !isfinite(bv))
          return fail(ctx, OSCAR_ERR_INVALID_ARG, "load_rotations: non-finite rotation entry");
        rvt[((size_t)h * kHeadDim + j) * kHeadDim + i] = bv;
      }
    // largest power of two with 2^8 * pscale * (2 clip_V / 3) * 1.01 <= 65504, at most
    // 2^7: decode feeds fp16 p * pscale * s_v to the tensor cores with p <= 2^8
    const double smax = 2.0 * clip_V[h] / 3.0 * 1.01 * 256.0;
    int ex = (int)floor(log2(65504.0 / smax));
    if (ex > 7) ex = 7;
    if (ex < -30) ex = -30;
    ps[h] = ldexpf(1.f, ex);
  }
  // prefill operands: 4 images of 128 x 128 bf16 per head
  std::vector<uint16_t> img((size_t)hkv * 4 * kHeadDim * kHeadDim);
  for (int h = 0; h < hkv; ++h) {
    uint16_t* base = img.data() + (size_t)h * 4 * kHeadDim * kHeadDim;
    const size_t m = (size_t)kHeadDim * kHeadDim;
    rotation_images(R_K + (size_t)h * m, false, base, base + m);
    rotation_images(R_V + (size_t)h * m, ctx->cfg.fold_rv != 0, base + 2 * m, base + 3 * m);
  }
  cudaError_t e = cudaMemcpy(ctx->images, img.data(), img.size() * sizeof(uint16_t), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(ctx->R_K, R_K, n * sizeof(float), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(ctx->R_V, R_V, n * sizeof(float), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(ctx->R_VT, rvt.data(), n * sizeof(float), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(ctx->clip_K, clip_K, hkv * sizeof(float), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(ctx->clip_V, clip_V, hkv * sizeof(float), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(ctx->pv_scale, ps.data(), hkv * sizeof(float), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "load_rotations");
  ctx->loaded = true;
  return OSCAR_OK;
}

static int append_impl(oscar_ctx* ctx, const int32_t* page_table, oscar_seq_state* state,
                       const void* k, const void* v, int32_t batch, int32_t n_new, float* trace,
                       int32_t trace_positions, void* stream, cudaEvent_t ev_before = nullptr,
                       cudaEvent_t ev_after = nullptr) {
  if (!ctx) return OSCAR_ERR_INVALID_ARG;
  if (!ctx->loaded) return fail(ctx, OSCAR_ERR_NOT_LOADED, "quant_append: rotations not loaded");
  if (!ctx->pool) return fail(ctx, OSCAR_ERR_NOT_BOUND, "quant_append: no cache bound");
  if (!page_table || !state || !k || !v)
    return fail(ctx, OSCAR_ERR_INVALID_ARG, "quant_append: null pointer");
  if (batch < 1 || n_new < 0) return fail(ctx, OSCAR_ERR_INVALID_ARG, "quant_append: batch >= 1, n_new >= 0");
  if (batch > ctx->cfg.max_batch)
    return fail(ctx, OSCAR_ERR_OUT_OF_RANGE, "quant_append: batch exceeds max_batch");
  if ((int64_t)n_new > (int64_t)ctx->cfg.max_pages_per_seq * kPage)
    return fail(ctx, OSCAR_ERR_OUT_OF_RANGE, "quant_append: n_new exceeds the page-table capacity");
  if (trace && trace_positions < 1)
    return fail(ctx, OSCAR_ERR_INVALID_ARG, "quant_append: trace_positions must be >= 1");
  if (n_new == 0) return OSCAR_OK;
  AppendParams p{};
  p.page_table = page_table;
  p.pt_stride = ctx->cfg.max_pages_per_seq;
  p.state = state;
  p.k = static_cast<const __nv_bfloat16*>(k);
  p.v = static_cast<const __nv_bfloat16*>(v);
  p.pool = ctx->pool;
  p.num_pages = ctx->num_pages;
  p.window = ctx->window;
  p.R_K = ctx->R_K;
  p.R_V = ctx->R_V;
  p.clip_K = ctx->clip_K;
  p.clip_V = ctx->clip_V;
  p.num_kv_heads = ctx->cfg.num_kv_heads;
  p.sink = ctx->cfg.sink;
  p.ngroups = kHeadDim / ctx->cfg.group_size;
  p.recent = ctx->cfg.recent;
  p.n_new = n_new;
  p.batch = batch;
  p.max_batch = ctx->cfg.max_batch;
  p.fold_rv = ctx->cfg.fold_rv;
  p.trace = trace;
  p.trace_positions = trace ? trace_positions : 0;
  p.err_flags = ctx->flags;
  p.counter = ctx->flags + 1;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // long appends: the tokens that go straight to INT2 run on the tensor cores,
  // the sink / ring / eviction tokens on the per-token kernel right after
  if (n_new >= ctx->cfg.sink + ctx->cfg.recent + 128 && prefill_supported(k, v)) {
    PrefillParams pp{};
    pp.page_table = page_table;
    pp.pt_stride = ctx->cfg.max_pages_per_seq;
    pp.state = state;
    pp.k = p.k;
    pp.v = p.v;
    pp.pool = ctx->pool;
    pp.num_pages = ctx->num_pages;
    pp.images = ctx->images;
    pp.clip_K = ctx->clip_K;
    pp.clip_V = ctx->clip_V;
    pp.num_kv_heads = ctx->cfg.num_kv_heads;
    pp.sink = ctx->cfg.sink;
    pp.ngroups = kHeadDim / ctx->cfg.group_size;
    pp.recent = ctx->cfg.recent;
    pp.n_new = n_new;
    pp.batch = batch;
    pp.max_batch = ctx->cfg.max_batch;
    pp.trace = p.trace;
    pp.trace_positions = p.trace_positions;
    pp.err_flags = ctx->flags;
    const int tiles = (n_new + 127) / 128 + 1;
    int cph = ctx->num_sms / (ctx->cfg.num_kv_heads * batch);
    if (cph < 1) cph = 1;
    if (cph > tiles) cph = tiles;
    cudaError_t e = launch_prefill_append(pp, cph, st, ev_before, ev_after);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "quant_append (tensor-core part) launch");
    p.tail_only = 1;
    ev_before = ev_after = nullptr;
  }
  cudaError_t e = launch_quant_append(p, st, ev_before, ev_after);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "quant_append launch");
  return OSCAR_OK;
}

int oscar_quant_append(oscar_ctx* ctx, const int32_t* page_table, oscar_seq_state* state,
                       const void* k, const void* v, int32_t batch, int32_t n_new, void* stream) {
  return append_impl(ctx, page_table, state, k, v, batch, n_new, nullptr, 0, stream);
}

int oscar_quant_append_traced(oscar_ctx* ctx, const int32_t* page_table, oscar_seq_state* state,
                              const void* k, const void* v, int32_t batch, int32_t n_new,
                              float* trace, int32_t trace_positions, void* stream) {
  if (!trace) return fail(ctx, OSCAR_ERR_INVALID_ARG, "quant_append_traced: null trace");
  return append_impl(ctx, page_table, state, k, v, batch, n_new, trace, trace_positions, stream);
}

int oscar_quant_append_timed(oscar_ctx* ctx, const int32_t* page_table, oscar_seq_state* state,
                             const void* k, const void* v, int32_t batch, int32_t n_new, void* stream,
                             void* ev_before, void* ev_after) {
  return append_impl(ctx, page_table, state, k, v, batch, n_new, nullptr, 0, stream,
                     static_cast<cudaEvent_t>(ev_before), static_cast<cudaEvent_t>(ev_after));
}

int oscar_decode_splits(const oscar_ctx* ctx, int32_t batch, int32_t* splits) {
  if (!ctx || !splits || batch < 1) return OSCAR_ERR_INVALID_ARG;
  *splits = auto_splits(ctx, batch);
  return OSCAR_OK;
}

// split counts of a shared-prefix call: the prefix pages are attended once per
// pack of requests (8 / g of them side by side in the tensor-core columns), the
// rest of every request as usual; both sets of slices fit the workspace
static void shared_prefix_splits(const oscar_ctx* ctx, int batch, int prefix_tokens, int* pack, int* prefix_splits,
                                 int* splits) {
  const int g = ctx->cfg.num_q_heads / ctx->cfg.num_kv_heads;
  *pack = std::min(kMaxGqa / g, (int)batch);
  const int64_t groups = (batch + *pack - 1) / *pack;
  const int64_t ppages = std::max(0, prefix_tokens / kPage - ctx->cfg.sink / kPage);
  const int64_t units = groups * ctx->cfg.num_kv_heads;
  int64_t by_wave = (kDecodeCtasPerSm * (int64_t)ctx->num_sms) / std::max<int64_t>(units, 1);
  int64_t by_pages = (ppages + kSplitPages - 1) / kSplitPages;
  int64_t ps = std::max(by_wave, by_pages);
  ps = std::min<int64_t>(ps, std::max<int64_t>((ppages + 7) / 8, 1));  // >= 8 pages per slice
  const int64_t spages = std::max<int64_t>(ctx->cfg.max_pages_per_seq - prefix_tokens / kPage, 1);
  int64_t ss = std::max<int64_t>((spages + kSplitPages - 1) / kSplitPages, 1);
  const int64_t cap = std::min<int64_t>(2 * ctx->max_splits, 256);
  ss = std::min(ss, cap - 1);
  ps = std::max<int64_t>(std::min(ps, cap - ss), 1);
  *prefix_splits = (int)ps;
  *splits = (int)ss;
}

// step_k / step_v non-null: a decode step (oscar_decode_step), the one-token
// append of every request done inside the call
static int decode_impl(oscar_ctx* ctx, const void* q, const int32_t* page_table, const oscar_seq_state* state,
                       float* o, int32_t batch, void* stream, cudaEvent_t ev_before, cudaEvent_t ev_after,
                       int32_t prefix_tokens = 0, const void* step_k = nullptr, const void* step_v = nullptr) {
  if (!ctx) return OSCAR_ERR_INVALID_ARG;
  if (!ctx->loaded) return fail(ctx, OSCAR_ERR_NOT_LOADED, "decode_attn: rotations not loaded");
  if (!ctx->pool) return fail(ctx, OSCAR_ERR_NOT_BOUND, "decode_attn: no cache bound");
  if (!q || !page_table || !state || !o) return fail(ctx, OSCAR_ERR_INVALID_ARG, "decode_attn: null pointer");
  if (batch < 1) return fail(ctx, OSCAR_ERR_INVALID_ARG, "decode_attn: batch >= 1");
  if (batch > ctx->cfg.max_batch) return fail(ctx, OSCAR_ERR_OUT_OF_RANGE, "decode_attn: batch exceeds max_batch");
  if (prefix_tokens < 0 || prefix_tokens % kPage != 0 ||
      (int64_t)prefix_tokens > (int64_t)ctx->cfg.max_pages_per_seq * kPage)
    return fail(ctx, OSCAR_ERR_INVALID_ARG, "decode_attn: prefix_tokens must be a multiple of 16 within the page table");
  DecodeParams p{};
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.page_table = page_table;
  p.pt_stride = ctx->cfg.max_pages_per_seq;
  p.state = state;
  p.pool = ctx->pool;
  p.num_pages = ctx->num_pages;
  p.window = ctx->window;
  p.R_K = ctx->R_K;
  p.R_VT = ctx->R_VT;
  p.qrec = ctx->qrec;
  p.part = ctx->part;
  p.o = o;
  p.pv_scale = ctx->pv_scale;
  p.num_q_heads = ctx->cfg.num_q_heads;
  p.num_kv_heads = ctx->cfg.num_kv_heads;
  p.gqa = ctx->cfg.num_q_heads / ctx->cfg.num_kv_heads;
  p.sink = ctx->cfg.sink;
  p.ngroups = kHeadDim / ctx->cfg.group_size;
  p.recent = ctx->cfg.recent;
  const bool step = step_k != nullptr;
  p.splits = auto_splits(ctx, batch, step ? 1 : 0);
  p.win_chunk = win_chunk_for(ctx, batch);
  p.win_slots = window_slots(ctx->cfg.sink + ctx->cfg.recent, p.win_chunk);
  p.batch = batch;
  p.prefix_tokens = 0;
  p.prefix_splits = 0;
  p.pack = 1;
  if (prefix_tokens > 0) {
    p.prefix_tokens = prefix_tokens;
    shared_prefix_splits(ctx, batch, prefix_tokens, &p.pack, &p.prefix_splits, &p.splits);
  }
  p.fold_rv = ctx->cfg.fold_rv;
  p.max_batch = ctx->cfg.max_batch;
  p.scale_log2 = ctx->cfg.softmax_scale * 1.4426950408889634f;
  p.err_flags = ctx->flags;
  if (step) {
    p.step_slots = 1;
    p.step_k = static_cast<const __nv_bfloat16*>(step_k);
    p.step_v = static_cast<const __nv_bfloat16*>(step_v);
    p.step_state = const_cast<oscar_seq_state*>(state);   // the caller's writable state (oscar_decode_step)
    p.step_pool = ctx->pool;
    p.step_window = ctx->window;
    p.R_V = ctx->R_V;
    p.clip_K = ctx->clip_K;
    p.clip_V = ctx->clip_V;
  }
  cudaError_t e = launch_decode(p, batch, static_cast<cudaStream_t>(stream), ev_before, ev_after);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "decode_attn launch");
  return OSCAR_OK;
}

int oscar_decode_attn(oscar_ctx* ctx, const void* q, const int32_t* page_table,
                      const oscar_seq_state* state, float* o, int32_t batch, void* stream) {
  return decode_impl(ctx, q, page_table, state, o, batch, stream, nullptr, nullptr);
}

int oscar_decode_attn_shared_prefix(oscar_ctx* ctx, const void* q, const int32_t* page_table,
                                    const oscar_seq_state* state, int32_t prefix_tokens, float* o, int32_t batch,
                                    void* stream) {
  return decode_impl(ctx, q, page_table, state, o, batch, stream, nullptr, nullptr, prefix_tokens);
}

int oscar_decode_attn_timed(oscar_ctx* ctx, const void* q, const int32_t* page_table,
                            const oscar_seq_state* state, float* o, int32_t batch, void* stream,
                            void* ev_before, void* ev_after) {
  return decode_impl(ctx, q, page_table, state, o, batch, stream, static_cast<cudaEvent_t>(ev_before),
                     static_cast<cudaEvent_t>(ev_after));
}

// one decode step on device buffers: the append and the attention in the same
// launches when k and v allow 16-byte copies, else the append kernel first
static int step_impl(oscar_ctx* ctx, const int32_t* page_table, oscar_seq_state* state, const void* q,
                     const void* k, const void* v, float* o, int32_t batch, void* stream) {
  if (!ctx) return OSCAR_ERR_INVALID_ARG;
  if (!k || !v) return fail(ctx, OSCAR_ERR_INVALID_ARG, "decode_step: null pointer");
  if (((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) & 15) == 0)
    return decode_impl(ctx, q, page_table, state, o, batch, stream, nullptr, nullptr, 0, k, v);
  const int st = append_impl(ctx, page_table, state, k, v, batch, 1, nullptr, 0, stream);
  if (st != OSCAR_OK) return st;
  return decode_impl(ctx, q, page_table, state, o, batch, stream, nullptr, nullptr);
}

int oscar_decode_step(oscar_ctx* ctx, const int32_t* page_table, oscar_seq_state* state, const void* q,
                      const void* k, const void* v, float* o, int32_t batch, void* stream) {
  return step_impl(ctx, page_table, state, q, k, v, o, batch, stream);
}

int oscar_decode_step_host(oscar_ctx* ctx, const int32_t* page_table, oscar_seq_state* state,
                           const void* h_qkv, void* d_qkv, float* o, float* h_o, int32_t batch,
                           void* stream) {
  if (!ctx) return OSCAR_ERR_INVALID_ARG;
  if (!h_qkv || !h_o) return fail(ctx, OSCAR_ERR_INVALID_ARG, "decode_step_host: null pointer");
  if (batch < 1) return fail(ctx, OSCAR_ERR_INVALID_ARG, "decode_step_host: batch >= 1");
  if (batch > ctx->cfg.max_batch)
    return fail(ctx, OSCAR_ERR_OUT_OF_RANGE, "decode_step_host: batch exceeds max_batch");
  // page-locked host memory is addressed by the kernels directly (over the
  // host-device link); other host memory goes through the staging buffer and
  // the device output with copies
  const uint8_t* in = static_cast<const uint8_t*>(mapped_host(h_qkv));
  float* out = static_cast<float*>(mapped_host(h_o));
  if (!in && !d_qkv) return fail(ctx, OSCAR_ERR_INVALID_ARG, "decode_step_host: null pointer (d_qkv)");
  if (!in && (reinterpret_cast<uintptr_t>(d_qkv) & 15))
    return fail(ctx, OSCAR_ERR_INVALID_ARG, "decode_step_host: d_qkv must be 16-byte aligned");
  if (!out && !o) return fail(ctx, OSCAR_ERR_INVALID_ARG, "decode_step_host: null pointer (o)");
  const size_t qbytes = (size_t)batch * ctx->cfg.num_q_heads * kHeadDim * sizeof(__nv_bfloat16);
  const size_t kbytes = (size_t)batch * ctx->cfg.num_kv_heads * kHeadDim * sizeof(__nv_bfloat16);
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (!in) {
    e = cudaMemcpyAsync(d_qkv, h_qkv, qbytes + 2 * kbytes, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "decode_step_host: input copy");
    in = static_cast<const uint8_t*>(d_qkv);
  }
  const int st = step_impl(ctx, page_table, state, in, in + qbytes, in + qbytes + kbytes, out ? out : o, batch, stream);
  if (st != OSCAR_OK) return st;
  if (!out) {
    e = cudaMemcpyAsync(h_o, o, (size_t)batch * ctx->cfg.num_q_heads * kHeadDim * sizeof(float),
                        cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "decode_step_host: output copy");
  }
  return OSCAR_OK;
}

int oscar_error_flags(oscar_ctx* ctx, uint32_t* flags, int32_t clear) {
  if (!ctx || !flags) return OSCAR_ERR_INVALID_ARG;
  cudaError_t e = cudaDeviceSynchronize();
  uint32_t f = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&f, ctx->flags, sizeof(uint32_t), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && clear) e = cudaMemset(ctx->flags, 0, sizeof(uint32_t));
  if (e != cudaSuccess) return cuda_fail(ctx, e, "error_flags");
  *flags = f;
  return OSCAR_OK;
}

const char* oscar_last_error(const oscar_ctx* ctx) {
  if (!ctx) return kNullCtxMsg;
  return ctx->last_error.c_str();
}

size_t oscar_calibration_workspace_bytes(int32_t n, int32_t num_q_heads) {
  if (n < 1 || num_q_heads < 1) return 0;
  return calib_workspace_bytes(n, num_q_heads);
}

int oscar_calibration_covariances(const void* q, const void* k, const void* v, int32_t n, int32_t num_q_heads,
                                  int32_t num_kv_heads, float softmax_scale, float* c_q, float* c_s,
                                  void* workspace, size_t workspace_bytes, void* stream) {
  if (!q || !k || !v || !c_q || !c_s || !workspace || n < 1 || num_kv_heads < 1 || num_q_heads < num_kv_heads ||
      num_q_heads % num_kv_heads != 0 || !(softmax_scale >= 0.f) || isinf(softmax_scale))
    return OSCAR_ERR_INVALID_ARG;
  if (workspace_bytes < calib_workspace_bytes(n, num_q_heads)) return OSCAR_ERR_OUT_OF_RANGE;
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.f / sqrtf((float)kHeadDim);
  cudaError_t e = launch_calib_covariances(static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
                                           static_cast<const __nv_bfloat16*>(v), n, num_q_heads, num_kv_heads, scale,
                                           c_q, c_s, static_cast<float*>(workspace), static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
}

}  // extern "C"
