// Decode attention for callers that cannot allocate device memory.
//
// Some hosts of this library cannot call cudaMalloc: code running inside a
// CUDA-graph capture that must not add allocation nodes, plug-ins whose
// device memory is budgeted by another runtime, or allocator-free embedded
// runtimes. oscar_decode_attn_noalloc gives them the fused decode attention
// without a context: every buffer the computation reads or writes is passed
// in, and the split-K workspace lives in a fixed array in this library's own
// device memory (oscar_noalloc_scratch below), reserved on every GPU that loads
// the library for as long as the process lives.
//
// The array is shared by all calls on a device and keeps whatever the last
// call left in it; each call rewrites the parts it reads (and clears the error
// word it uses) before reading them. Two calls whose work overlaps on the GPU
// (different streams, or different host threads on one stream without
// ordering) race on the array and may produce wrong results.
//
// The address of the array is looked up once per device, with that device
// current, on the first call made on it; make that first call before any
// stream capture begins.
#include <math.h>

#include <mutex>

#include "oscar_internal.cuh"

namespace oscar {

constexpr size_t kNoallocScratchBytes = OSCAR_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) uint8_t oscar_noalloc_scratch[kNoallocScratchBytes];

namespace {

std::mutex g_mu;
void* g_scratch[kMaxDevices] = {};

size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }

// same split rule as the context-based decode
int noalloc_splits(const oscar_config* c, int num_sms, int batch) {
  if (c->num_splits > 0) return c->num_splits;
  const int64_t units = (int64_t)batch * c->num_kv_heads;
  const int64_t pages = c->max_pages_per_seq;
  const int64_t wins = units * window_slots(c->sink + c->recent, window_chunk(c->sink + c->recent, units, num_sms));
  int64_t by_wave = (kDecodeCtasPerSm * (int64_t)num_sms - wins) / units;
  int64_t by_pages = (pages + kSplitPages - 1) / kSplitPages;
  int64_t s = by_wave > by_pages ? by_wave : by_pages;
  const int64_t cap = (pages + 7) / 8;
  if (s > cap) s = cap;
  if (s > 256) s = 256;
  if (s < 1) s = 1;
  return (int)s;
}

// per-call preparation inside the scratch array: R_V^T, the probability scale of
// each KV head (largest power of two p with 2^8 * p * (2 clip_V / 3) * 1.01 <=
// 65504, at most 2^7) and a cleared error word
__global__ void __launch_bounds__(256) oscar_noalloc_prep_kernel(const float* __restrict__ R_V,
                                                                  const float* __restrict__ clip_V,
                                                                  float* RVT, float* pv_scale,
                                                                  uint32_t* flags, int hkv) {
  const int h = blockIdx.x;
  const float* src = R_V + (size_t)h * kHeadDim * kHeadDim;
  float* dst = RVT + (size_t)h * kHeadDim * kHeadDim;
  for (int i = threadIdx.x; i < kHeadDim * kHeadDim; i += blockDim.x) {
    const int r = i / kHeadDim, c = i % kHeadDim;
    dst[c * kHeadDim + r] = src[i];
  }
  if (threadIdx.x == 0) {
    const double smax = 2.0 * (double)clip_V[h] / 3.0 * 1.01 * 256.0;
    int ex = (int)floor(log2(65504.0 / smax));
    if (ex > 7) ex = 7;
    if (ex < -30) ex = -30;
    pv_scale[h] = ldexpf(1.f, ex);
    if (h == 0 && flags) *flags = 0u;
  }
}

}  // namespace
}  // namespace oscar

using namespace oscar;

extern "C" int oscar_decode_attn_noalloc(const oscar_config* cfg, const void* q, const int32_t* page_table,
                                         const oscar_seq_state* state, float* o, int32_t batch,
                                         const void* int2_pool, int64_t num_pages, const void* window,
                                         const float* R_K, const float* R_V, const float* clip_V,
                                         uint32_t* err_flags, void* stream) {
  if (oscar_check_config(cfg) != OSCAR_OK) return oscar_check_config(cfg);
  if (!q || !page_table || !state || !o || !int2_pool || !window || !R_K || !R_V || !clip_V)
    return OSCAR_ERR_INVALID_ARG;
  if (batch < 1 || num_pages < 1 || num_pages > INT32_MAX) return OSCAR_ERR_INVALID_ARG;
  if (batch > cfg->max_batch) return OSCAR_ERR_OUT_OF_RANGE;
  if (((uintptr_t)int2_pool & 15) || ((uintptr_t)window & 15) || ((uintptr_t)R_K & 15) ||
      ((uintptr_t)R_V & 15))
    return OSCAR_ERR_INVALID_ARG;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return OSCAR_ERR_CUDA;
  int num_sms = 0;
  if (cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return OSCAR_ERR_CUDA;

  const int hkv = cfg->num_kv_heads, g = cfg->num_q_heads / cfg->num_kv_heads;
  const int splits = noalloc_splits(cfg, num_sms, batch);
  const int win_chunk = window_chunk(cfg->sink + cfg->recent, (int64_t)batch * cfg->num_kv_heads, num_sms);
  const int win_slots = window_slots(cfg->sink + cfg->recent, win_chunk);
  // scratch layout: R_V^T | pv_scale | error word | q~ records | split-K partials
  const size_t off_rvt = 0;
  const size_t off_pv = off_rvt + round256((size_t)hkv * kHeadDim * kHeadDim * sizeof(float));
  const size_t off_flags = off_pv + round256((size_t)hkv * sizeof(float));
  const size_t off_qrec = off_flags + 256;
  const size_t off_part = off_qrec + round256((size_t)batch * hkv * kQrecWords * sizeof(uint32_t));
  const size_t total =
      off_part + round256((size_t)batch * hkv * (win_slots + splits) * g * kPartFloats * sizeof(float));
  if (total > kNoallocScratchBytes) return OSCAR_ERR_OUT_OF_RANGE;

  uint8_t* base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch[dev]) {
      void* ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, oscar_noalloc_scratch) != cudaSuccess || !ptr) return OSCAR_ERR_CUDA;
      g_scratch[dev] = ptr;
    }
    base = static_cast<uint8_t*>(g_scratch[dev]);
  }

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* rvt = reinterpret_cast<float*>(base + off_rvt);
  float* pv = reinterpret_cast<float*>(base + off_pv);
  uint32_t* flags = err_flags ? err_flags : reinterpret_cast<uint32_t*>(base + off_flags);
  oscar_noalloc_prep_kernel<<<hkv, 256, 0, s>>>(R_V, clip_V, rvt, pv, err_flags ? nullptr : flags, hkv);
  if (cudaGetLastError() != cudaSuccess) return OSCAR_ERR_CUDA;

  DecodeParams p{};
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.page_table = page_table;
  p.pt_stride = cfg->max_pages_per_seq;
  p.state = state;
  p.pool = static_cast<const uint8_t*>(int2_pool);
  p.num_pages = num_pages;
  p.window = static_cast<const __nv_bfloat16*>(window);
  p.R_K = R_K;
  p.R_VT = rvt;
  p.qrec = reinterpret_cast<uint32_t*>(base + off_qrec);
  p.part = reinterpret_cast<float*>(base + off_part);
  p.o = o;
  p.pv_scale = pv;
  p.num_q_heads = cfg->num_q_heads;
  p.num_kv_heads = hkv;
  p.gqa = g;
  p.sink = cfg->sink;
  p.ngroups = kHeadDim / cfg->group_size;
  p.batch = batch;
  p.prefix_tokens = 0;
  p.prefix_splits = 0;
  p.pack = 1;
  p.recent = cfg->recent;
  p.splits = splits;
  p.fold_rv = cfg->fold_rv;
  p.max_batch = cfg->max_batch;
  p.win_slots = win_slots;
  p.win_chunk = win_chunk;
  const float scale = cfg->softmax_scale == 0.f ? 1.f / sqrtf((float)kHeadDim) : cfg->softmax_scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.err_flags = flags;
  if (launch_decode(p, batch, s) != cudaSuccess) return OSCAR_ERR_CUDA;
  return OSCAR_OK;
}
