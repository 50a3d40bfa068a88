// Internal declarations shared by the CUDA translation units of liboscar.
#pragma once

#include <cuda.h>   // CUtensorMap (header only: the encoder is fetched from the driver at run time)
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/oscar.h"
#include "per_device_once.h"

namespace oscar {

// a sequence state the kernels accept (see the invariants in oscar.h)
__host__ __device__ __forceinline__ bool state_ok(const oscar_seq_state& st, int S, int W, int max_batch) {
  const int L = st.seq_len, E = st.int2_end;
  return L >= 0 && E >= S && E <= (L > S ? L : S) && L - E <= W && st.window_row >= 0 &&
         st.window_row < max_batch;
}

constexpr int kHeadDim = 128;
constexpr int kPage = 16;
constexpr int kGroup = 32;                   // the default group size
constexpr int kGroups = kHeadDim / kGroup;   // 4 quantisation groups per token (at most)
constexpr int kBlockBytes = OSCAR_PAGE_BLOCK_BYTES;   // block of the default group size (the largest)

// Page block of a group size with ng = 128 / group_size groups per token: codes
// as for every group size, then the fp16 metadata (see include/oscar.h).
__host__ __device__ constexpr int block_bytes(int ng) { return 1024 + 128 * ng; }
// K scales: word gq of chunk t % 8 holds (scale of slot t % 8, scale of slot t % 8 + 8)
__host__ __device__ constexpr int kscale_off(int ng, int t, int gq) {
  return 1024 + 4 * ng * (t & 7) + 4 * gq + 2 * (t >> 3);
}
__host__ __device__ constexpr int kzero_off(int ng, int t, int gq) { return 1024 + 32 * ng + 2 * ng * t + 2 * gq; }
// V scales of slots (2b, 2b + 1) and (2b + 8, 2b + 9) in the first two words of chunk
// 4 gq + b, b = (t % 8) / 2; the zeros in the same order in the next two (vzero_off)
__host__ __device__ constexpr int vscale_off(int ng, int t, int gq) {
  return 1024 + 64 * ng + 16 * (4 * gq + ((t & 7) >> 1)) + 4 * (t >> 3) + 2 * (t & 1);
}
__host__ __device__ constexpr int vzero_off(int ng, int t, int gq) { return vscale_off(ng, t, gq) + 8; }
static_assert(block_bytes(kGroups) == kBlockBytes, "the default block size");
static_assert(block_bytes(2) == OSCAR_PAGE_BLOCK_BYTES_FOR(64), "the group-64 block size");
constexpr int kMaxGqa = 8;
// per-(request, KV head) record written by the query-rotation kernel:
// [0, 1024) fp16x2 mma column fragments of q~ (hi, lo), [1024, 1088) fragments of
// the per-group sums of q~ (hi/lo), [1088] the score scale, rest zero
constexpr int kQrecWords = 1104;
constexpr int kPartFloats = kHeadDim + 4;    // o[128], m, l, 2 pad (rows stay 16-byte aligned)
// BF16 window tokens per decode CTA: short chunks while the window CTAs are few
// (they then run beside the INT2 CTAs, and their latency is what counts), long
// ones when they are many (fewer CTAs: less fixed cost per token)
constexpr int kWindowChunkSmall = 64;
constexpr int kWindowChunkMax = 160;
// INT2 pages one decode CTA streams at most when the split count is automatic
#ifndef OSCAR_SPLIT_PAGES
#define OSCAR_SPLIT_PAGES 512
#endif
constexpr int kSplitPages = OSCAR_SPLIT_PAGES;
// decode CTAs resident per SM (registers and shared memory are sized for it)
constexpr int kDecodeCtasPerSm = 2;
// window chunk of a decode call with `units` (request, KV head) pairs
inline int window_chunk(int window_tokens, int64_t units, int num_sms) {
  const int64_t small = units * ((window_tokens + kWindowChunkSmall - 1) / kWindowChunkSmall);
  return 4 * small <= (int64_t)kDecodeCtasPerSm * num_sms ? kWindowChunkSmall : kWindowChunkMax;
}
inline int window_slots(int window_tokens, int chunk) { return (window_tokens + chunk - 1) / chunk; }

struct AppendParams {
  const int32_t* page_table;
  int32_t pt_stride;
  oscar_seq_state* state;
  const __nv_bfloat16* k;   // [B][n_new][Hkv][128]
  const __nv_bfloat16* v;
  uint8_t* pool;
  int64_t num_pages;
  __nv_bfloat16* window;    // [B][Hkv][2][S+W][128]
  const float* R_K;         // [Hkv][128][128]
  const float* R_V;
  const float* clip_K;      // [Hkv]
  const float* clip_V;
  int32_t num_kv_heads, sink, recent, n_new, batch, max_batch;
  int32_t ngroups;          // quantisation groups per token: 128 / group_size (4 or 2)
  int32_t fold_rv;          // 1: V arrives already rotated (R_V folded into the projection)
  float* trace;             // optional [B][trace_positions][Hkv][2][128]
  int32_t trace_positions;
  uint32_t* err_flags;
  uint32_t* counter;        // zero between launches
  // prefill split: when set, this launch handles only the first `sink` and the
  // last `recent` new tokens (virtual index v < sink -> token v, else token
  // n_new - recent + (v - sink)) and skips tokens that go straight to INT2
  int32_t tail_only;
  int32_t tokens_per_cta;   // set by launch_quant_append
};

// tokens that go straight from the input to INT2 during a long append
struct PrefillParams {
  CUtensorMap tmap_k;       // 4-D TMA maps of k / v: (channel, KV head, token, request), 64 x 1 x 128 x 1
  CUtensorMap tmap_v;       // boxes with a 128-byte swizzle (written by launch_prefill_append)
  const int32_t* page_table;
  int32_t pt_stride;
  const oscar_seq_state* state;
  const __nv_bfloat16* k;   // [B][n_new][Hkv][128]
  const __nv_bfloat16* v;
  uint8_t* pool;
  int64_t num_pages;
  const uint8_t* images;    // [Hkv][4][32 KiB]: R_K hi, R_K lo, R_V hi, R_V lo (bf16, swizzled)
  const float* clip_K;
  const float* clip_V;
  int32_t num_kv_heads, sink, recent, n_new, batch, max_batch;
  int32_t ngroups;          // quantisation groups per token: 128 / group_size (4 or 2)
  float* trace;
  int32_t trace_positions;
  uint32_t* err_flags;
};

struct DecodeParams {
  const __nv_bfloat16* q;   // [B][Hq][128]
  const int32_t* page_table;
  int32_t pt_stride;
  const oscar_seq_state* state;
  const uint8_t* pool;
  int64_t num_pages;
  const __nv_bfloat16* window;
  const float* R_K;         // [Hkv][128][128]
  const float* R_VT;        // [Hkv][128][128], R_VT[h][i][j] = R_V[h][j][i]
  uint32_t* qrec;           // [B][Hkv][kQrecWords]
  float* part;              // [B][Hkv][win_slots + splits][gqa][kPartFloats]
  float* o;                 // [B][Hq][128]
  const float* pv_scale;    // [Hkv] power of two applied to p * s_v before fp16 rounding
  int32_t num_q_heads, num_kv_heads, gqa, sink, recent, splits, fold_rv, max_batch;
  int32_t win_slots;        // CTAs over the BF16 window, win_chunk tokens each
  int32_t win_chunk;        // kWindowChunkSmall or kWindowChunkMax (window_chunk)
  int32_t ngroups;          // quantisation groups per token: 128 / group_size (4 or 2)
  int32_t batch;            // requests of this call
  // shared prefix: requests 0 .. batch-1 map positions [0, prefix_tokens) to the
  // same pages; prefix CTAs attend over that range once for `pack` requests at a
  // time (their query heads side by side in the tensor-core columns), split
  // prefix_splits ways; prefix_tokens = 0: no shared range
  int32_t prefix_tokens, prefix_splits, pack;
  float scale_log2;         // softmax_scale * log2(e)
  uint32_t* err_flags;
  // A decode step (oscar_decode_step): one new token per request is appended by
  // the call itself. step_slots = 1 adds, after the splits, the slot of the
  // position the step quantises (written by one more CTA per request and KV
  // head, which also writes the new token into the window); every other CTA
  // works from the state before the step, and the merge publishes the new one.
  // step_slots = 0 (a plain decode): the fields below are unused.
  int32_t step_slots;
  const __nv_bfloat16* step_k;   // [B][Hkv][128], 16-byte aligned
  const __nv_bfloat16* step_v;
  oscar_seq_state* step_state;   // = state, written by the merge
  uint8_t* step_pool;            // = pool, writable
  __nv_bfloat16* step_window;    // = window, writable
  const float* R_V;              // [Hkv][128][128]
  const float* clip_K;           // [Hkv]
  const float* clip_V;
};

// partial slots of a decode call per (request, KV head): window chunks, shared
// prefix splits, splits, and the slot of a step's newly quantised position
__host__ __device__ __forceinline__ int total_slots(const DecodeParams& p) {
  return p.win_slots + p.prefix_splits + p.splits + p.step_slots;
}

// Programmatic dependent launch: kernels launched with launch_pdl may start
// while the previous kernel on the stream is still running. Before its
// pdl_wait a kernel touches only constant data (rotations, their images), reads
// caller inputs that no kernel of this library writes (q, k, v) and host-set
// fields that kernels only rewrite unchanged (a request's window row), and
// issues level-2 prefetches, which return no data; every kernel calls pdl_wait
// before it exits. So a kernel's predecessor completes
// only after the predecessor's own predecessor did, and by induction everything
// after a kernel's pdl_wait runs once all earlier kernels on the stream have
// completed, wherever those kernels placed their pdl_trigger. The append lets
// its dependents start at once, so that the query rotation stages R_K and
// computes q~ beside it.
// A decode step's append CTA reads only R_K, R_V (level-2 prefetch) and the
// caller's q, k and v before its wait; its writes (window, page, partial) and the
// merge's state publication come after the waits.
// One exception to "constant data": the no-alloc decode keeps R_V^T and the
// probability scales in its shared scratch array and rewrites them at every
// call with an ordinary (non-overlapping) preparation launch, while the merge
// kernel stages R_V^T before its pdl_wait. That stays ordered because the
// decode kernel, the merge's predecessor, triggers its dependents only after
// its own pdl_wait, which runs after the query rotation and hence after the
// preparation kernel. A decode kernel that triggered before its wait would let
// the merge read the previous call's R_V^T.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;\n" ::); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// run `setup` (returning a cudaError_t) once for the current device
template <typename F>
cudaError_t once_for_current_device(PerDeviceOnce& once, F&& setup) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int r = once.run_on(dev, [&] { return (int)setup(); });
  return r < 0 ? cudaErrorInvalidDevice : (cudaError_t)r;
}

// launchers (return cudaGetLastError())
// ev_before / ev_after (may be null): recorded on s around the main launch
cudaError_t launch_quant_append(const AppendParams& p, cudaStream_t s, cudaEvent_t ev_before = nullptr,
                                cudaEvent_t ev_after = nullptr);
cudaError_t launch_prefill_append(const PrefillParams& p, int ctas_per_head, cudaStream_t s,
                                  cudaEvent_t ev_before = nullptr, cudaEvent_t ev_after = nullptr);
bool prefill_supported(const void* k, const void* v);   // TMA needs 16-byte aligned inputs
int prefill_image_bytes();
cudaError_t launch_decode(const DecodeParams& p, int batch, cudaStream_t s, cudaEvent_t ev_before = nullptr,
                          cudaEvent_t ev_after = nullptr);
int decode_smem_bytes();
// offline calibration: causal attention outputs of every query head into o_ws
// (calib_workspace_bytes), then C_Q and C_S per KV head (fp32 [hkv][128][128])
size_t calib_workspace_bytes(int n, int hq);
cudaError_t launch_calib_covariances(const __nv_bfloat16* q, const __nv_bfloat16* k, const __nv_bfloat16* v, int n,
                                     int hq, int hkv, float scale, float* c_q, float* c_s, float* o_ws,
                                     cudaStream_t s);

}  // namespace oscar
