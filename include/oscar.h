/*
 * oscar.h - C ABI of the OSCAR INT2 KV-cache serving library (GB300, sm_103a).
 *
 * The library implements the online serving path of OSCAR (Offline Spectral
 * Covariance-Aware Rotation): the write path that rotates each new key or value
 * vector by a fixed per-head rotation, clips it and stores it as packed 2-bit
 * groups in a paged cache, and the fused decode attention that reads BF16 sink
 * and recent tokens together with the INT2 history in one pass.
 *
 * Sources, cited by page title and section:
 *   [IT] "OSCAR: Offline Spectral Covariance-Aware Rotation for 2-bit KV Cache
 *        Quantization", gist.science explainer (Italian), "Riepilogo Tecnico".
 *   [ES] "Juntos, AI Open-Sources OSCAR: un sistema de cuantificación de caché KV
 *        de 2 bits consciente de la atención para servicios de LLM de contexto
 *        prolongado", 7minutos.es.
 *
 * Conventions shared by every call
 *   - Activations are row vectors; a rotation acts on the right: x_rot = x @ R,
 *     R row-major [d][d], x_rot[j] = sum_i x[i] * R[i][j].
 *   - Every function returns 0 (OSCAR_OK) or a negative oscar_status. No call
 *     aborts, throws or traps; the message of the last failure on a context is
 *     returned by oscar_last_error().
 *   - Device buffers (pool, window, page table, state, q, k, v, o) are owned by
 *     the caller. The library owns its device copies of the rotations and clip
 *     values and a split-K workspace allocated by oscar_create().
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Kernel work is asynchronous on that stream; errors found by the host are
 *     reported at once, errors found by the device are latched in a flag word
 *     read by oscar_error_flags().
 *   - Kernels are launched with programmatic dependent launch and let the next
 *     launch on the stream start only once their own inputs were complete. A
 *     caller's kernel that runs right before a call of this library and itself
 *     allows early dependent launch must likewise do so only after its own
 *     prerequisites completed (the query rotation of oscar_decode_attn reads q
 *     as soon as it starts).
 *   - Supported shapes: head_dim 128, page_size 16, group_size 32 or 64 (the
 *     same for K and V), and a query group (num_q_heads / num_kv_heads) of 1,
 *     2, 4 or 8. Anything else is OSCAR_ERR_UNSUPPORTED.
 *
 * Storage formats (owned by the library, allocated by the caller)
 *
 *   INT2 pool: num_pages * num_kv_heads blocks of BB = 1024 + 128 * NG bytes,
 *   NG = 128 / group_size groups per token (BB = 1536 for group_size 32, 1280
 *   for 64; OSCAR_PAGE_BLOCK_BYTES_FOR(group_size)); the block of page id p and
 *   KV head h starts at byte (p * num_kv_heads + h) * BB. A page holds 16
 *   consecutive positions, slot t = position % 16. Codes and metadata of one
 *   token are spread over the block so that each lane of a warp reads the
 *   exact operand fragment it feeds to the tensor cores:
 *     K code of slot t, channel c (2 bits, bytes [0, 512)):
 *       i = c/16, r = c%16, x = r/8, b = (r%8)/2, hi = r%2, a = t%8, th = t/8;
 *       32-bit little-endian word at byte 16*(4a+b) + 4*(2*th+x), bit 16*hi+2*i.
 *     V code of slot t, channel c (bytes [512, 1024)):
 *       i = c/16, r = c%16, x = r/8, a = r%8, tt = t/8, b = (t%8)/2, hi = t%2;
 *       word at byte 512 + 16*(4a+b) + 4*(2*tt+x), bit 16*hi+2*i.
 *     fp16 scale and zero of group gq (channels group_size*gq ..) of slot t,
 *       with a = t%8, b = (t%8)/2, pair = t/8, half = t%2 (bytes [1024, BB)):
 *       K scale at byte 1024 + 4*NG*a + 4*gq + 2*pair;
 *       K zero  at byte 1024 + 32*NG + 2*NG*t + 2*gq;
 *       V scale at byte 1024 + 64*NG + 16*(4*gq + b) + 4*pair + 2*half,
 *       V zero 8 bytes later.
 *   Slots of positions outside [sink, int2_end) are never read.
 *
 *   Window: bf16 [max_batch][num_kv_heads][2 (K, V)][sink + recent][128],
 *   row r = window_row of a request. Slot s < sink holds position s; slot
 *   sink + (pos % recent) holds a recent position pos.
 *
 *   Page table: int32 [batch][max_pages_per_seq]; entry n maps positions
 *   [16n, 16n+16) of the request to a page id. Several requests may map the
 *   same page id (shared prefix); such pages must not be appended to.
 *
 *   Sequence state: oscar_seq_state [batch] in device memory. seq_len = cached
 *   tokens L; int2_end = E, the first position still held in BF16 after the
 *   sink; window_row = the request's row of the BF16 window. A new request is
 *   {0, sink, row, 0}. Invariants: sink <= E, E <= max(L, sink), L - E <= recent,
 *   0 <= window_row < max_batch. Positions [0, min(sink, L)) are in the sink,
 *   [sink, E) are INT2, [E, L) are in the recent ring. Because every request
 *   carries its own window row, a call may pass any subset of requests (for
 *   example page_table + b * max_pages_per_seq and state + b with batch 1).
 */
#ifndef OSCAR_H
#define OSCAR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define OSCAR_ABI_VERSION 1
#define OSCAR_PAGE_BLOCK_BYTES 1536 /* group_size 32 */
#define OSCAR_PAGE_BLOCK_BYTES_FOR(group_size) (1024 + 128 * (128 / (group_size)))

typedef enum oscar_status {
  OSCAR_OK = 0,
  OSCAR_ERR_INVALID_ARG = -1,  /* null pointer, bad shape or size */
  OSCAR_ERR_NOT_LOADED = -2,   /* rotations not loaded */
  OSCAR_ERR_OUT_OF_RANGE = -3, /* batch or length beyond what the context was created for */
  OSCAR_ERR_CUDA = -4,         /* a CUDA runtime call failed; see oscar_last_error */
  OSCAR_ERR_UNSUPPORTED = -5,  /* shape the kernels are not built for */
  OSCAR_ERR_NOT_BOUND = -6     /* no cache bound to the context */
} oscar_status;

/* Device-side error flags (bit set = condition seen since the last clear). */
#define OSCAR_FLAG_BAD_PAGE_ID 1u   /* a page-table entry outside [0, num_pages); access skipped */
#define OSCAR_FLAG_BAD_STATE 2u     /* a sequence state breaking the invariants; request skipped */
#define OSCAR_FLAG_TIMEOUT 4u       /* a bounded wait inside a kernel expired; its remaining work skipped */

typedef struct oscar_config {
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;          /* 128 */
  int32_t page_size;         /* 16 */
  int32_t group_size;        /* 32 or 64: channels per quantisation group (K and V) */
  int32_t sink;              /* S >= 0: leading tokens kept in BF16 */
  int32_t recent;            /* W >= 1: trailing tokens kept in BF16 */
  int32_t max_batch;         /* requests per call, >= 1 */
  int32_t max_pages_per_seq; /* page-table row stride, >= 1 */
  float softmax_scale;       /* 0 selects 1/sqrt(head_dim) */
  int32_t fold_rv;           /* 1: R_V is folded into the model's value and output projections
                                ([ES] "El sistema de servicio"): values arrive already in the
                                R_V basis, so the write path does not rotate V and decode
                                returns its output in the R_V basis (no R_V^T applied) */
  int32_t num_splits;        /* INT2 splits per (request, KV head) in decode; 0 = automatic */
} oscar_config;

typedef struct oscar_seq_state {
  int32_t seq_len;    /* L */
  int32_t int2_end;   /* E */
  int32_t window_row; /* row of the BF16 window that holds this request, [0, max_batch) */
  int32_t reserved;   /* 0 */
} oscar_seq_state;

typedef struct oscar_ctx oscar_ctx;

/* ABI version (OSCAR_ABI_VERSION). */
int oscar_version(void);

/* Static text for a status code. */
const char* oscar_status_string(int status);

/* Host-only check of a configuration: OSCAR_OK, OSCAR_ERR_INVALID_ARG or
 * OSCAR_ERR_UNSUPPORTED. Touches no GPU. */
int oscar_check_config(const oscar_config* cfg);

/* Bytes the caller must allocate for an INT2 pool of num_pages pages and for
 * the BF16 window of cfg->max_batch requests. Host only. [IT] 2.2 B (paged
 * mixed-precision layout); [ES] "El sistema de servicio" (sink / recent / history). */
int oscar_cache_bytes(const oscar_config* cfg, int64_t num_pages, size_t* pool_bytes,
                      size_t* window_bytes);

/* Create a context on the current CUDA device: validates cfg, allocates the
 * rotation copies and the split-K workspace. *out is NULL on failure. */
int oscar_create(const oscar_config* cfg, oscar_ctx** out);

/* Free a context and everything it allocated (NULL is ignored). */
void oscar_destroy(oscar_ctx* ctx);

/* Bind caller-owned device memory: the INT2 pool (oscar_cache_bytes bytes,
 * 16-byte aligned) and the BF16 window. May be called again to rebind. */
int oscar_bind_cache(oscar_ctx* ctx, void* int2_pool, int64_t num_pages, void* window);

/* Load the fixed per-layer rotations and clip values computed offline.
 * [IT] 2.2 A (R_K = U_Q H_Had P_br, R_V = U_S H_Had P_br, clip thresholds from
 * the rotated calibration activations); [ES] "Lo que OSCAR hace diferente".
 * R_K, R_V: HOST float32 [num_kv_heads][128][128] row-major; clip_K, clip_V:
 * HOST float32 [num_kv_heads], > 0. Copied synchronously; the caller keeps
 * ownership of its arrays. */
int oscar_load_rotations(oscar_ctx* ctx, const float* R_K, const float* R_V,
                         const float* clip_K, const float* clip_V);

/* Write path: append n_new tokens to each of `batch` requests.
 * [ES] "El sistema de servicio": each token is rotated, clipped to the
 * calibrated threshold and quantised to asymmetric per-token INT2 groups;
 * sink and recent tokens stay in BF16.
 * k, v: DEVICE bf16 [batch][n_new][num_kv_heads][128] (positions L..L+n_new-1).
 * page_table: DEVICE int32 [batch][max_pages_per_seq]; it must map every
 * position below the new int2_end. state: DEVICE [batch], read and updated.
 * With E' = max(E, sink, L + n_new - recent): positions below sink go to the
 * sink, positions in [E, E') are rotated (x @ R), clipped to [-c, c],
 * quantised per group of group_size channels (32 or 64, from the config) with
 * s = fp16((max-min)/3), z = fp16(min),
 * code = clamp(rint((x - z) * fp32(1/s)), 0, 3) (0 when s == 0), and packed; taken from
 * the ring when already cached, else from k/v. The remaining new positions go
 * to the ring. Afterwards state = {L + n_new, E'}. */
int oscar_quant_append(oscar_ctx* ctx, const int32_t* page_table, oscar_seq_state* state,
                       const void* k, const void* v, int32_t batch, int32_t n_new,
                       void* stream);

/* oscar_quant_append that also records, for every token it quantises, the
 * rotated float32 value before clipping: trace DEVICE float32
 * [batch][trace_positions][num_kv_heads][2 (K, V)][128], indexed by absolute
 * position; positions >= trace_positions are not recorded. Same arithmetic. */
int oscar_quant_append_traced(oscar_ctx* ctx, const int32_t* page_table,
                              oscar_seq_state* state, const void* k, const void* v,
                              int32_t batch, int32_t n_new, float* trace,
                              int32_t trace_positions, void* stream);

/* Read path: one decode query per request over its whole cache.
 * [IT] 2.2 B "Integrazione del Kernel"; [ES] "El sistema de servicio" (unpack,
 * dequantise, undo the rotation and attend in one pass). Because R is
 * orthogonal the library rotates the query by R_K instead of de-rotating
 * every key, accumulates INT2 values in the R_V basis and applies R_V^T to
 * the merged output once (skipped when fold_rv = 1).
 * q: DEVICE bf16 [batch][num_q_heads][128]; o: DEVICE float32
 * [batch][num_q_heads][128]; query head j reads KV head j / (Hq/Hkv).
 * o = softmax(q K^T * softmax_scale) V over all L cached positions; a request
 * with L = 0 gets o = 0. */
int oscar_decode_attn(oscar_ctx* ctx, const void* q, const int32_t* page_table,
                      const oscar_seq_state* state, float* o, int32_t batch, void* stream);

/* Decode for requests that share a prefix: the same result as oscar_decode_attn,
 * with the INT2 positions of the shared range read once per pack of requests.
 * Prefix caching is kept in the paged cache ([ES] "El sistema de servicio"
 * keeps prefix caching and paged attention); this call adds reading an aliased
 * page once for several requests, which the pages leave open.
 * Contract: requests 0 .. batch-1 map positions [0, prefix_tokens) to the same
 * page ids (page_table rows equal on their first prefix_tokens / 16 entries,
 * as after a fork), and prefix_tokens <= int2_end <= seq_len for each of them.
 * prefix_tokens: a multiple of 16 (0 = no shared range: oscar_decode_attn).
 * The shared range [sink, prefix_tokens) is attended once for every 8 / g
 * requests (their g query heads side by side in the tensor-core columns), each
 * request's own positions after it as usual. A request breaking the contract
 * sets OSCAR_FLAG_BAD_STATE and gets no contribution from the shared range. */
int oscar_decode_attn_shared_prefix(oscar_ctx* ctx, const void* q, const int32_t* page_table,
                                    const oscar_seq_state* state, int32_t prefix_tokens, float* o,
                                    int32_t batch, void* stream);

/* One serving step on device buffers: every request gets one new token,
 * written to the cache, and one decode query over the cache that then holds it
 * ([ES] "El sistema de servicio": the new K / V enter the BF16 sink or ring,
 * the ring entry they replace is quantised to INT2, and the step attends over
 * sink, ring and INT2 history). The same cache contents, state and output as
 * oscar_quant_append(k, v, n_new = 1) followed by oscar_decode_attn(q), in the
 * decode call's launches: one more CTA per request and KV head writes the new
 * token, quantises the position that leaves the ring (the append kernel's
 * arithmetic, so the same bytes) and attends over it, while the other CTAs
 * attend over the rest; the state is published by the call's last launch.
 * q: DEVICE bf16 [batch][num_q_heads][128]; k, v: DEVICE bf16
 * [batch][num_kv_heads][128]; o: DEVICE float32 [batch][num_q_heads][128];
 * state: DEVICE [batch], read and updated as by oscar_quant_append. With k or v
 * not 16-byte aligned the call runs oscar_quant_append, then oscar_decode_attn.
 * A decode step may use one INT2 split fewer than oscar_decode_attn (its
 * append CTAs take their place in the wave). Statuses as for those calls. */
int oscar_decode_step(oscar_ctx* ctx, const int32_t* page_table, oscar_seq_state* state, const void* q,
                      const void* k, const void* v, float* o, int32_t batch, void* stream);

/* One serving step with host-side inputs and output: every request gets one
 * new token, written to the cache, then one decode query over the cache that
 * now holds it ([ES] "El sistema de servicio": the new K / V enter the BF16
 * ring and the oldest ring entry is quantised, then the step attends over sink,
 * ring and INT2 history).
 * h_qkv: HOST bf16, q [batch][num_q_heads][128], then k and v
 * [batch][num_kv_heads][128] each, back to back. h_o: HOST float32
 * [batch][num_q_heads][128], written. On `stream`: oscar_decode_step(q, k, v)
 * into the output; asynchronous, h_o holds the result once the stream has
 * passed the call.
 * Page-locked host memory (cudaHostAlloc / cudaHostRegister) is read and
 * written by the kernels in place over the host-device link: then d_qkv and o
 * are not used and may be NULL. Other host memory goes through copies: h_qkv
 * to d_qkv (DEVICE staging buffer of the same layout and size, 16-byte
 * aligned, caller-owned) before, and o (DEVICE float32 of h_o's size) to h_o
 * after. h_qkv must stay unchanged until the stream has passed the call.
 * Statuses as for those calls, and OSCAR_ERR_INVALID_ARG for a null pointer
 * that is needed or a misaligned staging buffer, OSCAR_ERR_CUDA for a failed
 * copy. */
int oscar_decode_step_host(oscar_ctx* ctx, const int32_t* page_table, oscar_seq_state* state,
                           const void* h_qkv, void* d_qkv, float* o, float* h_o, int32_t batch,
                           void* stream);

/* Number of INT2 splits per (request, KV head) decode uses for `batch`. */
int oscar_decode_splits(const oscar_ctx* ctx, int32_t batch, int32_t* splits);

/* Read (and optionally clear) the device error flags. Synchronises the
 * device. flags receives an OR of OSCAR_FLAG_* bits. */
int oscar_error_flags(oscar_ctx* ctx, uint32_t* flags, int32_t clear);

/* Message of the last failure on ctx ("" if none; a static text for NULL). */
const char* oscar_last_error(const oscar_ctx* ctx);

/* Measurement variants (no counterpart on the method's pages: a profiling aid of
 * this library). They do exactly what oscar_decode_attn / oscar_quant_append do
 * and in addition record two caller-created CUDA events (cudaEvent_t, passed as
 * void*, either may be NULL) on `stream`: ev_before just before and ev_after just
 * after the launch of the main kernel - the split-K attention kernel of the
 * decode call; the tensor-core kernel of a long append (an append short enough
 * to take only the per-token kernel records the events around that kernel). The
 * records order that launch after its predecessor and before its successor, so
 * the programmatic overlap between neighbouring launches is lost while timing.
 * Statuses and errors as for the untimed calls. */
int oscar_decode_attn_timed(oscar_ctx* ctx, const void* q, const int32_t* page_table,
                            const oscar_seq_state* state, float* o, int32_t batch, void* stream,
                            void* ev_before, void* ev_after);
int oscar_quant_append_timed(oscar_ctx* ctx, const int32_t* page_table, oscar_seq_state* state,
                             const void* k, const void* v, int32_t batch, int32_t n_new, void* stream,
                             void* ev_before, void* ev_after);

/* Offline calibration on the device (no context): the covariance targets of the
 * rotations of one layer, "OSCAR: Offline Spectral Covariance-Aware Rotation
 * ..." (gist.science, it), Riepilogo Tecnico 2.2 A "Stima della Covarianza".
 * q: DEVICE bf16 [n][num_q_heads][128], k, v: DEVICE bf16 [n][num_kv_heads][128]
 * (the calibration activations of the layer, token-major); c_q, c_s: DEVICE
 * float32 [num_kv_heads][128][128], written:
 *   c_q[h] = (1/(n g)) sum over h's g query heads j and tokens t of q_jt^T q_jt,
 *   c_s[h] = (1/(n g)) sum_j (S_j V_h)^T (S_j V_h), S_j = causal softmax of
 *            q_j k_h^T * softmax_scale (0: 1/sqrt(128)),
 * accumulated in float32. workspace: caller-owned DEVICE memory of at least
 * oscar_calibration_workspace_bytes(n, num_q_heads) bytes (the attention
 * outputs S_j V_h). Asynchronous on stream. The rotations follow on the host:
 * eigenvectors in descending eigenvalue order, R = U H P.
 * Returns OSCAR_ERR_INVALID_ARG for a null pointer or inconsistent sizes,
 * OSCAR_ERR_OUT_OF_RANGE for a workspace that is too small, OSCAR_ERR_CUDA
 * for a launch failure. */
size_t oscar_calibration_workspace_bytes(int32_t n, int32_t num_q_heads);
int oscar_calibration_covariances(const void* q, const void* k, const void* v, int32_t n, int32_t num_q_heads,
                                  int32_t num_kv_heads, float softmax_scale, float* c_q, float* c_s,
                                  void* workspace, size_t workspace_bytes, void* stream);

/* Size of the fixed device array behind oscar_decode_attn_noalloc. */
#define OSCAR_NOALLOC_SCRATCH_BYTES (32u << 20)

/* Decode attention that allocates nothing (no counterpart on the method's pages:
 * this is an integration aid of this library).
 *
 * For callers that cannot call cudaMalloc: code recorded into a CUDA graph that
 * must not contain allocations, plug-ins whose device memory is budgeted by a
 * host framework, or runtimes without a device allocator. The call needs no
 * context: it computes exactly what oscar_decode_attn computes, from buffers the
 * caller passes, with its split-K workspace in a fixed array of
 * OSCAR_NOALLOC_SCRATCH_BYTES inside this library's device image. That array
 * exists on every GPU that loads the library, for the life of the process.
 *
 * cfg: HOST configuration (as for oscar_create). q, page_table, state, o: as for
 * oscar_decode_attn. int2_pool (num_pages pages), window: the cache buffers, laid
 * out as for oscar_bind_cache (16-byte aligned). R_K, R_V: DEVICE float32
 * [num_kv_heads][128][128] (16-byte aligned); clip_V: DEVICE float32
 * [num_kv_heads]. err_flags: optional DEVICE uint32 that the kernels OR
 * OSCAR_FLAG_* bits into (never cleared by the call); NULL sends the flags to a
 * word of the fixed array that each call clears and no caller can read.
 *
 * Returns OSCAR_ERR_OUT_OF_RANGE when batch exceeds cfg->max_batch or when the
 * workspace of this call (growing with batch, num_kv_heads, the query group and
 * the number of splits) does not fit in OSCAR_NOALLOC_SCRATCH_BYTES; the other
 * statuses as for oscar_decode_attn. No cudaMalloc or cudaFree is ever made.
 *
 * The first call on each device looks up the array's device address with that
 * device current; make it before any stream capture. All calls on a device share
 * the array and it keeps the last call's contents (each call rewrites what it
 * reads); calls whose kernels can overlap on the GPU race on it. */
int oscar_decode_attn_noalloc(const oscar_config* cfg, const void* q, const int32_t* page_table,
                              const oscar_seq_state* state, float* o, int32_t batch,
                              const void* int2_pool, int64_t num_pages, const void* window,
                              const float* R_K, const float* R_V, const float* clip_V,
                              uint32_t* err_flags, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* OSCAR_H */
