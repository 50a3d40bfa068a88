// Read path of the OSCAR INT2 cache: fused paged decode attention.
//
// Sources: "OSCAR: Offline Spectral Covariance-Aware Rotation ..." (gist.science,
// it), Riepilogo Tecnico 2.2 B "Integrazione del Kernel" (one kernel unpacks,
// dequantises, undoes the rotation and attends over the INT2 history, paged,
// with no extra memory traffic); "Juntos, AI Open-Sources OSCAR ..."
// (7minutos.es), section "El sistema de servicio" (BF16 sink and recent
// tokens, INT2 history, inverse rotation on read).
//
// Three launches on one stream:
//   1. oscar_rotate_q_kernel   q~ = q R_K * scale * log2(e) per (request, KV head),
//      written as ready-to-use tensor-core operand fragments (fp16 hi + lo).
//   2. oscar_decode_kernel<NG, FEW, MERGED, STEP> grid (window chunks + prefix splits + splits, Hkv,
//      B), NG = 128 / group size: the first CTAs attend over the BF16 sink +
//      recent ring in the raw basis (64 or 160 tokens each, per call); the
//      others stream a slice of the INT2 pages, computing scores and the P.V
//      product on the tensor cores with exact 2-bit operands, in the R_V basis. With a shared prefix
//      (oscar_decode_attn_shared_prefix) the prefix CTAs attend over the shared
//      pages once for a pack of requests, their query heads side by side in the
//      tensor-core columns, and the per-request CTAs over what follows.
//   3. oscar_merge_kernel      log-sum-exp merge of all partials, R_V^T applied to
//      the INT2 part, normalisation.
//
// Because R_K is orthogonal, (x_hat R_K^T) . q = x_hat . (q R_K): rotating the
// query once replaces de-rotating every key; likewise sum_t p_t (v_hat_t R_V^T)
// = (sum_t p_t v_hat_t) R_V^T, so the INT2 values stay rotated until the merge.
//
// Operand encoding. A 2-bit code c placed in the low mantissa bits of an fp16
// lane is the subnormal c * 2^-24, an exact tensor-core operand; a code stored
// at bit 2i of a half (i <= 4) reads as c * 4^i * 2^-24 after one AND. Slots
// 5..7 are read after a 10-bit right shift. The pool layout (include/oscar.h)
// puts, for every lane, the 8 codes it needs per mma into one 32-bit word, and
// the factor 4^i of each slot is divided out of the query operand (scores) or
// out of the per-channel-block accumulator (values).
#include <math.h>

#include <type_traits>

#include "oscar_internal.cuh"
#include "token_quant.cuh"

namespace oscar {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
// pages in flight per warp (a power of two): the ring of cp.async page copies
#ifndef OSCAR_DEC_STAGES
#define OSCAR_DEC_STAGES 4
#endif
constexpr int kStages = OSCAR_DEC_STAGES;
constexpr int kStageBytes = kWarps * kStages * kBlockBytes;   // 48 KB with 4 stages
static_assert((kStages & (kStages - 1)) == 0 && kStages >= 2, "page ring depth must be a power of two");
constexpr int kMaxWindow = 1024;                                // sink + recent limit
constexpr int kWinChunk = kWindowChunkMax;                      // window tokens per CTA, at most

// factor of a code read from slot i (see the file comment)
__host__ __device__ constexpr float slot_factor(int i) {
  return i <= 4 ? (float)(1 << (2 * i)) : (float)(1 << (2 * (i - 5)));
}

// w: a code word, wh = w >> 10 (computed once per word, shared by slots 5..7)
template <int I>
__device__ __forceinline__ uint32_t slot_bits(uint32_t w, uint32_t wh) {
  if constexpr (I <= 4) {
    return w & (0x00030003u << (2 * I));
  } else {
    return wh & (0x00030003u << (2 * (I - 5)));
  }
}
__device__ __forceinline__ uint4 shr10(uint4 w) { return make_uint4(w.x >> 10, w.y >> 10, w.z >> 10, w.w >> 10); }

// d += a b (no side effects: not volatile, so the compiler may interleave
// independent products with the arithmetic around them)
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// d = a b (a zero accumulator without zeroing registers first)
__device__ __forceinline__ void mma16816_z(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                           uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};\n"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}

// d = a b with k = 8 (a: rows gid / gid + 8 at k 2 tig, 2 tig + 1; b: k 2 tig, 2 tig + 1
// of column gid)
__device__ __forceinline__ void mma1688_z(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
  asm("mma.sync.aligned.m16n8k8.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5}, {%6}, {%7,%7,%7,%7};\n"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(b0), "f"(0.f));
}

__device__ __forceinline__ uint32_t hmul2_bits(uint32_t a, uint32_t b) {
  __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

__device__ __forceinline__ uint32_t f2_to_h2_bits(float lo, float hi) {
  __half2 r = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&r);
}

__device__ __forceinline__ float2 h2_bits_to_f2(uint32_t a) {
  return __half22float2(*reinterpret_cast<const __half2*>(&a));
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem));
}
// the same with a shared-space address and a source size of 16 or 0 bytes (0:
// nothing is read, the 16 bytes are zero-filled)
__device__ __forceinline__ void cp_async16_s(uint32_t saddr, const void* gmem, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(saddr), "l"(gmem), "r"(src_bytes));
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}
__device__ __forceinline__ float warp_maxf(float x) {
#pragma unroll
  for (int o = 16; o; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

// --------------------------------------------------------------------------
// 1. query rotation and operand fragments
// --------------------------------------------------------------------------
constexpr int kRotThreads = 256;
constexpr int kRotSmem = kHeadDim * kHeadDim * 4;  // one 128 x 128 float matrix

// copy a 128 x 128 float matrix into shared memory with every copy in flight at
// once (cp.async does not go through registers); the caller waits and syncs
__device__ __forceinline__ void stage_matrix(float* dst, const float* src, int tid, int nthreads) {
  for (int i = tid; i < kHeadDim * kHeadDim / 4; i += nthreads) cp_async16(dst + 4 * i, src + 4 * i);
  cp_commit();
}

__global__ void __launch_bounds__(kRotThreads) oscar_rotate_q_kernel(DecodeParams p) {
  extern __shared__ __align__(16) uint8_t dsm[];
  float* Rs = reinterpret_cast<float*>(dsm);                  // R_K[h], [128][128]
  const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  const int c = tid & (kHeadDim - 1), half = tid >> 7;
  const int g = p.gqa;
  __shared__ float qs[kMaxGqa][kHeadDim];
  __shared__ float red[kMaxGqa][kHeadDim];
  __shared__ __half hs[2][kMaxGqa][kHeadDim];
  __shared__ float wsum[kMaxGqa][4];  // per head and warp: 2^(k-24) times the sum of its 32 channels of q~
  __shared__ float wmax[4];
  __shared__ int s_k;
  stage_matrix(Rs, p.R_K + (size_t)h * kHeadDim * kHeadDim, tid, kRotThreads);  // constant data
  // Everything up to the wait reads only R_K and the caller's q, which no
  // kernel of this library writes, so it may run beside earlier kernels (the
  // append lets this kernel start at once); qrec, which the previous decode
  // reads, is written only after the wait.
  for (int i = tid; i < g * kHeadDim; i += kRotThreads)
    qs[i >> 7][i & 127] = __bfloat162float(p.q[((size_t)b * p.num_q_heads + h * g) * kHeadDim + i]);
  cp_wait<0>();
  __syncthreads();
  // thread (half, c): rows [64 half, 64 half + 64) of q R_K for every head
  float acc[kMaxGqa];
#pragma unroll
  for (int m = 0; m < kMaxGqa; ++m) acc[m] = 0.f;
  const int i0 = half * 64;
#pragma unroll 8
  for (int i = 0; i < 64; ++i) {
    const float r = Rs[(i0 + i) * kHeadDim + c];
#pragma unroll
    for (int m = 0; m < kMaxGqa; ++m)
      if (m < g) acc[m] = fmaf(qs[m][i0 + i], r, acc[m]);
  }
  if (half == 1) {
#pragma unroll
    for (int m = 0; m < kMaxGqa; ++m) red[m][c] = acc[m];
  }
  __syncthreads();
  if (half == 0) {
    float amax = 0.f;
#pragma unroll
    for (int m = 0; m < kMaxGqa; ++m) {
      acc[m] = m < g ? (acc[m] + red[m][c]) * p.scale_log2 : 0.f;
      amax = fmaxf(amax, fabsf(acc[m]));
    }
    amax = warp_maxf(amax);
    if ((c & 31) == 0) wmax[c >> 5] = amax;
  }
  __syncthreads();
  if (half == 0) {
    const float amax = fmaxf(fmaxf(wmax[0], wmax[1]), fmaxf(wmax[2], wmax[3]));
    // operand scale 2^k keeps the largest entry in [2^13, 2^14): far from fp16
    // overflow, and the small entries of the lo part stay representable
    int e = 0;
    if (amax > 0.f) frexpf(amax, &e);
    const int k = amax > 0.f ? min(14 - e, 100) : 0;
    const float s2k = ldexpf(1.f, k);
    const float inv_f = 1.f / slot_factor(c >> 4);
#pragma unroll
    for (int m = 0; m < kMaxGqa; ++m) {
      const float a = acc[m] * s2k * inv_f;
      const __half hi = __float2half_rn(a);
      hs[0][m][c] = hi;
      hs[1][m][c] = __float2half_rn(a - __half2float(hi));
    }
    // sums of q~ per head and 32 channels, scaled like the mma results
    // (2^(k-24) sum q~); the group sums below are the zero-point operand
    const float gscale = ldexpf(1.f, k - 24);
#pragma unroll
    for (int m = 0; m < kMaxGqa; ++m) {
      const float sm = warp_sum(acc[m]) * gscale;
      if ((c & 31) == 0) wsum[m][c >> 5] = sm;
    }
    if (c == 0) s_k = k;
  }
  __syncthreads();
  pdl_wait();  // earlier kernels (the previous decode reads qrec) are complete
  pdl_trigger();
  uint32_t* rec = p.qrec + ((size_t)b * p.num_kv_heads + h) * kQrecWords;
  if (tid == 0) {
    rec[1088] = __float_as_uint(ldexpf(1.f, 24 - s_k));
    for (int w = 1089; w < kQrecWords; ++w) rec[w] = 0u;
  }
  // column fragments of m16n8k16 (k = channel, n = head): per slot kb and lane
  // (gid, tig) four words, hi parts of head gid at channels 16 kb + 2 tig (+1) and
  // + 8 (+9), then the lo parts at the same channels, so that each operand pair
  // is one aligned half of the 16-byte record entry. With g = 1, 2 or 4 heads the
  // hi words of the spare columns gid = g .. 2g - 1 carry the lo parts of heads
  // gid - g, so that one product per slot covers both parts (the merged scores)
  const bool merged = g == 1 || g == 2 || g == 4;
#pragma unroll
  for (int n = 0; n < 4; ++n) {
    const int widx = tid + kRotThreads * n;
    const int r = widx & 3, lane = (widx >> 2) & 31, kb = widx >> 7;
    const int gid = lane >> 2, tig = lane & 3;
    const int col = kb * 16 + 2 * tig + ((r & 1) ? 8 : 0);
    const bool spare_lo = merged && r < 2 && gid >= g && gid < 2 * g;
    const __half* src = spare_lo ? hs[1][gid - g] : hs[r >> 1][gid];
    const uint32_t lo = __half_as_ushort(src[col]);
    const uint32_t hi = __half_as_ushort(src[col + 1]);
    rec[widx] = lo | (hi << 16);
  }
  // zero-point column operand: per lane (gid, tig) a hi and a lo word, the fp16
  // hi / lo parts of the group sums of q~ for head gid, groups 2 tig and 2 tig + 1
  // (4 groups of 32 channels: tig < 2; 2 groups of 64: tig = 0)
  if (tid < 64) {
    const int lane = tid >> 1, r = tid & 1, gid = lane >> 2, tig = lane & 3;
    const int ng = p.ngroups;
    uint32_t w = 0u;
    if (2 * tig < ng) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int gq = 2 * tig + e;
        const float sm = ng == kGroups ? wsum[gid][gq] : wsum[gid][2 * gq] + wsum[gid][2 * gq + 1];
        const __half hi = __float2half_rn(sm);
        const __half part = r ? __float2half_rn(sm - __half2float(hi)) : hi;
        w |= (uint32_t)__half_as_ushort(part) << (16 * e);
      }
    }
    rec[1024 + tid] = w;
  }
}

// --------------------------------------------------------------------------
// 2a. BF16 sink + recent ring: CTA x < win_slots attends over window tokens
//     [c x, c x + c), c = p.win_chunk (sink first, then the ring in position
//     order)
// --------------------------------------------------------------------------
// Shared-memory rows are padded by 16 bytes so that the 8 rows an 8x8 matrix
// load reads fall into different banks.
constexpr int kWinRow = kHeadDim + 8;   // bf16 elements per staged window / query row (272 bytes)
constexpr int kWindowSmem = 2 * kWinChunk * kWinRow * 2 + kMaxGqa * kWinRow * 2 + (kMaxGqa * kWinChunk + 2 * kMaxGqa) * 4;
static_assert(kWinChunk % 16 == 0, "window chunks are whole 16-token tiles");

// four 8x8 b16 matrices from shared memory (lane l gives the row address of
// matrix l / 8), optionally transposed
__device__ __forceinline__ void ldsm_x4(uint32_t saddr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(saddr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t saddr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(saddr));
}
__device__ __forceinline__ void mma16816_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// a bf16 pair as an fp16 pair (exact for the window's values: 8-bit mantissas
// inside the fp16 range)
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t x) {
  return f2_to_h2_bits(__uint_as_float(x << 16), __uint_as_float(x & 0xffff0000u));
}

// The chunk's tokens as 16-token tiles (rows past the chunk zero-filled). Scores:
// warp w takes tiles w, w + 8 with the K rows as the bf16 row operand and the
// raw bf16 query heads as the column operand (exact products, fp32 sums), scaled
// to log2 units afterwards. Values: warp w takes channels 16 w .. 16 w + 15 for
// every tile, V^T as the row operand (fp16 after a conversion that is exact for
// values of magnitude 2^-14 .. 65504) and the fp16 probabilities as the column
// operand, as in the INT2 value product.
// newrow: with STEP, threads 0-15 / 16-31 hold 16-byte pieces of the step's new
// K / V row, loaded before the kernel's wait
template <bool STEP>
__device__ void window_attention(const DecodeParams& p, int b, int h, int chunk, uint8_t* smem, uint4 newrow) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int g = p.gqa, S = p.sink, W = p.recent;
  __nv_bfloat16* krows = reinterpret_cast<__nv_bfloat16*>(smem);             // [chunk][kWinRow]
  __nv_bfloat16* vrows = krows + kWinChunk * kWinRow;                         // [chunk][kWinRow]
  __nv_bfloat16* qb = vrows + kWinChunk * kWinRow;                            // [8][kWinRow]
  float* sc = reinterpret_cast<float*>(qb + kMaxGqa * kWinRow);               // [8][chunk]
  float* stat = sc + kMaxGqa * kWinChunk;                                     // [8][2]
  const int nslots = total_slots(p);
  float* part = p.part + (((size_t)b * p.num_kv_heads + h) * nslots + chunk) * g * kPartFloats;

  const oscar_seq_state st = p.state[b];
  const bool ok = state_ok(st, S, W, p.max_batch);
  int L = st.seq_len, E = st.int2_end;
  // a decode step attends over the window as its append leaves it: position L
  // added (read from the caller's k / v, since the append CTA writes the window
  // concurrently), the entry it evicts (or, without a ring, the token itself)
  // left to the append CTA's INT2 slot
  int newpos = -1;
  if (STEP && ok) {
    newpos = L;
    E = max(E, max(L + 1 - W, S));
    L = L + 1;
  }
  const int ns = ok ? min(S, L) : 0;
  const int rb = max(E, S);
  const int nr = ok && L > rb ? L - rb : 0;
  const int t0 = chunk * p.win_chunk;
  const int n = max(0, min(p.win_chunk, ns + nr - t0));
  const int ntiles = (n + 15) / 16;
  const size_t slots = (size_t)(S + W);
  const size_t wrow = ok ? (size_t)st.window_row : 0;
  const __nv_bfloat16* wk = p.window + ((wrow * p.num_kv_heads + h) * 2 + 0) * slots * kHeadDim;
  const __nv_bfloat16* wv = p.window + ((wrow * p.num_kv_heads + h) * 2 + 1) * slots * kHeadDim;

  for (int idx = tid; idx < ntiles * 16 * 16; idx += kThreads) {
    const int r = idx >> 4, u = idx & 15, t = t0 + r;
    const bool in = r < n;
    const int pos = t < ns ? t : rb + t - ns;
    if (STEP && in && pos == newpos) continue;  // the new token's row comes from registers (below)
    const int slot = !in ? 0 : (t < ns ? t : S + pos % W);
    cp_async16_s((uint32_t)__cvta_generic_to_shared(krows + r * kWinRow + 8 * u), wk + (size_t)slot * kHeadDim + 8 * u,
                 in ? 16u : 0u);
    cp_async16_s((uint32_t)__cvta_generic_to_shared(vrows + r * kWinRow + 8 * u), wv + (size_t)slot * kHeadDim + 8 * u,
                 in ? 16u : 0u);
  }
  cp_commit();
  if (STEP && newpos >= 0 && tid < 32) {
    // window token index of position L: in the sink, or after the sink in the ring
    const int r = (newpos < S ? newpos : ns + (newpos - rb)) - t0;
    if (r >= 0 && r < n) *reinterpret_cast<uint4*>(((tid >> 4) ? vrows : krows) + r * kWinRow + 8 * (tid & 15)) = newrow;
  }
  // the raw query heads of this KV head (element loads: q needs no alignment
  // beyond its element size); heads past g are zero
  for (int i = tid; i < kMaxGqa * kHeadDim; i += kThreads) {
    const int m = i >> 7, c = i & (kHeadDim - 1);
    qb[m * kWinRow + c] = m < g ? p.q[((size_t)b * p.num_q_heads + h * g + m) * kHeadDim + c] : __float2bfloat16(0.f);
  }
  cp_wait<0>();
  __syncthreads();
  const uint32_t ks = (uint32_t)__cvta_generic_to_shared(krows), vs = (uint32_t)__cvta_generic_to_shared(vrows);
  for (int t = warp; t < ntiles; t += kWarps) {
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    const int j = lane >> 3;
    const uint32_t arow = ks + (uint32_t)(((16 * t + (lane & 7) + 8 * (j & 1)) * kWinRow + 8 * (j >> 1)) * 2);
#pragma unroll
    for (int kk = 0; kk < kHeadDim / 16; ++kk) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4(arow + 32 * kk, a0, a1, a2, a3);
      const uint32_t b0 = *reinterpret_cast<const uint32_t*>(qb + gid * kWinRow + 16 * kk + 2 * tig);
      const uint32_t b1 = *reinterpret_cast<const uint32_t*>(qb + gid * kWinRow + 16 * kk + 2 * tig + 8);
      mma16816_bf16(d, a0, a1, a2, a3, b0, b1);
    }
    const int r0 = 16 * t + gid, h0 = 2 * tig;
    if (h0 < g) {
      sc[h0 * kWinChunk + r0] = d[0] * p.scale_log2;
      sc[h0 * kWinChunk + r0 + 8] = d[2] * p.scale_log2;
    }
    if (h0 + 1 < g) {
      sc[(h0 + 1) * kWinChunk + r0] = d[1] * p.scale_log2;
      sc[(h0 + 1) * kWinChunk + r0 + 8] = d[3] * p.scale_log2;
    }
  }
  __syncthreads();
  // softmax per head; the probabilities of the tile rows past the chunk are 0.
  // The sum adds the probabilities as the value product sees them (rounded to
  // fp16), so that numerator and denominator agree to the last bit of p.
  for (int m = warp; m < g; m += kWarps) {
    float mx = -INFINITY;
    for (int t = lane; t < n; t += 32) mx = fmaxf(mx, sc[m * kWinChunk + t]);
    mx = warp_maxf(mx);
    float l = 0.f;
    for (int t = lane; t < 16 * ntiles; t += 32) {
      const float e = t < n ? exp2f(sc[m * kWinChunk + t] - mx) : 0.f;
      sc[m * kWinChunk + t] = e;
      l += __half2float(__float2half_rn(e));
    }
    l = warp_sum(l);
    if (lane == 0) {
      stat[2 * m] = mx;
      stat[2 * m + 1] = l;
    }
  }
  __syncthreads();
  {
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    const int j = lane >> 3;
    const uint32_t vrow = vs + (uint32_t)((((lane & 7) + 8 * (j >> 1)) * kWinRow + 16 * warp + 8 * (j & 1)) * 2);
    const float* pg = sc + (gid < g ? gid : 0) * kWinChunk;
    for (int t = 0; t < ntiles; ++t) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4_t(vrow + (uint32_t)(16 * t * kWinRow * 2), a0, a1, a2, a3);
      const float2 p0 = *reinterpret_cast<const float2*>(pg + 16 * t + 2 * tig);
      const float2 p1 = *reinterpret_cast<const float2*>(pg + 16 * t + 2 * tig + 8);
      const uint32_t b0 = gid < g ? f2_to_h2_bits(p0.x, p0.y) : 0u;
      const uint32_t b1 = gid < g ? f2_to_h2_bits(p1.x, p1.y) : 0u;
      mma16816(d, bf16x2_to_f16x2(a0), bf16x2_to_f16x2(a1), bf16x2_to_f16x2(a2), bf16x2_to_f16x2(a3), b0, b1);
    }
    // rows: channels 16 warp + gid (+ 8), columns: heads 2 tig, 2 tig + 1
    const int c0 = 16 * warp + gid, h0 = 2 * tig;
    if (h0 < g) {
      part[(size_t)h0 * kPartFloats + c0] = d[0];
      part[(size_t)h0 * kPartFloats + c0 + 8] = d[2];
    }
    if (h0 + 1 < g) {
      part[(size_t)(h0 + 1) * kPartFloats + c0] = d[1];
      part[(size_t)(h0 + 1) * kPartFloats + c0 + 8] = d[3];
    }
    if (tid < g) {
      part[(size_t)tid * kPartFloats + kHeadDim] = stat[2 * tid];
      part[(size_t)tid * kPartFloats + kHeadDim + 1] = stat[2 * tid + 1];
    }
  }
}

// --------------------------------------------------------------------------
// 2b. INT2 pages: CTA x >= win_slots streams split x - win_slots of the pages
// --------------------------------------------------------------------------
// 2^x on the SFU (inputs here are <= 15; results below 2^-126 flush to 0)
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Lazy rescaling: the running maximum moves only when a score exceeds it by more
// than kLazyLog2 (log2 units), so probabilities relative to it stay <= 2^8.
constexpr float kLazyLog2 = 8.f;

// Scores of two staged pages A, B with the codes as the row operand: lane (gid,
// tig) gets tokens gid and gid + 8 of each page for heads 2 tig and 2 tig + 1,
// u[4 page + 2 (token is gid + 8) + (head is 2 tig + 1)], in units u = sum_gq s_k
// (q~ . code) + sum_gq z_k sum q~ (scaled by 2^(k-24)). The code fragment of slot
// KB for tokens (gid, gid + 8) is (kw.x, kw.z, kw.y, kw.w) masked to the slot;
// q~ hi and lo are two column operands accumulating into the same group result,
// so hi + lo needs no extra add. zqb: the zero-point column operand (group sums
// of q~, hi in k rows 0-3, lo in rows 4-7).
// NG: quantisation groups per token (4 of 32 channels, or 2 of 64).
// MERGED (query groups of 1, 2 or 4 heads): columns g .. 2g - 1 of the query
// operand hold the lo parts of heads 0 .. g - 1 (see oscar_rotate_q_kernel), so
// one product per slot covers hi and lo, and the two column halves are added
// afterwards (within a lane for g = 1, across lanes tig ^ (g / 2) otherwise).
template <int NG, bool MERGED>
__device__ __forceinline__ void pair_scores(const uint8_t* sbA, const uint8_t* sbB, const uint4* qs,
                                            uint32_t zqb, int lane, int g, float (&u)[8]) {
  const int gid = lane >> 2, tig = lane & 3;
  const uint4 kwA = *reinterpret_cast<const uint4*>(sbA + lane * 16);
  const uint4 kwB = *reinterpret_cast<const uint4*>(sbB + lane * 16);
  const uint4 kwAh = shr10(kwA), kwBh = shr10(kwB);
  {
    // K zeros of tokens gid and gid + 8: k rows 0 .. NG-1 of the zero-point
    // product pair with the hi, rows NG .. 2NG-1 with the lo copy of the group
    // sums (4 groups: groups 2 (tig & 1), +1 for every tig; 2 groups: groups 0, 1
    // for tig 0 and 1, nothing for tig 2 and 3)
    const int zo = kzero_off(NG, gid, NG == kGroups ? 2 * (tig & 1) : 0);
    constexpr int zpair = kzero_off(NG, 8, 0) - kzero_off(NG, 0, 0);  // token gid + 8
    const bool zon = NG == kGroups || tig < 2;
    float zA[4], zB[4];
    mma1688_z(zA, zon ? *reinterpret_cast<const uint32_t*>(sbA + zo) : 0u,
              zon ? *reinterpret_cast<const uint32_t*>(sbA + zo + zpair) : 0u, zqb);
    mma1688_z(zB, zon ? *reinterpret_cast<const uint32_t*>(sbB + zo) : 0u,
              zon ? *reinterpret_cast<const uint32_t*>(sbB + zo + zpair) : 0u, zqb);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      u[i] = zA[i];
      u[4 + i] = zB[i];
    }
  }
  // K scales of tokens gid and gid + 8: the two halves of word gq at kscale_off(gid, gq)
  const int so = kscale_off(NG, gid, 0);
#pragma unroll
  for (int gq = 0; gq < NG; ++gq) {
    float a[4], c[4];
#define OSCAR_QK(KB, MMA)                                                                          \
  {                                                                                                \
    const uint32_t xa = slot_bits<KB>(kwA.x, kwAh.x), ya = slot_bits<KB>(kwA.y, kwAh.y);           \
    const uint32_t za = slot_bits<KB>(kwA.z, kwAh.z), wa = slot_bits<KB>(kwA.w, kwAh.w);           \
    const uint32_t xb = slot_bits<KB>(kwB.x, kwBh.x), yb = slot_bits<KB>(kwB.y, kwBh.y);           \
    const uint32_t zb = slot_bits<KB>(kwB.z, kwBh.z), wb = slot_bits<KB>(kwB.w, kwBh.w);           \
    if constexpr (MERGED) {                                                                        \
      const uint2 q2 = reinterpret_cast<const uint2*>(qs)[2 * ((KB) * 32 + lane)];                 \
      MMA(a, xa, za, ya, wa, q2.x, q2.y);                                                          \
      MMA(c, xb, zb, yb, wb, q2.x, q2.y);                                                          \
    } else {                                                                                       \
      const uint4 q4 = qs[(KB) * 32 + lane];                                                       \
      MMA(a, xa, za, ya, wa, q4.x, q4.y);                                                          \
      mma16816(a, xa, za, ya, wa, q4.z, q4.w);                                                     \
      MMA(c, xb, zb, yb, wb, q4.x, q4.y);                                                          \
      mma16816(c, xb, zb, yb, wb, q4.z, q4.w);                                                     \
    }                                                                                              \
  }
    if constexpr (NG == kGroups) {
      if (gq == 0) { OSCAR_QK(0, mma16816_z) OSCAR_QK(1, mma16816) }
      if (gq == 1) { OSCAR_QK(2, mma16816_z) OSCAR_QK(3, mma16816) }
      if (gq == 2) { OSCAR_QK(4, mma16816_z) OSCAR_QK(5, mma16816) }
      if (gq == 3) { OSCAR_QK(6, mma16816_z) OSCAR_QK(7, mma16816) }
    } else {
      if (gq == 0) { OSCAR_QK(0, mma16816_z) OSCAR_QK(1, mma16816) OSCAR_QK(2, mma16816) OSCAR_QK(3, mma16816) }
      if (gq == 1) { OSCAR_QK(4, mma16816_z) OSCAR_QK(5, mma16816) OSCAR_QK(6, mma16816) OSCAR_QK(7, mma16816) }
    }
#undef OSCAR_QK
    const float2 sA = h2_bits_to_f2(*reinterpret_cast<const uint32_t*>(sbA + so + 4 * gq));  // (gid, gid + 8)
    const float2 sB = h2_bits_to_f2(*reinterpret_cast<const uint32_t*>(sbB + so + 4 * gq));
    u[0] = fmaf(sA.x, a[0], u[0]);
    u[1] = fmaf(sA.x, a[1], u[1]);
    u[2] = fmaf(sA.y, a[2], u[2]);
    u[3] = fmaf(sA.y, a[3], u[3]);
    u[4] = fmaf(sB.x, c[0], u[4]);
    u[5] = fmaf(sB.x, c[1], u[5]);
    u[6] = fmaf(sB.y, c[2], u[6]);
    u[7] = fmaf(sB.y, c[3], u[7]);
  }
  if constexpr (MERGED) {
    if (g == 1) {
      // column 0: hi, column 1: lo of the one head (lane tig = 0)
#pragma unroll
      for (int i = 0; i < 8; i += 2) u[i] = u[i + 1] = u[i] + u[i + 1];
    } else {
      // lanes tig and tig ^ (g / 2) hold the hi and lo columns of the same heads
      const int x = g >> 1;
#pragma unroll
      for (int i = 0; i < 8; ++i) u[i] += __shfl_xor_sync(0xffffffffu, u[i], x);
    }
  }
}

// transpose an 8 x 8 matrix of 16-bit values held one row pair per lane (lane
// (gid, tig) holds row gid, columns 2 tig and 2 tig + 1)
__device__ __forceinline__ uint32_t transpose8x8(uint32_t a) {
  uint32_t d;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

// acc[cb] += codes^T (p * s_v) and oz += z_v^T p for one staged page; P01 / P23
// hold fp16 p * pscale of my tokens (0 for masked tokens, whose value metadata
// the caller has zeroed). Rows gq < NG of oz are the value zero-point terms of
// group gq; row 4 of the zero-point row
// operand is all ones, so row 4 of oz sums the same fp16 probabilities the
// values are weighted with: the softmax denominator, consistent with the
// numerator to the last bit of p.
template <int NG>
__device__ __forceinline__ void page_values(const uint8_t* sb, int lane, uint32_t P01, uint32_t P23,
                                            float (&acc)[8][4], float (&oz)[4]) {
  const int gid = lane >> 2, tig = lane & 3;
  const uint4 vw = *reinterpret_cast<const uint4*>(sb + 512 + lane * 16);
  const uint4 vwh = shr10(vw);
  constexpr int vbase = vscale_off(NG, 0, 0);
#pragma unroll
  for (int gq = 0; gq < NG; ++gq) {
    // scales of tokens (2 tig, 2 tig + 1) and (2 tig + 8, 2 tig + 9): one 8-byte load
    const uint2 mv = *reinterpret_cast<const uint2*>(sb + vbase + 16 * (4 * gq + tig));
    const uint32_t B0 = hmul2_bits(P01, mv.x);
    const uint32_t B1 = hmul2_bits(P23, mv.y);
#define OSCAR_PV(CB)                                                                          \
  mma16816(acc[CB], slot_bits<CB>(vw.x, vwh.x), slot_bits<CB>(vw.y, vwh.y), slot_bits<CB>(vw.z, vwh.z),   \
           slot_bits<CB>(vw.w, vwh.w),                                                                    \
           B0, B1);
    if constexpr (NG == kGroups) {
      if (gq == 0) { OSCAR_PV(0) OSCAR_PV(1) }
      if (gq == 1) { OSCAR_PV(2) OSCAR_PV(3) }
      if (gq == 2) { OSCAR_PV(4) OSCAR_PV(5) }
      if (gq == 3) { OSCAR_PV(6) OSCAR_PV(7) }
    } else {
      if (gq == 0) { OSCAR_PV(0) OSCAR_PV(1) OSCAR_PV(2) OSCAR_PV(3) }
      if (gq == 1) { OSCAR_PV(4) OSCAR_PV(5) OSCAR_PV(6) OSCAR_PV(7) }
    }
#undef OSCAR_PV
  }
  // rows 0 .. NG-1: the value zeros of the groups; row 4: ones
  constexpr uint32_t kOnes = 0x3c003c00u;  // fp16 (1, 1)
  uint2 mz = make_uint2(gid == 4 ? kOnes : 0u, gid == 4 ? kOnes : 0u);
  if (gid < NG) mz = *reinterpret_cast<const uint2*>(sb + vbase + 16 * (4 * gid + tig) + 8);
  const uint32_t za0 = mz.x, za2 = mz.y;
  mma16816(oz, za0, 0u, za2, 0u, P01, P23);
}

// bits t of the tokens t in [0, 16) of a page at position pos that lie in [lo, hi)
__device__ __forceinline__ uint32_t page_token_bits(bool ok, int pos, int lo, int hi) {
  const int a = max(lo - pos, 0), e = min(hi - pos, kPage);
  return (ok && e > a) ? (((1u << (e - a)) - 1u) << a) : 0u;
}

// zero the value scales and zeros of the tokens of two staged pages whose bit in
// `valid` is clear (bit t: page A token t, bit 16 + t: page B token t); lane:
// page lane / 16, 16-byte chunk c = 4 g + bb of the value metadata, whose 32-bit
// word w holds tokens 8 (w % 2) + 2 bb and + 1 (scales for w < 2, zeros after)
template <int NG>
__device__ __forceinline__ void zero_masked_value_meta(uint8_t* sbA, uint8_t* sbB, uint32_t valid, int lane) {
  const int c = lane & 15;
  if (c >= 4 * NG) return;  // NG groups: 4 NG chunks
  const uint32_t vpage = (lane >> 4) ? (valid >> 16) : (valid & 0xffffu);
  uint4* chunk = reinterpret_cast<uint4*>(((lane >> 4) ? sbB : sbA) + vscale_off(NG, 0, 0) + 16 * c);
  uint32_t keep[4];
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const int tw = 8 * (w & 1) + 2 * (c & 3);
    keep[w] = (((vpage >> tw) & 1u) ? 0x0000ffffu : 0u) | (((vpage >> (tw + 1)) & 1u) ? 0xffff0000u : 0u);
  }
  uint4 x = *chunk;
  x.x &= keep[0];
  x.y &= keep[1];
  x.z &= keep[2];
  x.w &= keep[3];
  *chunk = x;
}

// INT2 positions [lo, hi) of KV head h, the split-th of nsplits slices of its
// pages, for nreq requests r0 .. r0 + nreq - 1 that share those pages (nreq > 1
// only over a shared prefix): column n of the tensor-core products is head n % g
// of request r0 + n / g. Page ids come from request r0's page-table row. okmask
// bit r: request r0 + r is consistent (else its partial is left empty). The
// result goes to partial slot `slot` of every request. PACK: nreq may exceed 1
// (otherwise both columns of a lane belong to request r0 and share its scale).
// FEW: every warp of the CTA streams at most 64 pages (splits of up to 512
// pages, the automatic split sizes), so all of a warp's page ids fit two
// registers per lane.
template <int NG, bool PACK, bool FEW, bool MERGED = false>
__device__ void int2_attention(const DecodeParams& p, int h, int split, int nsplits, int r0, int nreq,
                               uint32_t okmask, int lo, int hi, int slot, uint8_t* smem, uint4* qs,
                               int2* wbounds) {
  // qs [8 x 32]: q~ fragments of the packed requests, shared by all warps;
  // wbounds [kWarps]: each warp's [lo, hi) relative to its first page
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int g = p.gqa;

  int npages = 0, first = 0;
  if (okmask != 0u && hi > lo) {
    first = lo / kPage;
    npages = (hi - 1) / kPage - first + 1;
  }
  // split size rounded up to whole page pairs of every warp, so that all warps of
  // a split but the last one stream the same even number of pages
  const int chunk = ((npages + nsplits - 1) / nsplits + 2 * kWarps - 1) / (2 * kWarps) * (2 * kWarps);
  const int pbeg = first + split * chunk;
  const int pend = min(pbeg + chunk, first + npages);
  // Warp w takes pages pbeg + w + 8 j, nmine of them. Every warp runs the same
  // npw iterations (the CTA's count) so that the page loop's control flow is
  // the same in all warps; a warp's steps past its own pages read nothing and
  // are masked like tokens outside [lo, hi).
  const int nmine = pend - pbeg - warp > 0 ? (pend - pbeg - warp + kWarps - 1) / kWarps : 0;
  const int npw = pend > pbeg ? (pend - pbeg + kWarps - 1) / kWarps : 0;

  // query operand fragments (see oscar_rotate_q_kernel): column n = gid of lane
  // (gid, tig) takes the fragment of head gid % g of request r0 + gid / g
  auto record = [&](int r) { return p.qrec + ((size_t)(r0 + r) * p.num_kv_heads + h) * kQrecWords; };
  for (int i = tid; i < 8 * 32; i += kThreads) {
    if constexpr (PACK) {
      const int l = i & 31, cr = (l >> 2) / g;
      qs[i] = cr < nreq ? reinterpret_cast<const uint4*>(record(cr))[(i & ~31) | (4 * ((l >> 2) % g) + (l & 3))]
                        : make_uint4(0u, 0u, 0u, 0u);
    } else {
      qs[i] = reinterpret_cast<const uint4*>(record(0))[i];
    }
  }
  // zero-point column operand: k rows 2 tig, 2 tig + 1 of head gid = group sums of
  // q~ (hi for tig 0 / 1, lo for tig 2 / 3), taken from the record's row layout
  uint32_t zqb;
  {
    uint2 zq;
    if constexpr (PACK) {
      const int cr = gid / g;
      zq = cr < nreq ? reinterpret_cast<const uint2*>(record(cr) + 1024)[4 * (gid % g) + tig] : make_uint2(0u, 0u);
    } else {
      zq = reinterpret_cast<const uint2*>(record(0) + 1024)[lane];
    }
    const int src = NG == kGroups ? (lane & ~3) | (tig & 1) : lane & ~3;
    const uint32_t zx = __shfl_sync(0xffffffffu, zq.x, src);
    const uint32_t zy = __shfl_sync(0xffffffffu, zq.y, src);
    if constexpr (NG == kGroups)
      zqb = tig < 2 ? zx : zy;
    else
      zqb = tig == 0 ? zx : (tig == 1 ? zy : 0u);
  }
  // score units of columns 2 tig (index 0) and 2 tig + 1 (index 1): each request
  // has its own query operand scale
  const int cr0 = PACK ? (2 * tig) / g : 0, cr1 = PACK ? (2 * tig + 1) / g : 0;
  const float us0 = !PACK || cr0 < nreq ? __uint_as_float(record(cr0)[1088]) : 1.f;
  const float us1 = PACK ? (cr1 < nreq ? __uint_as_float(record(cr1)[1088]) : 1.f) : us0;
  const float tau0 = kLazyLog2 / us0, tau1 = PACK ? kLazyLog2 / us1 : tau0;
  // probabilities enter the value product as fp16 p * pscale with p <= 2^8 (lazy
  // maximum); pv_scale is the largest power of two keeping 2^8 * pv_scale * s_v
  // (s_v <= 2 clip_V / 3) below the fp16 maximum
  const float pscale = p.pv_scale[h];
  const float lg_ps = log2f(pscale);

  uint8_t* sbuf = smem + warp * kStages * kBlockBytes;
  const int32_t* ptrow = p.page_table + (size_t)r0 * p.pt_stride + pbeg + warp;
  constexpr int kBB = block_bytes(NG);
  const uint8_t* pool_h = p.pool + (size_t)h * kBB + lane * 16;
  const size_t page_stride = (size_t)p.num_kv_heads * kBB;
  // Page ids, two per lane for the first 64 pages of the warp (FEW: all of them),
  // -1 for a page the warp does not have; an id outside the pool is reported
  // after the loop and treated like a missing page: nothing is read (its ring
  // slot is zero-filled) and its tokens are masked.
  const uint32_t stride = (uint32_t)page_stride;   // heads x 1536 bytes, far below 2^32
  bool bad = false;
  auto load_id = [&](int j) {
    int id = -1;
    if (j < nmine) {
      id = ptrow[kWarps * j];
      if (id < 0 || id >= p.num_pages) {
        bad = true;
        id = -1;
      }
    }
    return id;
  };
  const int id0 = load_id(lane);
  const int id1 = load_id(lane + 32);
  // id of page j of the warp, -1 when it has none (or its id is outside the pool)
  auto page_id = [&](int j) {
    if (FEW || j < 64) return __shfl_sync(0xffffffffu, j < 32 ? id0 : id1, j & 31);
    return load_id(j);
  };
  // stage page j into ring slot sl (= j % kStages); nothing is read when `want`
  // is false (the slot is zero-filled)
  const uint32_t sring = (uint32_t)__cvta_generic_to_shared(sbuf) + lane * 16;
  auto issue = [&](int j, uint32_t slot_off, bool want) {
    const int id = want ? page_id(j) : -1;
    const uint32_t nb = id >= 0 ? 16u : 0u;
    const uint8_t* src = pool_h + (uint64_t)(uint32_t)max(id, 0) * stride;
    const uint32_t dst = sring + slot_off;
    cp_async16_s(dst, src, nb);
    cp_async16_s(dst + 512, src + 512, nb);
    if (NG == kGroups || lane < 16) cp_async16_s(dst + 1024, src + 1024, nb);  // metadata: 128 NG bytes
  };
  // pages j in [jlo, jhi) of the warp lie wholly inside [lo, hi) (page j starts
  // at position base + 128 j; only a split's first and last pages can be cut by
  // lo / hi) and every id is in the pool: pairs inside that range need no
  // masking. The bounds relative to the warp's first page live in shared memory
  // for the masking path, so that they hold no registers in the page loop.
  bool bad_id = __any_sync(0xffffffffu, bad);
  int jlo, jhi;
  {
    const int rlo = lo - (pbeg + warp) * kPage, rhi = hi - (pbeg + warp) * kPage;
    jlo = bad_id || (!FEW && nmine > 64) ? npw : (rlo <= 0 ? 0 : (rlo + kWarps * kPage - 1) / (kWarps * kPage));
    jhi = min(nmine, rhi < kPage ? 0 : (rhi - kPage) / (kWarps * kPage) + 1);
    if (lane == 0) wbounds[warp] = make_int2(rlo, rhi);
  }

#pragma unroll
  for (int s = 0; s < kStages; ++s) {
    issue(s, s * kBlockBytes, s < npw);
    cp_commit();
  }
  __syncthreads();  // q~ fragments and the bounds visible to every warp

  // running (lazy) max in score units u (log2 units = u * uscale), running sum and
  // accumulators in units of pscale
  // per lane: running maxima of heads 2 tig (index 0) and 2 tig + 1 (index 1); the
  // running sums are row 4 of oz (see page_values)
  float m0 = -INFINITY, m1 = -INFINITY;
  float acc[8][4];
  float oz[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int cb = 0; cb < 8; ++cb) acc[cb][0] = acc[cb][1] = acc[cb][2] = acc[cb][3] = 0.f;

  // Pages are consumed two at a time (one softmax update per pair), pair j in ring
  // slots SA, SA + 1 with SA = j % kStages; the loop below is unrolled over the two
  // slot pairs so that every ring address is a constant.
  static_assert(kStages == 4, "the page loop is unrolled over two slot pairs");
  // MASKED: the pair may hold tokens outside [lo, hi) or pages the warp does
  // not have; pairs wholly inside are consumed by the same code without masking
  auto consume_pair = [&](int j, auto masked_const) {
    constexpr bool MASKED = decltype(masked_const)::value;
    // ring slots j % kStages and the next (j is even): byte offset soff
    const uint32_t soff = (j & 2) ? 2 * kBlockBytes : 0;
    // the copy groups of pages j and j + 1 (empty when a page does not exist) are
    // the oldest two of the kStages in flight
    cp_wait<kStages - 2>();
    __syncwarp();
    uint8_t* sbA = sbuf + soff;
    uint8_t* sbB = sbA + kBlockBytes;

    float u[8];
    pair_scores<NG, MERGED>(sbA, sbB, qs, zqb, lane, g, u);
    if (MASKED) {
      // tokens outside [lo, hi), on a page the warp does not have or whose id is
      // outside the pool: scores -inf, and their value scales and zeros set to 0
      // in shared memory, so the value product is the same code for every pair
      const bool okA = page_id(j) >= 0;
      const bool okB = page_id(j + 1) >= 0;
      const int posA = kWarps * kPage * j;   // relative to the warp's first page, like rlo / rhi
      const int posB = posA + kWarps * kPage;
      const int2 rb = wbounds[warp];
      const uint32_t valid = page_token_bits(okA, posA, rb.x, rb.y) | (page_token_bits(okB, posB, rb.x, rb.y) << 16);
      const bool a0v = (valid >> gid) & 1u, a1v = (valid >> (gid + 8)) & 1u;
      const bool b0v = (valid >> (gid + 16)) & 1u, b1v = (valid >> (gid + 24)) & 1u;
      u[0] = a0v ? u[0] : -INFINITY;
      u[1] = a0v ? u[1] : -INFINITY;
      u[2] = a1v ? u[2] : -INFINITY;
      u[3] = a1v ? u[3] : -INFINITY;
      u[4] = b0v ? u[4] : -INFINITY;
      u[5] = b0v ? u[5] : -INFINITY;
      u[6] = b1v ? u[6] : -INFINITY;
      u[7] = b1v ? u[7] : -INFINITY;
      zero_masked_value_meta<NG>(sbA, sbB, valid, lane);
      __syncwarp();
    }

    // ---- online softmax over the pair, per head (lazy maximum) ------------------
    // The running maximum only has to bound every score seen to within kLazyLog2:
    // a warp vote on this lane's own scores decides whether it must move, and only
    // then is the maximum over the head's 16 lanes taken.
    float mx0 = fmaxf(fmaxf(u[0], u[2]), fmaxf(u[4], u[6]));
    float mx1 = fmaxf(fmaxf(u[1], u[3]), fmaxf(u[5], u[7]));
    if (__any_sync(0xffffffffu, mx0 > m0 + tau0 || mx1 > m1 + tau1)) {
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
      }
      const bool bump0 = mx0 > m0 + tau0, bump1 = mx1 > m1 + tau1;
      const float a0 = bump0 ? ex2((m0 - mx0) * us0) : 1.f;
      const float a1 = bump1 ? ex2((m1 - mx1) * us1) : 1.f;
      m0 = bump0 ? mx0 : m0;
      m1 = bump1 ? mx1 : m1;
#pragma unroll
      for (int cb = 0; cb < 8; ++cb) {
        acc[cb][0] *= a0;
        acc[cb][1] *= a1;
        acc[cb][2] *= a0;
        acc[cb][3] *= a1;
      }
      oz[0] *= a0;
      oz[1] *= a1;
      oz[2] *= a0;
      oz[3] *= a1;
    }
    // every head sees the same tokens: the maximum stays -inf until a valid
    // token has been seen, and the probabilities of such pairs are 0 (the
    // offset is 0 then, so that -inf scores give 2^-inf = 0)
    const float nb0 = m0 == -INFINITY ? 0.f : fmaf(-m0, us0, lg_ps);
    const float nb1 = m1 == -INFINITY ? 0.f : fmaf(-m1, us1, lg_ps);
    float pr[8];  // p * pscale, p <= 2^8
#pragma unroll
    for (int i = 0; i < 8; ++i) pr[i] = ex2(fmaf(u[i], (i & 1) ? us1 : us0, (i & 1) ? nb1 : nb0));
    // token-major probabilities -> the (token, head) column operand of P.V
    const uint32_t PA01 = transpose8x8(f2_to_h2_bits(pr[0], pr[1]));
    const uint32_t PA23 = transpose8x8(f2_to_h2_bits(pr[2], pr[3]));
    const uint32_t PB01 = transpose8x8(f2_to_h2_bits(pr[4], pr[5]));
    const uint32_t PB23 = transpose8x8(f2_to_h2_bits(pr[6], pr[7]));
    page_values<NG>(sbA, lane, PA01, PA23, acc, oz);
    page_values<NG>(sbB, lane, PB01, PB23, acc, oz);
    __syncwarp();
    // the pages kStages further on replace these two in the ring (copies past the
    // warp's last step read nothing)
    issue(j + kStages, soff, j + kStages < npw);
    cp_commit();
    issue(j + 1 + kStages, soff + kBlockBytes, j + 1 + kStages < npw);
    cp_commit();
  };
  // pairs j, j + 1 (j even) with j >= jlo and j + 1 < jhi need no masking: a
  // masked head (the split's first page may start before lo), the unmasked
  // middle, a masked tail
  int j = 0;
  for (; j < npw && j < jlo; j += 2) consume_pair(j, std::true_type{});
  for (; j + 1 < jhi; j += 2) consume_pair(j, std::false_type{});
  for (; j < npw; j += 2) consume_pair(j, std::true_type{});
  cp_wait<0>();
  if (__any_sync(0xffffffffu, bad_id) && lane == 0) atomicOr(p.err_flags, OSCAR_FLAG_BAD_PAGE_ID);

  // ---- per-warp partial -> shared memory, then CTA merge --------------------
  const float inv_ps = 1.f / pscale;
  __syncthreads();  // staging buffers are reused below
  // rows padded by 4 floats: the 32 lanes of a warp store (2 tig + e, 16 cb + gid)
  // into 32 different banks
  constexpr int kWRow = kHeadDim + 4;
  float* wpart = reinterpret_cast<float*>(smem);              // [8 warps][8 heads][kWRow]
  float* wml = wpart + kWarps * kMaxGqa * kWRow;              // [8 warps][8 heads][2]
  if (gid == 4) {
    // oz row 4: the sums of the probabilities of heads 2 tig, 2 tig + 1
    wml[(warp * kMaxGqa + 2 * tig) * 2] = m0 * us0;             // log2 units
    wml[(warp * kMaxGqa + 2 * tig) * 2 + 1] = oz[0] * inv_ps;
    wml[(warp * kMaxGqa + 2 * tig + 1) * 2] = m1 * us1;
    wml[(warp * kMaxGqa + 2 * tig + 1) * 2 + 1] = oz[1] * inv_ps;
  }
#pragma unroll
  for (int cb = 0; cb < 8; ++cb) {
    const int gq = cb / (8 / NG);
    const float ze = __shfl_sync(0xffffffffu, oz[0], 4 * gq + tig) * inv_ps;
    const float zo = __shfl_sync(0xffffffffu, oz[1], 4 * gq + tig) * inv_ps;
    const float sc = 16777216.f / slot_factor(cb) * inv_ps;
    const int ch = 16 * cb + gid;
    const int he = 2 * tig, ho = 2 * tig + 1;
    float* base = wpart + warp * kMaxGqa * kWRow;
    base[he * kWRow + ch] = fmaf(acc[cb][0], sc, ze);
    base[ho * kWRow + ch] = fmaf(acc[cb][1], sc, zo);
    base[he * kWRow + ch + 8] = fmaf(acc[cb][2], sc, ze);
    base[ho * kWRow + ch + 8] = fmaf(acc[cb][3], sc, zo);
  }
  __syncthreads();
  // per column n the weights of the 8 warps' partials, their running maximum and
  // the merged sum, once: thread (n, w) for the first 8 ncols threads, the 8 warps
  // of a column being 8 consecutive lanes
  const int ncols = (PACK ? nreq : 1) * g;
  float* wts = wml + kWarps * kMaxGqa * 2;   // [8 columns][8 warps], then [8 columns][2]: M, l
  if (warp < (kWarps * ncols + 31) / 32) {   // whole warps (the shuffles); lanes past the columns write nothing
    const int n = tid >> 3, w = tid & 7;   // n < 8 here
    const float mw = wml[(w * kMaxGqa + n) * 2];
    float M = mw;
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const bool okr = (okmask >> (PACK ? n / g : 0)) & 1u;
    const float sw = (!okr || mw == -INFINITY) ? 0.f : exp2f(mw - M);
    float l = sw * wml[(w * kMaxGqa + n) * 2 + 1];
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    if (n < ncols) {
      wts[n * kWarps + w] = sw;
      if (w == 0) {
        wts[kWarps * kMaxGqa + 2 * n] = okr ? M : -INFINITY;
        wts[kWarps * kMaxGqa + 2 * n + 1] = l;
      }
    }
  }
  __syncthreads();
  const int nslots = total_slots(p);
  for (int i = tid; i < ncols * kHeadDim; i += kThreads) {
    const int n = i / kHeadDim, c = i % kHeadDim;  // column n: head n % g of request r0 + n / g
    const int cr = PACK ? n / g : 0;
    float o = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) o = fmaf(wts[n * kWarps + w], wpart[(w * kMaxGqa + n) * kWRow + c], o);
    float* dst = p.part + ((((size_t)(r0 + cr) * p.num_kv_heads + h) * nslots + slot) * g + (PACK ? n % g : n)) *
                              kPartFloats;
    dst[c] = o;
    if (c == 0) {
      dst[kHeadDim] = wts[kWarps * kMaxGqa + 2 * n];
      dst[kHeadDim + 1] = wts[kWarps * kMaxGqa + 2 * n + 1];
    }
  }
}

// --------------------------------------------------------------------------
// 2c. A decode step's append (oscar_decode_step): the last CTA of every
//     (request, KV head) appends the request's new token. With L, E the state
//     before the step and E' = max(E, L + 1 - recent, sink), position L goes to
//     the sink (L < sink) or to the recent ring, whose slot first hands the
//     entry it held, position L - recent, to INT2 when that lies in [E, E');
//     without a ring (recent = 0) position L itself goes to INT2. That position
//     is rotated, clipped, quantised and packed with the append kernel's
//     arithmetic, and this CTA attends over it: its partial (the score of the
//     dequantised key in log2 units, weight 1, the dequantised value) takes the
//     call's last slot, in the R_V basis like the splits' partials.
//     Sources: "Juntos, AI Open-Sources OSCAR ..." (7minutos.es), section "El
//     sistema de servicio" (BF16 sink and recent ring, INT2 for the rest; the
//     write path's rotate, clip and group quantisation).
// --------------------------------------------------------------------------
constexpr int kStepSmem =
    (kHeadDim * kHeadDim + 2 * kMaxGqa * kHeadDim + 8 * kHeadDim + 16) * 4 + 2 * kHeadDim + 2 * kGroups * 2 * 2;

__device__ __forceinline__ float warp_minf(float x) {
#pragma unroll
  for (int o = 16; o; o >>= 1) x = fminf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

__device__ void step_append(const DecodeParams& p, int h, int b, uint8_t* smem) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = p.gqa, S = p.sink, W = p.recent, Hkv = p.num_kv_heads;
  // thread (kind, c): kind 0 = K, 1 = V (or, in the rotations, the half of the rows)
  const int kind = tid >> 7, c = tid & (kHeadDim - 1);
  float* Rs = reinterpret_cast<float*>(smem);                // [128][128]: R_K[h], later R_V[h]
  float* qf = Rs + kHeadDim * kHeadDim;                       // [8][128]: the raw query heads
  float* qt = qf + kMaxGqa * kHeadDim;                        // [8][128]: q~ in log2 units
  float* xs = qt + kMaxGqa * kHeadDim;                        // [2][128]: K, V of the position going to INT2
  float* red = xs + 2 * kHeadDim;                             // [2 kinds][2 halves][128]
  float* deq = red + 4 * kHeadDim;                            // [2][128]: its dequantised K, V (R basis)
  float* wmm = deq + 2 * kHeadDim;                            // [2 kinds][4 warps][2]: min, max
  uint8_t(*codes)[kHeadDim] = reinterpret_cast<uint8_t(*)[kHeadDim]>(wmm + 16);
  __half(*meta)[kGroups][2] = reinterpret_cast<__half(*)[kGroups][2]>(codes + 2);
  const size_t rmat = (size_t)h * kHeadDim * kHeadDim;

  // constant data and the caller's q, k, v before the wait: R_K staged, R_V into
  // the level-2 cache, this thread's element of the new K / V row, q~ = q R_K *
  // scale * log2(e) (thread (half, c) sums 64 rows)
  stage_matrix(Rs, p.R_K + rmat, tid, kThreads);
  const __nv_bfloat16 xin = ((kind ? p.step_v : p.step_k) + ((size_t)b * Hkv + h) * kHeadDim)[c];
  if (tid == 0 && !p.fold_rv)
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(p.R_V + rmat), "r"(kHeadDim * kHeadDim * 4)
                 : "memory");
  for (int i = tid; i < kMaxGqa * kHeadDim; i += kThreads)
    qf[i] = (i >> 7) < g ? __bfloat162float(p.q[((size_t)b * p.num_q_heads + h * g) * kHeadDim + i]) : 0.f;
  cp_wait<0>();
  __syncthreads();
  {
    const int i0 = 64 * kind;
    float acc[kMaxGqa];
#pragma unroll
    for (int m = 0; m < kMaxGqa; ++m) acc[m] = 0.f;
#pragma unroll 4
    for (int i = 0; i < 64; ++i) {
      const float r = Rs[(i0 + i) * kHeadDim + c];
#pragma unroll
      for (int m = 0; m < kMaxGqa; ++m)
        if (m < g) acc[m] = fmaf(qf[m * kHeadDim + i0 + i], r, acc[m]);
    }
    if (kind == 1) {
#pragma unroll
      for (int m = 0; m < kMaxGqa; ++m)
        if (m < g) qt[m * kHeadDim + c] = acc[m];
    }
    __syncthreads();
    if (kind == 0) {
#pragma unroll
      for (int m = 0; m < kMaxGqa; ++m)
        if (m < g) qt[m * kHeadDim + c] = (acc[m] + qt[m * kHeadDim + c]) * p.scale_log2;
    }
  }

  pdl_wait();  // the state, the window and the pages come from earlier kernels
  pdl_trigger();
  const oscar_seq_state st = p.state[b];
  const bool ok = state_ok(st, S, W, p.max_batch);
  if (!ok && tid == 0) atomicOr(p.err_flags, OSCAR_FLAG_BAD_STATE);
  const int L = st.seq_len, E = st.int2_end;
  const int E2 = max(E, max(L + 1 - W, S));
  // the window slot of position L (-1: none) and the position going to INT2
  // (-1: none), taken from the ring or from the caller's k / v
  int wslot = -1, qpos = -1;
  bool from_ring = false;
  if (ok) {
    if (L < S) {
      wslot = L;
    } else if (L < E2) {
      qpos = L;
    } else {
      const int pe = L - W;
      if (pe >= E && pe < E2 && pe >= S) {
        qpos = pe;
        from_ring = true;
      }
      wslot = S + L % W;
    }
  }
  const size_t slots = (size_t)(S + W);
  const size_t wrow = ok ? (size_t)st.window_row : 0;
  __nv_bfloat16* win = p.step_window + ((wrow * Hkv + h) * 2 + kind) * slots * kHeadDim;
  int page = -1;
  if (qpos >= 0) {
    xs[kind * kHeadDim + c] = __bfloat162float(from_ring ? win[(size_t)(S + qpos % W) * kHeadDim + c] : xin);
    const int pidx = qpos / kPage;
    page = pidx < p.pt_stride ? p.page_table[(size_t)b * p.pt_stride + pidx] : -1;
  }
  __syncthreads();  // the entry the new token evicts is read before the window write
  if (wslot >= 0) win[(size_t)wslot * kHeadDim + c] = xin;

  const int nslot = total_slots(p);
  float* part = p.part + (((size_t)b * Hkv + h) * nslot + nslot - 1) * g * kPartFloats;
  if (qpos < 0) {
    // nothing goes to INT2 in this step: an empty partial
    for (int i = tid; i < g * kPartFloats; i += kThreads) part[i] = i % kPartFloats == kHeadDim ? -INFINITY : 0.f;
    return;
  }
  // the rotation x R as in the append kernel: thread (half, c) sums 64 terms in
  // order and the halves are added afterwards; K with R_K, then V with R_V
  {
    const int i0 = 64 * kind;
    float acc = 0.f;
#pragma unroll 16
    for (int i = 0; i < 64; ++i) acc = fmaf(xs[i0 + i], Rs[(i0 + i) * kHeadDim + c], acc);
    red[kind * kHeadDim + c] = acc;
    float accv = 0.f;
    if (p.fold_rv) {
      accv = kind ? 0.f : xs[kHeadDim + c];  // identity: V is already in the R_V basis
    } else {
      __syncthreads();  // R_K is no longer read
      stage_matrix(Rs, p.R_V + rmat, tid, kThreads);
      cp_wait<0>();
      __syncthreads();
#pragma unroll 16
      for (int i = 0; i < 64; ++i) accv = fmaf(xs[kHeadDim + i0 + i], Rs[(i0 + i) * kHeadDim + c], accv);
    }
    red[(2 + kind) * kHeadDim + c] = accv;
  }
  __syncthreads();
  // thread (kind, c): clip, group minimum and maximum (a group of 32 channels is
  // one warp, one of 64 two warps), scale, zero and code
  const float x_rot = red[(2 * kind) * kHeadDim + c] + red[(2 * kind + 1) * kHeadDim + c];
  const float clip = (kind ? p.clip_V : p.clip_K)[h];
  const float x = fminf(fmaxf(x_rot, -clip), clip);
  float mn = warp_minf(x), mx = warp_maxf(x);
  if (p.ngroups != kGroups) {
    if (lane == 0) {
      wmm[(kind * 4 + (c >> 5)) * 2] = mn;
      wmm[(kind * 4 + (c >> 5)) * 2 + 1] = mx;
    }
    __syncthreads();
    const int w = (c >> 5) ^ 1;  // the other warp of a 64-channel group
    mn = fminf(mn, wmm[(kind * 4 + w) * 2]);
    mx = fmaxf(mx, wmm[(kind * 4 + w) * 2 + 1]);
  }
  __half s16, z16;
  group_scale_zero(mn, mx, s16, z16);
  const float sf = __half2float(s16), zf = __half2float(z16);
  const int code = group_code(x, sf, zf);
  codes[kind][c] = (uint8_t)code;
  const int gsz = kHeadDim / p.ngroups;
  if ((c & (gsz - 1)) == 0) {
    meta[kind][c / gsz][0] = s16;
    meta[kind][c / gsz][1] = z16;
  }
  deq[kind * kHeadDim + c] = fmaf(sf, (float)code, zf);
  __syncthreads();
  if (tid < 72) {
    if (page >= 0 && page < p.num_pages)
      store_token_block(p.step_pool + ((size_t)page * Hkv + h) * block_bytes(p.ngroups), qpos % kPage, tid,
                        p.ngroups, codes, meta);
    else if (tid == 0)
      atomicOr(p.err_flags, OSCAR_FLAG_BAD_PAGE_ID);
  }
  // the partial of that position (warp m: query head m)
  for (int m = warp; m < g; m += kWarps) {
    float sc = 0.f;
    for (int cc = lane; cc < kHeadDim; cc += 32) sc = fmaf(qt[m * kHeadDim + cc], deq[cc], sc);
    sc = warp_sum(sc);
    float* row = part + (size_t)m * kPartFloats;
    for (int cc = lane; cc < kHeadDim; cc += 32) row[cc] = deq[kHeadDim + cc];
    if (lane == 0) {
      row[kHeadDim] = sc;
      row[kHeadDim + 1] = 1.f;
    }
  }
}

// FEW: no split holds more than 64 pages per warp (kFewPages per CTA), so the
// INT2 CTAs keep all their page ids in registers; the host picks the instance
// from the page-table width and the split counts (few_pages_call)
constexpr int kFewPages = 64 * kWarps;
// STEP: the instance a decode step launches (the step's append CTAs; see 2c),
// separate so that plain decodes run code without them
template <int NG, bool FEW, bool MERGED, bool STEP>
__global__ void __launch_bounds__(kThreads, kDecodeCtasPerSm) oscar_decode_kernel(DecodeParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint4 qs[8 * 32];
  __shared__ int2 wb[kWarps];
  const int x = blockIdx.x, h = blockIdx.y, z = blockIdx.z;
  if constexpr (STEP) {
    if (x == total_slots(p) - 1) {
      step_append(p, h, z, smem);
      return;
    }
  }
  // R_V^T[h] (constant) into the level-2 cache for the merge, whose CTAs only
  // become resident as these retire: one bulk prefetch per KV head
  if (x == 0 && z == 0 && threadIdx.x == 0 && !p.fold_rv) {
    const float* rvt = p.R_VT + (size_t)h * kHeadDim * kHeadDim;
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(rvt), "r"(kHeadDim * kHeadDim * 4) : "memory");
  }
  // a decode step's new K / V row (the caller's input) is loaded before the
  // wait, so that the window CTA holding it does not read it after the wait
  uint4 newrow = make_uint4(0u, 0u, 0u, 0u);
  if constexpr (STEP) {
    if (x < p.win_slots && threadIdx.x < 32) {
      const size_t off = ((size_t)z * p.num_kv_heads + h) * kHeadDim + 8 * (threadIdx.x & 15);
      newrow = *reinterpret_cast<const uint4*>(((threadIdx.x >> 4) ? p.step_v : p.step_k) + off);
    }
  }
  pdl_wait();  // cache, state and q~ come from earlier kernels
  pdl_trigger();
  const int S = p.sink, W = p.recent, P = p.prefix_tokens;
  if (x < p.win_slots) {
    window_attention<STEP>(p, z, h, x, smem, newrow);
  } else if (x < p.win_slots + p.prefix_splits) {
    // the shared prefix [S, P) once for requests z pack .. z pack + pack - 1; every
    // one of them must hold [S, P) in INT2
    const int r0 = z * p.pack;
    if (r0 >= p.batch) return;
    const int nreq = min(p.pack, p.batch - r0);
    uint32_t okmask = 0u;
    for (int r = 0; r < nreq; ++r) {
      const oscar_seq_state st = p.state[r0 + r];
      const bool ok = state_ok(st, S, W, p.max_batch) && P <= min(st.int2_end, st.seq_len);
      okmask |= (uint32_t)ok << r;
    }
    if (okmask != (1u << nreq) - 1u && threadIdx.x == 0) atomicOr(p.err_flags, OSCAR_FLAG_BAD_STATE);
    int2_attention<NG, true, FEW>(p, h, x - p.win_slots, p.prefix_splits, r0, nreq, okmask, S, P, x, smem, qs, wb);
  } else {
    // the request's own INT2 positions after the shared prefix
    const oscar_seq_state st = p.state[z];
    const bool ok = state_ok(st, S, W, p.max_batch);
    const int lo = max(S, P), hi = min(st.int2_end, st.seq_len);
    int2_attention<NG, false, FEW, MERGED>(p, h, x - p.win_slots - p.prefix_splits, p.splits, z, 1, ok ? 1u : 0u, lo, hi,
                                   x, smem, qs, wb);
  }
}

// --------------------------------------------------------------------------
// 3. merge of the partials, un-rotation, normalisation; CTA z handles query
//    heads 2z and 2z + 1 of (request y, KV head x). The partial rows (o, m, l)
//    are staged in rounds of up to kMergeChunk slots, all in flight at once, and
//    folded in with a running maximum, so a call with up to kMergeChunk slots
//    waits for the level-2 cache once.
// --------------------------------------------------------------------------
constexpr int kMergeThreads = 256;
constexpr int kMaxSlots = 256 + kMaxWindow / kWindowChunkSmall + 1;   // INT2 splits + window chunks + a step's slot
constexpr int kMergeChunk = 64;                            // slots staged per round
// floats of the staged rows (also the un-rotation partials, 4 x 128 floats)
__host__ __device__ constexpr int merge_rows_floats(int nslots) {
  return (nslots < kMergeChunk ? nslots : kMergeChunk) * 2 * kPartFloats > 4 * kHeadDim
             ? (nslots < kMergeChunk ? nslots : kMergeChunk) * 2 * kPartFloats
             : 4 * kHeadDim;
}
__host__ __device__ constexpr int merge_smem_bytes(int nslots) {
  return kRotSmem + merge_rows_floats(nslots) * 4 + 2 * kHeadDim * 4;
}
constexpr int kMergeSmem = merge_smem_bytes(kMergeChunk);

// the state after a decode step's append, written by one merge CTA per request
// once every CTA of the decode kernel (which all read the state from before
// the step) has completed: {L + 1, max(E, L + 1 - recent, sink)}
__device__ __forceinline__ void publish_step_state(const DecodeParams& p, int b) {
  oscar_seq_state st = p.step_state[b];
  if (!state_ok(st, p.sink, p.recent, p.max_batch)) return;
  const int64_t nl = (int64_t)st.seq_len + 1;
  int64_t ne = nl - p.recent;
  if (ne < st.int2_end) ne = st.int2_end;
  if (ne < p.sink) ne = p.sink;
  st.seq_len = (int32_t)nl;
  st.int2_end = (int32_t)ne;
  p.step_state[b] = st;
}

__global__ void __launch_bounds__(kMergeThreads) oscar_merge_kernel(DecodeParams p) {
  extern __shared__ __align__(16) uint8_t dsm[];
  const int g = p.gqa, nslots = total_slots(p), nwin = p.win_slots;
  const int chunk = nslots < kMergeChunk ? nslots : kMergeChunk;
  float* RT = reinterpret_cast<float*>(dsm);                   // R_V^T[h], [128][128]
  float* rows = RT + kHeadDim * kHeadDim;                       // [chunk slots][2 heads][kPartFloats]
  float* orot = rows + merge_rows_floats(nslots);               // [2][128]
  const int h = blockIdx.x, b = blockIdx.y, m0 = 2 * blockIdx.z, tid = threadIdx.x;
  const int nh = min(2, g - m0);
  if (!p.fold_rv) stage_matrix(RT, p.R_VT + (size_t)h * kHeadDim * kHeadDim, tid, kMergeThreads);
  else cp_commit();
  const float* part = p.part + ((size_t)b * p.num_kv_heads + h) * nslots * g * kPartFloats;
  pdl_wait();  // the partials come from the decode kernel
  pdl_trigger();
  // warp hh < nh keeps the running maximum and row sum of head hh and writes the
  // round's slot weights; thread (head hh, channel c) keeps the weighted sums of
  // the window and INT2 partials, relative to the running maximum
  __shared__ float wts[kMergeChunk * 2];   // [slot][head] weights of the round
  __shared__ float resc[2], lsum[2];       // per head: the round's rescale factor, the row sum
  const int warp = tid >> 5, lane = tid & 31;
  const int c = tid & (kHeadDim - 1), hh = tid >> 7;
  float Mw = -INFINITY, lw = 0.f;
  float owin = 0.f, orr0 = 0.f, orr1 = 0.f;
  constexpr int kChunks16 = kPartFloats / 4;  // 16-byte pieces per row
  for (int s0 = 0; s0 < nslots; s0 += chunk) {
    const int n = min(chunk, nslots - s0);
    if (s0 > 0) __syncthreads();  // the previous round's rows and weights are consumed
    // a slot's rows of both heads are contiguous: one warp per slot, no divisions
    for (int r = warp; r < n; r += kMergeThreads / 32) {
      const float* src = part + ((size_t)(s0 + r) * g + m0) * kPartFloats;
      float* dst = rows + r * nh * kPartFloats;
      for (int u = lane; u < nh * kChunks16; u += 32) cp_async16(dst + 4 * u, src + 4 * u);
    }
    cp_commit();
    // while the first round's rows are in flight
    if (s0 == 0 && p.step_slots && h == 0 && blockIdx.z == 0 && tid == 0) publish_step_state(p, b);
    cp_wait<0>();
    __syncthreads();
    if (warp < nh) {
      float mx = Mw;
      for (int r = lane; r < n; r += 32) mx = fmaxf(mx, rows[(r * nh + warp) * kPartFloats + kHeadDim]);
      mx = warp_maxf(mx);
      const float a = Mw == -INFINITY ? 0.f : exp2f(Mw - mx);  // accumulators are 0 while Mw is -inf
      float ls = 0.f;
      for (int r = lane; r < n; r += 32) {
        const float* row = rows + (r * nh + warp) * kPartFloats;
        const float ms = row[kHeadDim];
        const float w = ms == -INFINITY ? 0.f : exp2f(ms - mx);
        wts[r * 2 + warp] = w;
        ls = fmaf(w, row[kHeadDim + 1], ls);
      }
      ls = warp_sum(ls);
      lw = fmaf(lw, a, ls);
      Mw = mx;
      if (lane == 0) {
        resc[warp] = a;
        lsum[warp] = lw;
      }
    }
    __syncthreads();
    if (hh < nh) {
      const float a = resc[hh];
      owin *= a;
      orr0 *= a;
      orr1 *= a;
      const int nw = min(max(nwin - s0, 0), n);  // the round's window slots come first
      for (int r = 0; r < nw; ++r) owin = fmaf(wts[r * 2 + hh], rows[(r * nh + hh) * kPartFloats + c], owin);
      int r = nw;
#pragma unroll 4
      for (; r + 1 < n; r += 2) {
        orr0 = fmaf(wts[r * 2 + hh], rows[(r * nh + hh) * kPartFloats + c], orr0);
        orr1 = fmaf(wts[r * 2 + 2 + hh], rows[((r + 1) * nh + hh) * kPartFloats + c], orr1);
      }
      if (r < n) orr0 = fmaf(wts[r * 2 + hh], rows[(r * nh + hh) * kPartFloats + c], orr0);
    }
  }
  const float orr = orr0 + orr1;
  if (hh < nh) orot[hh * kHeadDim + c] = orr;
  cp_wait<0>();
  __syncthreads();
  float oi = orr;
  if (!p.fold_rv) {
    // un-rotation: thread (channel c, half hh) takes rows j of its half for both
    // heads, so every R_V^T entry is read from shared memory once; the two halves
    // meet in shared memory (rows is free by now)
    float* acc2 = rows;   // [2 halves][2 heads][128]
    const int j0 = hh * (kHeadDim / 2);
    float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
#pragma unroll 4
    for (int j = j0; j < j0 + kHeadDim / 2; j += 4) {
      const float4 x0 = *reinterpret_cast<const float4*>(orot + j);
      const float4 x1 = *reinterpret_cast<const float4*>(orot + kHeadDim + j);
      const float r0 = RT[j * kHeadDim + c], r1 = RT[(j + 1) * kHeadDim + c];
      const float r2 = RT[(j + 2) * kHeadDim + c], r3 = RT[(j + 3) * kHeadDim + c];
      a0 = fmaf(x0.x, r0, a0);
      a1 = fmaf(x0.y, r1, a1);
      a0 = fmaf(x0.z, r2, a0);
      a1 = fmaf(x0.w, r3, a1);
      b0 = fmaf(x1.x, r0, b0);
      b1 = fmaf(x1.y, r1, b1);
      b0 = fmaf(x1.z, r2, b0);
      b1 = fmaf(x1.w, r3, b1);
    }
    acc2[(hh * 2 + 0) * kHeadDim + c] = a0 + a1;
    acc2[(hh * 2 + 1) * kHeadDim + c] = b0 + b1;
    __syncthreads();
    if (hh < nh) oi = acc2[(0 * 2 + hh) * kHeadDim + c] + acc2[(1 * 2 + hh) * kHeadDim + c];
  }
  if (hh < nh) {
    const float l = lsum[hh];
    p.o[((size_t)b * p.num_q_heads + h * g + m0 + hh) * kHeadDim + c] = l > 0.f ? (oi + owin) / l : 0.f;
  }
}

// --------------------------------------------------------------------------
// 3b. the same merge for calls with few (request, KV head) pairs: CTA z = 4 m + q
//     of (request y, KV head x) produces output channels 32 q .. 32 q + 31 of
//     query head m, from all of m's partial rows and the 32 columns of R_V^T it
//     needs, so that 8 times more CTAs share the work and each un-rotates 32
//     rows per thread instead of 64 (the merge of a small batch is a latency
//     chain, not a bandwidth bound); calls with up to kMergeChunk slots
// --------------------------------------------------------------------------
constexpr int kMergeColsThreads = 128;
constexpr int kMergeColsMaxCtas = 64;   // merge-kernel CTAs (2 query heads each) up to which it is used
constexpr int kMergeCols = 32;
constexpr int kMergeColsSmem =
    (kHeadDim * kMergeCols + kMergeChunk * kPartFloats + kMergeChunk + 2 * kHeadDim + 4 * kMergeCols) * 4;

__global__ void __launch_bounds__(kMergeColsThreads) oscar_merge_cols_kernel(DecodeParams p) {
  extern __shared__ __align__(16) uint8_t dsm[];
  const int g = p.gqa, nslots = total_slots(p), nwin = p.win_slots;
  float* RTc = reinterpret_cast<float*>(dsm);                  // [128 rows][32 columns] of R_V^T
  float* rows = RTc + kHeadDim * kMergeCols;                    // [nslots][kPartFloats]
  float* wts = rows + kMergeChunk * kPartFloats;                // [nslots]
  float* osum = wts + kMergeChunk;                              // [2][128]: INT2 sums, window sums
  float* red = osum + 2 * kHeadDim;                             // [4][32]
  __shared__ float lsum;
  const int h = blockIdx.x, b = blockIdx.y, m = blockIdx.z >> 2, q = blockIdx.z & 3;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int col0 = q * kMergeCols;
  if (!p.fold_rv) {
    // columns col0 .. col0 + 31 of every row of R_V^T[h] (constant data)
    const float* src = p.R_VT + (size_t)h * kHeadDim * kHeadDim + col0;
    for (int i = tid; i < kHeadDim * (kMergeCols / 4); i += kMergeColsThreads) {
      const int r = i / (kMergeCols / 4), u = i % (kMergeCols / 4);
      cp_async16(RTc + r * kMergeCols + 4 * u, src + (size_t)r * kHeadDim + 4 * u);
    }
  }
  cp_commit();
  // rows of query head m for every slot: slot s at ((b Hkv + h) nslots + s) g + m
  const float* part = p.part + (((size_t)b * p.num_kv_heads + h) * nslots * g + m) * kPartFloats;
  pdl_wait();  // the partials come from the decode kernel
  pdl_trigger();
  constexpr int kChunks16 = kPartFloats / 4;
  for (int i = tid; i < nslots * kChunks16; i += kMergeColsThreads) {
    const int sl = i / kChunks16, u = i % kChunks16;
    cp_async16(rows + sl * kPartFloats + 4 * u, part + (size_t)sl * g * kPartFloats + 4 * u);
  }
  cp_commit();
  // while the rows are in flight
  if (p.step_slots && h == 0 && blockIdx.z == 0 && tid == 0) publish_step_state(p, b);
  cp_wait<0>();
  __syncthreads();
  if (warp == 0) {
    float mx = -INFINITY;
    for (int sl = lane; sl < nslots; sl += 32) mx = fmaxf(mx, rows[sl * kPartFloats + kHeadDim]);
    mx = warp_maxf(mx);
    float ls = 0.f;
    for (int sl = lane; sl < nslots; sl += 32) {
      const float ms = rows[sl * kPartFloats + kHeadDim];
      const float w = ms == -INFINITY ? 0.f : exp2f(ms - mx);
      wts[sl] = w;
      ls = fmaf(w, rows[sl * kPartFloats + kHeadDim + 1], ls);
    }
    ls = warp_sum(ls);
    if (lane == 0) lsum = ls;
  }
  __syncthreads();
  {
    // thread c: the weighted sums of channel c over the INT2 and the window slots
    const int c = tid;
    float ow = 0.f, o0 = 0.f, o1 = 0.f;
    int sl = 0;
    for (; sl < nwin; ++sl) ow = fmaf(wts[sl], rows[sl * kPartFloats + c], ow);
#pragma unroll 4
    for (; sl + 1 < nslots; sl += 2) {
      o0 = fmaf(wts[sl], rows[sl * kPartFloats + c], o0);
      o1 = fmaf(wts[sl + 1], rows[(sl + 1) * kPartFloats + c], o1);
    }
    if (sl < nslots) o0 = fmaf(wts[sl], rows[sl * kPartFloats + c], o0);
    osum[c] = o0 + o1;
    osum[kHeadDim + c] = ow;
  }
  __syncthreads();
  // output channel col0 + j: warp w takes rows 32 w .. 32 w + 31 of the un-rotation
  const int j = lane;
  float oi;
  if (!p.fold_rv) {
    float a0 = 0.f, a1 = 0.f;
#pragma unroll 8
    for (int r = 32 * warp; r < 32 * warp + 32; r += 2) {
      a0 = fmaf(osum[r], RTc[r * kMergeCols + j], a0);
      a1 = fmaf(osum[r + 1], RTc[(r + 1) * kMergeCols + j], a1);
    }
    red[warp * kMergeCols + j] = a0 + a1;
    __syncthreads();
    oi = red[j] + red[kMergeCols + j] + red[2 * kMergeCols + j] + red[3 * kMergeCols + j];
  } else {
    oi = osum[col0 + j];
  }
  if (warp == 0) {
    const float l = lsum;
    p.o[((size_t)b * p.num_q_heads + h * g + m) * kHeadDim + col0 + j] =
        l > 0.f ? (oi + osum[kHeadDim + col0 + j]) / l : 0.f;
  }
}

int decode_smem_bytes() {
  const int window = kWindowSmem;
  const int merge = (kWarps * kMaxGqa * (kHeadDim + 4) + kWarps * kMaxGqa * 2 + kMaxGqa * kWarps + kMaxGqa * 2) * 4;
  int m = kStageBytes;
  if (window > m) m = window;
  if (merge > m) m = merge;
  if (kStepSmem > m) m = kStepSmem;
  return m;
}

// the decode kernel instance for ng groups per token (4 or 2), splits of at
// most kFewPages pages (few), merged hi / lo score columns (query groups of 1,
// 2 or 4 heads; only with few) and a decode step's append CTAs (step)
static void (*decode_instance(int ng, bool few, bool merged, bool step))(DecodeParams) {
  if (ng == kGroups) {
    if (!few) return step ? oscar_decode_kernel<kGroups, false, false, true> : oscar_decode_kernel<kGroups, false, false, false>;
    if (merged) return step ? oscar_decode_kernel<kGroups, true, true, true> : oscar_decode_kernel<kGroups, true, true, false>;
    return step ? oscar_decode_kernel<kGroups, true, false, true> : oscar_decode_kernel<kGroups, true, false, false>;
  }
  if (!few) return step ? oscar_decode_kernel<2, false, false, true> : oscar_decode_kernel<2, false, false, false>;
  if (merged) return step ? oscar_decode_kernel<2, true, true, true> : oscar_decode_kernel<2, true, true, false>;
  return step ? oscar_decode_kernel<2, true, false, true> : oscar_decode_kernel<2, true, false, false>;
}

cudaError_t launch_decode(const DecodeParams& p, int batch, cudaStream_t s, cudaEvent_t ev_before,
                          cudaEvent_t ev_after) {
  static PerDeviceOnce attrs;
  const int smem = decode_smem_bytes();
  cudaError_t ea = once_for_current_device(attrs, [&] {
    void (*const kernels[])(DecodeParams) = {
        decode_instance(kGroups, true, false, false), decode_instance(kGroups, false, false, false),
        decode_instance(2, true, false, false),       decode_instance(2, false, false, false),
        decode_instance(kGroups, true, true, false),  decode_instance(2, true, true, false),
        decode_instance(kGroups, true, false, true),  decode_instance(kGroups, false, false, true),
        decode_instance(2, true, false, true),        decode_instance(2, false, false, true),
        decode_instance(kGroups, true, true, true),   decode_instance(2, true, true, true)};
    cudaError_t e = cudaSuccess;
    for (auto k : kernels)
      if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(oscar_rotate_q_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kRotSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(oscar_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMergeSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(oscar_merge_cols_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMergeColsSmem);
    return e;
  });
  if (ea != cudaSuccess) return ea;
  if (total_slots(p) > kMaxSlots) return cudaErrorInvalidValue;
  if (p.win_chunk < 1 || p.win_chunk > kWinChunk) return cudaErrorInvalidValue;
  // every split of the call streams at most kFewPages pages: a request's INT2
  // pages fit its page-table row, the shared prefix its own page count
  const int64_t prefix_pages = (int64_t)(p.prefix_tokens + kPage - 1) / kPage;
  const bool few = (p.pt_stride + p.splits - 1) / p.splits <= kFewPages &&
                   (p.prefix_splits == 0 || (prefix_pages + p.prefix_splits - 1) / p.prefix_splits <= kFewPages);
  // one query-operand product per slot covers hi and lo (see pair_scores)
  const bool merged = p.gqa == 1 || p.gqa == 2 || p.gqa == 4;
  cudaError_t e = launch_pdl(oscar_rotate_q_kernel, dim3(p.num_kv_heads, batch), dim3(kRotThreads), kRotSmem,
                             s, p);
  if (e == cudaSuccess && ev_before) e = cudaEventRecord(ev_before, s);
  if (e == cudaSuccess)
    e = launch_pdl(decode_instance(p.ngroups, few, merged, p.step_slots != 0),
                   dim3(total_slots(p), p.num_kv_heads, batch), dim3(kThreads),
                   smem, s, p);
  if (e == cudaSuccess && ev_after) e = cudaEventRecord(ev_after, s);
  // few (request, KV head) pairs: the merge by columns (8 times the CTAs)
  const int nslots = total_slots(p);
  const bool by_cols = nslots <= kMergeChunk && (int64_t)batch * p.num_kv_heads * ((p.gqa + 1) / 2) <= kMergeColsMaxCtas;
  if (e == cudaSuccess) {
    if (by_cols)
      e = launch_pdl(oscar_merge_cols_kernel, dim3(p.num_kv_heads, batch, 4 * p.gqa), dim3(kMergeColsThreads),
                     kMergeColsSmem, s, p);
    else
      e = launch_pdl(oscar_merge_kernel, dim3(p.num_kv_heads, batch, (p.gqa + 1) / 2), dim3(kMergeThreads),
                     merge_smem_bytes(nslots), s, p);
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace oscar
