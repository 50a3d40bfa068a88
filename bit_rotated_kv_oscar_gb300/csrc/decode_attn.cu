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
//   2. oscar_decode_kernel     grid (1 + splits, Hkv, B): CTA x = 0 attends over
//      the BF16 sink + recent ring in the raw basis; CTA x >= 1 streams a slice of
//      the INT2 pages, computing scores and the P.V product on the tensor cores
//      with exact 2-bit operands, in the R_V basis.
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

#include "oscar_internal.cuh"

namespace oscar {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 4;
constexpr int kStageBytes = kWarps * kStages * kBlockBytes;   // 48 KB
constexpr int kMaxWindow = 1024;                                // sink + recent limit

__device__ __forceinline__ bool state_ok(int L, int E, int S, int W) {
  return L >= 0 && E >= S && E <= (L > S ? L : S) && L - E <= W;
}

// factor of a code read from slot i (see the file comment)
__host__ __device__ constexpr float slot_factor(int i) {
  return i <= 4 ? (float)(1 << (2 * i)) : (float)(1 << (2 * (i - 5)));
}

template <int I>
__device__ __forceinline__ uint32_t slot_bits(uint32_t w) {
  if constexpr (I <= 4) {
    return w & (0x00030003u << (2 * I));
  } else {
    return (w >> 10) & (0x00030003u << (2 * (I - 5)));
  }
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
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
__global__ void __launch_bounds__(128) oscar_rotate_q_kernel(DecodeParams p) {
  const int h = blockIdx.x, b = blockIdx.y, c = threadIdx.x;
  const int g = p.gqa;
  __shared__ float qs[kMaxGqa][kHeadDim];
  __shared__ __half hs[2][kMaxGqa][kHeadDim];
  __shared__ float wmax[4];
  for (int m = 0; m < g; ++m)
    qs[m][c] = __bfloat162float(p.q[((size_t)b * p.num_q_heads + h * g + m) * kHeadDim + c]);
  __syncthreads();
  float acc[kMaxGqa];
#pragma unroll
  for (int m = 0; m < kMaxGqa; ++m) acc[m] = 0.f;
  const float* R = p.R_K + (size_t)h * kHeadDim * kHeadDim;
#pragma unroll 8
  for (int i = 0; i < kHeadDim; ++i) {
    const float r = __ldg(&R[i * kHeadDim + c]);
#pragma unroll
    for (int m = 0; m < kMaxGqa; ++m)
      if (m < g) acc[m] = fmaf(qs[m][i], r, acc[m]);
  }
  float amax = 0.f;
#pragma unroll
  for (int m = 0; m < kMaxGqa; ++m) {
    acc[m] = m < g ? acc[m] * p.scale_log2 : 0.f;
    amax = fmaxf(amax, fabsf(acc[m]));
  }
  amax = warp_maxf(amax);
  if ((c & 31) == 0) wmax[c >> 5] = amax;
  __syncthreads();
  amax = fmaxf(fmaxf(wmax[0], wmax[1]), fmaxf(wmax[2], wmax[3]));
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
  uint32_t* rec = p.qrec + ((size_t)b * p.num_kv_heads + h) * kQrecWords;
  // group sums of q~ (per head) scaled like the mma results: 2^(k-24) sum q~
  const float gscale = ldexpf(1.f, k - 24);
#pragma unroll
  for (int m = 0; m < kMaxGqa; ++m) {
    const float s = warp_sum(acc[m]);
    if ((c & 31) == 0) rec[1024 + (c >> 5) * 8 + m] = __float_as_uint(s * gscale);
  }
  if (c == 0) {
    rec[1056] = __float_as_uint(ldexpf(1.f, 24 - k));
    for (int w = 1057; w < kQrecWords; ++w) rec[w] = 0u;
  }
  __syncthreads();
  // A fragments of m16n8k16: rows 0-7 = head hi parts, rows 8-15 = lo parts
#pragma unroll
  for (int n = 0; n < 8; ++n) {
    const int widx = c + 128 * n;
    const int r = widx & 3, lane = (widx >> 2) & 31, kb = widx >> 7;
    const int gid = lane >> 2, tig = lane & 3;
    const int col = kb * 16 + 2 * tig + (r >= 2 ? 8 : 0);
    const __half* src = hs[r & 1][gid];
    const uint32_t lo = __half_as_ushort(src[col]);
    const uint32_t hi = __half_as_ushort(src[col + 1]);
    rec[widx] = lo | (hi << 16);
  }
}

// --------------------------------------------------------------------------
// 2a. BF16 sink + recent ring (CTA x = 0)
// --------------------------------------------------------------------------
__device__ void window_attention(const DecodeParams& p, int b, int h, uint8_t* smem) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = p.gqa, S = p.sink, W = p.recent;
  float* qs = reinterpret_cast<float*>(smem);                 // [8][128]
  float* sc = qs + kMaxGqa * kHeadDim;                        // [8][kMaxWindow]
  float* stat = sc + kMaxGqa * kMaxWindow;                    // [8][2]
  float* part = p.part + (((size_t)b * p.num_kv_heads + h) * (p.splits + 1)) * g * kPartFloats;

  const oscar_seq_state st = p.state[b];
  const int L = st.seq_len, E = st.int2_end;
  const bool ok = state_ok(L, E, S, W);
  const int ns = ok ? min(S, L) : 0;
  const int rb = max(E, S);
  const int nr = ok && L > rb ? L - rb : 0;
  const int nw = ns + nr;
  const size_t slots = (size_t)(S + W);
  const __nv_bfloat16* wk = p.window + (((size_t)b * p.num_kv_heads + h) * 2 + 0) * slots * kHeadDim;
  const __nv_bfloat16* wv = p.window + (((size_t)b * p.num_kv_heads + h) * 2 + 1) * slots * kHeadDim;

  for (int i = tid; i < g * kHeadDim; i += kThreads)
    qs[i] = __bfloat162float(p.q[((size_t)b * p.num_q_heads + h * g) * kHeadDim + i]) * p.scale_log2;
  __syncthreads();
  // scores: thread per token, all heads
  for (int t = tid; t < nw; t += kThreads) {
    const int slot = t < ns ? t : S + (rb + t - ns) % W;
    const uint4* row = reinterpret_cast<const uint4*>(wk + (size_t)slot * kHeadDim);
    float acc[kMaxGqa];
#pragma unroll
    for (int m = 0; m < kMaxGqa; ++m) acc[m] = 0.f;
#pragma unroll 4
    for (int u = 0; u < kHeadDim / 8; ++u) {
      const uint4 w = row[u];
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 kv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ws[e]));
        const int cidx = u * 8 + 2 * e;
#pragma unroll
        for (int m = 0; m < kMaxGqa; ++m) {
          if (m < g) {
            acc[m] = fmaf(qs[m * kHeadDim + cidx], kv.x, acc[m]);
            acc[m] = fmaf(qs[m * kHeadDim + cidx + 1], kv.y, acc[m]);
          }
        }
      }
    }
#pragma unroll
    for (int m = 0; m < kMaxGqa; ++m)
      if (m < g) sc[m * kMaxWindow + t] = acc[m];
  }
  __syncthreads();
  if (warp < g) {
    float mx = -INFINITY;
    for (int t = lane; t < nw; t += 32) mx = fmaxf(mx, sc[warp * kMaxWindow + t]);
    mx = warp_maxf(mx);
    float l = 0.f;
    if (nw > 0) {
      for (int t = lane; t < nw; t += 32) {
        const float e = exp2f(sc[warp * kMaxWindow + t] - mx);
        sc[warp * kMaxWindow + t] = e;
        l += e;
      }
    }
    l = warp_sum(l);
    if (lane == 0) {
      stat[2 * warp] = mx;
      stat[2 * warp + 1] = l;
    }
  }
  __syncthreads();
  for (int i = tid; i < g * kHeadDim; i += kThreads) {
    const int m = i / kHeadDim, c = i % kHeadDim;
    float acc = 0.f;
    for (int t = 0; t < nw; ++t) {
      const int slot = t < ns ? t : S + (rb + t - ns) % W;
      acc = fmaf(sc[m * kMaxWindow + t], __bfloat162float(wv[(size_t)slot * kHeadDim + c]), acc);
    }
    float* dst = part + (size_t)m * kPartFloats;
    dst[c] = acc;
    if (c == 0) {
      dst[kHeadDim] = stat[2 * m];
      dst[kHeadDim + 1] = stat[2 * m + 1];
    }
  }
}

// --------------------------------------------------------------------------
// 2b. INT2 pages (CTA x >= 1)
// --------------------------------------------------------------------------
__device__ void int2_attention(const DecodeParams& p, int b, int h, int split, uint8_t* smem) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int g = p.gqa, S = p.sink, W = p.recent;
  __shared__ int ids[kWarps][kStages];

  const oscar_seq_state st = p.state[b];
  const int L = st.seq_len, E = st.int2_end;
  const bool ok = state_ok(L, E, S, W);
  const int lo = S, hi = min(E, L);
  int npages = 0, first = 0;
  if (ok && hi > lo) {
    first = lo / kPage;
    npages = (hi - 1) / kPage - first + 1;
  }
  const int chunk = (npages + p.splits - 1) / p.splits;
  const int pbeg = first + (split - 1) * chunk;
  const int pend = min(pbeg + chunk, first + npages);
  const int nmine = pend - pbeg - warp > 0 ? (pend - pbeg - warp + kWarps - 1) / kWarps : 0;

  // query operand fragments, group sums, score scale
  const uint32_t* rec = p.qrec + ((size_t)b * p.num_kv_heads + h) * kQrecWords;
  uint32_t qa[8][4];
#pragma unroll
  for (int kb = 0; kb < 8; ++kb) {
    const uint4 w = reinterpret_cast<const uint4*>(rec)[kb * 32 + lane];
    qa[kb][0] = w.x;
    qa[kb][1] = w.y;
    qa[kb][2] = w.z;
    qa[kb][3] = w.w;
  }
  float qsum[4];
#pragma unroll
  for (int gq = 0; gq < 4; ++gq) qsum[gq] = __uint_as_float(rec[1024 + gq * 8 + gid]);
  const float uscale = __uint_as_float(rec[1056]);
  // probabilities enter the value product as fp16 p * pscale; pscale is the
  // largest power of two keeping p * pscale * s_v (s_v <= 2 clip_V / 3) finite
  const float pscale = p.pv_scale[h];

  uint8_t* sbuf = smem + warp * kStages * kBlockBytes;
  const int32_t* ptrow = p.page_table + (size_t)b * p.pt_stride;

  auto issue = [&](int stage, int pidx) {
    int id = ptrow[pidx];
    if (id < 0 || id >= p.num_pages) {
      if (lane == 0) atomicOr(p.err_flags, OSCAR_FLAG_BAD_PAGE_ID);
      id = -1;
    }
    if (lane == 0) ids[warp][stage] = id;
    if (id >= 0) {
      const uint8_t* src = p.pool + ((int64_t)id * p.num_kv_heads + h) * kBlockBytes;
      uint8_t* dst = sbuf + stage * kBlockBytes;
      cp_async16(dst + lane * 16, src + lane * 16);
      cp_async16(dst + 512 + lane * 16, src + 512 + lane * 16);
      cp_async16(dst + 1024 + lane * 16, src + 1024 + lane * 16);
    }
  };

#pragma unroll
  for (int s = 0; s < kStages; ++s) {
    if (s < nmine) issue(s, pbeg + warp + kWarps * s);
    cp_commit();
  }

  float m_run = -INFINITY, l_run = 0.f;
  float acc[8][4];
  float oz[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int cb = 0; cb < 8; ++cb) acc[cb][0] = acc[cb][1] = acc[cb][2] = acc[cb][3] = 0.f;

  const int t0 = 2 * tig;  // my tokens: t0, t0+1, t0+8, t0+9

  for (int it = 0; it < nmine; ++it) {
    cp_wait<kStages - 1>();
    __syncwarp();
    const int stage = it % kStages;
    const int pidx = pbeg + warp + kWarps * it;
    const uint8_t* sb = sbuf + stage * kBlockBytes;
    const int id = ids[warp][stage];
    const int pos0 = pidx * kPage;
    const bool full = id >= 0 && pos0 >= lo && pos0 + kPage <= hi;
    bool vld[4] = {true, true, true, true};
    if (!full) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int pos = pos0 + t0 + (i & 1) + 8 * (i >> 1);
        vld[i] = id >= 0 && pos >= lo && pos < hi;
      }
    }
    if (id >= 0) {
      const uint4 kw = *reinterpret_cast<const uint4*>(sb + lane * 16);
      const uint4 vw = *reinterpret_cast<const uint4*>(sb + 512 + lane * 16);

      // ---- scores: u = sum_gq s_k * (q~ . code) + z_k * sum q~ -------------
      float u[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int gq = 0; gq < 4; ++gq) {
        const uint4 mk = *reinterpret_cast<const uint4*>(sb + 1024 + 16 * (4 * gq + tig));
        float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
#define OSCAR_QK(KB)                                                                              \
  mma16816(c0, qa[KB][0], qa[KB][1], qa[KB][2], qa[KB][3], slot_bits<KB>(kw.x), slot_bits<KB>(kw.y)); \
  mma16816(c1, qa[KB][0], qa[KB][1], qa[KB][2], qa[KB][3], slot_bits<KB>(kw.z), slot_bits<KB>(kw.w));
        if (gq == 0) { OSCAR_QK(0) OSCAR_QK(1) }
        if (gq == 1) { OSCAR_QK(2) OSCAR_QK(3) }
        if (gq == 2) { OSCAR_QK(4) OSCAR_QK(5) }
        if (gq == 3) { OSCAR_QK(6) OSCAR_QK(7) }
#undef OSCAR_QK
        const float2 s01 = h2_bits_to_f2(mk.x), z01 = h2_bits_to_f2(mk.y);
        const float2 s23 = h2_bits_to_f2(mk.z), z23 = h2_bits_to_f2(mk.w);
        u[0] += s01.x * (c0[0] + c0[2]) + z01.x * qsum[gq];
        u[1] += s01.y * (c0[1] + c0[3]) + z01.y * qsum[gq];
        u[2] += s23.x * (c1[0] + c1[2]) + z23.x * qsum[gq];
        u[3] += s23.y * (c1[1] + c1[3]) + z23.y * qsum[gq];
      }

      // ---- online softmax (log2 domain), per head gid -----------------------
      float s[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) s[i] = vld[i] ? u[i] * uscale : -INFINITY;
      float mx = fmaxf(fmaxf(s[0], s[1]), fmaxf(s[2], s[3]));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float m_new = fmaxf(m_run, mx);
      if (m_new != -INFINITY) {
        const float alpha = exp2f(m_run - m_new);
        float pr[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) pr[i] = exp2f(s[i] - m_new);
        l_run = l_run * alpha + ((pr[0] + pr[1]) + (pr[2] + pr[3]));
        m_run = m_new;
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
          const float ae = __shfl_sync(0xffffffffu, alpha, 8 * tig);
          const float ao = __shfl_sync(0xffffffffu, alpha, 8 * tig + 4);
#pragma unroll
          for (int cb = 0; cb < 8; ++cb) {
            acc[cb][0] *= ae;
            acc[cb][1] *= ao;
            acc[cb][2] *= ae;
            acc[cb][3] *= ao;
          }
          oz[0] *= ae;
          oz[1] *= ao;
          oz[2] *= ae;
          oz[3] *= ao;
        }
        const uint32_t P01 = f2_to_h2_bits(pr[0] * pscale, pr[1] * pscale);
        const uint32_t P23 = f2_to_h2_bits(pr[2] * pscale, pr[3] * pscale);
        const uint32_t m01 = (vld[0] ? 0x0000ffffu : 0u) | (vld[1] ? 0xffff0000u : 0u);
        const uint32_t m23 = (vld[2] ? 0x0000ffffu : 0u) | (vld[3] ? 0xffff0000u : 0u);

        // ---- values: acc[cb] += codes^T (p * s_v) ; oz += z_v^T p -------------
#pragma unroll
        for (int gq = 0; gq < 4; ++gq) {
          const uint4 mv = *reinterpret_cast<const uint4*>(sb + 1024 + 16 * (4 * (4 + gq) + tig));
          const uint32_t B0 = hmul2_bits(P01, mv.x & m01);
          const uint32_t B1 = hmul2_bits(P23, mv.z & m23);
#define OSCAR_PV(CB)                                                                          \
  mma16816(acc[CB], slot_bits<CB>(vw.x), slot_bits<CB>(vw.y), slot_bits<CB>(vw.z), slot_bits<CB>(vw.w), \
           B0, B1);
          if (gq == 0) { OSCAR_PV(0) OSCAR_PV(1) }
          if (gq == 1) { OSCAR_PV(2) OSCAR_PV(3) }
          if (gq == 2) { OSCAR_PV(4) OSCAR_PV(5) }
          if (gq == 3) { OSCAR_PV(6) OSCAR_PV(7) }
#undef OSCAR_PV
        }
        const uint4 mz = *reinterpret_cast<const uint4*>(sb + 1024 + 16 * (4 * (4 + (gid & 3)) + tig));
        const uint32_t za0 = gid < 4 ? (mz.y & m01) : 0u;
        const uint32_t za2 = gid < 4 ? (mz.w & m23) : 0u;
        mma16816(oz, za0, 0u, za2, 0u, P01, P23);
      }
    }
    __syncwarp();
    const int nxt = it + kStages;
    if (nxt < nmine) issue(stage, pbeg + warp + kWarps * nxt);
    cp_commit();
  }
  cp_wait<0>();

  // ---- per-warp partial -> shared memory, then CTA merge --------------------
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
  __syncthreads();  // staging buffers are reused below
  float* wpart = reinterpret_cast<float*>(smem);              // [8 warps][8 heads][128]
  float* wml = wpart + kWarps * kMaxGqa * kHeadDim;           // [8 warps][8 heads][2]
  if (tig == 0) {
    wml[(warp * kMaxGqa + gid) * 2] = m_run;
    wml[(warp * kMaxGqa + gid) * 2 + 1] = l_run;
  }
#pragma unroll
  for (int cb = 0; cb < 8; ++cb) {
    const int gq = cb >> 1;
    const float ze = __shfl_sync(0xffffffffu, oz[0], 4 * gq + tig) / pscale;
    const float zo = __shfl_sync(0xffffffffu, oz[1], 4 * gq + tig) / pscale;
    const float sc = 16777216.f / (slot_factor(cb) * pscale);
    const int ch = 16 * cb + gid;
    const int he = 2 * tig, ho = 2 * tig + 1;
    float* base = wpart + warp * kMaxGqa * kHeadDim;
    base[he * kHeadDim + ch] = acc[cb][0] * sc + ze;
    base[ho * kHeadDim + ch] = acc[cb][1] * sc + zo;
    base[he * kHeadDim + ch + 8] = acc[cb][2] * sc + ze;
    base[ho * kHeadDim + ch + 8] = acc[cb][3] * sc + zo;
  }
  __syncthreads();
  float* part = p.part + (((size_t)b * p.num_kv_heads + h) * (p.splits + 1) + split) * g * kPartFloats;
  for (int i = tid; i < g * kHeadDim; i += kThreads) {
    const int m = i / kHeadDim, c = i % kHeadDim;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, wml[(w * kMaxGqa + m) * 2]);
    float o = 0.f, l = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float mw = wml[(w * kMaxGqa + m) * 2];
        const float sw = mw == -INFINITY ? 0.f : exp2f(mw - M);
        o += sw * wpart[(w * kMaxGqa + m) * kHeadDim + c];
        l += sw * wml[(w * kMaxGqa + m) * 2 + 1];
      }
    }
    float* dst = part + (size_t)m * kPartFloats;
    dst[c] = o;
    if (c == 0) {
      dst[kHeadDim] = M;
      dst[kHeadDim + 1] = l;
    }
  }
}

__global__ void __launch_bounds__(kThreads, 2) oscar_decode_kernel(DecodeParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  if (split == 0)
    window_attention(p, b, h, smem);
  else
    int2_attention(p, b, h, split, smem);
}

// --------------------------------------------------------------------------
// 3. merge of the partials, un-rotation, normalisation
// --------------------------------------------------------------------------
__global__ void __launch_bounds__(128) oscar_merge_kernel(DecodeParams p) {
  const int h = blockIdx.x, b = blockIdx.y, c = threadIdx.x;
  const int g = p.gqa, nslots = p.splits + 1;
  __shared__ float orot[kMaxGqa][kHeadDim];
  const float* part = p.part + ((size_t)b * p.num_kv_heads + h) * nslots * g * kPartFloats;
  float ow[kMaxGqa], lsum[kMaxGqa];
#pragma unroll
  for (int m = 0; m < kMaxGqa; ++m) {
    ow[m] = 0.f;
    lsum[m] = 0.f;
    if (m >= g) continue;
    float M = -INFINITY;
    for (int s = 0; s < nslots; ++s) M = fmaxf(M, part[((size_t)s * g + m) * kPartFloats + kHeadDim]);
    float orr = 0.f;
    if (M != -INFINITY) {
      for (int s = 0; s < nslots; ++s) {
        const float* ps = part + ((size_t)s * g + m) * kPartFloats;
        const float ms = ps[kHeadDim];
        if (ms == -INFINITY) continue;
        const float w = exp2f(ms - M);
        lsum[m] += w * ps[kHeadDim + 1];
        const float v = w * ps[c];
        if (s == 0)
          ow[m] = v;
        else
          orr += v;
      }
    }
    orot[m][c] = orr;
  }
  __syncthreads();
  const float* RT = p.R_VT + (size_t)h * kHeadDim * kHeadDim;
  float oi[kMaxGqa];
#pragma unroll
  for (int m = 0; m < kMaxGqa; ++m) oi[m] = 0.f;
  if (p.fold_rv) {
#pragma unroll
    for (int m = 0; m < kMaxGqa; ++m)
      if (m < g) oi[m] = orot[m][c];
  } else {
#pragma unroll 4
    for (int i = 0; i < kHeadDim; ++i) {
      const float r = __ldg(&RT[i * kHeadDim + c]);
#pragma unroll
      for (int m = 0; m < kMaxGqa; ++m)
        if (m < g) oi[m] = fmaf(orot[m][i], r, oi[m]);
    }
  }
#pragma unroll
  for (int m = 0; m < kMaxGqa; ++m) {
    if (m >= g) continue;
    const float val = lsum[m] > 0.f ? (oi[m] + ow[m]) / lsum[m] : 0.f;
    p.o[((size_t)b * p.num_q_heads + h * g + m) * kHeadDim + c] = val;
  }
}


int decode_smem_bytes() {
  const int window = (kMaxGqa * kHeadDim + kMaxGqa * kMaxWindow + 2 * kMaxGqa) * 4;
  const int merge = (kWarps * kMaxGqa * kHeadDim + kWarps * kMaxGqa * 2) * 4;
  int m = kStageBytes;
  if (window > m) m = window;
  if (merge > m) m = merge;
  return m;
}

cudaError_t launch_decode(const DecodeParams& p, int batch, cudaStream_t s) {
  static bool attr_set = false;
  const int smem = decode_smem_bytes();
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(oscar_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  oscar_rotate_q_kernel<<<dim3(p.num_kv_heads, batch), 128, 0, s>>>(p);
  oscar_decode_kernel<<<dim3(p.splits + 1, p.num_kv_heads, batch), kThreads, smem, s>>>(p);
  oscar_merge_kernel<<<dim3(p.num_kv_heads, batch), 128, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace oscar
