// Offline calibration on the device: the two covariance targets of OSCAR's
// rotations for one layer.
//
// Sources: "OSCAR: Offline Spectral Covariance-Aware Rotation ..." (gist.science,
// it), Riepilogo Tecnico 2.1 (value error weighted by the scores S) and 2.2 A
// ("Stima della Covarianza": C_Q from the queries, C_S from the score-weighted
// values); "Juntos, AI Open-Sources OSCAR ..." (7minutos.es), section "Lo que
// OSCAR hace diferente".
//
// Per KV head h, averaged over its g query heads j:
//   C_Q[h] = (1 / (N g)) sum_j sum_n q_jn^T q_jn
//   C_S[h] = (1 / (N g)) sum_j (S_j V_h)^T (S_j V_h),  S_j = causal softmax(q_j k_h^T * scale)
// Two kernels: the causal attention output O_j = S_j V_h of every query head
// (fp32, an online softmax over 64-key blocks, written to the caller's
// workspace), then the symmetric 128 x 128 products sum X^T X of Q and O. The
// eigendecomposition that turns them into rotations stays on the host.
#include <math.h>

#include "oscar_internal.cuh"

namespace oscar {

namespace {

constexpr int kCalRows = 64;     // queries per attention CTA
constexpr int kCalKeys = 64;     // keys per block
constexpr int kCalThreads = 128; // two threads per query row
constexpr int kCalSmem = (kCalRows + 2 * kCalKeys) * kHeadDim * 4 + kCalRows * kCalKeys * 4;

// rows [i0, i0 + 64) of O_j for query head j = blockIdx.y
__global__ void __launch_bounds__(kCalThreads) oscar_calib_attention_kernel(
    const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ v,
    int n, int hq, int hkv, float scale_log2, float* __restrict__ o) {
  extern __shared__ __align__(16) float cs[];
  float* Qs = cs;                               // [64][128]
  float* Ks = Qs + kCalRows * kHeadDim;         // [64][128]
  float* Vs = Ks + kCalKeys * kHeadDim;         // [64][128]
  float* Ps = Vs + kCalKeys * kHeadDim;         // [64 rows][64 keys]
  const int tid = threadIdx.x, j = blockIdx.y, h = j / (hq / hkv);
  const int i0 = blockIdx.x * kCalRows;
  const int r = tid >> 1, half = tid & 1;       // my row; my half of keys / channels
  for (int e = tid; e < kCalRows * kHeadDim; e += kCalThreads) {
    const int rr = e / kHeadDim, c = e % kHeadDim, i = i0 + rr;
    Qs[e] = i < n ? __bfloat162float(q[((size_t)i * hq + j) * kHeadDim + c]) * scale_log2 : 0.f;
  }
  float m = -INFINITY, l = 0.f;                 // running max (log2 units) and sum of my row
  float acc[64];                                // channels 64 half .. 64 half + 63 of my row
#pragma unroll
  for (int c = 0; c < 64; ++c) acc[c] = 0.f;
  const int i = i0 + r;
  const int kend = min(n, i0 + kCalRows);       // causal: keys < the block's last query + 1
  for (int t0 = 0; t0 < kend; t0 += kCalKeys) {
    __syncthreads();                            // previous blocks consumed
    for (int e = tid; e < kCalKeys * kHeadDim; e += kCalThreads) {
      const int tt = e / kHeadDim, c = e % kHeadDim, t = t0 + tt;
      Ks[e] = t < n ? __bfloat162float(k[((size_t)t * hkv + h) * kHeadDim + c]) : 0.f;
      Vs[e] = t < n ? __bfloat162float(v[((size_t)t * hkv + h) * kHeadDim + c]) : 0.f;
    }
    __syncthreads();
    // scores of my row for keys 32 half .. 32 half + 31 (log2 units), staged in Ps
    float* prow = Ps + r * kCalKeys + 32 * half;
    float mx = -INFINITY;
#pragma unroll 4
    for (int kk = 0; kk < 32; ++kk) {
      const int tk = 32 * half + kk, t = t0 + tk;
      float d = 0.f;
      const float* qr = Qs + r * kHeadDim;
      const float* kr = Ks + tk * kHeadDim;
#pragma unroll 16
      for (int c = 0; c < kHeadDim; ++c) d = fmaf(qr[c], kr[c], d);
      d = (t <= i && t < n) ? d : -INFINITY;
      prow[kk] = d;
      mx = fmaxf(mx, d);
    }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    const float mnew = fmaxf(m, mx);
    const float alpha = (mnew == -INFINITY) ? 1.f : exp2f(m - mnew);
    float ls = 0.f;
#pragma unroll 4
    for (int kk = 0; kk < 32; ++kk) {
      const float sv = prow[kk];
      const float pv = sv == -INFINITY ? 0.f : exp2f(sv - mnew);
      prow[kk] = pv;
      ls += pv;
    }
    ls += __shfl_xor_sync(0xffffffffu, ls, 1);
    l = l * alpha + ls;
    m = mnew;
#pragma unroll
    for (int c = 0; c < 64; ++c) acc[c] *= alpha;
    __syncwarp();
    // O row += P row V over the block's keys, my 64 channels
    for (int tk = 0; tk < kCalKeys; ++tk) {
      const float pv = Ps[r * kCalKeys + tk];
      const float* vr = Vs + tk * kHeadDim + 64 * half;
#pragma unroll
      for (int c = 0; c < 64; ++c) acc[c] = fmaf(pv, vr[c], acc[c]);
    }
  }
  if (i < n) {
    const float inv = l > 0.f ? 1.f / l : 0.f;
    float* dst = o + ((size_t)j * n + i) * kHeadDim + 64 * half;
#pragma unroll
    for (int c = 0; c < 64; ++c) dst[c] = acc[c] * inv;
  }
}

// C[h] (+)= sum over the g query heads and n rows of x^T x / (n g), rows 32 rb ..
// 32 rb + 31 of the 128 x 128 result; x = q (bf16 [n][hq][128]) for which = 0,
// x = O (fp32 [hq][n][128]) for which = 1
constexpr int kCovThreads = 256;
constexpr int kCovChunk = 64;    // samples staged per round
__global__ void __launch_bounds__(kCovThreads) oscar_calib_cov_kernel(const __nv_bfloat16* __restrict__ q,
                                                                      const float* __restrict__ o, int n, int hq,
                                                                      int hkv, float* __restrict__ c_q,
                                                                      float* __restrict__ c_s) {
  __shared__ float xs[kCovChunk][kHeadDim];
  const int tid = threadIdx.x, rb = blockIdx.x, h = blockIdx.y, which = blockIdx.z;
  const int g = hq / hkv;
  const int row = 32 * rb + (tid >> 3), c0 = (tid & 7) * 16;
  float acc[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) acc[e] = 0.f;
  for (int jj = 0; jj < g; ++jj) {
    const int j = h * g + jj;
    for (int s0 = 0; s0 < n; s0 += kCovChunk) {
      __syncthreads();
      for (int e = tid; e < kCovChunk * kHeadDim; e += kCovThreads) {
        const int ss = e / kHeadDim, c = e % kHeadDim, s = s0 + ss;
        float x = 0.f;
        if (s < n)
          x = which == 0 ? __bfloat162float(q[((size_t)s * hq + j) * kHeadDim + c])
                         : o[((size_t)j * n + s) * kHeadDim + c];
        xs[ss][c] = x;
      }
      __syncthreads();
#pragma unroll 4
      for (int ss = 0; ss < kCovChunk; ++ss) {
        const float xi = xs[ss][row];
#pragma unroll
        for (int e = 0; e < 16; ++e) acc[e] = fmaf(xi, xs[ss][c0 + e], acc[e]);
      }
    }
  }
  const float inv = 1.f / ((float)n * (float)g);
  float* dst = (which == 0 ? c_q : c_s) + ((size_t)h * kHeadDim + row) * kHeadDim + c0;
#pragma unroll
  for (int e = 0; e < 16; ++e) dst[e] = acc[e] * inv;
}

}  // namespace

size_t calib_workspace_bytes(int n, int hq) { return (size_t)hq * n * kHeadDim * sizeof(float); }

cudaError_t launch_calib_covariances(const __nv_bfloat16* q, const __nv_bfloat16* k, const __nv_bfloat16* v, int n,
                                     int hq, int hkv, float scale, float* c_q, float* c_s, float* o_ws,
                                     cudaStream_t s) {
  static PerDeviceOnce attrs;
  const cudaError_t ea = once_for_current_device(attrs, [] {
    return cudaFuncSetAttribute(oscar_calib_attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kCalSmem);
  });
  if (ea != cudaSuccess) return ea;
  oscar_calib_attention_kernel<<<dim3((n + kCalRows - 1) / kCalRows, hq), kCalThreads, kCalSmem, s>>>(
      q, k, v, n, hq, hkv, scale * 1.4426950408889634f, o_ws);
  oscar_calib_cov_kernel<<<dim3(kHeadDim / 32, hkv, 2), kCovThreads, 0, s>>>(q, o_ws, n, hq, hkv, c_q, c_s);
  return cudaGetLastError();
}

}  // namespace oscar
