// Prefill write path on the 5th-generation tensor cores: rotate a batch of new
// tokens (x R as a BF16 GEMM with R = R_hi + R_lo and fp32 accumulation in tensor
// memory), then clip, group-quantise and pack them into their INT2 pages.
//
// Sources: "Juntos, AI Open-Sources OSCAR ..." (7minutos.es), section "El
// sistema de servicio" (write path: rotate, clip to the calibrated threshold,
// asymmetric per-token INT2 groups); "OSCAR: Offline Spectral Covariance-Aware
// Rotation ..." (gist.science, it), Riepilogo Tecnico 2.2 A (R = U H P).
//
// Work split. Only the tokens that go straight from the input to INT2 (positions
// [max(L, S), E') of an append) are handled here; sink tokens, ring occupants
// and the ring entries they evict stay with oscar_quant_append_kernel. Tiles are
// 128 page-aligned positions (8 pages) of one KV head of one request; a CTA
// owns a strided set of tiles of one (request, KV head) and walks them as jobs
// (tile, K) and (tile, V).
//
// Per CTA (256 threads, one per SM): shared memory holds the four rotation
// images (R_K hi/lo, R_V hi/lo; bf16, K-major, 128-byte swizzle, 32 KiB each),
// two 32 KiB token-tile buffers and the packing scratch. Thread 0 issues the 16
// tcgen05.mma (M 128, N 128, K 16; hi then lo) of a job into one of two
// 128-column TMEM accumulators and commits them to an mbarrier; while they run,
// all eight warps quantise the previous job: warp w reads TMEM lanes
// 32 (w % 4) .. +31 (one token each) and columns 64 (w / 4) .. +63 (two groups),
// and the next tile streams in with cp.async. Every mbarrier wait is bounded:
// on expiry the kernel raises OSCAR_FLAG_TIMEOUT and stops issuing work.
#include <math.h>

#include "oscar_internal.cuh"

namespace oscar {

constexpr int kPfThreads = 256;
constexpr int kTileM = 128;
constexpr int kImageBytes = kHeadDim * kHeadDim * 2;     // one bf16 128 x 128 operand: 32 KiB
constexpr int kAtomBytes = kTileM * 128;                 // 64 bf16 columns of 128 rows: 16 KiB
constexpr int kPfSmemImages = 4 * kImageBytes;            // R_K hi, R_K lo, R_V hi, R_V lo
constexpr int kPfSmemX = 2 * kImageBytes;                 // two token tiles
constexpr int kPfSmemPack = 2 * kTileM * 8 * 4 + 2 * kTileM * 16 * 2;  // partial K words, V half-words
constexpr int kPfSmem = 1024 + kPfSmemImages + kPfSmemX + kPfSmemPack + 64;
constexpr uint32_t kTmemCols = 256;
constexpr long kSpinLimit = 1L << 20;

// ---- PTX wrappers ------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void cp16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(smem)), "l"(gmem));
}
__device__ __forceinline__ void cp_commit_pf() { asm volatile("cp.async.commit_group;\n" ::); }
__device__ __forceinline__ void cp_wait_all_pf() { asm volatile("cp.async.wait_group 0;\n" ::); }
__device__ __forceinline__ void cp_wait_one_pf() { asm volatile("cp.async.wait_group 1;\n" ::); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }

__device__ __forceinline__ void mbar_init(uint32_t addr, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(addr), "r"(count));
}
// bounded wait on an mbarrier phase; false when the limit expires
__device__ __forceinline__ bool mbar_wait(uint32_t addr, uint32_t parity) {
  for (long it = 0; it < kSpinLimit; ++it) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(addr), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

// shared-memory matrix descriptor: K-major operand, 128-byte swizzle, 8-row
// groups 1024 bytes apart
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFF) >> 4);        // start address
  d |= (uint64_t)1 << 16;                         // leading byte offset (unused with this swizzle)
  d |= (uint64_t)(1024 >> 4) << 32;               // stride byte offset
  d |= (uint64_t)1 << 46;                         // descriptor version
  d |= (uint64_t)2 << 61;                         // 128-byte swizzle
  return d;
}

// instruction descriptor: D f32, A and B bf16, both K-major, M = 128, N = 128
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(128 >> 3) << 17) |
                            ((uint32_t)(128 >> 4) << 24);

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(kIdesc), "r"(accumulate));
}
__device__ __forceinline__ void umma_commit(uint32_t mbar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(mbar)
               : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Scale, zero and the 2-bit codes of one group of 32 rotated values, packed in
// place into the page-block words (kw: K words, vh: V half-words) of the token.
//
// The quantiser is code = clamp(rint(fp32(fp32(xc - zf) * fp32(1 / sf))), 0, 3)
// on the clipped value xc. Every step is monotone in x and the clip bounds map
// to the extreme codes (they are the group's min / max after clipping), so the
// code of the unclipped value clamped to [0, 3] is the same and only the min /
// max are clipped. rint (nearest, ties to even) is an add of 1.5 * 2^23.
template <int KIND, int GQ>
__device__ __forceinline__ void group_quantise(const float (&v)[32], float clip, __half& s16, __half& z16,
                                               uint32_t (&kw)[8], uint32_t (&vh)[16]) {
  float mn = v[0], mx = v[0];
#pragma unroll
  for (int i = 1; i < 32; ++i) {
    mn = fminf(mn, v[i]);
    mx = fmaxf(mx, v[i]);
  }
  mn = fminf(fmaxf(mn, -clip), clip);
  mx = fminf(fmaxf(mx, -clip), clip);
  s16 = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), 3.0f));
  z16 = __float2half_rn(mn);
  const float sf = __half2float(s16), zf = __half2float(z16);
  const float rsf = sf != 0.f ? __frcp_rn(sf) : 0.f;  // sf == 0: every code is 0
  constexpr float kMagic = 12582912.f;                 // 1.5 * 2^23
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const float u = fminf(fmaxf(__fmul_rn(__fsub_rn(v[i], zf), rsf), 0.f), 3.f);
    const uint32_t code = __float_as_uint(__fadd_rn(u, kMagic)) & 3u;
    constexpr int kCh0 = 32 * GQ;
    const int ch = kCh0 + i;                            // compile-time
    const int si = ch >> 4, r = ch & 15;
    if (KIND == 0)
      kw[2 * ((r & 7) >> 1) + (r >> 3)] |= code << (16 * (r & 1) + 2 * si);
    else
      vh[2 * (r & 7) + (r >> 3)] |= code << (2 * si);
  }
}

// Quantise job j from tensor memory: the warp reads TMEM lanes 32 (warp % 4) ..
// (one token per thread) and the 64 columns of its HALF (two groups); codes go
// to the partial-word scratch, scale / zero straight to the page block. All
// channel indices are compile-time, so the packing stays in registers.
template <int HALF, int KIND>
__device__ __forceinline__ void pf_epilogue(const PrefillParams& p, int j, int c, int warp, int lane, int h,
                                            int b, int64_t P0, int64_t d0, int64_t d1, uint32_t tmem,
                                            uint32_t* kpart, uint16_t* vpart) {
  const int tile = c + (j >> 1) * (int)gridDim.x;
  constexpr int kind = KIND;
  const int row = 32 * (warp & 3) + lane;
  const int64_t pos = P0 + (int64_t)tile * kTileM + row;
  const bool valid = pos >= d0 && pos < d1;
  const uint32_t acc = tmem + (uint32_t)((j & 1) * kHeadDim) + ((uint32_t)(32 * (warp & 3)) << 16);
  const float clip = (kind ? p.clip_V : p.clip_K)[h];
  const int Hkv = p.num_kv_heads;
  uint8_t* blk = nullptr;
  if (valid) {
    const int64_t pidx = pos / kPage;
    const int32_t id = pidx < p.pt_stride ? p.page_table[(int64_t)b * p.pt_stride + pidx] : -1;
    if (id >= 0 && id < p.num_pages)
      blk = p.pool + ((int64_t)id * Hkv + h) * kBlockBytes;
    else
      atomicOr(p.err_flags, OSCAR_FLAG_BAD_PAGE_ID);
  }
  const int t = (int)(pos % kPage);
  const int bb = (t & 7) >> 1, pair = t >> 3, th = t & 1;
  uint32_t kw[8];
  uint32_t vh[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) kw[i] = 0u;
#pragma unroll
  for (int i = 0; i < 16; ++i) vh[i] = 0u;
#pragma unroll
  for (int gg = 0; gg < 2; ++gg) {
    const int gq = 2 * HALF + gg;
    float v[32];
    tmem_ld32(acc + (uint32_t)(32 * gq), v);
    if (valid && p.trace && pos < p.trace_positions) {
      float* tr = p.trace + ((((size_t)b * p.trace_positions + pos) * Hkv + h) * 2 + kind) * kHeadDim + 32 * gq;
#pragma unroll
      for (int i = 0; i < 32; ++i) tr[i] = v[i];
    }
    __half s16, z16;
    if (gg == 0)
      group_quantise<KIND, 2 * HALF>(v, clip, s16, z16, kw, vh);
    else
      group_quantise<KIND, 2 * HALF + 1>(v, clip, s16, z16, kw, vh);
    if (blk) {
      if (kind == 0) {
        *reinterpret_cast<__half*>(blk + 1024 + 32 * bb + 8 * gq + 4 * pair + 2 * th) = s16;
        *reinterpret_cast<__half*>(blk + 1152 + 4 * (2 * t + (gq >> 1)) + 2 * (gq & 1)) = z16;
      } else {
        uint8_t* m = blk + 1280 + 16 * (4 * gq + bb) + 4 * (2 * pair) + 2 * th;
        *reinterpret_cast<__half*>(m) = s16;
        *reinterpret_cast<__half*>(m + 4) = z16;
      }
    }
  }
  // combine the two column halves of every token, then store its codes
  if (kind == 0) {
#pragma unroll
    for (int i = 0; i < 8; ++i) kpart[(HALF * kTileM + row) * 8 + i] = kw[i];
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) vpart[(HALF * kTileM + row) * 16 + i] = (uint16_t)vh[i];
  }
  tc_fence_before();
  __syncthreads();
  if (HALF == 0 && blk) {
    const int a = t & 7, tt = t >> 3;
    if (kind == 0) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int b2 = i >> 1, x = i & 1;
        const uint32_t w = kpart[row * 8 + i] | kpart[(kTileM + row) * 8 + i];
        *reinterpret_cast<uint32_t*>(blk + 16 * (4 * a + b2) + 4 * (2 * tt + x)) = w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int a2 = i >> 1, x = i & 1;
        const uint16_t w = (uint16_t)(vpart[row * 16 + i] | vpart[(kTileM + row) * 16 + i]);
        *reinterpret_cast<uint16_t*>(blk + 512 + 16 * (4 * a2 + bb) + 4 * (2 * tt + x) + 2 * th) = w;
      }
    }
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kPfThreads, 1) oscar_prefill_append_kernel(PrefillParams p) {
  extern __shared__ uint8_t dsm_raw[];
  // 1024-byte alignment for the swizzled operands
  uint8_t* dsm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t* img = dsm;                                     // 4 rotation images
  uint8_t* xbuf = img + kPfSmemImages;                    // 2 token tiles
  uint32_t* kpart = reinterpret_cast<uint32_t*>(xbuf + kPfSmemX);       // [2][128][8]
  uint16_t* vpart = reinterpret_cast<uint16_t*>(kpart + 2 * kTileM * 8);  // [2][128][16]
  uint64_t* mbar = reinterpret_cast<uint64_t*>(vpart + 2 * kTileM * 16);  // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mbar + 2);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int S = p.sink, W = p.recent, Hkv = p.num_kv_heads;

  // rotation images are constant: stage them before waiting for earlier kernels
  {
    const uint8_t* src = p.images + (size_t)h * kPfSmemImages;
    for (int i = tid; i < kPfSmemImages / 16; i += kPfThreads) cp16(img + 16 * i, src + 16 * i);
    cp_commit_pf();
  }
  pdl_trigger();
  pdl_wait();

  __shared__ oscar_seq_state s_st;
  if (tid == 0) s_st = p.state[b];
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::);
  }
  if (tid == 0) {
    mbar_init(smem_u32(&mbar[0]), 1);
    mbar_init(smem_u32(&mbar[1]), 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  cp_wait_all_pf();
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const oscar_seq_state st = s_st;
  const bool ok = state_ok(st, S, W, p.max_batch);
  const int L = st.seq_len, E = st.int2_end;
  int64_t E2 = (int64_t)L + p.n_new - W;
  if (E2 < E) E2 = E;
  if (E2 < S) E2 = S;
  const int64_t d0 = L > S ? L : S;            // first position quantised straight from the input
  const int64_t d1 = ok ? E2 : d0;             // end of that range
  const int64_t P0 = (d0 / kPage) * kPage;     // tiles are page aligned
  const int ntiles = d1 > d0 ? (int)((d1 - P0 + kTileM - 1) / kTileM) : 0;
  const int nmine = ntiles > c ? (ntiles - c + (int)gridDim.x - 1) / (int)gridDim.x : 0;
  const int njobs = 2 * nmine;

  const size_t tok_stride = (size_t)Hkv * kHeadDim;    // elements between tokens of the input
  const __nv_bfloat16* xbase_k = p.k + ((size_t)b * p.n_new * Hkv + h) * kHeadDim;
  const __nv_bfloat16* xbase_v = p.v + ((size_t)b * p.n_new * Hkv + h) * kHeadDim;

  // stage the token rows of job j into tile buffer j & 1 (128-byte swizzle, K-major)
  auto load_job = [&](int j) {
    const int tile = c + (j >> 1) * (int)gridDim.x;
    const __nv_bfloat16* xb = (j & 1) ? xbase_v : xbase_k;
    uint8_t* buf = xbuf + (size_t)(j & 1) * kImageBytes;
    for (int i = tid; i < kTileM * 16; i += kPfThreads) {
      const int r = i >> 4, chunk = i & 15;
      const int64_t pos = P0 + (int64_t)tile * kTileM + r;
      if (pos < d0 || pos >= d1) continue;
      const __nv_bfloat16* src = xb + (size_t)(pos - L) * tok_stride + 8 * chunk;
      const int atom = chunk >> 3, cc = chunk & 7;
      cp16(buf + atom * kAtomBytes + r * 128 + ((cc ^ (r & 7)) << 4), src);
    }
    cp_commit_pf();
  };

  bool alive = true;
  if (njobs > 0) load_job(0);

  auto epilogue = [&](int j) {
    if (warp < 4) {
      if (j & 1)
        pf_epilogue<0, 1>(p, j, c, warp, lane, h, b, P0, d0, d1, tmem, kpart, vpart);
      else
        pf_epilogue<0, 0>(p, j, c, warp, lane, h, b, P0, d0, d1, tmem, kpart, vpart);
    } else {
      if (j & 1)
        pf_epilogue<1, 1>(p, j, c, warp, lane, h, b, P0, d0, d1, tmem, kpart, vpart);
      else
        pf_epilogue<1, 0>(p, j, c, warp, lane, h, b, P0, d0, d1, tmem, kpart, vpart);
    }
  };

  for (int j = 0; j < njobs && alive; ++j) {
    // (a) the MMAs of job j - 1 are done: its tile buffer and accumulator are readable
    if (j >= 1) {
      const bool done = mbar_wait(smem_u32(&mbar[(j - 1) & 1]), ((j - 1) >> 1) & 1);
      alive = __syncthreads_and(done) != 0;  // one decision for the whole CTA
      if (!alive) {
        if (tid == 0) atomicOr(p.err_flags, OSCAR_FLAG_TIMEOUT);
        break;
      }
    }
    // (b) prefetch job j + 1 into the buffer job j - 1 used
    if (j + 1 < njobs) {
      load_job(j + 1);
      cp_wait_one_pf();
    } else {
      cp_wait_all_pf();
    }
    // (c) job j's tile is in shared memory
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // (d) issue job j
    if (tid == 0) {
      const int kind = j & 1;
      const uint32_t a_base = smem_u32(xbuf + (size_t)(j & 1) * kImageBytes);
      const uint32_t hi_base = smem_u32(img + (size_t)(2 * kind) * kImageBytes);
      const uint32_t lo_base = smem_u32(img + (size_t)(2 * kind + 1) * kImageBytes);
      const uint32_t d_tmem = tmem + (uint32_t)((j & 1) * kHeadDim);
#pragma unroll
      for (int term = 0; term < 2; ++term) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (uint32_t)((kk >> 2) * kAtomBytes + (kk & 3) * 32);
          umma_bf16(d_tmem, sw128_desc(a_base + off), sw128_desc((term ? lo_base : hi_base) + off),
                    (term | kk) ? 1u : 0u);
        }
      }
      umma_commit(smem_u32(&mbar[j & 1]));
    }
    // (e) quantise job j - 1 while job j runs
    if (j >= 1) {
      tc_fence_after();
      epilogue(j - 1);
    }
  }
  if (alive && njobs > 0) {
    const int j = njobs - 1;
    const bool done = mbar_wait(smem_u32(&mbar[j & 1]), (j >> 1) & 1);
    if (__syncthreads_and(done)) {
      tc_fence_after();
      epilogue(j);
    } else if (tid == 0) {
      atomicOr(p.err_flags, OSCAR_FLAG_TIMEOUT);
    }
  }
  cp_wait_all_pf();
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(kTmemCols));
  }
}

cudaError_t launch_prefill_append(const PrefillParams& p, int ctas_per_head, cudaStream_t s) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(oscar_prefill_append_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kPfSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaError_t e = launch_pdl(oscar_prefill_append_kernel, dim3(ctas_per_head, p.num_kv_heads, p.batch),
                             dim3(kPfThreads), kPfSmem, s, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

int prefill_image_bytes() { return kPfSmemImages; }

}  // namespace oscar
