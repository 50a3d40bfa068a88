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
// (one per SM) owns a strided set of tiles of one (request, KV head) and walks
// them as jobs (tile, K), (tile, V), ...
//
// Warp roles (576 threads), all hand-offs on mbarriers, no CTA-wide barrier in
// the steady state:
//   warp 16 (one lane) TMA producer: each job's 128 x 128 bf16 token tile, as two
//                      64-channel boxes with a 128-byte swizzle, into a 3-stage
//                      ring of 32 KiB shared-memory slots;
//   warp 17 (one lane) MMA issuer: 16 tcgen05.mma (M 128, N 128, K 16; R_hi then
//                      R_lo) per job into one of four 128-column accumulators
//                      (512 TMEM columns), committed to the slot's "empty" and
//                      the accumulator's "full" barrier;
//   warps 0-15         epilogue, one warpgroup per accumulator (jobs j = g mod 4
//                      for warpgroup g, so warpgroups 0 / 2 see K, 1 / 3 see V):
//                      warp w reads TMEM lanes 32 (w % 4) .. +31, one token per
//                      thread and all 128 columns, frees the accumulator, then
//                      quantises and packs whole page-block words, so no partial
//                      words are combined across warps. K and V run the same
//                      instructions up to the final stores.
// The four rotation images (R_K hi/lo, R_V hi/lo; bf16, K-major, 128-byte
// swizzle) stay in shared memory for the whole kernel. Every mbarrier wait is
// bounded: on expiry the kernel raises OSCAR_FLAG_TIMEOUT, the other roles stop
// at their next wait, copies and MMAs already issued are waited for (again with
// a limit) and tensor memory is released.
#include <cudaTypedefs.h>
#include <math.h>

#include <mutex>

#include "oscar_internal.cuh"
#include "tc_ptx.cuh"

namespace oscar {

constexpr int kPfThreads = 576;
constexpr int kProducerTid = 512;                        // lane 0 of warp 16
constexpr int kMmaTid = 544;                             // lane 0 of warp 17
constexpr int kTileM = 128;
constexpr int kImageBytes = kHeadDim * kHeadDim * 2;     // one bf16 128 x 128 operand: 32 KiB
constexpr int kAtomBytes = kTileM * 128;                 // 64 bf16 columns of 128 rows: 16 KiB
constexpr int kStages = 3;                                // token-tile slots
constexpr int kAccBufs = 4;                               // 128-column accumulators
constexpr int kPfSmemImages = 4 * kImageBytes;            // R_K hi, R_K lo, R_V hi, R_V lo
constexpr int kPfSmemStages = kStages * kImageBytes;
constexpr int kPfSmemBars = (2 * (kStages + kAccBufs) + 1) * 8 + 16;
constexpr int kPfSmem = 1024 + kPfSmemImages + kPfSmemStages + kPfSmemBars;
constexpr uint32_t kTmemCols = kAccBufs * kHeadDim;       // 512
// ---- PTX wrappers ------------------------------------------------------------
__device__ __forceinline__ void cp16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(smem)), "l"(gmem));
}
__device__ __forceinline__ void cp_commit_pf() { asm volatile("cp.async.commit_group;\n" ::); }
__device__ __forceinline__ void cp_wait_all_pf() { asm volatile("cp.async.wait_group 0;\n" ::); }

// one 64-channel x 128-token box of a 4-D tensor map into shared memory,
// completing on an mbarrier; the input is read once, so it is marked for early
// eviction from L2
__device__ __forceinline__ void tma_load_box(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2, int c3,
                                             uint32_t mbar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(mbar), "l"(policy)
      : "memory");
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
// ---- quantiser -----------------------------------------------------------------
// The code of a value is clamp(rint(fp32(fp32(xc - zf) * fp32(1 / sf))), 0, 3) on
// the clipped value xc (rint: nearest, ties to even). Adding 1.5 * 2^23 rounds a
// float in (-2^22, 2^22) to the nearest integer with ties to even and leaves
// that integer in the low mantissa bits, so the code is carried as the float
// kMagic + code. Every step is monotone in x, so clipping x and clamping to
// [0, 3] together equal clamping the unclipped value's code to
// [code(min_c), code(max_c)], the codes of the group's clipped extremes; that
// is the only clamp applied per element.
//
// Packing: the bits of kMagic + code are kMagicBits + code, whose low 16 bits
// are the code itself (two's complement for the negative codes of values that
// the clamp will raise). Every code of a token goes to a 2-bit field of one of
// 16 half-words: channel ch = 16 si + rr to half-word 2 (rr % 8) + rr / 8 at bit
// 2 si (the V layout); a K word (b2, x) is the pair of half-words 4 b2 + x (low)
// and 4 b2 + 2 + x (high). The eight K words are accumulated in 32-bit
// registers; the clamped codes never carry into the next field.
constexpr float kMagic = 12582912.f;        // 1.5 * 2^23
constexpr uint32_t kMagicBits = 0x4B400000u; // its bit pattern

__device__ __forceinline__ void chunk_minmax(const uint32_t (&r)[32], float& mn, float& mx) {
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    mn = fminf(mn, __uint_as_float(r[i]));
    mx = fmaxf(mx, __uint_as_float(r[i]));
  }
}

// scale and zero of a group from the minimum and maximum of its rotated values
// (clipping is monotonic, so the clipped extremes are the clipped minimum and
// maximum), and the bounds the codes of the group's values are clamped to
struct GroupQ {
  __half s16, z16;
  float zf, rsf, lo, hi;
  uint32_t lo2, hi2;   // the codes of lo and hi in both 16-bit halves
  bool small;          // every value's code before the clamp fits a signed 16-bit half
};
__device__ __forceinline__ GroupQ group_params(float mn, float mx, float clip) {
  GroupQ q;
  const float mn_raw = mn, mx_raw = mx;
  mn = fminf(fmaxf(mn, -clip), clip);
  mx = fminf(fmaxf(mx, -clip), clip);
  q.s16 = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), 3.0f));
  q.z16 = __float2half_rn(mn);
  const float sf = __half2float(q.s16);
  q.zf = __half2float(q.z16);
  q.rsf = sf != 0.f ? __frcp_rn(sf) : 0.f;  // sf == 0: every code is 0
  q.lo = fminf(fmaxf(__fadd_rn(__fmul_rn(__fsub_rn(mn, q.zf), q.rsf), kMagic), kMagic), kMagic + 3.f);
  q.hi = fminf(fmaxf(__fadd_rn(__fmul_rn(__fsub_rn(mx, q.zf), q.rsf), kMagic), kMagic), kMagic + 3.f);
  q.lo2 = (__float_as_uint(q.lo) - kMagicBits) * 0x10001u;
  q.hi2 = (__float_as_uint(q.hi) - kMagicBits) * 0x10001u;
  // the unclipped extremes bound every value's scaled offset (all steps are monotone)
  const float umin = __fmul_rn(__fsub_rn(mn_raw, q.zf), q.rsf);
  const float umax = __fmul_rn(__fsub_rn(mx_raw, q.zf), q.rsf);
  q.small = umin > -16384.f && umax < 16384.f;
  return q;
}

// fp32(fp32(x - zf) * rsf) for two values at once: the packed fp32 pair
// instructions round every lane to nearest like the scalar ones. kMagic is
// added by the caller with a scalar add: a packed add right after the packed
// multiply may be contracted into one fused multiply-add (one rounding instead
// of two), which changes the code of a product that rounds to a tie.
__device__ __forceinline__ void scaled_pair(uint32_t x0, uint32_t x1, uint64_t zz, uint64_t rr, float& u0, float& u1) {
  asm("{\n .reg .b64 t;\n mov.b64 t, {%2, %3};\n sub.rn.f32x2 t, t, %4;\n mul.rn.f32x2 t, t, %5;\n"
      " mov.b64 {%0, %1}, t;\n}\n"
      : "=f"(u0), "=f"(u1)
      : "r"(x0), "r"(x1), "l"(zz), "l"(rr));
}
__device__ __forceinline__ uint64_t pair_of(float f) {
  const uint64_t u = __float_as_uint(f);
  return u | (u << 32);
}

// codes of the 32 channels 32 CH .. 32 CH + 31 into the packed K words.
// Channels 2 k and 2 k + 1 go to the low and high half of the same word at the
// same shift, so a pair of codes is packed into one register (the low 16 bits
// of kMagic + code are the code) and added at once. SMALL: the codes before the
// clamp fit signed 16-bit halves, so both are clamped with one pair of 16-bit
// SIMD min / max; otherwise each is clamped as a float first.
template <int CH, bool SMALL>
__device__ __forceinline__ void chunk_codes_t(const uint32_t (&r)[32], const GroupQ& q, uint32_t (&acc)[8]) {
  const uint64_t zz = pair_of(q.zf), rr = pair_of(q.rsf);
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    float u0, u1;
    scaled_pair(r[i], r[i + 1], zz, rr, u0, u1);
    float m0 = __fadd_rn(u0, kMagic), m1 = __fadd_rn(u1, kMagic);
    if (!SMALL) {
      m0 = fminf(fmaxf(m0, q.lo), q.hi);
      m1 = fminf(fmaxf(m1, q.lo), q.hi);
    }
    uint32_t pr = __byte_perm(__float_as_uint(m0), __float_as_uint(m1), 0x5410);
    if (SMALL) {
      asm("max.s16x2 %0, %0, %1;" : "+r"(pr) : "r"(q.lo2));
      asm("min.s16x2 %0, %0, %1;" : "+r"(pr) : "r"(q.hi2));
    }
    constexpr int kCh0 = 32 * CH;
    const int ch = kCh0 + i;                            // even, compile-time
    const int si = ch >> 4, rr4 = ch & 15;
    const int hw = 2 * (rr4 & 7) + (rr4 >> 3);         // half-word of the even channel
    const int word = 2 * (hw >> 2) + (hw & 1);
    acc[word] += pr << (2 * si);
  }
}
template <int CH>
__device__ __forceinline__ void chunk_codes(const uint32_t (&r)[32], const GroupQ& q, uint32_t (&acc)[8]) {
  if (__all_sync(0xffffffffu, q.small))
    chunk_codes_t<CH, true>(r, q, acc);
  else
    chunk_codes_t<CH, false>(r, q, acc);
}

// ---- epilogue: one token of one kind per thread ----------------------------------
// page id of a token's position: kNoPage when the position is not one this launch
// writes, -1 when it lies past the request's page-table row; token_block reports
// every id outside the pool and returns no block for it
constexpr int32_t kNoPage = INT32_MIN;
__device__ __forceinline__ int32_t token_page(const PrefillParams& p, int64_t pos, bool valid, int b) {
  if (!valid) return kNoPage;
  const int64_t pidx = pos / kPage;
  return pidx < p.pt_stride ? p.page_table[(int64_t)b * p.pt_stride + pidx] : -1;
}
__device__ __forceinline__ uint8_t* token_block(const PrefillParams& p, int32_t id, int h) {
  if (id >= 0 && id < p.num_pages) return p.pool + ((int64_t)id * p.num_kv_heads + h) * block_bytes(p.ngroups);
  if (id != kNoPage) atomicOr(p.err_flags, OSCAR_FLAG_BAD_PAGE_ID);
  return nullptr;
}

__device__ __forceinline__ void trace_group(const PrefillParams& p, const uint32_t (&r)[32], int64_t pos, bool valid,
                                            int h, int b, int kind, int gq) {
  if (valid && p.trace && pos < p.trace_positions) {
    float* tr = p.trace + ((((size_t)b * p.trace_positions + pos) * p.num_kv_heads + h) * 2 + kind) * kHeadDim;
#pragma unroll
    for (int i = 0; i < 32; ++i) tr[32 * gq + i] = __uint_as_float(r[i]);
  }
}

// words: the eight packed K words; sz[g]: scale (low half)
// and zero (high half) of group g; ng groups per token
__device__ __forceinline__ void store_token(uint8_t* blk, int kind, int64_t pos, const uint32_t (&words)[8],
                                            const uint32_t (&sz)[kGroups], int ng) {
  const int t = (int)(pos % kPage);
  const int a = t & 7, bb = (t & 7) >> 1, th = t & 1, tt = t >> 3;
  if (kind == 0) {
    // codes: words (b2, x) at 16 (4 a + b2) + 4 (2 tt + x)
#pragma unroll
    for (int b2 = 0; b2 < 4; ++b2)
      *reinterpret_cast<uint2*>(blk + 16 * (4 * a + b2) + 8 * tt) = make_uint2(words[2 * b2], words[2 * b2 + 1]);
#pragma unroll
    for (int g = 0; g < kGroups; ++g)
      if (g < ng) *reinterpret_cast<uint16_t*>(blk + kscale_off(ng, t, g)) = (uint16_t)sz[g];
    // the zeros of a token are contiguous
    if (ng == kGroups)
      *reinterpret_cast<uint2*>(blk + kzero_off(ng, t, 0)) =
          make_uint2(__byte_perm(sz[0], sz[1], 0x7632), __byte_perm(sz[2], sz[3], 0x7632));
    else
      *reinterpret_cast<uint32_t*>(blk + kzero_off(ng, t, 0)) = __byte_perm(sz[0], sz[1], 0x7632);
  } else {
    // half-word i of the V layout is half (i / 2) % 2 of word 2 (i / 4) + i % 2
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int a2 = i >> 1, x = i & 1;
      const uint32_t w = words[2 * (i >> 2) + (i & 1)];
      *reinterpret_cast<uint16_t*>(blk + 512 + 16 * (4 * a2 + bb) + 4 * (2 * tt + x) + 2 * th) =
          (uint16_t)(((i >> 1) & 1) ? (w >> 16) : w);
    }
#pragma unroll
    for (int g = 0; g < kGroups; ++g) {
      if (g < ng) {
        *reinterpret_cast<uint16_t*>(blk + vscale_off(ng, t, g)) = (uint16_t)sz[g];
        *reinterpret_cast<uint16_t*>(blk + vzero_off(ng, t, g)) = (uint16_t)(sz[g] >> 16);
      }
    }
  }
}

// NG: quantisation groups per token (p.ngroups), 4 (groups of 32) or 2 (of 64)
template <int NG>
__global__ void __launch_bounds__(kPfThreads, 1) oscar_prefill_append_kernel(const __grid_constant__ PrefillParams p) {
  extern __shared__ uint8_t dsm_raw[];
  // 1024-byte alignment for the swizzled operands
  uint8_t* dsm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t* img = dsm;                                      // 4 rotation images
  uint8_t* slot = img + kPfSmemImages;                     // kStages token tiles
  uint64_t* bars = reinterpret_cast<uint64_t*>(slot + kPfSmemStages);
  uint64_t* full = bars;                                   // [kStages] tile landed (TMA bytes)
  uint64_t* empty = full + kStages;                        // [kStages] tile consumed (MMA commit)
  uint64_t* accf = empty + kStages;                        // [kAccBufs] accumulator ready (MMA commit)
  uint64_t* acce = accf + kAccBufs;                        // [kAccBufs] accumulator read (4 warps)
  uint64_t* drainb = acce + kAccBufs;                      // teardown after an abort
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drainb + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  __shared__ oscar_seq_state s_st;
  __shared__ int s_loads, s_mmas;                          // jobs issued by the producer / MMA issuer

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int S = p.sink, W = p.recent;

  // rotation images are constant: stage them before waiting for earlier kernels
  {
    const uint8_t* src = p.images + (size_t)h * kPfSmemImages;
    for (int i = tid; i < kPfSmemImages / 16; i += kPfThreads) cp16(img + 16 * i, src + 16 * i);
    cp_commit_pf();
  }
  if (tid == kProducerTid) {
    asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&p.tmap_k)) : "memory");
    asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&p.tmap_v)) : "memory");
  }
  pdl_wait();
  pdl_trigger();

  if (tid == 0) s_st = p.state[b];
  if (warp == kMmaTid / 32) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::);
  }
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(smem_u32(&full[i]), 1);
      mbar_init(smem_u32(&empty[i]), 1);
    }
    for (int i = 0; i < kAccBufs; ++i) {
      mbar_init(smem_u32(&accf[i]), 1);
      mbar_init(smem_u32(&acce[i]), 4);
    }
    mbar_init(smem_u32(drainb), 1);
    *abort_flag = 0;
    s_loads = 0;
    s_mmas = 0;
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
  auto tile_start = [&](int j) { return P0 + (int64_t)(c + (j >> 1) * (int)gridDim.x) * kTileM; };

  if (warp == kProducerTid / 32) {
    // ---- TMA producer --------------------------------------------------------
    if (lane == 0) {
      uint64_t policy;
      asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(policy));
      for (int j = 0; j < njobs; ++j) {
        const int s = j % kStages;
        if (j >= kStages && !mbar_wait(smem_u32(&empty[s]), (uint32_t)((j / kStages - 1) & 1), abort_flag)) {
          *abort_flag = 1;
          break;
        }
        const CUtensorMap* map = (j & 1) ? &p.tmap_v : &p.tmap_k;
        const int tok = (int)(tile_start(j) - L);   // row of the tile's first position in the input
        const uint32_t dst = smem_u32(slot + (size_t)s * kImageBytes);
        const uint32_t fb = smem_u32(&full[s]);
        mbar_expect_tx(fb, (uint32_t)kImageBytes);
        tma_load_box(dst, map, 0, h, tok, b, fb, policy);
        tma_load_box(dst + kAtomBytes, map, 64, h, tok, b, fb, policy);
        s_loads = j + 1;
      }
    }
  } else if (warp == kMmaTid / 32) {
    // ---- MMA issuer ----------------------------------------------------------
    if (lane == 0) {
      for (int j = 0; j < njobs; ++j) {
        const int s = j % kStages, a = j % kAccBufs;
        if (!mbar_wait(smem_u32(&full[s]), (uint32_t)((j / kStages) & 1), abort_flag) ||
            (j >= kAccBufs &&
             !mbar_wait(smem_u32(&acce[a]), (uint32_t)((j / kAccBufs - 1) & 1), abort_flag))) {
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const int kind = j & 1;
        const uint32_t a_base = smem_u32(slot + (size_t)s * kImageBytes);
        const uint32_t hi_base = smem_u32(img + (size_t)(2 * kind) * kImageBytes);
        const uint32_t lo_base = smem_u32(img + (size_t)(2 * kind + 1) * kImageBytes);
        const uint32_t d_tmem = tmem + (uint32_t)(a * kHeadDim);
#pragma unroll
        for (int term = 0; term < 2; ++term) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (uint32_t)((kk >> 2) * kAtomBytes + (kk & 3) * 32);
            umma_bf16(d_tmem, sw128_desc(a_base + off), sw128_desc((term ? lo_base : hi_base) + off),
                      (term | kk) ? 1u : 0u);
          }
        }
        umma_commit(smem_u32(&empty[s]));
        umma_commit(smem_u32(&accf[a]));
        s_mmas = j + 1;
      }
    }
  } else {
    // ---- epilogue: warpgroup g takes the jobs j = g (mod 4), accumulator g -------
    const int g = warp >> 2, kind = g & 1;
    const int row = 32 * (warp & 3) + lane;
    const float clip = (kind ? p.clip_V : p.clip_K)[h];
    const uint32_t taddr = tmem + (uint32_t)(g * kHeadDim) + ((uint32_t)(32 * (warp & 3)) << 16);
    for (int j = g; j < njobs; j += kAccBufs) {
      const bool ready = mbar_wait(smem_u32(&accf[g]), (uint32_t)((j / kAccBufs) & 1), abort_flag);
      if (!__all_sync(0xffffffffu, ready)) {
        if (lane == 0) *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const int64_t pos = tile_start(j) + row;
      const bool valid = pos >= d0 && pos < d1;
      // the page id of this token's position is read now and used after the
      // arithmetic, so that its latency is hidden
      const int32_t page = token_page(p, pos, valid, b);
      uint32_t acc[8];   // packed K words
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0u;
      uint32_t sz[kGroups];   // scale (low half) and zero (high half) of each group
      uint32_t r[32];
      auto load_chunk = [&](int ch) {
        tmem_ld32(taddr + 32 * ch, r);
        asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
        tmem_regs_ready(r);
      };
      auto release = [&]() {
        // every column this thread needs is in registers: the accumulator may be overwritten
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&acce[g]));
      };
      if constexpr (NG == kGroups) {
        // groups of 32 channels: one TMEM chunk each
#pragma unroll
        for (int gq = 0; gq < kGroups; ++gq) {
          load_chunk(gq);
          if (gq == kGroups - 1) release();
          trace_group(p, r, pos, valid, h, b, kind, gq);
          float mn = __uint_as_float(r[0]), mx = mn;
          chunk_minmax(r, mn, mx);
          const GroupQ q = group_params(mn, mx, clip);
          if (gq == 0) chunk_codes<0>(r, q, acc);
          if (gq == 1) chunk_codes<1>(r, q, acc);
          if (gq == 2) chunk_codes<2>(r, q, acc);
          if (gq == 3) chunk_codes<3>(r, q, acc);
          sz[gq] = (uint32_t)__half_as_ushort(q.s16) | ((uint32_t)__half_as_ushort(q.z16) << 16);
        }
      } else {
        // groups of 64 channels: the extremes of both chunks first, then the codes
        // of the second chunk (in registers) and of the first (read again)
#pragma unroll
        for (int gq = 0; gq < 2; ++gq) {
          load_chunk(2 * gq);
          trace_group(p, r, pos, valid, h, b, kind, 2 * gq);
          float mn = __uint_as_float(r[0]), mx = mn;
          chunk_minmax(r, mn, mx);
          load_chunk(2 * gq + 1);
          trace_group(p, r, pos, valid, h, b, kind, 2 * gq + 1);
          chunk_minmax(r, mn, mx);
          const GroupQ q = group_params(mn, mx, clip);
          if (gq == 0) chunk_codes<1>(r, q, acc);
          if (gq == 1) chunk_codes<3>(r, q, acc);
          load_chunk(2 * gq);
          if (gq == 1) release();
          if (gq == 0) chunk_codes<0>(r, q, acc);
          if (gq == 1) chunk_codes<2>(r, q, acc);
          sz[gq] = (uint32_t)__half_as_ushort(q.s16) | ((uint32_t)__half_as_ushort(q.z16) << 16);
        }
        sz[2] = sz[3] = 0u;
      }
      uint8_t* blk = token_block(p, page, h);
      if (blk) store_token(blk, kind, pos, acc, sz, NG);
    }
  }

  // ---- teardown ------------------------------------------------------------------
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    if (tid == 0) atomicOr(p.err_flags, OSCAR_FLAG_TIMEOUT);
    if (tid == kProducerTid) {
      // tiles still landing in shared memory
      for (int j = s_mmas; j < s_loads; ++j) mbar_drain(smem_u32(&full[j % kStages]), (uint32_t)((j / kStages) & 1));
    }
    if (tid == kMmaTid) {
      // MMAs still writing tensor memory: a commit tracks every MMA issued before it
      umma_commit(smem_u32(drainb));
      mbar_drain(smem_u32(drainb), 0u);
    }
    __syncthreads();
  }
  if (warp == kMmaTid / 32) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(kTmemCols));
  }
}

// ---- host side -------------------------------------------------------------------
namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

// k or v [batch][n_new][Hkv][128] bf16 as a 4-D map (channel, head, token, request)
// with 64 x 1 x 128 x 1 boxes: each box is one 16 KiB swizzled operand atom
bool encode_map(CUtensorMap* map, const void* base, int hkv, int n_new, int batch) {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode) return false;
  const cuuint64_t dims[4] = {(cuuint64_t)kHeadDim, (cuuint64_t)hkv, (cuuint64_t)n_new, (cuuint64_t)batch};
  const cuuint64_t row = (cuuint64_t)kHeadDim * 2;
  const cuuint64_t strides[3] = {row, row * hkv, row * hkv * (cuuint64_t)n_new};
  const cuuint32_t box[4] = {64, 1, (cuuint32_t)kTileM, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool prefill_supported(const void* k, const void* v) {
  return ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) & 15) == 0;
}

cudaError_t launch_prefill_append(const PrefillParams& p_in, int ctas_per_head, cudaStream_t s,
                                  cudaEvent_t ev_before, cudaEvent_t ev_after) {
  static PerDeviceOnce attrs;
  const cudaError_t ea = once_for_current_device(attrs, [] {
    cudaError_t e = cudaFuncSetAttribute(oscar_prefill_append_kernel<kGroups>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kPfSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(oscar_prefill_append_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, kPfSmem);
    return e;
  });
  if (ea != cudaSuccess) return ea;
  if (p_in.ngroups != kGroups && p_in.ngroups != 2) return cudaErrorInvalidValue;
  PrefillParams p = p_in;
  if (!encode_map(&p.tmap_k, p.k, p.num_kv_heads, p.n_new, p.batch) ||
      !encode_map(&p.tmap_v, p.v, p.num_kv_heads, p.n_new, p.batch))
    return cudaErrorInvalidValue;
  if (ev_before && cudaEventRecord(ev_before, s) != cudaSuccess) return cudaGetLastError();
  cudaError_t e = launch_pdl(p.ngroups == kGroups ? oscar_prefill_append_kernel<kGroups> : oscar_prefill_append_kernel<2>,
                             dim3(ctas_per_head, p.num_kv_heads, p.batch), dim3(kPfThreads), kPfSmem, s, p);
  if (e != cudaSuccess) return e;
  if (ev_after && (e = cudaEventRecord(ev_after, s)) != cudaSuccess) return e;
  return cudaGetLastError();
}

int prefill_image_bytes() { return kPfSmemImages; }

}  // namespace oscar
