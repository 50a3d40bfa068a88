// Write path of the OSCAR INT2 cache: rotate, clip, group-quantise, pack.
//
// One CTA of 512 threads handles a run of consecutive new tokens of one request
// and one KV head (K and V together), one token after another. Depending on a
// token's position it either copies the token into the BF16 sink, quantises it
// straight into its INT2 page, or places it in the BF16 recent ring after
// quantising the ring entry it evicts. Sources: "Juntos, AI Open-Sources OSCAR ..." (7minutos.es), section
// "El sistema de servicio" (write path: rotate, clip to the calibrated
// threshold, asymmetric per-token INT2 groups; sink and recent tokens in BF16);
// "OSCAR: Offline Spectral Covariance-Aware Rotation ..." (gist.science, it),
// Riepilogo Tecnico 2.2 B (mixed-precision paged layout).
#include "oscar_internal.cuh"
#include "token_quant.cuh"

namespace oscar {

constexpr int kThreads = 512;

__device__ __forceinline__ float warp_min(float x) {
#pragma unroll
  for (int o = 16; o; o >>= 1) x = fminf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const uint32_t sa = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(sa), "l"(gmem));
}

// page block for page-table entry `id` (nullptr and a flag when out of range)
__device__ __forceinline__ uint8_t* block_of(const AppendParams& p, int32_t id, int h) {
  if (id < 0 || id >= p.num_pages) {
    atomicOr(p.err_flags, OSCAR_FLAG_BAD_PAGE_ID);
    return nullptr;
  }
  return p.pool + ((int64_t)id * p.num_kv_heads + h) * block_bytes(p.ngroups);
}

constexpr int kMaxTokensPerCta = 16;

// whether a tail_only CTA with virtual tokens [j0, j1) quantises anything: a
// ring token at position q >= E2 evicts the entry at q - W ((q - L) / W + 1),
// which goes to INT2 when it lies in [max(E, S), E2) (the token loop's rule)
__device__ __forceinline__ bool any_quantised(const AppendParams& p, int j0, int j1, int L, int E, int64_t E2) {
  const int S = p.sink, W = p.recent;
  for (int jv = j0; jv < j1; ++jv) {
    const int j = jv < S ? jv : p.n_new - W + (jv - S);
    const int64_t q = (int64_t)L + j;
    if (q >= E2) {
      const int64_t pe = q - (int64_t)W * ((q - L) / W + 1);
      if (pe >= E && pe < E2 && pe >= S) return true;
    }
  }
  return false;
}
constexpr int kAppendSmem = 2 * kHeadDim * kHeadDim * 4;  // R_K[h] and R_V[h]

__global__ void __launch_bounds__(kThreads, 1)
oscar_quant_append_kernel(AppendParams p) {
  extern __shared__ __align__(16) uint8_t dsm[];
  float* Rs = reinterpret_cast<float*>(dsm);  // [2][128][128]: R_K[h], R_V[h]
  const int tid = threadIdx.x;
  const int h = blockIdx.y, b = blockIdx.z;
  // token indices of this CTA: all new tokens, or with tail_only only the first
  // `sink` and the last `recent` of them (virtual indices, see AppendParams)
  const int nvirt = p.tail_only ? p.sink + p.recent : p.n_new;
  const int j0 = blockIdx.x * p.tokens_per_cta;
  const int j1 = min(j0 + p.tokens_per_cta, nvirt);
  const int S = p.sink, W = p.recent;
  const int Hkv = p.num_kv_heads;

  __shared__ oscar_seq_state s_st;
  __shared__ int s_page;
  __shared__ __align__(16) __nv_bfloat16 s_in[2][kHeadDim];   // K, V of the CTA's first token
  __shared__ float xs[2][kHeadDim];            // token being quantised, K and V
  __shared__ float red[2][2][kHeadDim];        // partial dot products
  __shared__ uint8_t codes[2][kHeadDim];
  __shared__ __half meta[2][kGroups][2];
  __shared__ float wmm[2][4][2];  // per kind and warp: min, max of its 32 clipped channels

  // copies of 16 bytes need 16-byte aligned inputs (otherwise read in place)
  const bool staged = j0 < j1 && ((reinterpret_cast<uintptr_t>(p.k) | reinterpret_cast<uintptr_t>(p.v)) & 15) == 0;
  // the rotations are constant: stage them before waiting for earlier kernels.
  // A launch for the sink / ring tokens of a long append (tail_only) quantises
  // only ring entries that the new tokens evict, usually none: it stages them
  // after reading the state, and only when it needs them.
  auto stage_rotations = [&]() {
    const float* rk = p.R_K + (size_t)h * kHeadDim * kHeadDim;
    const float* rv = p.R_V + (size_t)h * kHeadDim * kHeadDim;
    constexpr int n4 = kHeadDim * kHeadDim / 4;
    for (int i = tid; i < n4; i += kThreads) {
      cp_async16(Rs + 4 * i, rk + 4 * i);
      if (!p.fold_rv) cp_async16(Rs + kHeadDim * kHeadDim + 4 * i, rv + 4 * i);
    }
  };
  {
    if (!p.tail_only) stage_rotations();
    // the CTA's first new token: the caller's input, which no kernel of this
    // library writes, so it is read before waiting for earlier kernels
    if (staged && tid < 2 * (kHeadDim / 8)) {
      const int jf = !p.tail_only ? j0 : (j0 < S ? j0 : p.n_new - W + (j0 - S));
      const size_t off = (((size_t)b * p.n_new + jf) * Hkv + h) * kHeadDim;
      const int kind = tid >> 4, u = tid & 15;
      cp_async16(&s_in[kind][8 * u], (kind ? p.v : p.k) + off + 8 * u);
    }
    asm volatile("cp.async.commit_group;\n" ::);
  }
  // level-2 prefetches (they return no data): the request's BF16 window rows of
  // this head, where the entry a token evicts is read, and the request's page
  // table row (host-written). The window row index is set by the host; kernels
  // only ever rewrite it unchanged.
  if (blockIdx.x == 0) {
    const int wr = p.state[b].window_row;
    if (wr >= 0 && wr < p.max_batch) {
      const size_t slots = (size_t)(S + W);
      const char* wbase = reinterpret_cast<const char*>(p.window + ((size_t)wr * Hkv + h) * 2 * slots * kHeadDim);
      const size_t wbytes = 2 * slots * kHeadDim * sizeof(__nv_bfloat16);
      for (size_t off = (size_t)tid * 128; off < wbytes; off += (size_t)kThreads * 128)
        asm volatile("prefetch.global.L2 [%0];\n" ::"l"(wbase + off));
    }
    if (h == 0) {
      const char* pt = reinterpret_cast<const char*>(p.page_table + (size_t)b * p.pt_stride);
      const size_t pbytes = (size_t)p.pt_stride * sizeof(int32_t);
      for (size_t off = (size_t)tid * 128; off < pbytes; off += (size_t)kThreads * 128)
        asm volatile("prefetch.global.L2 [%0];\n" ::"l"(pt + off));
    }
  }
  // dependents may start now: before their own wait they touch only constant
  // data and caller inputs
  pdl_trigger();
  pdl_wait();
  // ticket: taken once the state is read; its value is needed only at the end,
  // where the CTA holding the last one publishes the new states
  unsigned ticket = 0u;
  if (tid == 0) {
    s_st = p.state[b];
    asm volatile("fence.acq_rel.gpu;\n" ::: "memory");   // the state read comes before the ticket
    ticket = atomicAdd(p.counter, 1u);
  }
  asm volatile("cp.async.wait_group 0;\n" ::);  // rotations staged, visible after the barrier
  __syncthreads();
  const oscar_seq_state st = s_st;
  const int L = st.seq_len, E = st.int2_end;
  const bool ok = state_ok(st, S, W, p.max_batch);
  if (!ok && tid == 0 && blockIdx.x == 0 && h == 0) atomicOr(p.err_flags, OSCAR_FLAG_BAD_STATE);

  if (ok) {
    int64_t E2 = (int64_t)L + p.n_new - W;
    if (E2 < E) E2 = E;
    if (E2 < S) E2 = S;
    const size_t slots = (size_t)(S + W);
    const size_t wrow = (size_t)st.window_row;
    __nv_bfloat16* win_k = p.window + ((wrow * Hkv + h) * 2 + 0) * slots * kHeadDim;
    __nv_bfloat16* win_v = p.window + ((wrow * Hkv + h) * 2 + 1) * slots * kHeadDim;
    if (p.tail_only) {
      // the ring entries this CTA's ring tokens evict that go to INT2 (see the
      // token loop below); stage the rotations if there are any
      const bool need = any_quantised(p, j0, j1, L, E, E2);
      if (need) {
        stage_rotations();
        asm volatile("cp.async.commit_group;\n" ::);
        asm volatile("cp.async.wait_group 0;\n" ::);
        __syncthreads();
      }
    }
    // Without entries to quantise the sink and ring tokens are plain copies:
    // all of the CTA's tokens at once, 16 bytes per thread (a long append's
    // inputs are 16-byte aligned), instead of one token after another.
    const bool copies_only = p.tail_only && !any_quantised(p, j0, j1, L, E, E2);
    if (copies_only) {
      for (int idx = tid; idx < (j1 - j0) * 32; idx += kThreads) {
        const int jv = j0 + (idx >> 5), kind = (idx >> 4) & 1, ch = idx & 15;
        const int j = jv < S ? jv : p.n_new - W + (jv - S);
        const int64_t q = (int64_t)L + j;
        int64_t slot = -1;
        if (q < S) slot = q;
        else if (q >= E2) slot = S + q % W;
        if (slot >= 0) {
          const size_t in_off = (((size_t)b * p.n_new + j) * Hkv + h) * kHeadDim + 8 * ch;
          const uint4 x = *reinterpret_cast<const uint4*>((kind ? p.v : p.k) + in_off);
          *reinterpret_cast<uint4*>((kind ? win_v : win_k) + (size_t)slot * kHeadDim + 8 * ch) = x;
        }
      }
    }


    for (int jv = copies_only ? j1 : j0; jv < j1; ++jv) {
      const int j = !p.tail_only ? jv : (jv < S ? jv : p.n_new - W + (jv - S));
      const int64_t q = (int64_t)L + j;
      // with tail_only the tokens going straight to INT2 belong to the prefill kernel
      if (p.tail_only && q >= S && q < E2) continue;
      const size_t in_off = (((size_t)b * p.n_new + j) * Hkv + h) * kHeadDim;
      const __nv_bfloat16* in_k = staged && jv == j0 ? s_in[0] : p.k + in_off;
      const __nv_bfloat16* in_v = staged && jv == j0 ? s_in[1] : p.v + in_off;
      // what this token quantises: -1 none, else the position, and where it comes from
      int64_t qpos = -1;
      const __nv_bfloat16* src_k = nullptr;
      const __nv_bfloat16* src_v = nullptr;
      int64_t ring_slot_new = -1;
      if (q < S) {
        // sink token: BF16 copy
        if (tid < kHeadDim) {
          win_k[(size_t)q * kHeadDim + tid] = in_k[tid];
          win_v[(size_t)q * kHeadDim + tid] = in_v[tid];
        }
      } else if (q < E2) {
        qpos = q;
        src_k = in_k;
        src_v = in_v;
      } else {
        // ring occupant; the entry at its slot may have to be quantised first
        const int64_t pe = q - (int64_t)W * ((q - L) / W + 1);
        if (pe >= E && pe < E2 && pe >= S) {
          qpos = pe;
          const size_t sl = (size_t)(S + pe % W) * kHeadDim;
          src_k = win_k + sl;
          src_v = win_v + sl;
        }
        ring_slot_new = S + q % W;
      }

      if (qpos >= 0) {
        if (tid == 2 * kHeadDim) {
          // page-table entry of the quantised position, fetched while the token loads
          const int64_t pidx = qpos / kPage;
          s_page = pidx < p.pt_stride ? p.page_table[(int64_t)b * p.pt_stride + pidx] : -1;
        }
        if (tid < 2 * kHeadDim) {
          const int kind = tid >> 7, c = tid & 127;
          xs[kind][c] = __bfloat162float((kind ? src_v : src_k)[c]);
        }
      }
      __syncthreads();  // ring entry read (and rotations staged) before the ring write

      if (ring_slot_new >= 0 && tid < 2 * kHeadDim) {
        const int kind = tid >> 7, c = tid & 127;
        __nv_bfloat16* dst = (kind ? win_v : win_k) + (size_t)ring_slot_new * kHeadDim;
        dst[c] = (kind ? in_v : in_k)[c];
      }

      if (qpos >= 0) {
        // rotation x @ R: thread (kind, half, c) sums 64 terms, the halves added in order
        {
          const int kind = tid >> 8, half = (tid >> 7) & 1, c = tid & 127;
          const float* R = Rs + kind * kHeadDim * kHeadDim + c;
          const int i0 = half * 64;
          float acc = 0.f;
          if (kind == 1 && p.fold_rv) {
            acc = half ? 0.f : xs[1][c];  // identity: V is already in the R_V basis
          } else {
#pragma unroll 16
            for (int i = 0; i < 64; ++i) acc = fmaf(xs[kind][i0 + i], R[(i0 + i) * kHeadDim], acc);
          }
          red[kind][half][c] = acc;
        }
        __syncthreads();
        // thread (kind, c) < 128 per kind: clip, then the group minimum and maximum
        // (a group of 32 channels is one warp; a group of 64 two warps, combined
        // through shared memory)
        const bool qthread = (tid & 255) < kHeadDim;
        const int kind = tid >> 8, c = tid & 127;
        float x = 0.f, mn = 0.f, mx = 0.f;
        if (qthread) {
          const float x_rot = red[kind][0][c] + red[kind][1][c];
          if (p.trace && qpos < p.trace_positions) {
            p.trace[((((size_t)b * p.trace_positions + qpos) * Hkv + h) * 2 + kind) * kHeadDim + c] = x_rot;
          }
          const float clip = (kind ? p.clip_V : p.clip_K)[h];
          x = fminf(fmaxf(x_rot, -clip), clip);
          mn = warp_min(x);
          mx = warp_max(x);
          if (p.ngroups != kGroups && (c & 31) == 0) {
            wmm[kind][c >> 5][0] = mn;
            wmm[kind][c >> 5][1] = mx;
          }
        }
        if (p.ngroups != kGroups) {
          __syncthreads();
          if (qthread) {
            const int w = (c >> 5) ^ 1;  // the other warp of a 64-channel group
            mn = fminf(mn, wmm[kind][w][0]);
            mx = fmaxf(mx, wmm[kind][w][1]);
          }
        }
        if (qthread) {
          __half s16, z16;
          group_scale_zero(mn, mx, s16, z16);
          codes[kind][c] = (uint8_t)group_code(x, __half2float(s16), __half2float(z16));
          const int gsz = kHeadDim / p.ngroups;
          if ((c & (gsz - 1)) == 0) {
            meta[kind][c / gsz][0] = s16;
            meta[kind][c / gsz][1] = z16;
          }
        }
        __syncthreads();
        uint8_t* blk = tid < 72 ? block_of(p, s_page, h) : nullptr;
        if (blk) store_token_block(blk, (int)(qpos % kPage), tid, p.ngroups, codes, meta);
        __syncthreads();  // codes / meta / xs reused by the next token
      }
    }
  }

  // the CTA that took the last ticket publishes the new state of every request
  if (tid == 0 && ticket == gridDim.x * gridDim.y * gridDim.z - 1u) {
    // every other CTA read its state before taking its ticket; the writes below
    // come after all of those reads (kernel completion publishes them)
    asm volatile("fence.acq_rel.gpu;\n" ::: "memory");
    for (int bb = 0; bb < p.batch; ++bb) {
      oscar_seq_state sb = bb == b ? s_st : p.state[bb];   // this CTA's own request is at hand
      if (!state_ok(sb, S, W, p.max_batch)) continue;
      const int64_t nl = (int64_t)sb.seq_len + p.n_new;
      int64_t ne = nl - W;
      if (ne < sb.int2_end) ne = sb.int2_end;
      if (ne < S) ne = S;
      sb.seq_len = (int32_t)nl;
      sb.int2_end = (int32_t)ne;
      p.state[bb] = sb;
    }
    *p.counter = 0u;
  }
}

cudaError_t launch_quant_append(const AppendParams& p, cudaStream_t s, cudaEvent_t ev_before,
                                cudaEvent_t ev_after) {
  static PerDeviceOnce attrs;
  static PerDeviceValue sm_count;
  const cudaError_t ea = once_for_current_device(attrs, [] {
    return cudaFuncSetAttribute(oscar_quant_append_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kAppendSmem);
  });
  if (ea != cudaSuccess) return ea;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaGetLastError();
  const int num_sms = sm_count.get(dev, [dev] {
    int n = 0;
    return cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0 ? n : 1;
  });
  // tokens are walked one after another inside a CTA: spread them over one wave
  // of CTAs (one per SM), at most kMaxTokensPerCta each
  AppendParams q = p;
  const int64_t nvirt = p.tail_only ? p.sink + p.recent : p.n_new;
  const int64_t units = (int64_t)p.num_kv_heads * p.batch;
  int64_t tpc = (nvirt * units + num_sms - 1) / num_sms;
  if (tpc < 1) tpc = 1;
  if (tpc > kMaxTokensPerCta) tpc = kMaxTokensPerCta;
  q.tokens_per_cta = (int32_t)tpc;
  dim3 grid((unsigned)((nvirt + tpc - 1) / tpc), (unsigned)p.num_kv_heads, (unsigned)p.batch);
  if (ev_before && cudaEventRecord(ev_before, s) != cudaSuccess) return cudaGetLastError();
  cudaError_t e = launch_pdl(oscar_quant_append_kernel, grid, dim3(kThreads), kAppendSmem, s, q);
  if (e != cudaSuccess) return e;
  if (ev_after && (e = cudaEventRecord(ev_after, s)) != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace oscar
