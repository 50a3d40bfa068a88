// Quantisation of one token's rotated K and V into its page block: the steps the
// per-token append kernel and the one-token append of a decode step share, so
// that both write the same bytes for the same rotated values.
//
// Source: "Juntos, AI Open-Sources OSCAR ..." (7minutos.es), section "El
// sistema de servicio" (clip to the calibrated threshold, asymmetric per-token
// INT2 groups with an fp16 scale and zero); the page block layout is the one in
// include/oscar.h.
#pragma once

#include "oscar_internal.cuh"

namespace oscar {

// scale and zero of a group with clipped extremes mn <= mx:
// s = fp16((mx - mn) / 3), z = fp16(mn)
__device__ __forceinline__ void group_scale_zero(float mn, float mx, __half& s16, __half& z16) {
  s16 = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), 3.0f));
  z16 = __float2half_rn(mn);
}

// code of a clipped value x in a group with scale sf and zero zf (fp16 values):
// clamp(rint((x - z) * fp32(1 / s)), 0, 3), 0 when s == 0
__device__ __forceinline__ int group_code(float x, float sf, float zf) {
  if (sf == 0.f) return 0;
  float u = rintf(__fmul_rn(__fsub_rn(x, zf), __frcp_rn(sf)));
  u = fminf(fmaxf(u, 0.f), 3.f);
  return (int)u;
}

// The share of thread `role` in storing token t (position mod 16) of a page
// block with ng groups per token: roles 0-7 write the 8 words of K codes, 32-47
// the 16 half-words of V codes, 64-71 the K and V scales and zeros; other roles
// write nothing. codes[kind][channel] (kind 0 = K, 1 = V) and
// meta[kind][group] = {scale, zero} hold the token's quantisation.
__device__ __forceinline__ void store_token_block(uint8_t* blk, int t, int role, int ng,
                                                  const uint8_t (*codes)[kHeadDim],
                                                  const __half (*meta)[kGroups][2]) {
  if (role < 8) {
    // K word (bb, x): channels 16 i + 2 bb + 8 x (low half-word) and the next
    // channel (high half-word), slot i at bits 2 i
    const int bb = role >> 1, x = role & 1;
    uint32_t w = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int ch = 16 * i + 2 * bb + 8 * x;
      w |= (uint32_t)codes[0][ch] << (2 * i);
      w |= (uint32_t)codes[0][ch + 1] << (16 + 2 * i);
    }
    const int a = t & 7, th = t >> 3;
    *reinterpret_cast<uint32_t*>(blk + 16 * (4 * a + bb) + 4 * (2 * th + x)) = w;
  } else if (role >= 32 && role < 48) {
    // V half-word (a, x): channels 16 i + a + 8 x, slot i at bits 2 i
    const int u = role - 32, a = u >> 1, x = u & 1;
    uint32_t hw = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) hw |= (uint32_t)codes[1][16 * i + a + 8 * x] << (2 * i);
    const int tt = t >> 3, bb = (t & 7) >> 1, hi = t & 1;
    *reinterpret_cast<uint16_t*>(blk + 512 + 16 * (4 * a + bb) + 4 * (2 * tt + x) + 2 * hi) = (uint16_t)hw;
  } else if (role >= 64 && role < 72) {
    const int u = role - 64, kind = u >> 2, gq = u & 3;
    if (gq < ng) {
      if (kind == 0) {
        *reinterpret_cast<__half*>(blk + kscale_off(ng, t, gq)) = meta[0][gq][0];
        *reinterpret_cast<__half*>(blk + kzero_off(ng, t, gq)) = meta[0][gq][1];
      } else {
        *reinterpret_cast<__half*>(blk + vscale_off(ng, t, gq)) = meta[1][gq][0];
        *reinterpret_cast<__half*>(blk + vzero_off(ng, t, gq)) = meta[1][gq][1];
      }
    }
  }
}

}  // namespace oscar
