"""Shared set-up for the GPU parity tests: one attention layer driven through
the C ABI next to the CPU oracle, both fed from the same seeded inputs."""

from __future__ import annotations

import numpy as np
import torch

import oracle
from bit_rotated_kv_oscar_gb300 import abi
from bit_rotated_kv_oscar_gb300.cache import PagedCache
from synth import draw_kv, draw_page_pool, draw_queries

D = 128
# attention-output tolerance against the float64 oracle
REL_L2 = 2e-3
MAX_ABS = 1e-2
# rotated values: |gpu - oracle| <= ROT_REL * max_j |oracle_j| per token-head vector
ROT_REL = 1e-5


def rel_l2(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def _fp16_interval(lo, hi):
    """fp16 values (RNE) reachable by rounding any real in [lo, hi] (as the set of the two ends)."""
    return np.float16(lo), np.float16(hi)


def resolve_group_ties(x64, clip, eps, g_codes, g_s16, g_z16, group=32):
    """Validate GPU quantisation decisions against exact rotated values x64 known to
    +-eps, and return them (codes, scales, zeros) for use by the oracle.

    A GPU fp16 scale / zero is valid if it is the fp16 rounding of some value
    within the error interval of the exact quantity; a code is valid if it is the
    rounding of (x - z) / s for some x within +-eps (either neighbour at a tie)."""
    n, hkv, d = x64.shape
    xc = np.clip(x64, -clip, clip)
    xg = xc.reshape(n, hkv, d // group, group)
    eg = eps.reshape(n, hkv, 1)
    mn, mx = xg.min(-1), xg.max(-1)
    # scale: fp16((mx - mn) / 3), the float32 steps are exact to ~1e-7 relative
    rng_lo = (mx - mn - 2 * eg) / 3 * (1 - 1e-6)
    rng_hi = (mx - mn + 2 * eg) / 3 * (1 + 1e-6)
    s_lo, s_hi = _fp16_interval(rng_lo, rng_hi)
    gs = g_s16.astype(np.float64)
    assert np.all((gs >= np.minimum(s_lo, s_hi).astype(np.float64)) &
                  (gs <= np.maximum(s_lo, s_hi).astype(np.float64))), "scale outside its tie interval"
    z_lo, z_hi = _fp16_interval(mn - eg * (1 + 1e-6), mn + eg * (1 + 1e-6))
    gz = g_z16.astype(np.float64)
    assert np.all((gz >= z_lo.astype(np.float64)) & (gz <= z_hi.astype(np.float64))), \
        "zero outside its tie interval"
    sf = np.repeat(gs, group, axis=-1)
    zf = np.repeat(gz, group, axis=-1)
    safe = np.where(sf == 0, 1.0, sf)
    u_lo = (xc - eps - zf) / safe
    u_hi = (xc + eps - zf) / safe
    want_lo = np.clip(np.rint(u_lo), 0, 3)
    want_hi = np.clip(np.rint(u_hi), 0, 3)
    gc = g_codes.astype(np.float64)
    ok = (gc >= np.minimum(want_lo, want_hi)) & (gc <= np.maximum(want_lo, want_hi))
    ok = np.where(sf == 0, gc == 0, ok)
    assert np.all(ok), "code outside its tie interval at %d elements" % int((~ok).sum())
    return g_codes.copy(), g_s16.copy(), g_z16.copy()


class Layer:
    """One layer: calibration (oracle), device context + cache, host copies of
    every token appended so the oracle can rebuild the same cache."""

    def __init__(self, hq, hkv, sink, recent, max_batch, max_tokens, seed=0, n_cal=512,
                 shuffled=True, fold_rv=0, num_splits=0, extra_pages=0, spikes=False,
                 device="cuda", group=32, clip_percentiles=(99.9, 99.9), device_calibration=False):
        self.hq, self.hkv, self.sink, self.recent = hq, hkv, sink, recent
        self.group = group
        self.seed, self.spikes, self.device = seed, spikes, device
        q_cal = draw_queries(seed, 900, n_cal, hq, hkv, D).numpy()
        k_cal, v_cal = (t.numpy() for t in draw_kv(seed, 900, n_cal, hkv, D, spikes))
        if device_calibration:
            # the library's device covariances, rotations and clips on the host; the
            # oracle then runs with these float32 rotations like with its own
            from bit_rotated_kv_oscar_gb300.calibrate import calibrate_device
            d = calibrate_device(q_cal, k_cal, v_cal, clip_percentile_k=clip_percentiles[0],
                                 clip_percentile_v=clip_percentiles[1])
            self.cal = {"R_K32": d["R_K"], "R_V32": d["R_V"], "clip_K32": d["clip_K"], "clip_V32": d["clip_V"],
                        "C_Q": d["C_Q"], "C_S": d["C_S"]}
        else:
            self.cal = oracle.calibrate(q_cal, k_cal, v_cal, clip_percentile_k=clip_percentiles[0],
                                        clip_percentile_v=clip_percentiles[1])
        self.fold_rv = fold_rv
        max_pages = (max_tokens + 15) // 16
        self.cfg = abi.make_config(hq, hkv, sink, recent, max_batch, max_pages, fold_rv=fold_rv,
                                   num_splits=num_splits, group_size=group)
        self.ctx = abi.Context(self.cfg)
        r_v = np.broadcast_to(np.eye(D, dtype=np.float32), (hkv, D, D)) if fold_rv else self.cal["R_V32"]
        self.r_v32 = np.ascontiguousarray(r_v)
        self.ctx.load_rotations(self.cal["R_K32"], self.r_v32, self.cal["clip_K32"], self.cal["clip_V32"])
        num_pages = max_batch * max_pages + extra_pages
        order = draw_page_pool(seed, num_pages, shuffled)
        self.cache = PagedCache(self.ctx, num_pages, device=device, page_order=order)
        self.k_host = [np.zeros((0, hkv, D), np.float32) for _ in range(max_batch)]
        self.v_host = [np.zeros((0, hkv, D), np.float32) for _ in range(max_batch)]
        self.len = [0] * max_batch
        self.e = [sink] * max_batch
        self.stream_id = 0

    # ------------------------------------------------------------------ write
    def draw(self, n):
        self.stream_id += 1
        return draw_kv(self.seed, self.stream_id, n, self.hkv, D, self.spikes)

    def new_trace(self, positions):
        return torch.full((1, positions, self.hkv, 2, D), float("nan"), device=self.device)

    def append(self, b, k, v, trace=None):
        """Append tokens k, v (float32 bf16-exact [n, hkv, D]) to request b; the rotated
        values of every token quantised are recorded in `trace` when given."""
        n = k.shape[0]
        self.cache.reserve(b, self.len[b] + n)
        kd = k.to(torch.bfloat16).to(self.device).contiguous()
        vd = v.to(torch.bfloat16).to(self.device).contiguous()
        if trace is not None:
            trace_positions = trace.shape[1]
            self.ctx.quant_append_traced(self.cache.page_table[b:], self.cache.state[b:], kd, vd, 1, n,
                                         trace, trace_positions)
        else:
            self.ctx.quant_append(self.cache.page_table[b:], self.cache.state[b:], kd, vd, 1, n)
        self._record(b, k, v)

    def append_batch(self, k, v):
        """Append one block of n tokens to every request: k, v [B, n, hkv, D]."""
        bsz, n = k.shape[:2]
        for b in range(bsz):
            self.cache.reserve(b, self.len[b] + n, upload=False)
        self.cache.upload()
        kd = k.to(torch.bfloat16).to(self.device).contiguous()
        vd = v.to(torch.bfloat16).to(self.device).contiguous()
        self.ctx.quant_append(self.cache.page_table, self.cache.state, kd, vd, bsz, n)
        for b in range(bsz):
            self._record(b, k[b], v[b])

    def _record(self, b, k, v):
        self.k_host[b] = np.concatenate([self.k_host[b], k.cpu().numpy()])
        self.v_host[b] = np.concatenate([self.v_host[b], v.cpu().numpy()])
        self.len[b], self.e[b] = oracle.next_state(self.len[b], self.e[b], k.shape[0], self.recent, self.sink)

    # ------------------------------------------------------------------- read
    def decode(self, q):
        """q float32 [B, hq, D] (bf16-exact) -> device output [B, hq, D] as numpy."""
        bsz = q.shape[0]
        qd = q.to(torch.bfloat16).to(self.device).contiguous()
        o = torch.full((bsz, self.hq, D), float("nan"), device=self.device)
        self.ctx.decode_attn(qd, self.cache.page_table, self.cache.state, o, bsz)
        torch.cuda.synchronize()
        return o.cpu().numpy()

    def oracle_cache(self, b):
        r_k = self.cal["R_K32"]
        return oracle.OracleCache(r_k, self.r_v32, self.cal["clip_K32"], self.cal["clip_V32"],
                                  self.sink, self.group).build(self.k_host[b], self.v_host[b], self.len[b],
                                                               self.e[b])

    def oracle_decode(self, q, b, resolve_ties=True):
        cache = self.oracle_cache_resolved(b) if resolve_ties else self.oracle_cache(b)
        return oracle.decode_attention(np.asarray(q, dtype=np.float64), cache)

    def oracle_cache_resolved(self, b):
        """The oracle's own cache of request b in which every decision that sits at
        a rounding tie of the oracle's float64 rotation (within the 1e-5 rotation
        bound) takes the GPU's choice, after checking that the choice is one of
        the valid ones there. Every other code, scale and zero must already be
        equal; a GPU decision that is neither raises AssertionError."""
        cache = self.oracle_cache(b)
        S, E = self.sink, min(self.e[b], self.len[b])
        if E <= S:
            return cache
        dec = self.int2_codes(b, S, E)
        for kind in range(2):
            x = (cache.k if kind == 0 else cache.v)[S:E]
            r = cache.r_k if kind == 0 else cache.r_v
            clip = (cache.clip_k if kind == 0 else cache.clip_v).reshape(1, -1, 1).astype(np.float64)
            x64 = np.einsum("nhi,hij->nhj", x, r)
            eps = ROT_REL * np.abs(x64).max(-1, keepdims=True)                 # [n, hkv, 1]
            codes, s16, z16 = resolve_group_ties(x64, clip, eps, dec[kind], dec[2 + 2 * kind],
                                                 dec[3 + 2 * kind], group=self.group)
            if kind == 0:
                cache.k_codes, cache.k_scale, cache.k_zero = codes, s16, z16
            else:
                cache.v_codes, cache.v_scale, cache.v_zero = codes, s16, z16
        return cache

    def device_state(self):
        return self.cache.state.cpu().numpy()

    def blocks_of_pages(self, page_ids):
        """Pool blocks of the given page ids as numpy [n, hkv, block bytes]."""
        pool = self.cache.pool.view(-1, self.hkv, abi.page_block_bytes(self.group))
        idx = torch.as_tensor(np.asarray(page_ids, dtype=np.int64), device=pool.device)
        return pool[idx].cpu().numpy()

    def int2_codes(self, b, lo, hi):
        """Decoded (k_codes, v_codes, k_s, k_z, v_s, v_z) of positions [lo, hi) of request b,
        each [hi - lo, hkv, ...], read through the oracle's restatement of the layout."""
        pt = self.cache.page_table_host[b]
        n0, n1 = lo // 16, (hi - 1) // 16 + 1
        dec = oracle.decode_page_block(self.blocks_of_pages(pt[n0:n1]), group=self.group)
        res = []
        for x in dec:
            x = np.moveaxis(x, 2, 1)
            x = x.reshape((-1,) + x.shape[2:])
            res.append(x[lo - n0 * 16:hi - n0 * 16])
        return res

    def window_rows(self, b):
        """BF16 window of request b as float32 numpy [hkv, 2, sink + recent, D]."""
        w = self.cache.window.view(self.cfg.max_batch, self.hkv, 2, self.sink + self.recent, D)
        return w[b].float().cpu().numpy()

    def queries(self, bsz, stream):
        return draw_queries(self.seed, stream, bsz, self.hq, self.hkv, D)
