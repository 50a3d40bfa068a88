"""Seeded generators for the synthetic Qwen3-shaped attention-layer workloads.

Every draw goes through ``torch.Generator`` so the same call produces the same
numbers on the CPU; on a CUDA device it produces a different (but equally
seeded) stream, which is what the large GPU workloads use. A test always takes
both sides' inputs from ONE call, so the two generators never have to agree.

Distributions (the method's pages quantise real Qwen3/GLM activations; these
stand in for them, taking only their shapes):
  * K and V: i.i.d. N(0, 1) with four fixed channels per KV head (drawn once,
    separately for K and V) multiplied by 20; optionally 1% of tokens
    multiplied by 8 (token spikes).
  * Q: z @ diag(0.9**i)**0.5 @ B^T with z ~ N(0, I) and B a random orthonormal
    basis per KV head, shared by that head's query heads (anisotropic queries).
  * Everything that enters the cache is rounded to bfloat16 (round to nearest
    even); arrays are returned as float32 holding bf16-exact values.
"""

from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch


# --------------------------------------------------------------------------
# Workload shapes
# --------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class WorkloadSpec:
    """One synthetic attention-layer workload (sizes only)."""

    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    batch: int
    context: int            # tokens per request before decoding (or max of a range)
    context_min: int        # lower end of a ragged length range (== context if fixed)
    page_size: int = 16
    group_size: int = 32
    sink: int = 4
    recent: int = 128
    calib_tokens: int = 2048
    token_spikes: bool = False
    shuffled_pages: bool = True
    seed: int = 0
    decode_steps: int = 1
    prefix_shared: int = 0  # tokens of a shared prefix (prefix-sharing workload)
    suffix: int = 0         # private tokens per request after the shared prefix
    clip_percentile_k: float = 99.9
    clip_percentile_v: float = 99.9

    @property
    def int2_token_bytes(self) -> int:
        """Bytes of one INT2 token of one KV head: K and V codes plus fp16
        scale and zero per group."""
        return 2 * (self.head_dim // 4) + 2 * (self.head_dim // self.group_size) * 4

    @property
    def gqa(self) -> int:
        return self.num_q_heads // self.num_kv_heads


WORKLOADS = {
    # single layer, 2 query heads / 1 KV head, 1024 tokens, 64-token recent window
    "tiny_1k": WorkloadSpec("tiny_1k", 2, 1, 128, 1, 1024, 1024, recent=64,
                            shuffled_pages=False, seed=0),
    # Qwen3-8B layer shape, batch 1 at 32768 tokens, 100 decode steps
    "qwen3_8b_bs1_32k": WorkloadSpec("qwen3_8b_bs1_32k", 32, 8, 128, 1, 32768, 32768,
                                     seed=1, decode_steps=100),
    # Qwen3-8B layer shape, 16 requests with lengths uniform in [8192, 32768]
    "qwen3_8b_bs16_ragged": WorkloadSpec("qwen3_8b_bs16_ragged", 32, 8, 128, 16, 32768, 8192,
                                         token_spikes=True, seed=2),
    # Qwen3-32B layer shape, 28 requests of 100000 tokens
    "qwen3_32b_bs28_100k": WorkloadSpec("qwen3_32b_bs28_100k", 64, 8, 128, 28, 100000, 100000,
                                        seed=3),
    # the same two decode workloads with the pages' own constants: groups of 64
    # channels, sink 64, recent window 256, clips at the 96th / 92nd percentile
    "qwen3_8b_bs1_32k_pages": WorkloadSpec("qwen3_8b_bs1_32k_pages", 32, 8, 128, 1, 32768, 32768,
                                           seed=1, decode_steps=100, group_size=64, sink=64, recent=256,
                                           clip_percentile_k=96.0, clip_percentile_v=92.0),
    "qwen3_32b_bs28_100k_pages": WorkloadSpec("qwen3_32b_bs28_100k_pages", 64, 8, 128, 28, 100000, 100000,
                                              seed=3, group_size=64, sink=64, recent=256,
                                              clip_percentile_k=96.0, clip_percentile_v=92.0),
    # 131072-token prefill, then 16 requests sharing its first 65536 tokens
    # through aliased pages, each with a private 4096-token suffix
    "prefill_128k_prefix16": WorkloadSpec("prefill_128k_prefix16", 32, 8, 128, 16, 131072, 131072,
                                          seed=4, prefix_shared=65536, suffix=4096),
}


# --------------------------------------------------------------------------
# Rounding helpers (input preparation, not part of the method)
# --------------------------------------------------------------------------

def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); float32 out."""
    return (bf16_bits(x).astype(np.uint32) << 16).view(np.float32)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) of float32 values, round to nearest even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def _gen(seed: int, stream: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    # splitmix-style mixing so (seed, stream) pairs give unrelated streams
    z = (seed * 0x9E3779B97F4A7C15 + stream * 0xBF58476D1CE4E5B9 + 0x94D049BB133111EB) & (2**63 - 1)
    g.manual_seed(z)
    return g


# --------------------------------------------------------------------------
# K / V / Q
# --------------------------------------------------------------------------

def kv_outlier_channels(seed: int, num_kv_heads: int, head_dim: int, n_out: int = 4) -> np.ndarray:
    """Outlier channel indices, shape [2 (K,V), num_kv_heads, n_out]."""
    g = _gen(seed, 11)
    out = np.empty((2, num_kv_heads, n_out), dtype=np.int64)
    for kind in range(2):
        for h in range(num_kv_heads):
            out[kind, h] = torch.randperm(head_dim, generator=g)[:n_out].numpy()
    return out


def query_basis(seed: int, num_kv_heads: int, head_dim: int) -> np.ndarray:
    """Random orthonormal bases [num_kv_heads, d, d] (float64), QR with sign fix."""
    g = _gen(seed, 13)
    out = np.empty((num_kv_heads, head_dim, head_dim), dtype=np.float64)
    for h in range(num_kv_heads):
        a = torch.randn(head_dim, head_dim, generator=g, dtype=torch.float64)
        qm, rm = torch.linalg.qr(a)
        qm = qm * torch.sign(torch.diagonal(rm)).unsqueeze(0)
        out[h] = qm.numpy()
    return out


def draw_kv(seed: int, stream: int, n_tokens: int, num_kv_heads: int, head_dim: int,
            token_spikes: bool = False, device="cpu", outlier_mult: float = 20.0,
            spike_prob: float = 0.01, spike_mult: float = 8.0):
    """Keys and values, bf16-exact float32 tensors [n_tokens, num_kv_heads, head_dim].

    ``stream`` separates independent draws (calibration, each request, each
    decode step). Returns torch tensors on ``device``.
    """
    outl = torch.as_tensor(kv_outlier_channels(seed, num_kv_heads, head_dim))
    g = _gen(seed, 1000 + stream, device)
    res = []
    for kind in range(2):
        x = torch.randn(n_tokens, num_kv_heads, head_dim, generator=g, device=device,
                        dtype=torch.float32)
        mult = torch.ones(num_kv_heads, head_dim, dtype=torch.float32)
        for h in range(num_kv_heads):
            mult[h, outl[kind, h]] = outlier_mult
        x = x * mult.to(device)
        if token_spikes:
            u = torch.rand(n_tokens, generator=g, device=device)
            x = torch.where((u < spike_prob)[:, None, None], x * spike_mult, x)
        res.append(x.to(torch.bfloat16).to(torch.float32).contiguous())
    return res[0], res[1]


def draw_queries(seed: int, stream: int, n_tokens: int, num_q_heads: int, num_kv_heads: int,
                 head_dim: int, device="cpu", decay: float = 0.9):
    """Queries, bf16-exact float32 [n_tokens, num_q_heads, head_dim], covariance B diag(decay**i) B^T."""
    basis = torch.as_tensor(query_basis(seed, num_kv_heads, head_dim), dtype=torch.float32)
    sd = torch.tensor([decay ** (0.5 * i) for i in range(head_dim)], dtype=torch.float32)
    g = _gen(seed, 5000 + stream, device)
    z = torch.randn(n_tokens, num_q_heads, head_dim, generator=g, device=device, dtype=torch.float32)
    grp = num_q_heads // num_kv_heads
    bmat = basis.to(device)[torch.arange(num_q_heads, device=device) // grp]  # [Hq, d, d]
    q = torch.einsum("nhi,hji->nhj", z * sd.to(device), bmat)
    return q.to(torch.bfloat16).to(torch.float32).contiguous()


def draw_shared_direction_qk(seed: int, stream: int, n_tokens: int, head_dim: int,
                             n_shared: int = 4, shared_mult: float = 20.0, decay: float = 0.9):
    """One head's queries and keys that share their leading directions.

    Queries as in ``draw_queries`` (covariance B diag(decay**i) B^T, B the random
    orthonormal basis of KV head 0); keys i.i.d. N(0, 1) plus independent
    N(0, shared_mult**2) components along the first ``n_shared`` columns of B,
    so the keys' large components lie along the queries' high-energy
    directions, the structure query and key projections of one attention head
    have in common. Returns bf16-exact float32 tensors (q [n, d], k [n, d]).
    """
    basis = torch.as_tensor(query_basis(seed, 1, head_dim)[0], dtype=torch.float32)
    sd = torch.tensor([decay ** (0.5 * i) for i in range(head_dim)], dtype=torch.float32)
    g = _gen(seed, 7000 + stream)
    q = (torch.randn(n_tokens, head_dim, generator=g) * sd) @ basis.T
    k = torch.randn(n_tokens, head_dim, generator=g)
    k = k + (torch.randn(n_tokens, n_shared, generator=g) * shared_mult) @ basis[:, :n_shared].T
    return (q.to(torch.bfloat16).to(torch.float32).contiguous(),
            k.to(torch.bfloat16).to(torch.float32).contiguous())


# --------------------------------------------------------------------------
# Paging
# --------------------------------------------------------------------------

def draw_page_pool(seed: int, num_pages: int, shuffled: bool = True) -> np.ndarray:
    """A permutation of page ids [0, num_pages) (identity if not shuffled)."""
    if not shuffled:
        return np.arange(num_pages, dtype=np.int32)
    g = _gen(seed, 17)
    return torch.randperm(num_pages, generator=g).numpy().astype(np.int32)


def draw_ragged_lengths(seed: int, batch: int, lo: int, hi: int) -> np.ndarray:
    """Per-request context lengths uniform in [lo, hi] (inclusive)."""
    if lo == hi:
        return np.full(batch, lo, dtype=np.int64)
    g = _gen(seed, 19)
    return torch.randint(lo, hi + 1, (batch,), generator=g).numpy().astype(np.int64)


def pages_for(n_tokens: int, page_size: int) -> int:
    return int(math.ceil(n_tokens / page_size))
