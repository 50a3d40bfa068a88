"""Offline calibration of one layer's fixed rotations and clip values.

Host setup, run once per layer before serving (not part of the per-token
path). Written with torch float64 on the CPU.

Steps ("OSCAR: Offline Spectral Covariance-Aware Rotation ..." (gist.science,
it), Riepilogo Tecnico 2.2 A; "Juntos, AI Open-Sources OSCAR ..." (7minutos.es),
section "Lo que OSCAR hace diferente"):
  C_Q = (1/N) sum q_n^T q_n and C_S = (1/N) V^T S^T S V per KV head (averaged
  over the head's query heads, S the causal scores at scale 1/sqrt(d));
  eigenbases U_Q, U_S with eigenvalues in descending order (each eigenvector's
  largest entry positive); R = U H P with H the orthonormal Sylvester
  Hadamard matrix and P the bit-reversal permutation; one clip per layer at a
  percentile of |x R| over the calibration activations.
"""

from __future__ import annotations

import numpy as np
import torch


def _hadamard(d: int) -> torch.Tensor:
    h = torch.tensor([[1.0]], dtype=torch.float64)
    base = torch.tensor([[1.0, 1.0], [1.0, -1.0]], dtype=torch.float64)
    while h.shape[0] < d:
        h = torch.kron(base, h)
    return h / d ** 0.5


def _bit_reversal(d: int) -> torch.Tensor:
    bits = d.bit_length() - 1
    idx = torch.arange(d)
    rev = torch.zeros(d, dtype=torch.long)
    for k in range(bits):
        rev |= ((idx >> k) & 1) << (bits - 1 - k)
    p = torch.zeros(d, d, dtype=torch.float64)
    p[idx, rev] = 1.0
    return p


def _eigvecs_desc(c: torch.Tensor) -> torch.Tensor:
    w, u = torch.linalg.eigh(c)
    order = torch.argsort(w, descending=True, stable=True)
    u = u[:, order]
    piv = u.abs().argmax(dim=0)
    sgn = torch.sign(u[piv, torch.arange(u.shape[1])])
    sgn[sgn == 0] = 1
    return u * sgn


def _percentile(x: torch.Tensor, pct: float) -> float:
    # linear interpolation between order statistics
    v = torch.sort(x.reshape(-1)).values
    pos = (v.numel() - 1) * pct / 100.0
    lo = int(np.floor(pos))
    hi = min(lo + 1, v.numel() - 1)
    return float(v[lo] + (v[hi] - v[lo]) * (pos - lo))


def calibrate(q_cal, k_cal, v_cal, percentile: float = 99.9, scale: float | None = None,
              clip_percentile_k: float | None = None, clip_percentile_v: float | None = None) -> dict:
    """q_cal [N, Hq, d], k_cal / v_cal [N, Hkv, d] -> float32 R_K, R_V [Hkv, d, d], clip_K, clip_V [Hkv].
    clip_percentile_k / _v override the clip percentile per kind (the pages'
    typical cK = 0.96, cV = 0.92 read as the 96th / 92nd percentiles)."""
    q = torch.as_tensor(q_cal).to(torch.float64)
    k = torch.as_tensor(k_cal).to(torch.float64)
    v = torch.as_tensor(v_cal).to(torch.float64)
    n, hq, d = q.shape
    hkv = k.shape[1]
    g = hq // hkv
    if scale is None:
        scale = d ** -0.5
    causal = torch.ones(n, n, dtype=torch.bool).triu(1)
    c_q = torch.zeros(hkv, d, d, dtype=torch.float64)
    c_s = torch.zeros(hkv, d, d, dtype=torch.float64)
    for h in range(hkv):
        for j in range(h * g, (h + 1) * g):
            qj = q[:, j]
            c_q[h] += qj.T @ qj / n
            logits = (qj @ k[:, h].T * scale).masked_fill(causal, float("-inf"))
            sv = torch.softmax(logits, dim=1) @ v[:, h]
            c_s[h] += sv.T @ sv / n
    return _rotations_and_clips(c_q / g, c_s / g, k, v, percentile, clip_percentile_k, clip_percentile_v)


def calibrate_device(q_cal, k_cal, v_cal, percentile: float = 99.9, scale: float | None = None,
                     clip_percentile_k: float | None = None, clip_percentile_v: float | None = None) -> dict:
    """calibrate() with the covariances C_Q, C_S accumulated on the GPU by the
    library (float32); eigendecomposition, rotations and clips on the host.
    q_cal [N, Hq, d], k_cal / v_cal [N, Hkv, d]: the calibration activations."""
    from . import abi

    dev = torch.device("cuda")
    q = torch.as_tensor(q_cal).to(dev, torch.bfloat16).contiguous()
    k = torch.as_tensor(k_cal).to(dev, torch.bfloat16).contiguous()
    v = torch.as_tensor(v_cal).to(dev, torch.bfloat16).contiguous()
    c_q, c_s = abi.calibration_covariances(q, k, v, 0.0 if scale is None else float(scale))
    torch.cuda.synchronize()
    return _rotations_and_clips(c_q.cpu().to(torch.float64), c_s.cpu().to(torch.float64),
                                k.cpu().to(torch.float64), v.cpu().to(torch.float64), percentile,
                                clip_percentile_k, clip_percentile_v)


def _rotations_and_clips(c_q, c_s, k, v, percentile, clip_percentile_k, clip_percentile_v) -> dict:
    """R = U H P per KV head from the covariances [Hkv, d, d] (float64), then the
    per-layer clips from the rotated calibration keys and values."""
    hkv, d = c_q.shape[0], c_q.shape[1]
    hp = _hadamard(d) @ _bit_reversal(d)
    r_k = torch.empty(hkv, d, d, dtype=torch.float64)
    r_v = torch.empty(hkv, d, d, dtype=torch.float64)
    for h in range(hkv):
        r_k[h] = _eigvecs_desc(c_q[h]) @ hp
        r_v[h] = _eigvecs_desc(c_s[h]) @ hp
    pk = percentile if clip_percentile_k is None else clip_percentile_k
    pv = percentile if clip_percentile_v is None else clip_percentile_v
    clip_k = _percentile(torch.einsum("nhi,hij->nhj", k, r_k).abs(), pk)
    clip_v = _percentile(torch.einsum("nhi,hij->nhj", v, r_v).abs(), pv)
    return {
        "C_Q": c_q.numpy(), "C_S": c_s.numpy(),
        "R_K": r_k.to(torch.float32).numpy(),
        "R_V": r_v.to(torch.float32).numpy(),
        "clip_K": np.full(hkv, clip_k, dtype=np.float32),
        "clip_V": np.full(hkv, clip_v, dtype=np.float32),
    }
