"""OSCAR oracle: offline calibration, composite rotation, INT2 group quantiser,
mixed-precision cache model and decode attention, in plain NumPy.

TEST INFRASTRUCTURE ONLY (see the package docstring). Floating point is
float64 except the group quantiser, which follows a fixed float32 operation
sequence so that an integer decision (a 2-bit code) is taken in the same
precision on both sides of a parity test.

Conventions: activations are row vectors, a rotation acts on the right
(x_rot = x @ R), R is [d, d] row-major; positions are 0-based.

Sources are cited as [IT] / [ES] / [JA] with the section on that page; the
page titles are listed in the package docstring.
"""

from __future__ import annotations

import numpy as np

F32 = np.float32


# --------------------------------------------------------------------------
# Fixed transforms
# --------------------------------------------------------------------------

def hadamard(d: int) -> np.ndarray:
    """Orthonormal Walsh-Hadamard matrix of order d, Sylvester (natural) order.

    [IT] Riepilogo Tecnico 2.2 A (third factor of the composite rotation);
    [ES] "Lo que OSCAR hace diferente" (Lemma 1 on H_Had). The pages do not fix
    the ordering or the normalisation; the Sylvester recursion scaled by
    1/sqrt(d) is the orthonormal reading.
    """
    if d < 1 or d & (d - 1):
        raise ValueError("Hadamard order must be a power of two")
    h = np.ones((1, 1), dtype=np.float64)
    while h.shape[0] < d:
        h = np.block([[h, h], [h, -h]])
    return h / np.sqrt(d)


def bit_reverse_index(d: int) -> np.ndarray:
    """br(i): i with its log2(d) bits written in reverse order.

    [IT] 2.2 A (P_br interleaves high- and low-variance channels); [ES] "Lo que
    OSCAR hace diferente" (each power-of-two group receives one channel of
    every importance tier).
    """
    if d < 1 or d & (d - 1):
        raise ValueError("order must be a power of two")
    nbits = d.bit_length() - 1
    idx = np.arange(d, dtype=np.int64)
    out = np.zeros(d, dtype=np.int64)
    for b in range(nbits):
        out |= ((idx >> b) & 1) << (nbits - 1 - b)
    return out


def bit_reversal_matrix(d: int) -> np.ndarray:
    """Permutation matrix P_br with P[i, br(i)] = 1 (so (x @ P)[br(i)] = x[i])."""
    p = np.zeros((d, d), dtype=np.float64)
    p[np.arange(d), bit_reverse_index(d)] = 1.0
    return p


# --------------------------------------------------------------------------
# Offline calibration
# --------------------------------------------------------------------------

def query_covariance(q: np.ndarray) -> np.ndarray:
    """C_Q = (1/N) sum_n q_n^T q_n for row vectors q_n, i.e. (1/N) Q^T Q.

    [IT] 2.2 A "Stima della Covarianza" (query-aware key target); [ES] "Lo que
    OSCAR hace diferente" (the logit error is weighted by Q^T Q).
    """
    q = np.asarray(q, dtype=np.float64)
    return q.T @ q / q.shape[0]


def causal_softmax_scores(q: np.ndarray, k: np.ndarray, scale: float) -> np.ndarray:
    """Attention score matrix S [N, N]: row-softmax of q k^T * scale, causal."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    logits = (q @ k.T) * scale
    n = logits.shape[0]
    mask = np.triu(np.ones((n, n), dtype=bool), k=1)
    logits = np.where(mask, -np.inf, logits)
    logits = logits - logits.max(axis=1, keepdims=True)
    e = np.exp(logits)
    return e / e.sum(axis=1, keepdims=True)


def score_weighted_value_covariance(q: np.ndarray, k: np.ndarray, v: np.ndarray,
                                    scale: float) -> np.ndarray:
    """C_S = (1/N) V^T S^T S V with S the causal attention scores of (q, k).

    [IT] 2.1 (value distortion is weighted by the scores S) and 2.2 A
    (score-aware value target); [ES] "Lo que OSCAR hace diferente". The pages
    do not state the mask or the scale: causal, 1/sqrt(d) is our reading.
    """
    s = causal_softmax_scores(q, k, scale)
    sv = s @ np.asarray(v, dtype=np.float64)
    return sv.T @ sv / sv.shape[0]


def eig_desc(c: np.ndarray):
    """Eigen-decomposition of a symmetric matrix, eigenvalues descending.

    Each eigenvector's sign is fixed so that its largest-magnitude entry is
    positive (the pages fix neither order nor sign). Returns (w, U) with
    C = U diag(w) U^T and the columns of U the eigenvectors.
    """
    w, u = np.linalg.eigh(np.asarray(c, dtype=np.float64))
    order = np.argsort(-w, kind="stable")
    w = w[order]
    u = u[:, order]
    for j in range(u.shape[1]):
        i = int(np.argmax(np.abs(u[:, j])))
        if u[i, j] < 0:
            u[:, j] = -u[:, j]
    return w, u


def composite_rotation(u: np.ndarray) -> np.ndarray:
    """R = U @ H_Had @ P_br ([IT] 2.2 A formula; [ES] R_K, R_V; [JA] 2.2 A.3)."""
    d = u.shape[0]
    return np.asarray(u, dtype=np.float64) @ hadamard(d) @ bit_reversal_matrix(d)


def clip_threshold(rotated_abs: np.ndarray, percentile: float = 99.9) -> float:
    """Symmetric clip value: a percentile of |rotated calibration activations|.

    [IT] 2.2 A "Soglie di Clipping" (per-layer thresholds from the rotated
    calibration activations); [ES] "El sistema de servicio" (percentile clip).
    Which percentile is used is not printed; 99.9 with linear interpolation is
    our reading. parity unpinned.
    """
    return float(np.percentile(np.asarray(rotated_abs, dtype=np.float64), percentile))


def calibrate(q_cal: np.ndarray, k_cal: np.ndarray, v_cal: np.ndarray,
              percentile: float = 99.9, scale: float | None = None,
              clip_percentile_k: float | None = None, clip_percentile_v: float | None = None) -> dict:
    """Offline calibration for one layer.

    q_cal [N, Hq, d], k_cal / v_cal [N, Hkv, d] (float). Per KV head h:
    C_Q is averaged over the h's query heads, C_S likewise; R_K = U_Q H P,
    R_V = U_S H P. One clip value per layer for K and one for V (percentile of
    |x @ R| over all calibration tokens, channels and KV heads), broadcast to
    every head. clip_percentile_k / _v override the percentile for K / V: the
    pages print typical clips "cK = 0.96, cV = 0.92" ([ES] "El sistema de
    servicio"), read here as the 96th / 92nd percentiles for that preset.
    Returns float64 arrays plus float32 copies for the device.
    """
    q_cal = np.asarray(q_cal, dtype=np.float64)
    k_cal = np.asarray(k_cal, dtype=np.float64)
    v_cal = np.asarray(v_cal, dtype=np.float64)
    n, hq, d = q_cal.shape
    hkv = k_cal.shape[1]
    g = hq // hkv
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    r_k = np.empty((hkv, d, d))
    r_v = np.empty((hkv, d, d))
    c_q = np.empty((hkv, d, d))
    c_s = np.empty((hkv, d, d))
    for h in range(hkv):
        heads = range(h * g, (h + 1) * g)
        c_q[h] = sum(query_covariance(q_cal[:, j]) for j in heads) / g
        c_s[h] = sum(score_weighted_value_covariance(q_cal[:, j], k_cal[:, h], v_cal[:, h], scale)
                     for j in heads) / g
        r_k[h] = composite_rotation(eig_desc(c_q[h])[1])
        r_v[h] = composite_rotation(eig_desc(c_s[h])[1])
    k_rot = np.einsum("nhi,hij->nhj", k_cal, r_k)
    v_rot = np.einsum("nhi,hij->nhj", v_cal, r_v)
    clip_k = clip_threshold(np.abs(k_rot), percentile if clip_percentile_k is None else clip_percentile_k)
    clip_v = clip_threshold(np.abs(v_rot), percentile if clip_percentile_v is None else clip_percentile_v)
    return {
        "R_K": r_k, "R_V": r_v, "C_Q": c_q, "C_S": c_s,
        "clip_K": np.full(hkv, clip_k), "clip_V": np.full(hkv, clip_v),
        "R_K32": r_k.astype(F32), "R_V32": r_v.astype(F32),
        "clip_K32": np.full(hkv, clip_k, dtype=F32), "clip_V32": np.full(hkv, clip_v, dtype=F32),
    }


# --------------------------------------------------------------------------
# Write path: rotate, clip, asymmetric per-token group quantisation
# --------------------------------------------------------------------------

def rotate(x: np.ndarray, r: np.ndarray) -> np.ndarray:
    """x @ R in float64 (x [..., d], R [d, d])."""
    return np.asarray(x, dtype=np.float64) @ np.asarray(r, dtype=np.float64)


def quantize_groups(x_rot32: np.ndarray, clip32, group: int = 32):
    """Clip, then asymmetric min/max INT2 quantisation per group of ``group`` channels.

    [ES] "El sistema de servicio": each token is rotated, clipped to a
    calibrated threshold and quantised to asymmetric per-token INT2 groups.
    The exact float32 sequence (our reading; the pages give no formula):
        x  = min(max(x_rot, -c), c)
        s  = fp16((mx - mn) / 3)      z = fp16(mn)      (fp32 divide, then RNE to fp16)
        r  = fp32(1 / s)                                (correctly rounded reciprocal)
        q  = 0 if s == 0 else clamp(rint_half_even(fp32(fp32(x - z) * r)), 0, 3)
    with z and s taken back to float32 before use: dividing by the scale is
    taken as multiplying by its float32 reciprocal, one fixed rounding per
    value. Returns (codes uint8 [..., d], scale float16 [..., d/group], zero
    float16 [..., d/group]).
    """
    x = np.asarray(x_rot32, dtype=F32)
    c = np.asarray(clip32, dtype=F32)
    xc = np.minimum(np.maximum(x, -c), c).astype(F32)
    d = xc.shape[-1]
    xg = xc.reshape(xc.shape[:-1] + (d // group, group))
    mn = xg.min(axis=-1)
    mx = xg.max(axis=-1)
    rng = (mx - mn).astype(F32)
    with np.errstate(over="ignore"):
        s16 = (rng / F32(3.0)).astype(F32).astype(np.float16)
        z16 = mn.astype(np.float16)
    sf = s16.astype(F32)
    zf = z16.astype(F32)
    diff = (xg - zf[..., None]).astype(F32)
    safe = np.where(sf == 0, F32(1.0), sf).astype(F32)
    with np.errstate(over="ignore", invalid="ignore"):
        rinv = (F32(1.0) / safe).astype(F32)
        u = (diff * rinv[..., None]).astype(F32)
    code = np.clip(np.rint(u), 0, 3)
    code = np.where((sf == 0)[..., None], 0, code)
    return code.reshape(x.shape).astype(np.uint8), s16, z16


def dequantize_groups(codes: np.ndarray, scale16: np.ndarray, zero16: np.ndarray,
                      group: int = 32) -> np.ndarray:
    """x_hat = code * s + z in float64 (per group)."""
    codes = np.asarray(codes, dtype=np.float64)
    d = codes.shape[-1]
    cg = codes.reshape(codes.shape[:-1] + (d // group, group))
    out = cg * np.asarray(scale16, dtype=np.float64)[..., None] + \
        np.asarray(zero16, dtype=np.float64)[..., None]
    return out.reshape(codes.shape)


# --------------------------------------------------------------------------
# Mixed-precision cache model
# --------------------------------------------------------------------------

def cache_regions(seq_len: int, int2_end: int, sink: int):
    """Position ranges (half-open) of the three regions of one request.

    [IT] 2.2 B "Layout a Precisione Mista"; [ES] "El sistema de servicio"
    (sink tokens and recent tokens in BF16, the history between them INT2).
    Sink = [0, min(S, L)), INT2 = [S, E), recent ring = [E, L) with E >= S.
    """
    return (0, min(sink, seq_len)), (sink, max(sink, int2_end)), (max(sink, int2_end), seq_len)


def next_state(seq_len: int, int2_end: int, n_new: int, recent: int, sink: int):
    """State after appending n_new tokens: the INT2 frontier follows the window.

    Tokens that fall out of the last ``recent`` positions are quantised; the
    frontier never moves back and never below the sink.
    """
    new_len = seq_len + n_new
    return new_len, max(int2_end, sink, new_len - recent)


class OracleCache:
    """One request's cache, modelled by position (history does not matter:
    quantisation is per token, so the INT2 content of a position depends only
    on that token's K/V)."""

    def __init__(self, r_k32, r_v32, clip_k32, clip_v32, sink: int, group: int = 32):
        self.r_k = np.asarray(r_k32, dtype=np.float64)
        self.r_v = np.asarray(r_v32, dtype=np.float64)
        self.clip_k = np.asarray(clip_k32, dtype=F32)
        self.clip_v = np.asarray(clip_v32, dtype=F32)
        self.sink = sink
        self.group = group

    def build(self, k_tokens: np.ndarray, v_tokens: np.ndarray, seq_len: int, int2_end: int):
        """k_tokens / v_tokens [>= L, Hkv, d] (bf16-exact). Quantises [S, E)."""
        self.k = np.asarray(k_tokens[:seq_len], dtype=np.float64)
        self.v = np.asarray(v_tokens[:seq_len], dtype=np.float64)
        self.seq_len = seq_len
        self.int2_end = max(int2_end, self.sink)
        lo, hi = self.sink, min(self.int2_end, seq_len)
        self.int2_lo, self.int2_hi = lo, max(lo, hi)
        hkv = self.k.shape[1]
        if self.int2_hi > self.int2_lo:
            kk = self.k[lo:hi]
            vv = self.v[lo:hi]
            krot = np.einsum("nhi,hij->nhj", kk, self.r_k).astype(F32)
            vrot = np.einsum("nhi,hij->nhj", vv, self.r_v).astype(F32)
            ck = self.clip_k.reshape(1, hkv, 1)
            cv = self.clip_v.reshape(1, hkv, 1)
            self.k_codes, self.k_scale, self.k_zero = quantize_groups(krot, ck, self.group)
            self.v_codes, self.v_scale, self.v_zero = quantize_groups(vrot, cv, self.group)
        return self

    def raw_kv(self, h: int):
        """K_hat, V_hat [L, d] float64 in the raw (un-rotated) basis for KV head h."""
        k = self.k[:, h].copy()
        v = self.v[:, h].copy()
        lo, hi = self.int2_lo, self.int2_hi
        if hi > lo:
            kq = dequantize_groups(self.k_codes[:, h], self.k_scale[:, h], self.k_zero[:, h], self.group)
            vq = dequantize_groups(self.v_codes[:, h], self.v_scale[:, h], self.v_zero[:, h], self.group)
            k[lo:hi] = kq @ self.r_k[h].T
            v[lo:hi] = vq @ self.r_v[h].T
        return k, v


def decode_attention(q: np.ndarray, cache: OracleCache, scale: float | None = None) -> np.ndarray:
    """Naive float64 softmax attention of one decode query over the whole cache.

    q [Hq, d] (bf16-exact). KV head of query head j is j // (Hq / Hkv). INT2
    keys and values are de-rotated (x_hat @ R^T) before use, as the pages'
    read path describes ([IT] 2.2 B "Integrazione del Kernel"; [ES] "El sistema
    de servicio": unpack, dequantise, inverse rotation, attention).
    Returns o [Hq, d] float64; an empty cache gives zeros.
    """
    q = np.asarray(q, dtype=np.float64)
    hq, d = q.shape
    hkv = cache.k.shape[1]
    g = hq // hkv
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    out = np.zeros((hq, d))
    if cache.seq_len == 0:
        return out
    for h in range(hkv):
        kh, vh = cache.raw_kv(h)
        for j in range(h * g, (h + 1) * g):
            logits = kh @ q[j] * scale
            p = np.exp(logits - logits.max())
            out[j] = (p / p.sum()) @ vh
    return out


# --------------------------------------------------------------------------
# Analysis helpers used by the pins
# --------------------------------------------------------------------------

def logit_error(q: np.ndarray, k: np.ndarray, k_hat: np.ndarray) -> float:
    """||Q K^T - Q K_hat^T||_F^2 computed directly from the logits."""
    q = np.asarray(q, dtype=np.float64)
    diff = q @ np.asarray(k, dtype=np.float64).T - q @ np.asarray(k_hat, dtype=np.float64).T
    return float(np.sum(diff * diff))


def logit_error_from_covariance(c_q: np.ndarray, n_queries: int, k: np.ndarray,
                                k_hat: np.ndarray) -> float:
    """N * tr((K - K_hat) C_Q (K - K_hat)^T), the right-hand side of the
    logit-error identity ([ES] "Lo que OSCAR hace diferente")."""
    e = np.asarray(k, dtype=np.float64) - np.asarray(k_hat, dtype=np.float64)
    return float(n_queries * np.trace(e @ c_q @ e.T))


def footprint_bits_per_element(group: int, seq_len: int, sink: int, recent: int,
                               meta_bits_per_group: int = 32, code_bits: int = 2,
                               bf16_bits: int = 16) -> float:
    """Average stored bits per K/V element of one request.

    BF16 sink and recent tokens cost 16 bits; every other token costs the
    code bits plus its share of the per-group metadata (fp16 scale + fp16
    zero = 32 bits by default).
    """
    n_bf16 = min(seq_len, sink + recent)
    n_int2 = seq_len - n_bf16
    bits = n_int2 * (code_bits + meta_bits_per_group / group) + n_bf16 * bf16_bits
    return bits / seq_len
