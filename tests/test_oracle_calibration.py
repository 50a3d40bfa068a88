"""Pins of the oracle's offline calibration (C_Q, C_S, eigenbases, clip, R).

Cited passages: "Juntos, AI Open-Sources OSCAR ..." (7minutos.es), section "Lo
que OSCAR hace diferente" (logit-error identity, C_Q, C_S); "OSCAR: Offline
Spectral Covariance-Aware Rotation ..." (gist.science, it), Riepilogo Tecnico
2.1 and 2.2 A (covariance estimation, eigen-decomposition, clip thresholds).
"""

import math

import numpy as np
import pytest

from oracle import (calibrate, causal_softmax_scores, composite_rotation, eig_desc,
                    logit_error, logit_error_from_covariance, query_covariance,
                    score_weighted_value_covariance)
from synth import draw_kv, draw_queries, query_basis


@pytest.mark.parametrize("seed", range(4))
def test_logit_error_identity_pins_query_covariance(seed):
    # ||Q K^T - Q K_hat^T||_F^2 = tr((K - K_hat) Q^T Q (K - K_hat)^T) and
    # Q^T Q = N C_Q; a transposed or mis-normalised C_Q fails this
    rng = np.random.default_rng(seed)
    n, m, d = 37, 23, 16
    q = rng.normal(size=(n, d))
    k = rng.normal(size=(m, d))
    k_hat = k + 0.1 * rng.normal(size=(m, d))
    lhs = logit_error(q, k, k_hat)
    rhs = logit_error_from_covariance(query_covariance(q), n, k, k_hat)
    assert abs(lhs - rhs) <= 1e-10 * lhs


def test_query_covariance_closed_form_on_generator():
    # the generator's queries have covariance B diag(0.9^i) B^T (per KV head);
    # at large N the estimate's eigenpairs approach it within sampling error
    d = 128
    n = 40000
    q = draw_queries(seed=7, stream=0, n_tokens=n, num_q_heads=1, num_kv_heads=1,
                     head_dim=d).numpy()[:, 0].astype(np.float64)
    c = query_covariance(q)
    w, u = eig_desc(c)
    lam = 0.9 ** np.arange(d)
    assert np.allclose(w[:8], lam[:8], rtol=0.05)
    assert abs(np.trace(c) - lam.sum()) < 0.03 * lam.sum()
    b = query_basis(7, 1, d)[0]
    for i in range(4):
        assert abs(u[:, i] @ b[:, i]) > 0.95


def test_score_weighted_value_covariance_brute_force():
    # C_S = (1/N) V^T S^T S V by explicit loops over tiny sizes
    rng = np.random.default_rng(3)
    n, d = 6, 4
    q, k, v = (rng.normal(size=(n, d)) for _ in range(3))
    scale = 1 / math.sqrt(d)
    s = np.zeros((n, n))
    for i in range(n):
        logits = [sum(q[i, a] * k[j, a] for a in range(d)) * scale for j in range(i + 1)]
        mx = max(logits)
        e = [math.exp(x - mx) for x in logits]
        for j in range(i + 1):
            s[i, j] = e[j] / sum(e)
    want = np.zeros((d, d))
    for a in range(d):
        for b in range(d):
            tot = 0.0
            for i in range(n):
                ya = sum(s[i, j] * v[j, a] for j in range(n))
                yb = sum(s[i, j] * v[j, b] for j in range(n))
                tot += ya * yb
            want[a, b] = tot / n
    assert np.allclose(causal_softmax_scores(q, k, scale), s, rtol=1e-12, atol=1e-15)
    assert np.allclose(score_weighted_value_covariance(q, k, v, scale), want, rtol=1e-12, atol=1e-15)


def test_calibrate_tiny_layer():
    d, hq, hkv, n = 128, 4, 2, 256
    q = draw_queries(1, 0, n, hq, hkv, d).numpy()
    k, v = (t.numpy() for t in draw_kv(1, 0, n, hkv, d))
    cal = calibrate(q, k, v)
    for name in ("R_K", "R_V"):
        for h in range(hkv):
            r = cal[name][h]
            assert np.max(np.abs(r.T @ r - np.eye(d))) < 1e-12
    for h in range(hkv):
        g = hq // hkv
        cq = sum(query_covariance(q[:, j].astype(np.float64)) for j in range(h * g, h * g + g)) / g
        assert np.allclose(cal["C_Q"][h], cq, rtol=1e-12, atol=1e-14)
        assert np.allclose(cal["R_K"][h], composite_rotation(eig_desc(cq)[1]), atol=1e-12)
        # Lemma 1 on the calibrated key rotation
        r = cal["R_K"][h]
        assert np.allclose(np.diag(r.T @ cq @ r), np.trace(cq) / d, rtol=1e-9)
    # the clip is the 99.9th percentile of |k R_K|: 0.1 % of values lie above it
    krot = np.einsum("nhi,hij->nhj", k.astype(np.float64), cal["R_K"])
    frac = np.mean(np.abs(krot) > cal["clip_K"][0])
    assert abs(frac - 0.001) <= 2.0 / krot.size
    assert cal["clip_K"][0] > 0 and cal["clip_V"][0] > 0
    assert cal["R_K32"].dtype == np.float32 and cal["clip_K32"].dtype == np.float32
