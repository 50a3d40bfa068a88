"""Pins of the oracle's fixed transforms: Hadamard, bit reversal, composite rotation.

Cited passages: "OSCAR: Offline Spectral Covariance-Aware Rotation for 2-bit KV
Cache Quantization" (gist.science, it), Riepilogo Tecnico 2.2 A (R = U H P);
"Juntos, AI Open-Sources OSCAR ..." (7minutos.es), section "Lo que OSCAR hace
diferente" (Lemma 1: every diagonal entry of H^T Lambda H is tr(Lambda)/d; P_br
gives each power-of-two group one channel of every tier).
"""

import numpy as np
import pytest
import scipy.linalg

from oracle import (bit_reversal_matrix, bit_reverse_index, composite_rotation, eig_desc,
                    hadamard)
from tests.conftest import read_golden


@pytest.mark.parametrize("d", [1, 2, 4, 8, 16, 64, 128, 256])
def test_hadamard_is_scipy_sylvester(d):
    # scipy.linalg.hadamard builds the same Sylvester-ordered +-1 matrix
    assert np.array_equal(hadamard(d) * np.sqrt(d), scipy.linalg.hadamard(d).astype(float))


@pytest.mark.parametrize("d", [8, 128])
def test_hadamard_orthonormal(d):
    h = hadamard(d)
    assert np.max(np.abs(h @ h.T - np.eye(d))) < 1e-12
    assert np.allclose(np.abs(h), 1 / np.sqrt(d), atol=0, rtol=1e-15)


@pytest.mark.parametrize("seed", range(4))
def test_lemma1_uniform_diagonal(seed):
    # Lemma 1: diag(H^T Lambda H) = tr(Lambda)/d for any diagonal Lambda
    d = 128
    rng = np.random.default_rng(seed)
    lam = np.diag(rng.exponential(size=d) * 10 ** rng.uniform(-3, 3, size=d))
    h = hadamard(d)
    diag = np.diag(h.T @ lam @ h)
    assert np.allclose(diag, np.trace(lam) / d, rtol=1e-12, atol=0)


def test_bit_reversal_textbook_d8():
    rows = read_golden("bit_reversal_d8.txt")
    want = np.array([int(r[1]) for r in rows])
    assert np.array_equal(bit_reverse_index(8), want)


@pytest.mark.parametrize("d", [2, 8, 64, 128])
def test_bit_reversal_involution_symmetric(d):
    br = bit_reverse_index(d)
    assert np.array_equal(br[br], np.arange(d))
    p = bit_reversal_matrix(d)
    assert np.array_equal(p, p.T)
    assert np.array_equal(p @ p, np.eye(d))


@pytest.mark.parametrize("group", [2, 4, 8, 16, 32, 64, 128])
def test_bit_reversal_one_channel_per_tier(group):
    # channels ranked by importance 0..d-1 form `group` tiers of d/group channels;
    # after x -> x @ P each block of `group` consecutive outputs holds channel
    # br(j) at position j, and those channels must cover every tier once
    d = 128
    br = bit_reverse_index(d)
    x = np.arange(d, dtype=float)  # x[i] = importance rank of channel i
    y = x @ bit_reversal_matrix(d)
    assert np.array_equal(y, br.astype(float))
    tier_size = d // group
    for blk in range(d // group):
        tiers = sorted(int(v) // tier_size for v in y[blk * group:(blk + 1) * group])
        assert tiers == list(range(group))


def test_composite_rotation_identity_basis_is_hadamard_only():
    d = 128
    r = composite_rotation(np.eye(d))
    assert np.array_equal(r, hadamard(d) @ bit_reversal_matrix(d))


@pytest.mark.parametrize("seed", range(3))
def test_eig_desc(seed):
    d = 32
    rng = np.random.default_rng(seed)
    a = rng.normal(size=(d, d))
    c = a @ a.T
    w, u = eig_desc(c)
    assert np.all(np.diff(w) <= 0)
    assert np.max(np.abs(u @ np.diag(w) @ u.T - c)) < 1e-10 * np.max(np.abs(c))
    assert np.max(np.abs(u.T @ u - np.eye(d))) < 1e-12
    for j in range(d):
        assert u[np.argmax(np.abs(u[:, j])), j] > 0


@pytest.mark.parametrize("seed", range(3))
def test_composite_rotation_orthogonal_and_equalises(seed):
    # R = U H P with U the eigenbasis of C: R^T R = I, and by Lemma 1 the
    # importance metric seen by every rotated channel, diag(R^T C R), is tr(C)/d.
    # A wrong factor order (e.g. H U P) or a transposed U breaks the second check.
    d = 128
    rng = np.random.default_rng(seed)
    basis, _ = np.linalg.qr(rng.normal(size=(d, d)))
    c = basis @ np.diag(0.9 ** np.arange(d)) @ basis.T
    w, u = eig_desc(c)
    r = composite_rotation(u)
    assert np.max(np.abs(r.T @ r - np.eye(d))) < 1e-12
    assert np.allclose(np.diag(r.T @ c @ r), np.trace(c) / d, rtol=1e-10, atol=0)
    r_bad = hadamard(d) @ u @ bit_reversal_matrix(d)
    assert not np.allclose(np.diag(r_bad.T @ c @ r_bad), np.trace(c) / d, rtol=1e-3)


@pytest.mark.parametrize("group", [16, 32, 64])
def test_leading_axes_become_group_offsets(group):
    # why R = U_Q H P_br protects the queries' leading directions at INT2: after
    # U_Q (eigenvalues descending) those directions are the first coordinate
    # axes; H maps axis i to the i-th Sylvester row, and after P_br rows
    # 0 .. d/group - 1 are constant inside every group of `group` consecutive
    # channels, so a key component along them is a per-group offset that the
    # asymmetric zero point absorbs. Checked row by row: exactly those rows are
    # group-constant.
    d = 128
    hp = hadamard(d) @ bit_reversal_matrix(d)
    const = [i for i in range(d) if np.all(np.ptp(hp[i].reshape(-1, group), axis=1) == 0)]
    assert const == list(range(d // group))
