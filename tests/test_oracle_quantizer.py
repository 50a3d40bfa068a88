"""Pins of the oracle's clip + asymmetric per-token INT2 group quantiser.

Cited passage: "Juntos, AI Open-Sources OSCAR ..." (7minutos.es), section "El
sistema de servicio": each token is rotated, clipped to a calibrated
percentile threshold and quantised with asymmetric per-token INT2 groups.
"""

import itertools

import numpy as np
import pytest

from oracle import dequantize_groups, quantize_groups

F32 = np.float32


def _exact_levels(s16, z16):
    sf = np.float64(np.float32(s16))
    zf = np.float64(np.float32(z16))
    return np.array([zf + c * sf for c in range(4)])


@pytest.mark.parametrize("group", [4, 8])
@pytest.mark.parametrize("seed", range(6))
def test_brute_force_all_code_vectors(group, seed):
    # d = 8: enumerate all 4^8 code vectors; given the group's (scale, zero)
    # the chosen vector minimises the squared reconstruction error
    rng = np.random.default_rng(seed)
    x = (rng.normal(size=8) * rng.uniform(0.1, 5)).astype(F32)
    clip = F32(np.inf)
    codes, s16, z16 = quantize_groups(x, clip, group)
    ng = 8 // group
    allv = np.array(list(itertools.product(range(4), repeat=8)), dtype=np.float64)
    sf = np.repeat(np.asarray(s16, np.float64), group)
    zf = np.repeat(np.asarray(z16, np.float64), group)
    recon = allv * sf + zf
    err = ((recon - x.astype(np.float64)) ** 2).sum(axis=1)
    best = err.min()
    mine = (((codes.astype(np.float64) * sf + zf) - x) ** 2).sum()
    # equal up to float32 rounding of the division at exact ties
    assert mine <= best * (1 + 1e-6) + 1e-12
    assert ng == len(s16)


@pytest.mark.parametrize("seed", range(10))
def test_error_bound_and_extremes(seed):
    rng = np.random.default_rng(seed)
    x = (rng.normal(size=(64, 128)) * 3).astype(F32)
    c = F32(np.percentile(np.abs(x), 99.0))
    codes, s16, z16 = quantize_groups(x, c, 32)
    xc = np.clip(x, -c, c).astype(np.float64)
    xhat = dequantize_groups(codes, s16, z16, 32)
    sf = np.repeat(s16.astype(np.float64), 32, axis=-1)
    # |x - x_hat| <= s/2 for every clipped value inside [z, z + 3 s]
    zf = np.repeat(z16.astype(np.float64), 32, axis=-1)
    inside = (xc >= zf) & (xc <= zf + 3 * sf)
    assert np.all(np.abs(xc - xhat)[inside] <= sf[inside] * (0.5 + 1e-3))
    # outside the fp16-rounded range the error is at most the fp16 rounding of z / s
    assert np.all(np.abs(xc - xhat) <= sf * (0.5 + 1e-3) + np.abs(zf) * 2 ** -10 + 3 * sf * 2 ** -10)
    # every non-degenerate group uses both extreme codes
    g = codes.reshape(64, 4, 32)
    assert np.all(g.min(axis=-1) == 0) and np.all(g.max(axis=-1) == 3)
    assert codes.max() <= 3


def test_clip_applies():
    x = np.array([[-10.0] + [0.1 * i for i in range(31)]], dtype=F32)
    codes, s16, z16 = quantize_groups(x, F32(1.0), 32)
    assert np.float32(z16[0, 0]) == np.float32(np.float16(-1.0))
    assert codes[0, 0] == 0


def test_degenerate_group_scale_zero():
    x = np.full((1, 32), 0.7, dtype=F32)
    codes, s16, z16 = quantize_groups(x, F32(5.0), 32)
    assert s16[0, 0] == 0 and np.all(codes == 0)
    assert z16[0, 0] == np.float16(0.7)


def test_textbook_minmax_quantiser_when_unclipped():
    # with no clipping and exactly representable extremes the rule is the
    # textbook asymmetric min-max quantiser: round((x - min) / ((max - min)/3))
    x = np.array([[0.0, 3.0, 1.0, 2.0, 0.4, 0.6, 1.49, 1.51, 2.5 - 2 ** -10, 2.5 + 2 ** -10]
                  + [1.0] * 22], dtype=F32)
    codes, s16, z16 = quantize_groups(x, F32(np.inf), 32)
    assert float(s16[0, 0]) == 1.0 and float(z16[0, 0]) == 0.0
    want = np.rint(x[0].astype(np.float64) / 1.0).clip(0, 3)
    assert np.array_equal(codes[0], want.astype(np.uint8))


def test_half_to_even_ties():
    # (x - z)/s landing exactly on .5 rounds to even codes: 0.5 -> 0, 1.5 -> 2, 2.5 -> 2
    x = np.array([[0.0, 3.0, 0.5, 1.5, 2.5] + [1.0] * 27], dtype=F32)
    codes, _, _ = quantize_groups(x, F32(np.inf), 32)
    assert list(codes[0, :5]) == [0, 3, 0, 2, 2]
