"""Pins of the oracle's restatement of the INT2 page-block byte layout."""

import numpy as np
import pytest

from oracle import (PAGE_BLOCK_BYTES, decode_page_block, encode_page_block, k_code_location,
                    meta_location, v_code_location)
from tests.conftest import read_golden


def test_hand_worked_locations():
    kinds = {"KS": (0, 0), "KZ": (0, 1), "VS": (1, 0), "VZ": (1, 1)}
    for kind, t, c, _, byte, bit in read_golden("page_block_locations.txt"):
        t, c, byte, bit = int(t), int(c), int(byte), int(bit)
        if kind == "K":
            assert k_code_location(t, c) == (byte, bit), (kind, t, c)
        elif kind == "V":
            assert v_code_location(t, c) == (byte, bit), (kind, t, c)
        else:
            kd, f = kinds[kind]
            assert meta_location(kd, t, c, f) == byte, (kind, t, c)


def test_layout_is_a_bijection():
    seen = set()
    for t in range(16):
        for c in range(128):
            for loc in (k_code_location(t, c), v_code_location(t, c)):
                byte, bit = loc
                assert 0 <= byte < 1024 and bit % 2 == 0
                seen.add(loc)
    assert len(seen) == 16 * 128 * 2 == 1024 * 4
    meta = set()
    for kind in range(2):
        for t in range(16):
            for gq in range(4):
                for f in range(2):
                    b = meta_location(kind, t, gq, f)
                    assert 1024 <= b < PAGE_BLOCK_BYTES and b % 2 == 0
                    meta.add(b)
    assert len(meta) == 256


@pytest.mark.parametrize("seed", range(3))
def test_round_trip(seed):
    rng = np.random.default_rng(seed)
    shape = (3, 2)
    kc = rng.integers(0, 4, size=shape + (16, 128), dtype=np.uint8)
    vc = rng.integers(0, 4, size=shape + (16, 128), dtype=np.uint8)
    ms = [rng.normal(size=shape + (16, 4)).astype(np.float16) for _ in range(4)]
    blk = encode_page_block(kc, vc, *ms)
    assert blk.shape == shape + (PAGE_BLOCK_BYTES,) and blk.dtype == np.uint8
    out = decode_page_block(blk)
    assert np.array_equal(out[0], kc) and np.array_equal(out[1], vc)
    for a, b in zip(out[2:], ms):
        assert np.array_equal(a.view(np.uint16), b.view(np.uint16))


def test_invalid_slots_stay_zero():
    kc = np.full((16, 128), 3, dtype=np.uint8)
    ms = [np.ones((16, 4), dtype=np.float16)] * 4
    valid = np.zeros(16, dtype=bool)
    valid[5] = True
    blk = encode_page_block(kc, kc, *ms, valid=valid)
    dk = decode_page_block(blk)
    assert np.all(dk[0][5] == 3) and dk[0].sum() == 3 * 128
    assert np.all(dk[2][5] == 1) and float(dk[2].astype(np.float32).sum()) == 4.0
