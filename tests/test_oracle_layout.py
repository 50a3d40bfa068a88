"""Pins of the oracle's restatement of the INT2 page-block byte layout."""

import numpy as np
import pytest

from oracle import (PAGE_BLOCK_BYTES, decode_page_block, encode_page_block, k_code_location,
                    meta_location, page_block_bytes, v_code_location)
from tests.conftest import read_golden


@pytest.mark.parametrize("group,fixture", [(32, "page_block_locations.txt"),
                                           (64, "page_block_locations_g64.txt")])
def test_hand_worked_locations(group, fixture):
    kinds = {"KS": (0, 0), "KZ": (0, 1), "VS": (1, 0), "VZ": (1, 1)}
    for kind, t, c, _, byte, bit in read_golden(fixture):
        t, c, byte, bit = int(t), int(c), int(byte), int(bit)
        if kind == "K":
            assert k_code_location(t, c) == (byte, bit), (kind, t, c)
        elif kind == "V":
            assert v_code_location(t, c) == (byte, bit), (kind, t, c)
        else:
            kd, f = kinds[kind]
            assert meta_location(kd, t, c, f, group) == byte, (kind, t, c)


@pytest.mark.parametrize("group", [32, 64])
def test_layout_is_a_bijection(group):
    seen = set()
    for t in range(16):
        for c in range(128):
            for loc in (k_code_location(t, c), v_code_location(t, c)):
                byte, bit = loc
                assert 0 <= byte < 1024 and bit % 2 == 0
                seen.add(loc)
    assert len(seen) == 16 * 128 * 2 == 1024 * 4
    ng = 128 // group
    assert page_block_bytes(group) == 1024 + 128 * ng and page_block_bytes(32) == PAGE_BLOCK_BYTES
    meta = set()
    for kind in range(2):
        for t in range(16):
            for gq in range(ng):
                for f in range(2):
                    b = meta_location(kind, t, gq, f, group)
                    assert 1024 <= b < page_block_bytes(group) and b % 2 == 0
                    meta.add(b)
    assert len(meta) == 64 * ng  # every metadata byte pair used once


@pytest.mark.parametrize("seed,group", [(0, 32), (1, 32), (2, 32), (0, 64), (1, 64)])
def test_round_trip(seed, group):
    rng = np.random.default_rng(seed)
    shape = (3, 2)
    ng = 128 // group
    kc = rng.integers(0, 4, size=shape + (16, 128), dtype=np.uint8)
    vc = rng.integers(0, 4, size=shape + (16, 128), dtype=np.uint8)
    ms = [rng.normal(size=shape + (16, ng)).astype(np.float16) for _ in range(4)]
    blk = encode_page_block(kc, vc, *ms, group=group)
    assert blk.shape == shape + (page_block_bytes(group),) and blk.dtype == np.uint8
    out = decode_page_block(blk, group=group)
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
