"""Byte layout of one INT2 page block, restated from the library header.

TEST INFRASTRUCTURE ONLY. The CUDA library defines how one page of 16 tokens
of one KV head is stored (1536 bytes: K codes, V codes, fp16 scale/zero
metadata); the header ``include/oscar.h`` states that format in words. This
module is an independent restatement of the same statement, used to read the
device pool back and to build expected bytes. It is specific to head_dim 128
and page size 16; the group size is 32 (the default, 1536-byte blocks) or 64
(1280-byte blocks).

Code of token t in channel c is a 2-bit field at (byte, bit) inside the block;
every 32-bit word is little-endian.

  K codes, bytes [0, 512): i = c // 16, r = c % 16, x = r // 8, b = (r % 8) // 2,
      hi = r % 2, a = t % 8, th = t // 8
      byte = 16 * (4a + b) + 4 * (2 th + x) + (16 hi + 2 i) // 8
  V codes, bytes [512, 1024): i = c // 16, r = c % 16, x = r // 8, a = r % 8,
      tt = t // 8, b = (t % 8) // 2, hi = t % 2
      byte = 512 + 16 * (4a + b) + 4 * (2 tt + x) + (16 hi + 2 i) // 8
  bit inside that byte = (16 hi + 2 i) % 8
  metadata, bytes [1024, 1024 + 128 NG) with NG = 128 / group groups per token,
      one fp16 each; a = t % 8, b = (t % 8) // 2, pair = t // 8, half = t % 2, group gq:
      K scale: 1024 + 4 NG a + 4 gq + 2 pair
      K zero:  1024 + 32 NG + 2 NG t + 2 gq
      V scale: 1024 + 64 NG + 16 (4 gq + b) + 4 pair + 2 half;  V zero: 8 bytes after it
"""

from __future__ import annotations

import numpy as np

PAGE = 16
HEAD_DIM = 128
GROUP = 32
N_GROUPS = HEAD_DIM // GROUP
PAGE_BLOCK_BYTES = 1536


def page_block_bytes(group: int = GROUP) -> int:
    """Bytes of one page block: 1024 code bytes, then 2 x 2 x 2 bytes of
    metadata per token and group."""
    return 1024 + 128 * (HEAD_DIM // group)


def k_code_location(t: int, c: int):
    """(byte, bit) of the K code of token slot t, channel c."""
    i, r = divmod(c, 16)
    x, r8 = divmod(r, 8)
    b, hi = divmod(r8, 2)
    a, th = t % 8, t // 8
    bitpos = 16 * hi + 2 * i
    return 16 * (4 * a + b) + 4 * (2 * th + x) + bitpos // 8, bitpos % 8


def v_code_location(t: int, c: int):
    """(byte, bit) of the V code of token slot t, channel c."""
    i, r = divmod(c, 16)
    x, a = divmod(r, 8)
    tt, t8 = divmod(t, 8)
    b, hi = divmod(t8, 2)
    bitpos = 16 * hi + 2 * i
    return 512 + 16 * (4 * a + b) + 4 * (2 * tt + x) + bitpos // 8, bitpos % 8


def meta_location(kind: int, t: int, gq: int, field: int, group: int = GROUP) -> int:
    """Byte offset of the fp16 scale (field 0) or zero (field 1) of group gq,
    token slot t, kind 0 = K / 1 = V."""
    ng = HEAD_DIM // group
    a, b, pair, half = t % 8, (t % 8) // 2, t // 8, t % 2
    if kind == 0 and field == 0:
        return 1024 + 4 * ng * a + 4 * gq + 2 * pair
    if kind == 0:
        return 1024 + 32 * ng + 2 * ng * t + 2 * gq
    return 1024 + 64 * ng + 16 * (4 * gq + b) + 8 * field + 4 * pair + 2 * half


def _tables(group: int = GROUP):
    ng = HEAD_DIM // group
    kb = np.empty((PAGE, HEAD_DIM), dtype=np.int64)
    ks = np.empty((PAGE, HEAD_DIM), dtype=np.int64)
    vb = np.empty((PAGE, HEAD_DIM), dtype=np.int64)
    vs = np.empty((PAGE, HEAD_DIM), dtype=np.int64)
    for t in range(PAGE):
        for c in range(HEAD_DIM):
            kb[t, c], ks[t, c] = k_code_location(t, c)
            vb[t, c], vs[t, c] = v_code_location(t, c)
    mb = np.empty((2, PAGE, ng, 2), dtype=np.int64)
    for kind in range(2):
        for t in range(PAGE):
            for gq in range(ng):
                for f in range(2):
                    mb[kind, t, gq, f] = meta_location(kind, t, gq, f, group)
    return kb, ks, vb, vs, mb


_TABLES = {}


def _tables_for(group: int):
    if group not in _TABLES:
        _TABLES[group] = _tables(group)
    return _TABLES[group]


_KB, _KS, _VB, _VS, _MB = _tables_for(GROUP)


def encode_page_block(k_codes, v_codes, k_scale, k_zero, v_scale, v_zero, valid=None, group: int = GROUP):
    """Build page blocks.

    k_codes / v_codes [..., 16, 128] uint8 in 0..3; scales / zeros [..., 16, 128 / group]
    float16; valid [..., 16] bool (invalid token slots are left zero).
    Returns uint8 [..., page_block_bytes(group)].
    """
    kb_, ks_, vb_, vs_, mb_ = _tables_for(group)
    ng, nbytes = HEAD_DIM // group, page_block_bytes(group)
    k_codes = np.asarray(k_codes, dtype=np.uint8)
    lead = k_codes.shape[:-2]
    if valid is None:
        valid = np.ones(lead + (PAGE,), dtype=bool)
    valid = np.asarray(valid, dtype=bool)
    out = np.zeros(lead + (nbytes,), dtype=np.uint32)
    flat = out.reshape(-1, nbytes)
    vmask = valid.reshape(-1, PAGE)
    for codes, byt, sh in ((k_codes, kb_, ks_), (np.asarray(v_codes, dtype=np.uint8), vb_, vs_)):
        cf = codes.reshape(-1, PAGE, HEAD_DIM).astype(np.uint32) * vmask[:, :, None]
        vals = cf << sh[None].astype(np.uint32)
        for n in range(flat.shape[0]):
            np.add.at(flat[n], byt.ravel(), vals[n].ravel())
    for kind, (sc, ze) in enumerate(((k_scale, k_zero), (v_scale, v_zero))):
        for f, arr in enumerate((sc, ze)):
            bits = np.asarray(arr, dtype=np.float16).view(np.uint16).reshape(-1, PAGE, ng)
            bits = bits.astype(np.uint32) * vmask[:, :, None]
            pos = mb_[kind, :, :, f]
            for n in range(flat.shape[0]):
                flat[n, pos.ravel()] = bits[n].ravel() & 0xFF
                flat[n, pos.ravel() + 1] = bits[n].ravel() >> 8
    return out.astype(np.uint8)


def decode_page_block(blocks, group: int = GROUP):
    """Inverse of encode_page_block: uint8 [..., page_block_bytes(group)] ->
    (k_codes, v_codes [..., 16, 128] uint8, k_scale, k_zero, v_scale, v_zero
    [..., 16, 128 / group] float16)."""
    kb_, ks_, vb_, vs_, mb_ = _tables_for(group)
    ng = HEAD_DIM // group
    blocks = np.asarray(blocks, dtype=np.uint8)
    assert blocks.shape[-1] == page_block_bytes(group)
    lead = blocks.shape[:-1]
    kc = (blocks[..., kb_] >> ks_) & 3
    vc = (blocks[..., vb_] >> vs_) & 3
    meta = []
    for kind in range(2):
        for f in range(2):
            pos = mb_[kind, :, :, f]
            lo = blocks[..., pos].astype(np.uint16)
            hi = blocks[..., pos + 1].astype(np.uint16)
            meta.append((lo | (hi << 8)).view(np.float16).reshape(lead + (PAGE, ng)))
    return (kc.astype(np.uint8), vc.astype(np.uint8), meta[0], meta[1], meta[2], meta[3])
