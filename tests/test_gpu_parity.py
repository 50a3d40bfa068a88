"""GPU parity of the write path and the fused decode attention against the oracle.

Every case drives the CUDA library through its C ABI and compares with the
float64 oracle on the same seeded inputs:
  * rotated values: |gpu - oracle| <= 1e-5 * max |oracle| per token-head vector;
  * 2-bit codes, fp16 scales and zeros: bit-exact when the oracle quantises the
    GPU's own rotated float32 values (the quantiser is a float decision, taken
    by both sides in float32), and equal except at rounding ties when the
    oracle quantises its own float64 rotation;
  * BF16 sink / recent windows: bit-exact copies;
  * attention output: rel-L2 <= 2e-3 and max-abs <= 1e-2 against the float64
    oracle built from the same tokens.
"""

import numpy as np
import pytest
import torch

import oracle
from bit_rotated_kv_oscar_gb300 import abi, build
from tests.gpu_harness import D, MAX_ABS, REL_L2, ROT_REL, Layer, rel_l2

pytestmark = pytest.mark.gpu

F32 = np.float32


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "the gpu-marked tests need a CUDA device"
    build.build()
    abi.lib()


# ---------------------------------------------------------------------------
# checks
# ---------------------------------------------------------------------------

def check_window(layer, b):
    L, E, S, W = layer.len[b], layer.e[b], layer.sink, layer.recent
    w = layer.window_rows(b)
    for pos in range(min(S, L)):
        assert np.array_equal(w[:, 0, pos], layer.k_host[b][pos]), pos
        assert np.array_equal(w[:, 1, pos], layer.v_host[b][pos]), pos
    for pos in range(max(E, S), L):
        slot = S + pos % W
        assert np.array_equal(w[:, 0, slot], layer.k_host[b][pos]), pos
        assert np.array_equal(w[:, 1, slot], layer.v_host[b][pos]), pos


def check_int2(layer, b, trace, lo=None, hi=None):
    """Codes of positions [lo, hi) (default the whole INT2 region) against the oracle."""
    S, E = layer.sink, layer.e[b]
    lo = S if lo is None else lo
    hi = E if hi is None else hi
    if hi <= lo:
        return
    dec = layer.int2_codes(b, lo, hi)
    tr = trace[0, lo:hi].cpu().numpy()
    assert not np.isnan(tr).any(), "some INT2 position was never quantised"
    for kind in range(2):
        x = (layer.k_host[b] if kind == 0 else layer.v_host[b])[lo:hi].astype(np.float64)
        r = (layer.cal["R_K32"] if kind == 0 else layer.r_v32).astype(np.float64)
        clip = (layer.cal["clip_K32"] if kind == 0 else layer.cal["clip_V32"]).reshape(1, -1, 1)
        ref = np.einsum("nhi,hij->nhj", x, r)
        got = tr[:, :, kind]
        err = np.abs(got - ref).max(-1)
        assert np.all(err <= ROT_REL * np.abs(ref).max(-1)), float((err / np.abs(ref).max(-1)).max())
        codes, s16, z16 = dec[kind], dec[2 + 2 * kind], dec[3 + 2 * kind]
        # (1) the oracle quantises the GPU's rotated float32 values: bit-exact
        oc, os_, oz = oracle.quantize_groups(got.astype(F32), clip.astype(F32), layer.group)
        assert np.array_equal(codes, oc)
        assert np.array_equal(s16.view(np.uint16), os_.view(np.uint16))
        assert np.array_equal(z16.view(np.uint16), oz.view(np.uint16))
        # (2) the oracle quantises its own rotation: equal away from rounding ties
        ic, is_, iz = oracle.quantize_groups(ref.astype(F32), clip.astype(F32), layer.group)
        mism = ic != codes
        assert mism.mean() < 1e-3, mism.mean()
        if mism.any():
            sf = np.repeat(is_.astype(np.float64), layer.group, axis=-1)
            zf = np.repeat(iz.astype(np.float64), layer.group, axis=-1)
            xc = np.clip(ref.astype(F32), -clip, clip).astype(np.float64)
            u = (xc - zf) / np.where(sf == 0, 1, sf)
            same_meta = (np.repeat(is_, layer.group, -1) == np.repeat(os_, layer.group, -1)) & \
                        (np.repeat(iz, layer.group, -1) == np.repeat(oz, layer.group, -1))
            # near a tie: within the rotation error bound (in units of the scale)
            # of a .5 boundary, and never closer than 1e-3 (the float32 steps)
            near = np.maximum(1e-3, ROT_REL * np.abs(ref).max(-1, keepdims=True) / np.where(sf == 0, 1, sf))
            tie = np.abs(u - np.floor(u) - 0.5) < near
            assert np.all(tie[mism & same_meta]), "code mismatch away from a rounding tie"


def check_decode(layer, bsz, stream=77):
    q = layer.queries(bsz, stream)
    o = layer.decode(q)
    assert np.isfinite(o).all()
    worst = (0.0, 0.0)
    for b in range(bsz):
        ref = layer.oracle_decode(q[b].numpy(), b)
        r, m = rel_l2(o[b], ref), float(np.abs(o[b] - ref).max())
        worst = (max(worst[0], r), max(worst[1], m))
        assert r <= REL_L2 and m <= MAX_ABS, (b, r, m)
    return worst


# ---------------------------------------------------------------------------
# write path
# ---------------------------------------------------------------------------

def test_prefill_tiny_single_layer():
    # single layer, 2 query heads / 1 KV head, 1024 tokens, sink 4, recent 64
    layer = Layer(2, 1, 4, 64, 1, 1024, seed=0, n_cal=2048, shuffled=False)
    k, v = layer.draw(1024)
    trace = layer.new_trace(1024)
    layer.append(0, k, v, trace)
    assert tuple(layer.device_state()[0][:2]) == (1024, 960)
    check_window(layer, 0)
    check_int2(layer, 0, trace)
    check_decode(layer, 1)
    assert layer.ctx.error_flags() == 0


def test_incremental_appends_evict_through_the_ring():
    layer = Layer(32, 8, 4, 128, 1, 4096, seed=5)
    trace = layer.new_trace(4096)
    for n in (1000, 1, 1, 500, 127, 129, 1, 1372, 3):
        k, v = layer.draw(n)
        layer.append(0, k, v, trace)
        assert tuple(layer.device_state()[0][:2]) == (layer.len[0], layer.e[0])
    check_window(layer, 0)
    check_int2(layer, 0, trace)
    check_decode(layer, 1)
    assert layer.ctx.error_flags() == 0


def test_decode_steps_slide_the_window():
    layer = Layer(8, 2, 4, 64, 2, 2048, seed=6)
    for b in range(2):
        k, v = layer.draw(300 + 211 * b)
        layer.append(b, k, v)
    for step in range(40):
        k, v = layer.draw(2)
        layer.append_batch(k.view(2, 1, 2, D), v.view(2, 1, 2, D))
        if step % 13 == 0:
            check_decode(layer, 2, stream=1000 + step)
    for b in range(2):
        check_window(layer, b)
    assert [tuple(s[:2]) for s in layer.device_state()] == [(340, 276), (551, 487)]


# ---------------------------------------------------------------------------
# read path
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 8), (32, 8), (64, 8), (4, 2)])
def test_gqa_group_sizes(hq, hkv):
    layer = Layer(hq, hkv, 4, 128, 1, 777, seed=hq + hkv)
    k, v = layer.draw(777)
    layer.append(0, k, v)
    check_decode(layer, 1)


@pytest.mark.parametrize("L", [1, 3, 4, 5, 100, 132, 133, 135, 147, 148, 149, 163, 164, 165, 420])
def test_lengths_around_the_window_and_page_edges(L):
    layer = Layer(8, 2, 4, 128, 1, 512, seed=L)
    k, v = layer.draw(L)
    trace = layer.new_trace(512)
    layer.append(0, k, v, trace)
    check_window(layer, 0)
    check_int2(layer, 0, trace)
    check_decode(layer, 1)


@pytest.mark.parametrize("sink,recent", [(0, 128), (16, 128), (64, 256), (4, 1), (7, 33)])
def test_window_sizes(sink, recent):
    layer = Layer(8, 2, sink, recent, 1, 1200, seed=sink * 7 + recent)
    trace = layer.new_trace(1200)
    for n in (700, 1, 300, 17):
        k, v = layer.draw(n)
        layer.append(0, k, v, trace)
    check_window(layer, 0)
    check_int2(layer, 0, trace)
    check_decode(layer, 1)


def test_empty_request_gives_zero():
    layer = Layer(8, 2, 4, 128, 2, 512, seed=3)
    k, v = layer.draw(300)
    layer.append(1, k, v)
    q = layer.queries(2, 5)
    o = layer.decode(q)
    assert np.all(o[0] == 0)
    ref = layer.oracle_decode(q[1].numpy(), 1)
    assert rel_l2(o[1], ref) <= REL_L2


def test_ragged_batch_shuffled_pool():
    lengths = [200, 1500, 3000, 17, 900, 2222]
    layer = Layer(32, 8, 4, 128, len(lengths), 3100, seed=11, spikes=True)
    for b, n in enumerate(lengths):
        k, v = layer.draw(n)
        layer.append(b, k, v)
    check_decode(layer, len(lengths))
    for step in range(3):
        k, v = layer.draw(len(lengths))
        layer.append_batch(k.view(len(lengths), 1, 8, D), v.view(len(lengths), 1, 8, D))
    check_decode(layer, len(lengths), stream=99)


@pytest.mark.parametrize("splits", [1, 2, 7, 64, 200])
def test_split_counts(splits):
    layer = Layer(32, 8, 4, 128, 1, 5000, seed=21, num_splits=splits)
    k, v = layer.draw(5000)
    layer.append(0, k, v)
    check_decode(layer, 1)


@pytest.mark.parametrize("splits", [1, 2])
def test_long_splits(splits):
    # 12000 tokens in one split of 750 pages (more than 64 per warp: the kernel
    # instance for long splits, page ids past the first 64 loaded on use) and in
    # two splits of 375 pages
    layer = Layer(32, 8, 4, 128, 1, 12000, seed=23, num_splits=splits)
    k, v = layer.draw(12000)
    layer.append(0, k, v)
    check_decode(layer, 1)


def test_fold_rv_keeps_values_rotated():
    layer = Layer(8, 2, 4, 64, 1, 1000, seed=31, fold_rv=1)
    k, v = layer.draw(1000)
    trace = layer.new_trace(1000)
    layer.append(0, k, v, trace)
    check_int2(layer, 0, trace)
    check_decode(layer, 1)


def test_shared_prefix_fork():
    layer = Layer(16, 4, 4, 128, 3, 3000, seed=41)
    k, v = layer.draw(2000)
    layer.append(0, k, v)
    q0 = layer.queries(3, 8)
    before = layer.decode(q0)[0]
    for dst in (1, 2):
        layer.cache.fork(0, dst, 1024)
        layer.k_host[dst] = layer.k_host[0][:1024].copy()
        layer.v_host[dst] = layer.v_host[0][:1024].copy()
        layer.len[dst], layer.e[dst] = 1024, 1024
        assert tuple(layer.device_state()[dst][:2]) == (1024, 1024)
    for dst, n in ((1, 300), (2, 77)):
        k, v = layer.draw(n)
        layer.append(dst, k, v)
    check_decode(layer, 3, stream=8)
    # appends to the forks left the shared pages alone
    assert np.array_equal(layer.decode(q0)[0], before)
    assert (layer.cache.page_table_host[1, :64] == layer.cache.page_table_host[0, :64]).all()


# ---------------------------------------------------------------------------
# errors: statuses from the host, flags from the device, never a fault
# ---------------------------------------------------------------------------

def test_status_codes():
    cfg = abi.make_config(8, 2, 4, 64, 2, 64)
    ctx = abi.Context(cfg)
    q = torch.zeros(2, 8, D, dtype=torch.bfloat16, device="cuda")
    o = torch.zeros(2, 8, D, device="cuda")
    pt = torch.zeros(2, 64, dtype=torch.int32, device="cuda")
    st = torch.zeros(2, 4, dtype=torch.int32, device="cuda")
    with pytest.raises(abi.OscarError) as e:
        ctx.decode_attn(q, pt, st, o, 2)
    assert e.value.status == -2
    eye = np.broadcast_to(np.eye(D, dtype=np.float32), (2, D, D))
    ctx.load_rotations(eye, eye, np.ones(2, np.float32), np.ones(2, np.float32))
    with pytest.raises(abi.OscarError) as e:
        ctx.decode_attn(q, pt, st, o, 2)
    assert e.value.status == -6
    with pytest.raises(abi.OscarError) as e:
        ctx.load_rotations(eye, eye, np.zeros(2, np.float32), np.ones(2, np.float32))
    assert e.value.status == -1
    from bit_rotated_kv_oscar_gb300.cache import PagedCache
    PagedCache(ctx, 64, device="cuda")
    with pytest.raises(abi.OscarError) as e:
        ctx.decode_attn(q, pt, st, o, 3)
    assert e.value.status == -3
    with pytest.raises(abi.OscarError) as e:
        ctx.decode_attn(None, pt, st, o, 2)
    assert e.value.status == -1


def test_bad_page_ids_raise_a_flag_not_a_fault():
    layer = Layer(8, 2, 4, 64, 1, 1024, seed=51)
    k, v = layer.draw(600)
    layer.append(0, k, v)
    assert layer.ctx.error_flags() == 0
    layer.cache.page_table[0, 3] = 10 ** 6
    layer.cache.page_table[0, 5] = -7
    o = layer.decode(layer.queries(1, 3))
    assert np.isfinite(o).all()
    assert layer.ctx.error_flags() & abi.FLAG_BAD_PAGE_ID
    k, v = layer.draw(100)
    layer.cache.reserve(0, 700)
    layer.cache.page_table[0, 35] = 10 ** 7  # positions 560..575, quantised by this append
    kd = k.to(torch.bfloat16).cuda()
    layer.ctx.quant_append(layer.cache.page_table, layer.cache.state, kd, kd, 1, 100)
    assert layer.ctx.error_flags() & abi.FLAG_BAD_PAGE_ID
    assert layer.ctx.error_flags() == 0  # cleared by the previous read


def test_bad_state_raises_a_flag():
    layer = Layer(8, 2, 4, 64, 1, 1024, seed=52)
    k, v = layer.draw(300)
    layer.append(0, k, v)
    layer.cache.state[0] = torch.tensor([300, 2, 0, 0], dtype=torch.int32)  # int2_end below the sink
    o = layer.decode(layer.queries(1, 3))
    assert np.all(o == 0)
    kd = k[:1].to(torch.bfloat16).cuda()
    layer.ctx.quant_append(layer.cache.page_table, layer.cache.state, kd, kd, 1, 1)
    assert layer.ctx.error_flags() & abi.FLAG_BAD_STATE
    assert tuple(layer.device_state()[0][:2]) == (300, 2)
