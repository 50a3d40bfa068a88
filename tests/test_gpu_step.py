"""GPU parity of the decode step (oscar_decode_step), whose one-token append runs
inside the decode call's launches.

Two twin layers (same seed, calibration and page order) take the same appends;
then one of them steps through oscar_quant_append + oscar_decode_attn, the other
through oscar_decode_step. The step must leave the same cache behind, byte for
byte (INT2 codes, scales and zeros, BF16 window rows, state), and its output
must meet the attention tolerance against the float64 oracle."""

import numpy as np
import pytest
import torch

from bit_rotated_kv_oscar_gb300 import abi, build
from tests.gpu_harness import D, MAX_ABS, REL_L2, Layer, rel_l2
from tests.test_gpu_parity import check_window

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "the gpu-marked tests need a CUDA device"
    build.build()
    abi.lib()


def _twins(*args, **kw):
    return Layer(*args, **kw), Layer(*args, **kw)


def _prefill(layers, lengths):
    for b, n in enumerate(lengths):
        if n:
            for layer in layers:
                layer.stream_id = 10 * b
                k, v = layer.draw(n)
                layer.append(b, k, v)


def _step_both(ref, stp, bsz, stream, aligned=True):
    """One step of every request: ref through the two calls, stp through the
    fused step; returns (q, o_ref, o_step) as numpy."""
    ref.stream_id = stp.stream_id = 1000 + stream
    k, v = ref.draw(bsz)
    stp.draw(bsz)
    q = ref.queries(bsz, stream)
    for layer in (ref, stp):
        for b in range(bsz):
            layer.cache.reserve(b, layer.len[b] + 1, upload=False)
        layer.cache.upload()
    kd = k.view(bsz, ref.hkv, D).to(torch.bfloat16).cuda()
    vd = v.view(bsz, ref.hkv, D).to(torch.bfloat16).cuda()
    qd = q.to(torch.bfloat16).cuda().contiguous()
    o_ref = torch.full((bsz, ref.hq, D), float("nan"), device="cuda")
    o_stp = torch.full((bsz, ref.hq, D), float("nan"), device="cuda")
    ref.ctx.quant_append(ref.cache.page_table, ref.cache.state, kd.view(bsz, 1, ref.hkv, D).contiguous(),
                         vd.view(bsz, 1, ref.hkv, D).contiguous(), bsz, 1)
    ref.ctx.decode_attn(qd, ref.cache.page_table, ref.cache.state, o_ref, bsz)
    if aligned:
        ks, vs = kd.contiguous(), vd.contiguous()
    else:
        # element-aligned views 2 bytes into larger buffers: the call falls back to
        # the append kernel followed by the decode
        kb = torch.zeros(kd.numel() + 8, dtype=torch.bfloat16, device="cuda")
        vb = torch.zeros(vd.numel() + 8, dtype=torch.bfloat16, device="cuda")
        kb[1:1 + kd.numel()] = kd.reshape(-1)
        vb[1:1 + vd.numel()] = vd.reshape(-1)
        ks, vs = kb[1:1 + kd.numel()], vb[1:1 + vd.numel()]
    stp.ctx.decode_step(stp.cache.page_table, stp.cache.state, qd, ks, vs, o_stp, bsz)
    torch.cuda.synchronize()
    for layer in (ref, stp):
        for b in range(bsz):
            layer._record(b, k[b:b + 1].view(1, ref.hkv, D), v[b:b + 1].view(1, ref.hkv, D))
    return q.numpy(), o_ref.cpu().numpy(), o_stp.cpu().numpy()


def _same_cache(ref, stp, b):
    assert np.array_equal(stp.device_state()[b], ref.device_state()[b])
    assert tuple(stp.device_state()[b][:2]) == (stp.len[b], stp.e[b])
    S, E = stp.sink, min(stp.e[b], stp.len[b])
    if E > S:
        for x, y in zip(ref.int2_codes(b, S, E), stp.int2_codes(b, S, E)):
            assert np.array_equal(np.ascontiguousarray(x).view(np.uint8), np.ascontiguousarray(y).view(np.uint8))
    check_window(stp, b)


def _check_output(stp, q, o, bsz):
    assert np.isfinite(o).all()
    for b in range(bsz):
        ref = stp.oracle_decode(q[b], b)
        r, m = rel_l2(o[b], ref), float(np.abs(o[b] - ref).max())
        assert r <= REL_L2 and m <= MAX_ABS, (b, r, m)


def _run(ref, stp, lengths, steps, check_every=1, aligned=True):
    bsz = len(lengths)
    _prefill((ref, stp), lengths)
    for s in range(steps):
        q, o_ref, o_stp = _step_both(ref, stp, bsz, s, aligned)
        for b in range(bsz):
            _same_cache(ref, stp, b)
        if s % check_every == 0 or s == steps - 1:
            _check_output(stp, q, o_stp, bsz)
            assert rel_l2(o_stp, o_ref) <= REL_L2
    assert ref.ctx.error_flags() == 0
    assert stp.ctx.error_flags() == 0


def test_step_evicts_through_the_ring_and_crosses_pages():
    # full ring from the start: every step quantises the entry the new token replaces
    ref, stp = _twins(32, 8, 4, 128, 1, 4096, seed=41)
    _run(ref, stp, [1000], 24, check_every=4)


def test_step_from_an_empty_request():
    # sink filling, ring filling, then evictions
    ref, stp = _twins(8, 2, 4, 16, 1, 512, seed=42)
    _run(ref, stp, [0], 40, check_every=5)


@pytest.mark.parametrize("sink,recent", [(0, 128), (4, 1), (7, 33), (64, 256)])
def test_step_window_sizes(sink, recent):
    ref, stp = _twins(16, 4, sink, recent, 1, 2048, seed=43 + sink + recent)
    _run(ref, stp, [sink + recent + 300], 6, check_every=2)


@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 8), (64, 8), (4, 2)])
def test_step_gqa_group_sizes(hq, hkv):
    ref, stp = _twins(hq, hkv, 4, 128, 1, 1024, seed=44 + hq)
    _run(ref, stp, [700], 4, check_every=1)


def test_step_ragged_batch():
    # an empty request, one in its sink, one with the ring filling, two evicting
    ref, stp = _twins(16, 4, 4, 64, 5, 2048, seed=45)
    _run(ref, stp, [0, 2, 40, 333, 1500], 8, check_every=3)


def test_step_group64_and_fold_rv():
    ref, stp = _twins(16, 4, 4, 64, 2, 1024, seed=46, group=64)
    _run(ref, stp, [500, 69], 5, check_every=2)
    ref, stp = _twins(16, 4, 4, 64, 1, 1024, seed=47, fold_rv=1)
    _run(ref, stp, [600], 5, check_every=2)


@pytest.mark.parametrize("splits", [1, 37])
def test_step_split_counts(splits):
    ref, stp = _twins(32, 8, 4, 128, 1, 4096, seed=48, num_splits=splits)
    _run(ref, stp, [3000], 3)


def test_step_unaligned_inputs_take_the_two_kernel_path():
    ref, stp = _twins(8, 2, 4, 32, 2, 512, seed=49)
    _run(ref, stp, [100, 37], 4, aligned=False)


def test_step_statuses():
    cfg = abi.make_config(8, 2, 4, 64, 2, 64)
    ctx = abi.Context(cfg)
    q = torch.zeros(2, 8, D, dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros(2, 2, D, dtype=torch.bfloat16, device="cuda")
    o = torch.zeros(2, 8, D, device="cuda")
    pt = torch.zeros(2, 64, dtype=torch.int32, device="cuda")
    st = torch.zeros(2, 4, dtype=torch.int32, device="cuda")
    with pytest.raises(abi.OscarError) as e:
        ctx.decode_step(pt, st, q, kv, kv, o, 2)
    assert e.value.status == -2          # rotations not loaded
    eye = np.broadcast_to(np.eye(D, dtype=np.float32), (2, D, D))
    ctx.load_rotations(eye, eye, np.ones(2, np.float32), np.ones(2, np.float32))
    with pytest.raises(abi.OscarError) as e:
        ctx.decode_step(pt, st, q, kv, kv, o, 2)
    assert e.value.status == -6          # no cache bound
    from bit_rotated_kv_oscar_gb300.cache import PagedCache
    PagedCache(ctx, 64, device="cuda")
    with pytest.raises(abi.OscarError) as e:
        ctx.decode_step(pt, st, q, kv, kv, o, 3)
    assert e.value.status == -3          # batch above max_batch
    with pytest.raises(abi.OscarError) as e:
        ctx.decode_step(pt, st, q, None, kv, o, 2)
    assert e.value.status == -1
    with pytest.raises(abi.OscarError) as e:
        ctx.decode_step(pt, st, None, kv, kv, o, 2)
    assert e.value.status == -1
    torch.cuda.synchronize()
    assert ctx.error_flags() == 0


def test_step_bad_page_id_raises_a_flag_not_a_fault():
    # a full ring: the step quantises position L - recent = 536 into page 33
    layer = Layer(8, 2, 4, 64, 1, 1024, seed=53)
    k, v = layer.draw(600)
    layer.append(0, k, v)
    assert layer.ctx.error_flags() == 0
    layer.cache.reserve(0, 601)
    layer.cache.page_table[0, 33] = 10 ** 6
    k1, v1 = layer.draw(1)
    q = layer.queries(1, 4).to(torch.bfloat16).cuda()
    o = torch.full((1, 8, D), float("nan"), device="cuda")
    layer.ctx.decode_step(layer.cache.page_table, layer.cache.state, q, k1.to(torch.bfloat16).cuda(),
                          v1.to(torch.bfloat16).cuda(), o, 1)
    torch.cuda.synchronize()
    assert torch.isfinite(o).all()
    assert layer.ctx.error_flags() & abi.FLAG_BAD_PAGE_ID
    assert tuple(layer.device_state()[0][:2]) == (601, 537)


def test_step_bad_state_raises_a_flag():
    layer = Layer(8, 2, 4, 64, 1, 1024, seed=54)
    k, v = layer.draw(300)
    layer.append(0, k, v)
    layer.cache.state[0] = torch.tensor([300, 2, 0, 0], dtype=torch.int32)  # int2_end below the sink
    q = layer.queries(1, 5).to(torch.bfloat16).cuda()
    o = torch.full((1, 8, D), float("nan"), device="cuda")
    kd = k[:1].to(torch.bfloat16).cuda()
    layer.ctx.decode_step(layer.cache.page_table, layer.cache.state, q, kd, kd, o, 1)
    torch.cuda.synchronize()
    assert torch.all(o == 0)
    assert layer.ctx.error_flags() & abi.FLAG_BAD_STATE
    assert tuple(layer.device_state()[0][:2]) == (300, 2)
