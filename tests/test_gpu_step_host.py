"""oscar_decode_step_host (one serving step with host-side inputs and output)
against the same step on device tensors (oscar_decode_step, or, for inputs that
are not 16-byte aligned, oscar_quant_append + oscar_decode_attn, which the step
then runs): bit-identical outputs and states over steps that evict through the
ring and cross page boundaries, with page-locked host buffers (read and written
by the kernels in place) and with pageable ones (copied through the staging
buffer), the resulting cache against the float64 oracle, and the argument
statuses."""

import ctypes

import pytest
import torch

from bit_rotated_kv_oscar_gb300 import abi, build
from tests.gpu_harness import D, Layer
from tests.test_gpu_parity import check_decode

pytestmark = pytest.mark.gpu

INVALID_ARG, OUT_OF_RANGE = -1, -3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "the gpu-marked tests need a CUDA device"
    build.build()
    abi.lib()


def _vp(t, offset=0):
    return ctypes.c_void_p(t.data_ptr() + offset)


@pytest.mark.parametrize("group,pinned,fold_rv,offset",
                         [(32, True, 0, 0), (64, True, 0, 0), (32, False, 0, 0), (32, True, 1, 0),
                          (64, True, 0, 2)])
def test_step_host_matches_device_step(group, pinned, fold_rv, offset):
    """offset: bytes the inputs start after a 16-byte boundary of the page-locked
    buffer (2: the step runs the append kernel, which reads them with plain
    loads, then the decode)."""
    bsz, hq, hkv = 3, 16, 4
    a = Layer(hq, hkv, 4, 64, bsz, 1400, seed=21, group=group, fold_rv=fold_rv)
    b = Layer(hq, hkv, 4, 64, bsz, 1400, seed=21, group=group, fold_rv=fold_rv)
    for r, n in enumerate((700, 300, 65)):
        k, v = a.draw(n)
        a.append(r, k, v)
        b.append(r, k, v)
    dev = a.device
    nq, nk = bsz * hq * D, bsz * hkv * D
    d_qkv = torch.empty(nq + 2 * nk, dtype=torch.bfloat16, device=dev)
    o_a = torch.empty(bsz, hq, D, device=dev)
    o_b = torch.empty_like(o_a)
    h_o = torch.empty(bsz, hq, D)
    if pinned:
        h_o = h_o.pin_memory()
    for i in range(20):  # ring evictions every step, page boundaries every 16
        q = a.queries(bsz, 300 + i)
        k, v = a.draw(bsz)
        for layer in (a, b):
            for r in range(bsz):
                layer.cache.reserve(r, layer.len[r] + 1, upload=False)
            layer.cache.upload()
        qd = q.to(torch.bfloat16).to(dev).contiguous()
        kd = k.to(torch.bfloat16).reshape(bsz, 1, hkv, D).to(dev).contiguous()
        vd = v.to(torch.bfloat16).reshape(bsz, 1, hkv, D).to(dev).contiguous()
        if offset % 16 == 0:
            a.ctx.decode_step(a.cache.page_table, a.cache.state, qd, kd, vd, o_a, bsz)
        else:
            a.ctx.quant_append(a.cache.page_table, a.cache.state, kd, vd, bsz, 1)
            a.ctx.decode_attn(qd, a.cache.page_table, a.cache.state, o_a, bsz)
        h_qkv = torch.cat([qd.reshape(-1), kd.reshape(-1), vd.reshape(-1)]).cpu()
        if pinned:
            pad = offset // 2
            buf = torch.zeros(h_qkv.numel() + pad, dtype=torch.bfloat16).pin_memory()
            buf[pad:].copy_(h_qkv)
            h_qkv = buf[pad:]
            assert h_qkv.data_ptr() % 16 == offset
            b.ctx.decode_step_host(b.cache.page_table, b.cache.state, h_qkv, None, None, h_o, bsz)
        else:
            b.ctx.decode_step_host(b.cache.page_table, b.cache.state, h_qkv, d_qkv, o_b, h_o, bsz)
        torch.cuda.synchronize()
        assert torch.equal(o_a.cpu(), h_o), i
        if not pinned:
            assert torch.equal(o_a, o_b), i
        assert torch.equal(a.cache.state, b.cache.state), i
        for layer in (a, b):
            for r in range(bsz):
                layer._record(r, k[r:r + 1], v[r:r + 1])
    assert torch.equal(a.cache.window, b.cache.window)
    check_decode(b, bsz, stream=77)
    assert a.ctx.error_flags() == 0 and b.ctx.error_flags() == 0


def test_step_host_statuses():
    layer = Layer(8, 2, 4, 32, 1, 256, seed=3)
    k, v = layer.draw(40)
    layer.append(0, k, v)
    d = torch.empty(8 * D + 4 * D + 16, dtype=torch.bfloat16, device="cuda")
    o = torch.empty(1, 8, D, device="cuda")
    h = torch.zeros(8 * D + 4 * D, dtype=torch.bfloat16)          # pageable: copies
    h_o = torch.empty(1, 8, D)
    lib, ctx = abi.lib(), layer.ctx.handle
    pt, st = _vp(layer.cache.page_table), _vp(layer.cache.state)
    assert lib.oscar_decode_step_host(ctx, pt, st, None, _vp(d), _vp(o), _vp(h_o), 1, None) == INVALID_ARG
    assert lib.oscar_decode_step_host(ctx, pt, st, _vp(h), _vp(d), _vp(o), None, 1, None) == INVALID_ARG
    assert lib.oscar_decode_step_host(ctx, pt, st, _vp(h), None, _vp(o), _vp(h_o), 1, None) == INVALID_ARG
    assert lib.oscar_decode_step_host(ctx, pt, st, _vp(h), _vp(d), None, _vp(h_o), 1, None) == INVALID_ARG
    assert lib.oscar_decode_step_host(ctx, pt, st, _vp(h), _vp(d, 2), _vp(o), _vp(h_o), 1, None) == INVALID_ARG
    assert "aligned" in layer.ctx.last_error()
    assert lib.oscar_decode_step_host(ctx, pt, st, _vp(h), _vp(d), _vp(o), _vp(h_o), 0, None) == INVALID_ARG
    assert lib.oscar_decode_step_host(ctx, pt, st, _vp(h), _vp(d), _vp(o), _vp(h_o), 2, None) == OUT_OF_RANGE
    assert lib.oscar_decode_step_host(None, pt, st, _vp(h), _vp(d), _vp(o), _vp(h_o), 1, None) == INVALID_ARG
    torch.cuda.synchronize()
    # nothing was launched by the rejected calls
    assert tuple(layer.device_state()[0][:2]) == (layer.len[0], layer.e[0])
    # page-locked buffers need neither the staging buffer nor the device output
    hp, hop = h.pin_memory(), h_o.pin_memory()
    layer.cache.reserve(0, layer.len[0] + 1)
    assert lib.oscar_decode_step_host(ctx, pt, st, _vp(hp), None, None, _vp(hop), 1, None) == 0
    torch.cuda.synchronize()
    assert tuple(layer.device_state()[0][:2]) == (layer.len[0] + 1, max(layer.e[0], layer.len[0] + 1 - 32))
    assert torch.isfinite(hop).all()
    assert layer.ctx.error_flags() == 0


def test_decode_query_needs_only_element_alignment():
    # q two bytes past a 16-byte boundary gives the same output as an aligned q
    layer = Layer(16, 4, 4, 64, 2, 900, seed=8)
    for r, n in enumerate((500, 130)):
        k, v = layer.draw(n)
        layer.append(r, k, v)
    q = layer.queries(2, 5).to(torch.bfloat16).cuda().contiguous()
    buf = torch.zeros(q.numel() + 1, dtype=torch.bfloat16, device="cuda")
    buf[1:].copy_(q.reshape(-1))
    q_off = buf[1:].view(q.shape)
    assert q_off.data_ptr() % 16 == 2
    o1 = torch.empty(2, 16, D, device="cuda")
    o2 = torch.empty_like(o1)
    layer.ctx.decode_attn(q, layer.cache.page_table, layer.cache.state, o1, 2)
    layer.ctx.decode_attn(q_off, layer.cache.page_table, layer.cache.state, o2, 2)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)
    assert layer.ctx.error_flags() == 0
