"""GPU parity of long appends, whose tokens going straight to INT2 are rotated on
the tensor cores (bf16 hi + lo GEMM, fp32 accumulation) and quantised in the
tensor-memory epilogue, next to the per-token kernel for sink / ring tokens.

Same bar as the per-token path: rotated values within 1e-5 of the float64
rotation, codes / scales / zeros bit-exact when the oracle quantises the GPU's
rotated values, decode output within the attention tolerance."""

import numpy as np
import pytest
import torch

from bit_rotated_kv_oscar_gb300 import abi, build
from tests.gpu_harness import D, Layer
from tests.test_gpu_parity import check_decode, check_int2, check_window

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "the gpu-marked tests need a CUDA device"
    build.build()
    abi.lib()


@pytest.mark.parametrize("n", [388, 2000, 4095])
def test_prefill_single_request(n):
    layer = Layer(8, 2, 4, 128, 1, 4096, seed=100 + n)
    k, v = layer.draw(n)
    trace = layer.new_trace(4096)
    layer.append(0, k, v, trace)
    assert tuple(layer.device_state()[0][:2]) == (layer.len[0], layer.e[0])
    check_window(layer, 0)
    check_int2(layer, 0, trace)
    check_decode(layer, 1)
    assert layer.ctx.error_flags() == 0


def test_prefill_onto_an_existing_sequence():
    layer = Layer(32, 8, 4, 128, 1, 4096, seed=7)
    trace = layer.new_trace(4096)
    for n in (300, 1500, 1, 700):
        k, v = layer.draw(n)
        layer.append(0, k, v, trace)
        assert tuple(layer.device_state()[0][:2]) == (layer.len[0], layer.e[0])
    check_window(layer, 0)
    check_int2(layer, 0, trace)
    check_decode(layer, 1)
    assert layer.ctx.error_flags() == 0


def test_prefill_batch_of_requests():
    layer = Layer(16, 4, 16, 64, 3, 2048, seed=8)
    for b, n in enumerate((0, 50, 333)):
        if n:
            k, v = layer.draw(n)
            layer.append(b, k, v)
    k, v = layer.draw(3 * 900)
    layer.append_batch(k.view(3, 900, 4, D), v.view(3, 900, 4, D))
    for b in range(3):
        check_window(layer, b)
    check_decode(layer, 3)
    assert layer.ctx.error_flags() == 0


def test_prefill_fold_rv():
    layer = Layer(8, 2, 4, 64, 1, 2048, seed=9, fold_rv=1)
    k, v = layer.draw(1500)
    trace = layer.new_trace(2048)
    layer.append(0, k, v, trace)
    check_int2(layer, 0, trace)
    check_decode(layer, 1)


@pytest.mark.parametrize("frac", [0.15, 0.02, 1e-5])
def test_prefill_heavy_clipping(frac):
    """Clip values far below the calibrated ones: most groups have clipped
    extremes (and some are clipped whole), so codes of values beyond the clip
    must come out as the codes of the clip itself. At 1e-5 the values beyond
    the clip sit tens of thousands of scale steps past it, outside the 16-bit
    range in which the epilogue clamps two codes at once."""
    layer = Layer(8, 2, 4, 64, 1, 2048, seed=11 + int(frac * 100))
    for key in ("clip_K32", "clip_V32", "clip_K", "clip_V"):
        layer.cal[key] = layer.cal[key] * frac
    layer.ctx.load_rotations(layer.cal["R_K32"], layer.r_v32, layer.cal["clip_K32"], layer.cal["clip_V32"])
    k, v = layer.draw(1700)
    trace = layer.new_trace(2048)
    layer.append(0, k, v, trace)
    check_int2(layer, 0, trace)
    check_decode(layer, 1)
    assert layer.ctx.error_flags() == 0
