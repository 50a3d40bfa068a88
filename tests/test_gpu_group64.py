"""GPU parity of the pages' own constants as a preset: quantisation groups of 64
channels (K and V), sink 64, recent window 256, clips at the 96th / 92nd
percentile ("Juntos, AI Open-Sources OSCAR ...", section "El sistema de
servicio": S0 = 64, W = 256, default group GK = 64, typical cK = 0.96,
cV = 0.92).

Same bar as the group-32 layout: rotated values within 1e-5, codes / scales /
zeros bit-exact against the oracle quantising the GPU's rotated values, output
rel-L2 <= 2e-3 and max-abs <= 1e-2 against the float64 oracle."""

import numpy as np
import pytest
import torch

from bit_rotated_kv_oscar_gb300 import abi, build
from tests.gpu_harness import D, Layer
from tests.test_gpu_parity import check_decode, check_int2, check_window

pytestmark = pytest.mark.gpu

PRESET = dict(sink=64, recent=256, group=64, clip_percentiles=(96.0, 92.0))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "the gpu-marked tests need a CUDA device"
    build.build()
    abi.lib()


def pages_layer(hq, hkv, max_batch, max_tokens, seed, **kw):
    return Layer(hq, hkv, PRESET["sink"], PRESET["recent"], max_batch, max_tokens, seed=seed,
                 group=PRESET["group"], clip_percentiles=PRESET["clip_percentiles"], **kw)


def test_block_size_of_the_preset():
    cfg = abi.make_config(32, 8, 64, 256, 1, 16, group_size=64)
    pool, _ = abi.cache_bytes(cfg, 10)
    assert pool == 10 * 8 * 1280 == 10 * 8 * abi.page_block_bytes(64)


@pytest.mark.parametrize("n", [300, 2000, 4095])
def test_long_append_single_request(n):
    # long appends: the tensor-core prefill kernel for the INT2 tokens
    layer = pages_layer(8, 2, 1, 4096, seed=200 + n)
    k, v = layer.draw(n)
    trace = layer.new_trace(4096)
    layer.append(0, k, v, trace)
    assert tuple(layer.device_state()[0][:2]) == (layer.len[0], layer.e[0])
    check_window(layer, 0)
    check_int2(layer, 0, trace)
    check_decode(layer, 1)
    assert layer.ctx.error_flags() == 0


def test_token_by_token_appends_evict_through_the_ring():
    layer = pages_layer(32, 8, 1, 2048, seed=31)
    trace = layer.new_trace(2048)
    for n in (400, 1, 1, 257, 3, 1, 511):
        k, v = layer.draw(n)
        layer.append(0, k, v, trace)
        assert tuple(layer.device_state()[0][:2]) == (layer.len[0], layer.e[0])
    check_window(layer, 0)
    check_int2(layer, 0, trace)
    check_decode(layer, 1)
    assert layer.ctx.error_flags() == 0


@pytest.mark.parametrize("hq,hkv", [(8, 8), (32, 8), (64, 8), (4, 2)])
def test_gqa_group_sizes(hq, hkv):
    layer = pages_layer(hq, hkv, 1, 1500, seed=hq * 3 + hkv)
    k, v = layer.draw(1500)
    layer.append(0, k, v)
    check_decode(layer, 1)


@pytest.mark.parametrize("L", [1, 64, 320, 321, 337, 352, 353, 1000])
def test_lengths_around_the_window_and_page_edges(L):
    layer = pages_layer(8, 2, 1, 1024, seed=L)
    k, v = layer.draw(L)
    trace = layer.new_trace(1024)
    layer.append(0, k, v, trace)
    check_window(layer, 0)
    check_int2(layer, 0, trace)
    check_decode(layer, 1)


def test_ragged_batch_decode_steps():
    lengths = [330, 1700, 3000, 70, 905]
    layer = pages_layer(32, 8, len(lengths), 3100, seed=41, spikes=True)
    for b, n in enumerate(lengths):
        k, v = layer.draw(n)
        layer.append(b, k, v)
    check_decode(layer, len(lengths))
    for step in range(3):
        k, v = layer.draw(len(lengths))
        layer.append_batch(k.view(len(lengths), 1, 8, D), v.view(len(lengths), 1, 8, D))
    check_decode(layer, len(lengths), stream=77)


@pytest.mark.parametrize("splits", [1, 5, 64])
def test_split_counts(splits):
    layer = pages_layer(32, 8, 1, 5000, seed=51, num_splits=splits)
    k, v = layer.draw(5000)
    layer.append(0, k, v)
    check_decode(layer, 1)
