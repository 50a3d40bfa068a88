"""The BF16 window's CTAs cover 64 tokens each while they are few and 160 while
they are many (one call's choice); both against the float64 oracle at window
sizes around the 160-token chunk (132, 160, 161 and 320 tokens), with 8 KV heads
at one request (64-token chunks) and at four (160-token chunks)."""

import pytest
import torch

from bit_rotated_kv_oscar_gb300 import abi, build
from tests.gpu_harness import Layer
from tests.test_gpu_parity import check_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "the gpu-marked tests need a CUDA device"
    build.build()
    abi.lib()


@pytest.mark.parametrize("sink,recent", [(4, 128), (4, 156), (4, 157), (64, 256)])
@pytest.mark.parametrize("batch", [1, 4])
def test_window_chunks(sink, recent, batch):
    layer = Layer(32, 8, sink, recent, batch, 1400, seed=60 + recent + batch)
    lengths = [1300, 700, sink + recent + 5, 90][:batch]
    for b, n in enumerate(lengths):
        k, v = layer.draw(n)
        layer.append(b, k, v)
    check_decode(layer, batch, stream=61)
    # one more token per request: the ring slides by one
    k, v = layer.draw(batch)
    layer.append_batch(k.view(batch, 1, 8, 128), v.view(batch, 1, 8, 128))
    check_decode(layer, batch, stream=62)
    assert layer.ctx.error_flags() == 0
