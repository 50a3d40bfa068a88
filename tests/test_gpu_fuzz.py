"""Randomised GPU parity sweep: seeded random shapes and histories through the
whole write and read path, each checked against the float64 oracle like the
hand-picked cases (codes bit-exact against the oracle quantising the GPU's
rotated values, rotated values within 1e-5, output rel-L2 <= 2e-3 and max-abs
<= 1e-2). Every draw is reproducible from its case number."""

import numpy as np
import pytest
import torch

from bit_rotated_kv_oscar_gb300 import abi, build
from tests.gpu_harness import D, Layer
from tests.test_gpu_parity import check_decode, check_int2, check_window
from tests.test_gpu_shared_prefix import check_against_oracle, shared_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "the gpu-marked tests need a CUDA device"
    build.build()
    abi.lib()


def draw_case(case):
    rng = np.random.default_rng(10_000 + case)
    hkv = int(rng.choice([1, 2, 4, 8]))
    g = int(rng.choice([1, 2, 4, 8]))
    sink = int(rng.choice([0, 4, 16, 64]))
    recent = int(rng.choice([1, 32, 128, 256]))
    group = int(rng.choice([32, 64]))
    splits = int(rng.choice([0, 0, 1, 3, 9]))
    nreq = int(rng.integers(1, 4))
    appends = [[int(x) for x in rng.integers(1, 900, size=int(rng.integers(1, 4)))] for _ in range(nreq)]
    return dict(hq=hkv * g, hkv=hkv, sink=sink, recent=recent, group=group, splits=splits, appends=appends,
                spikes=bool(rng.integers(0, 2)))


@pytest.mark.parametrize("case", range(16))
def test_random_layer(case):
    c = draw_case(case)
    total = max(sum(a) for a in c["appends"]) + 16
    layer = Layer(c["hq"], c["hkv"], c["sink"], c["recent"], len(c["appends"]), total, seed=case,
                  num_splits=c["splits"], group=c["group"], spikes=c["spikes"])
    trace = layer.new_trace(total)
    for b, ns in enumerate(c["appends"]):
        for n in ns:
            k, v = layer.draw(n)
            layer.append(b, k, v, trace if b == 0 else None)
    for b in range(len(c["appends"])):
        check_window(layer, b)
    check_int2(layer, 0, trace)
    check_decode(layer, len(c["appends"]), stream=case)
    assert layer.ctx.error_flags() == 0


@pytest.mark.parametrize("case", range(6))
def test_random_shared_prefix(case):
    rng = np.random.default_rng(20_000 + case)
    hkv = int(rng.choice([2, 8]))
    g = int(rng.choice([1, 2, 4, 8]))
    group = int(rng.choice([32, 64]))
    nreq = int(rng.integers(2, 7))
    prefix = 16 * int(rng.integers(20, 100))
    source = prefix + int(rng.integers(200, 800))
    suffixes = [int(x) for x in rng.integers(0, 500, size=nreq - 1)]
    layer = Layer(hkv * g, hkv, 4, 128, nreq, source + max(suffixes) + 64, seed=100 + case, group=group)
    k, v = layer.draw(source)
    layer.append(0, k, v)
    for dst in range(1, nreq):
        layer.cache.fork(0, dst, prefix)
        layer.k_host[dst] = layer.k_host[0][:prefix].copy()
        layer.v_host[dst] = layer.v_host[0][:prefix].copy()
        layer.len[dst], layer.e[dst] = prefix, prefix
        if suffixes[dst - 1]:
            k, v = layer.draw(suffixes[dst - 1])
            layer.append(dst, k, v)
    q = layer.queries(nreq, 30 + case)
    check_against_oracle(layer, q, shared_decode(layer, q, prefix))
    assert layer.ctx.error_flags() == 0
