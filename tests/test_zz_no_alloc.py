"""GPU test of oscar_decode_attn_noalloc, the decode entry point that allocates nothing.

Callers that cannot allocate device memory (code being captured into a CUDA
graph, plug-ins whose device memory belongs to a host framework, runtimes
without a device allocator) call this context-free variant; its split-K
workspace is a fixed array inside the library. Each of two consecutive calls
must reproduce the context-based oscar_decode_attn within the parity
tolerance. Kept in its own file, collected last, so a failure here never hides
the rest of the suite.
"""

import numpy as np
import pytest
import torch

from bit_rotated_kv_oscar_gb300 import abi, build
from tests.gpu_harness import D, MAX_ABS, REL_L2, Layer, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "the gpu-marked tests need a CUDA device"
    build.build()
    abi.lib()


@pytest.mark.parametrize("group", [32, 64])
def test_noalloc_matches_context_decode_twice(group):
    lengths = [2500, 700, 1900]
    layer = Layer(32, 8, 4, 128, len(lengths), 3000, seed=61, group=group)
    for b, n in enumerate(lengths):
        k, v = layer.draw(n)
        layer.append(b, k, v)
    q = layer.queries(len(lengths), 5)
    o_ctx = layer.decode(q)
    r_k = torch.tensor(layer.cal["R_K32"], device="cuda")
    r_v = torch.tensor(layer.r_v32, device="cuda")
    clip_v = torch.tensor(layer.cal["clip_V32"], device="cuda")
    qd = q.to(torch.bfloat16).cuda().contiguous()
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(2):
        o = torch.full((len(lengths), 32, D), float("nan"), device="cuda")
        abi.decode_attn_noalloc(layer.cfg, qd, layer.cache.page_table, layer.cache.state, o, len(lengths),
                                layer.cache.pool, layer.cache.num_pages, layer.cache.window, r_k, r_v,
                                clip_v, flags)
        torch.cuda.synchronize()
        got = o.cpu().numpy()
        assert np.isfinite(got).all()
        for b in range(len(lengths)):
            assert rel_l2(got[b], o_ctx[b]) <= REL_L2
            assert float(np.abs(got[b] - o_ctx[b]).max()) <= MAX_ABS
    assert int(flags.item()) == 0
    # and against the oracle for one request
    ref = layer.oracle_decode(q[1].numpy(), 1)
    assert rel_l2(got[1], ref) <= REL_L2


def test_noalloc_rejects_a_workspace_beyond_its_array():
    cfg = abi.make_config(64, 8, 4, 128, 4096, 64)
    t = torch.zeros(4096, dtype=torch.int32, device="cuda")
    f = torch.zeros(8 * 128 * 128, device="cuda")
    with pytest.raises(abi.OscarError) as e:
        abi.decode_attn_noalloc(cfg, t, t, t, f, 4096, t, 1, t, f, f, f)
    assert e.value.status == -3
