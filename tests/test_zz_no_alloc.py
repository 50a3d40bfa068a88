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


def _window_chunk_is_long(batch, hkv, window):
    # the library's window policy: 64-token window CTAs while they fill at most a
    # quarter of the two resident decode CTAs per SM, 160-token CTAs otherwise
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return 4 * batch * hkv * ((window + 63) // 64) > 2 * sms


# (group, request lengths): three requests keep the 64-token window chunk; five
# requests of 8 KV heads (40 window units) take the 160-token chunk
CASES = [(32, [2500, 700, 1900]), (64, [2500, 700, 1900]), (32, [2500, 700, 1900, 1200, 3000]),
         (64, [1500, 2900, 800, 2200, 3000])]


@pytest.mark.parametrize("group, lengths", CASES)
def test_noalloc_matches_context_decode_twice(group, lengths):
    B = len(lengths)
    layer = Layer(32, 8, 4, 128, B, 3100, seed=61, group=group)
    assert _window_chunk_is_long(B, 8, 4 + 128) == (B >= 5)
    for b, n in enumerate(lengths):
        k, v = layer.draw(n)
        layer.append(b, k, v)
    q = layer.queries(B, 5)
    o_ctx = layer.decode(q)
    r_k = torch.tensor(layer.cal["R_K32"], device="cuda")
    r_v = torch.tensor(layer.r_v32, device="cuda")
    clip_v = torch.tensor(layer.cal["clip_V32"], device="cuda")
    qd = q.to(torch.bfloat16).cuda().contiguous()
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    # the first call reports into the caller's flag word, the second into the
    # word kept inside the library's array (err_flags = NULL)
    for call, fl in enumerate((flags, None)):
        o = torch.full((B, 32, D), float("nan"), device="cuda")
        abi.decode_attn_noalloc(layer.cfg, qd, layer.cache.page_table, layer.cache.state, o, B,
                                layer.cache.pool, layer.cache.num_pages, layer.cache.window, r_k, r_v,
                                clip_v, fl)
        torch.cuda.synchronize()
        got = o.cpu().numpy()
        assert np.isfinite(got).all(), call
        for b in range(B):
            assert rel_l2(got[b], o_ctx[b]) <= REL_L2, (call, b)
            assert float(np.abs(got[b] - o_ctx[b]).max()) <= MAX_ABS, (call, b)
    assert int(flags.item()) == 0
    # and against the float64 oracle for two requests
    for b in (1, B - 1):
        ref = layer.oracle_decode(q[b].numpy(), b)
        assert rel_l2(got[b], ref) <= REL_L2, b
        assert float(np.abs(got[b] - ref).max()) <= MAX_ABS, b


def test_noalloc_rejects_a_workspace_beyond_its_array():
    cfg = abi.make_config(64, 8, 4, 128, 4096, 64)
    t = torch.zeros(4096, dtype=torch.int32, device="cuda")
    f = torch.zeros(8 * 128 * 128, device="cuda")
    with pytest.raises(abi.OscarError) as e:
        abi.decode_attn_noalloc(cfg, t, t, t, f, 4096, t, 1, t, f, f, f)
    assert e.value.status == -3
