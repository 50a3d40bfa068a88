"""GPU parity of the shared-prefix decode (oscar_decode_attn_shared_prefix): the
INT2 positions of a prefix that several requests map to the same pages are
attended once per pack of requests (8 / g of them side by side in the
tensor-core columns), each request's own positions as usual. Prefix caching on
a paged cache is the pages' ("Juntos, AI Open-Sources OSCAR ...", section "El
sistema de servicio"); the result must equal the plain decode's: output rel-L2
<= 2e-3 and max-abs <= 1e-2 against the float64 oracle of every request."""

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


def forked_layer(hq, hkv, nreq, prefix, source_len, suffixes, seed, **kw):
    """Request 0 holds source_len tokens; requests 1.. fork its first `prefix`
    positions and append their own suffix lengths."""
    layer = Layer(hq, hkv, kw.pop("sink", 4), kw.pop("recent", 128), nreq, source_len + max(suffixes) + 64,
                  seed=seed, **kw)
    k, v = layer.draw(source_len)
    layer.append(0, k, v)
    for dst in range(1, nreq):
        layer.cache.fork(0, dst, prefix)
        layer.k_host[dst] = layer.k_host[0][:prefix].copy()
        layer.v_host[dst] = layer.v_host[0][:prefix].copy()
        layer.len[dst], layer.e[dst] = prefix, prefix
        n = suffixes[dst - 1]
        if n:
            k, v = layer.draw(n)
            layer.append(dst, k, v)
    return layer


def shared_decode(layer, q, prefix):
    bsz = q.shape[0]
    qd = q.to(torch.bfloat16).to(layer.device).contiguous()
    o = torch.full((bsz, layer.hq, D), float("nan"), device=layer.device)
    layer.ctx.decode_attn_shared_prefix(qd, layer.cache.page_table, layer.cache.state, prefix, o, bsz)
    torch.cuda.synchronize()
    return o.cpu().numpy()


def check_against_oracle(layer, q, o):
    for b in range(q.shape[0]):
        ref = layer.oracle_decode(q[b].numpy(), b)
        r, m = rel_l2(o[b], ref), float(np.abs(o[b] - ref).max())
        assert r <= REL_L2 and m <= MAX_ABS, (b, r, m)


@pytest.mark.parametrize("hq,hkv", [(32, 8), (8, 8), (16, 8), (64, 8), (4, 2)])
def test_shared_prefix_matches_the_oracle(hq, hkv):
    layer = forked_layer(hq, hkv, 5, 2048, 2600, [0, 1, 130, 1000], seed=hq + 7 * hkv)
    q = layer.queries(5, 11)
    o = shared_decode(layer, q, 2048)
    assert np.isfinite(o).all()
    check_against_oracle(layer, q, o)
    # the plain decode of the same cache agrees with it to within the tolerance
    plain = layer.decode(q)
    assert rel_l2(o, plain) <= REL_L2
    assert layer.ctx.error_flags() == 0


def test_shared_prefix_of_the_pages_preset():
    layer = forked_layer(32, 8, 3, 1536, 2000, [300, 17], seed=5, sink=64, recent=256, group=64,
                         clip_percentiles=(96.0, 92.0))
    q = layer.queries(3, 12)
    check_against_oracle(layer, q, shared_decode(layer, q, 1536))
    assert layer.ctx.error_flags() == 0


def test_shared_prefix_with_values_folded_into_the_projection():
    layer = forked_layer(32, 8, 4, 1024, 1500, [100, 0, 333], seed=29, fold_rv=1)
    q = layer.queries(4, 16)
    check_against_oracle(layer, q, shared_decode(layer, q, 1024))
    assert layer.ctx.error_flags() == 0


@pytest.mark.parametrize("prefix", [0, 16, 512])
def test_shorter_declared_prefix(prefix):
    # declaring less than what is shared is still correct: the rest is read per request
    layer = forked_layer(32, 8, 4, 1024, 1500, [5, 200, 0], seed=13)
    q = layer.queries(4, 13)
    check_against_oracle(layer, q, shared_decode(layer, q, prefix))
    assert layer.ctx.error_flags() == 0


def test_contract_violation_raises_a_flag_not_a_fault():
    layer = forked_layer(32, 8, 3, 1024, 1500, [5, 40], seed=17)
    q = layer.queries(3, 14)
    # request 1 holds only 1029 positions, int2_end 1024: a declared prefix of
    # 1280 is not INT2 in it (nor mapped to the same pages)
    o = shared_decode(layer, q, 1280)
    assert np.isfinite(o).all()
    assert layer.ctx.error_flags() & abi.FLAG_BAD_STATE


def test_prefix_must_be_page_aligned():
    layer = forked_layer(8, 2, 2, 512, 700, [10], seed=19)
    q = layer.queries(2, 15)
    with pytest.raises(abi.OscarError) as e:
        shared_decode(layer, q, 100)
    assert e.value.status == -1
