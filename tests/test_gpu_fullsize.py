"""Full-size parity: every workload at its own sizes, driven the way the
benchmark drives it (16384-token population chunks, one 131072-token append,
the full decode batch with the automatic split count), and checked on samples
the oracle computes one by one (the 32k workload runs its 100 decode steps;
the batch-28 workload populates three of its requests independently):
  * the codes, scales and zeros of sampled pages bit-exact against the oracle
    quantising the GPU's rotated values, and those rotated values within 1e-5
    of the float64 rotation;
  * decode outputs of sampled (request, KV head) pairs within rel-L2 2e-3 and
    max-abs 1e-2 of the float64 oracle over the oracle's own cache of that
    head, with rounding ties of its float64 rotation resolved to the GPU's
    (valid) choice.
"""

import numpy as np
import pytest
import torch

import oracle
from bit_rotated_kv_oscar_gb300 import abi, build
from synth import WORKLOADS, draw_kv, draw_queries, draw_ragged_lengths
from tests.gpu_harness import D, MAX_ABS, REL_L2, ROT_REL, Layer, rel_l2, resolve_group_ties
from tests.test_gpu_parity import check_int2, check_window

pytestmark = pytest.mark.gpu

CHUNK = 16384   # population chunk of the benchmark


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "the gpu-marked tests need a CUDA device"
    build.build()
    abi.lib()


def spec_layer(spec, max_batch, max_tokens):
    return Layer(spec.num_q_heads, spec.num_kv_heads, spec.sink, spec.recent, max_batch, max_tokens,
                 seed=spec.seed, n_cal=spec.calib_tokens, shuffled=spec.shuffled_pages,
                 spikes=spec.token_spikes)


def populate(layer, b, n, stream0, trace=None, chunk=CHUNK):
    """Append n fresh tokens to request b in chunks of `chunk`."""
    pos = 0
    while pos < n:
        m = min(chunk, n - pos)
        k, v = draw_kv(layer.seed, stream0 + pos // chunk, m, layer.hkv, D, layer.spikes)
        layer.append(b, k, v, trace)
        pos += m


def sample_pages(rng, layer, b, count):
    """Page-aligned position ranges inside request b's INT2 region."""
    S, E = layer.sink, min(layer.e[b], layer.len[b])
    first, last = S // 16, (E - 1) // 16
    pages = rng.choice(np.arange(first, last + 1), size=min(count, last - first + 1), replace=False)
    return [(max(16 * int(p), S), min(16 * int(p) + 16, E)) for p in sorted(pages)]


def check_sampled_int2(layer, b, trace, rng, count=8):
    for lo, hi in sample_pages(rng, layer, b, count):
        check_int2(layer, b, trace, lo, hi)


def oracle_head(layer, b, h):
    """The oracle's cache of KV head h of request b, its float64-rotation ties
    resolved to the GPU's choice after checking the choice is a valid one."""
    cal, S = layer.cal, layer.sink
    L, E = layer.len[b], layer.e[b]
    cache = oracle.OracleCache(cal["R_K32"][h:h + 1], layer.r_v32[h:h + 1], cal["clip_K32"][h:h + 1],
                               cal["clip_V32"][h:h + 1], S)
    cache.build(layer.k_host[b][:, h:h + 1], layer.v_host[b][:, h:h + 1], L, E)
    hi = min(E, L)
    if hi <= S:
        return cache
    pt = layer.cache.page_table_host[b]
    n0, n1 = S // 16, (hi - 1) // 16 + 1
    blocks = layer.blocks_of_pages(pt[n0:n1])[:, h:h + 1]
    dec = []
    for x in oracle.decode_page_block(blocks):
        x = np.moveaxis(x, 2, 1)
        x = x.reshape((-1,) + x.shape[2:])
        dec.append(x[S - n0 * 16:hi - n0 * 16])
    for kind in range(2):
        x = (cache.k if kind == 0 else cache.v)[S:hi]
        r = cache.r_k if kind == 0 else cache.r_v
        clip = (cache.clip_k if kind == 0 else cache.clip_v).reshape(1, -1, 1).astype(np.float64)
        x64 = (x[:, 0] @ r[0])[:, None]
        eps = ROT_REL * np.abs(x64).max(-1, keepdims=True)
        codes, s16, z16 = resolve_group_ties(x64, clip, eps, dec[kind], dec[2 + 2 * kind], dec[3 + 2 * kind])
        if kind == 0:
            cache.k_codes, cache.k_scale, cache.k_zero = codes, s16, z16
        else:
            cache.v_codes, cache.v_scale, cache.v_zero = codes, s16, z16
    return cache


def decode_rows(layer, q, row0):
    """decode_attn for requests row0 .. row0 + len(q) - 1 (q float32 [B, hq, D])."""
    bsz = q.shape[0]
    qd = q.to(torch.bfloat16).to(layer.device).contiguous()
    o = torch.full((bsz, layer.hq, D), float("nan"), device=layer.device)
    layer.ctx.decode_attn(qd, layer.cache.page_table[row0:], layer.cache.state[row0:], o, bsz)
    torch.cuda.synchronize()
    return o.cpu().numpy()


def check_sampled_decode(layer, q, o, pairs, row0=0, caches=None):
    g = layer.hq // layer.hkv
    worst = (0.0, 0.0)
    for i, h in pairs:
        b = row0 + i
        cache = caches[h] if caches is not None else oracle_head(layer, b, h)
        ref = oracle.decode_attention(q[i, h * g:(h + 1) * g].numpy().astype(np.float64), cache)
        got = o[i, h * g:(h + 1) * g]
        assert np.isfinite(got).all()
        r, m = rel_l2(got, ref), float(np.abs(got - ref).max())
        worst = (max(worst[0], r), max(worst[1], m))
        assert r <= REL_L2 and m <= MAX_ABS, (b, h, r, m)
    return worst


def clone_request(layer, src, dst):
    """Request dst gets a copy of request src's pages, window rows and state
    (distinct pages, same contents), as the benchmark fills its batch."""
    L, E, S, W, hkv = layer.len[src], layer.e[src], layer.sink, layer.recent, layer.hkv
    layer.cache.reserve(dst, L)
    pool = layer.cache.pool.view(-1, hkv, abi.PAGE_BLOCK_BYTES)
    npg = (L + 15) // 16
    src_ids = torch.as_tensor(layer.cache.page_table_host[src, :npg].astype(np.int64), device=pool.device)
    dst_ids = torch.as_tensor(layer.cache.page_table_host[dst, :npg].astype(np.int64), device=pool.device)
    pool[dst_ids] = pool[src_ids]
    win = layer.cache.window.view(layer.cfg.max_batch, hkv, 2, S + W, D)
    win[dst].copy_(win[src])
    layer.cache.state[dst] = torch.tensor([L, E, dst, 0], dtype=torch.int32, device=pool.device)
    layer.k_host[dst], layer.v_host[dst] = layer.k_host[src], layer.v_host[src]
    layer.len[dst], layer.e[dst] = L, E
    torch.cuda.synchronize()


# ---------------------------------------------------------------------------
# Qwen3-8B layer, batch 1 x 32768 tokens, then decode steps with appends
# ---------------------------------------------------------------------------

def test_fullsize_qwen3_8b_bs1_32k():
    # the workload's 100 decode steps as the benchmark runs them (oscar_decode_step:
    # one token appended, which evicts the oldest recent token into INT2, and the
    # decode query, in the same launches), next to a twin layer that takes the
    # same steps as quant_append (traced) + decode_attn: the step's cache must
    # equal the twin's byte for byte, the twin's evicted codes are checked against
    # the oracle through its trace, and the step's outputs of every KV head against
    # the oracle at steps 0, 50 and 99
    spec = WORKLOADS["qwen3_8b_bs1_32k"]
    n, steps = spec.context, spec.decode_steps
    assert steps == 100
    layer = spec_layer(spec, 1, n + steps + 16)
    twin = spec_layer(spec, 1, n + steps + 16)
    trace = layer.new_trace(n + steps)
    populate(layer, 0, n, 10_000, trace)
    populate(twin, 0, n, 10_000)
    rng = np.random.default_rng(1)
    check_sampled_int2(layer, 0, trace, rng)
    check_window(layer, 0)
    for step in range(steps):
        k, v = draw_kv(layer.seed, 100 + step, 1, layer.hkv, D, layer.spikes)
        q = draw_queries(layer.seed, 100 + step, 1, layer.hq, layer.hkv, D)
        layer.append(0, k.view(1, layer.hkv, D), v.view(1, layer.hkv, D), trace)
        o_two = decode_rows(layer, q, 0)
        twin.cache.reserve(0, twin.len[0] + 1)
        o = torch.full((1, twin.hq, D), float("nan"), device=twin.device)
        twin.ctx.decode_step(twin.cache.page_table, twin.cache.state, q.to(torch.bfloat16).to(twin.device),
                             k.view(1, twin.hkv, D).to(torch.bfloat16).to(twin.device),
                             v.view(1, twin.hkv, D).to(torch.bfloat16).to(twin.device), o, 1)
        torch.cuda.synchronize()
        twin._record(0, k.view(1, twin.hkv, D), v.view(1, twin.hkv, D))
        o = o.cpu().numpy()
        assert np.isfinite(o).all(), step
        assert rel_l2(o, o_two) <= REL_L2, step
        if step in (0, 50, 99):
            check_sampled_decode(twin, q, o, [(0, h) for h in range(twin.hkv)])
    assert (layer.len[0], layer.e[0]) == (n + steps, n + steps - spec.recent)
    assert tuple(twin.device_state()[0][:2]) == (n + steps, n + steps - spec.recent)
    # the tokens the steps evicted into INT2: the twin's against the oracle, the
    # step's against the twin's
    lo, hi = n - spec.recent, layer.e[0]
    check_int2(layer, 0, trace, lo, hi)
    for x, y in zip(layer.int2_codes(0, lo, hi), twin.int2_codes(0, lo, hi)):
        assert np.array_equal(np.ascontiguousarray(x).view(np.uint8), np.ascontiguousarray(y).view(np.uint8))
    check_window(layer, 0)
    check_window(twin, 0)
    assert layer.ctx.error_flags() == 0 and twin.ctx.error_flags() == 0


# ---------------------------------------------------------------------------
# Qwen3-8B layer, batch 16 with ragged lengths in 8k-32k and token spikes
# ---------------------------------------------------------------------------

def test_fullsize_qwen3_8b_bs16_ragged():
    spec = WORKLOADS["qwen3_8b_bs16_ragged"]
    lengths = draw_ragged_lengths(spec.seed, spec.batch, spec.context_min, spec.context)
    layer = spec_layer(spec, spec.batch, int(lengths.max()) + 16)
    trace = layer.new_trace(int(lengths.max()))
    rng = np.random.default_rng(2)
    for b in range(spec.batch):
        trace.fill_(float("nan"))
        populate(layer, b, int(lengths[b]), 20_000 + 100 * b, trace)
        if b in (0, 7, 15):
            check_sampled_int2(layer, b, trace, rng, count=4)
            check_window(layer, b)
    q = draw_queries(layer.seed, 3, spec.batch, layer.hq, layer.hkv, D)
    o = decode_rows(layer, q, 0)
    assert np.isfinite(o).all()
    check_sampled_decode(layer, q, o, [(0, 0), (3, 7), (7, 3), (11, 5), (15, 1)])
    assert layer.ctx.error_flags() == 0


# ---------------------------------------------------------------------------
# Qwen3-32B layer, batch 28 x ~100000 tokens: three requests populated
# independently (their own seeds and lengths), the others copies of request 0
# ---------------------------------------------------------------------------

def test_fullsize_qwen3_32b_bs28_100k():
    spec = WORKLOADS["qwen3_32b_bs28_100k"]
    n, B = spec.context, spec.batch
    own = {0: n, 13: n - 37, 27: n - 1000}      # request -> its own length
    layer = spec_layer(spec, B, n + 16)
    trace = layer.new_trace(n)
    populate(layer, 0, n, 10_000, trace)
    rng = np.random.default_rng(3)
    check_sampled_int2(layer, 0, trace, rng)
    del trace
    for b, length in own.items():
        if b:
            populate(layer, b, length, 30_000 + 100 * b)
    for b in range(1, B):
        if b not in own:
            clone_request(layer, 0, b)
    q = draw_queries(layer.seed, 3, B, layer.hq, layer.hkv, D)
    o = decode_rows(layer, q, 0)
    assert np.isfinite(o).all()
    heads = (0, 5)
    for b in own:
        caches = {h: oracle_head(layer, b, h) for h in heads}
        check_sampled_decode(layer, q, o, [(b, h) for h in heads], caches=caches)
    # a copied request reads the same cache as request 0 through other pages
    caches = {h: oracle_head(layer, 0, h) for h in heads}
    check_sampled_decode(layer, q, o, [(b, h) for b in (5, 20) for h in heads], caches=caches)
    del caches
    # one decode step of all 28 requests through oscar_decode_step, the launch
    # configuration the benchmark times at this size (the step's append CTAs
    # beside the splits): every request's ring entry goes to INT2
    k1, v1 = draw_kv(layer.seed, 50_000, B, layer.hkv, D, layer.spikes)
    q1 = draw_queries(layer.seed, 4, B, layer.hq, layer.hkv, D)
    for b in range(B):
        layer.cache.reserve(b, layer.len[b] + 1, upload=False)
    layer.cache.upload()
    dev = layer.device
    o1 = torch.full((B, layer.hq, D), float("nan"), device=dev)
    layer.ctx.decode_step(layer.cache.page_table, layer.cache.state, q1.to(torch.bfloat16).to(dev),
                          k1.to(torch.bfloat16).to(dev).contiguous(), v1.to(torch.bfloat16).to(dev).contiguous(),
                          o1, B)
    torch.cuda.synchronize()
    for b in range(B):
        layer._record(b, k1[b:b + 1], v1[b:b + 1])
    o1 = o1.cpu().numpy()
    assert np.isfinite(o1).all()
    state = layer.device_state()
    for b in (0, 20, 27):
        assert tuple(state[b][:2]) == (layer.len[b], layer.e[b])
    check_sampled_decode(layer, q1, o1, [(b, h) for b in (0, 20, 27) for h in heads])
    assert layer.ctx.error_flags() == 0


# ---------------------------------------------------------------------------
# 131072-token prefill, 16 forks at 65536 tokens with 4096-token suffixes
# ---------------------------------------------------------------------------

def test_fullsize_prefill_128k_prefix16():
    spec = WORKLOADS["prefill_128k_prefix16"]
    n, fork, suf, nreq = spec.context, spec.prefix_shared, spec.suffix, spec.batch
    layer = spec_layer(spec, nreq + 1, n + 16)
    trace = layer.new_trace(n)
    k, v = draw_kv(layer.seed, 1, n, layer.hkv, D, layer.spikes)
    layer.append(0, k, v, trace)                 # one long append: the tensor-core path
    rng = np.random.default_rng(4)
    check_sampled_int2(layer, 0, trace, rng, count=12)
    check_window(layer, 0)
    del trace
    for r in range(1, nreq + 1):
        layer.cache.fork(0, r, fork)
        layer.cache.reserve(r, fork + suf, upload=False)
    layer.cache.upload()
    ks, vs = draw_kv(layer.seed, 2, nreq * suf, layer.hkv, D, layer.spikes)
    ks, vs = ks.view(nreq, suf, layer.hkv, D), vs.view(nreq, suf, layer.hkv, D)
    layer.ctx.quant_append(layer.cache.page_table[1:], layer.cache.state[1:],
                           ks.to(torch.bfloat16).to(layer.device).contiguous(),
                           vs.to(torch.bfloat16).to(layer.device).contiguous(), nreq, suf)
    for r in range(1, nreq + 1):
        layer.k_host[r] = np.concatenate([layer.k_host[0][:fork], ks[r - 1].numpy()])
        layer.v_host[r] = np.concatenate([layer.v_host[0][:fork], vs[r - 1].numpy()])
        layer.len[r], layer.e[r] = oracle.next_state(fork, fork, suf, layer.recent, layer.sink)
    assert tuple(layer.device_state()[1][:2]) == (layer.len[1], layer.e[1])
    check_window(layer, 1)
    check_window(layer, nreq)
    q = draw_queries(layer.seed, 3, nreq, layer.hq, layer.hkv, D)
    o = decode_rows(layer, q, 1)
    assert np.isfinite(o).all()
    check_sampled_decode(layer, q, o, [(0, 0), (5, 6), (15, 3)], row0=1)
    assert layer.ctx.error_flags() == 0
