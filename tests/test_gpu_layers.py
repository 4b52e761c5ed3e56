"""Multi-layer appends (kv_quant_append_layers): one call writes the same new tokens into every
layer's cache with two kernel launches in all.

Three layers with different R_K, page orders and clip factors take a bulk append, chunked appends
that push tokens out of the window, one-token appends (the per-channel kernel) and an append that
leaves one request empty, each as ONE batched call; twin caches take the same tokens through one
kv_quant_append per layer.  After every append the pools, BF16 regions and per-request metadata
(lengths and recorded value-scale maxima) of each layer must be identical byte for byte, and at
the end every layer's stored INT2 and BF16 bytes are checked against its own oracle cache.
Errors: caches whose lengths differ, a cache given twice, a short workspace.
Source of the write path: axbrief.com OSCAR page, section "attention-statistics rotation + Triton
kernels" (per-layer R_K, per-token asymmetric INT2).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import int2_rotated_paged_gb300 as K
from gpu_util import check_bf16_bytes, check_int2_bytes, oracle_rk, pages_needed

pytestmark = pytest.mark.gpu

B, HQ, HKV, L = 3, 16, 2, 3


@pytest.fixture(scope="module", autouse=True)
def _built():
    from int2_rotated_paged_gb300 import build
    build.build()
    oracle.build()
    assert torch.cuda.is_available()


def _layer_tokens(layer, n, start):
    k, v = synth.kv_block(500 + layer, n, start, HKV, device="cuda")
    return k, v


def test_batched_layers_store_the_bytes_of_per_layer_appends():
    per_seq = pages_needed(2600) + 1
    total = per_seq * B + 2
    clips = [(0.96, 0.92), (1.0, 1.0), (0.9, 0.95)]
    rks = [oracle_rk(40 + l, HKV, 1024) for l in range(L)]
    rk_dev = [torch.tensor(r, device="cuda") for r in rks]

    def caches(tag):
        cs = [K.Cache(B, HQ, HKV, total, per_seq, page_order=synth.page_order(60 + l, total, "permuted"),
                      clip_k=clips[l][0], clip_v=clips[l][1]) for l in range(L)]
        for c in cs:
            c.pool.zero_()      # whole pools are compared below, unwritten bytes included
        return cs
    batched, single = caches("batched"), caches("single")
    ws = torch.empty(K.kv_quant_append_layers_workspace_bytes(L), dtype=torch.uint8, device="cuda")
    plan = [[1500, 700, 400], [1, 1, 1], [70, 5, 0], [300, 0, 64], [1, 0, 1], [0, 0, 0], [700, 1300, 30]]
    done = [0] * B
    for n in plan:
        toks = [_layer_tokens(l, n, done) for l in range(L)]
        K.kv_quant_append_layers(batched, [t[0] for t in toks], [t[1] for t in toks], n, rk_dev, ws)
        for l in range(L):
            single[l].append(toks[l][0], toks[l][1], n, rk_dev[l])
        torch.cuda.synchronize()
        for l in range(L):
            assert torch.equal(batched[l].pool, single[l].pool), (n, l)
            assert torch.equal(batched[l].bf16, single[l].bf16), (n, l)
            assert torch.equal(batched[l].seq_lens, single[l].seq_lens), (n, l)
        done = [done[b] + n[b] for b in range(B)]
    for l in range(L):
        for b in range(B):
            assert batched[l].length(b) == done[b]
    # every layer against its own oracle (one KV head per request)
    for l in range(L):
        for b in range(B):
            h = (l + b) % HKV
            oc = oracle.OracleCache(rks[l][h], clip_k=clips[l][0], clip_v=clips[l][1])
            oc.append(synth.bf16_bits(synth.keys(500 + l, b, h, 0, done[b], device="cuda")),
                      synth.bf16_bits(synth.values(500 + l, b, h, 0, done[b], device="cuda")))
            check_int2_bytes(batched[l], oc, b, h)
            check_bf16_bytes(batched[l], oc, b, h)


def test_batched_layers_errors():
    per_seq = pages_needed(1000) + 1
    cs = [K.Cache(B, HQ, HKV, per_seq * B, per_seq) for _ in range(2)]
    rk = torch.eye(128, device="cuda").repeat(HKV, 1, 1).contiguous()
    ws = torch.empty(K.kv_quant_append_layers_workspace_bytes(2), dtype=torch.uint8, device="cuda")
    k, v = synth.kv_block(1, [10, 10, 10], [0, 0, 0], HKV, device="cuda")
    cs[0].append(k, v, [10, 10, 10], rk)
    with pytest.raises(K.OscarError) as e:        # lengths differ between the layers
        K.kv_quant_append_layers(cs, [k, k], [v, v], [10, 10, 10], [rk, rk], ws)
    assert e.value.code == K.OSCAR_EINVAL
    cs[1].append(k, v, [10, 10, 10], rk)
    with pytest.raises(K.OscarError) as e:        # the same cache twice
        K.kv_quant_append_layers([cs[0], cs[0]], [k, k], [v, v], [10, 10, 10], [rk, rk], ws)
    assert e.value.code == K.OSCAR_EINVAL
    with pytest.raises(K.OscarError) as e:        # workspace too small
        K.kv_quant_append_layers(cs, [k, k], [v, v], [10, 10, 10], [rk, rk], ws[:64])
    assert e.value.code == K.OSCAR_EWORKSPACE
    K.kv_quant_append_layers(cs, [k, k], [v, v], [10, 10, 10], [rk, rk], ws)   # now it goes through
    torch.cuda.synchronize()
    assert cs[0].length(0) == cs[1].length(0) == 20
