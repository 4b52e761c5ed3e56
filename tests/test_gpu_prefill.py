"""GPU parity of chunked-prefill attention (oscar_prefill_attention) against the oracle's causal view.

Each request appends a chunk of n_q tokens through the write path; the chunk's queries then attend,
each over the cached positions up to its own, in the precision the cache holds them in after the
append (BF16 sink and window, INT2 history).  The oracle is OracleCache.attend_upto (pinned in
tests/test_oracle_prefill.py).  Covered: chunks that stay in the BF16 window, chunks whose append
pushes tokens into INT2 pages, long contexts, 1 .. 256 queries, GQA groups whose queries share a
request slot in different packings (G = 1, 3, 4, 8, 12), bf16 queries and outputs, and the errors.
Bars: rel-L2 <= 1e-3 and max-abs <= 2e-3 per (request, KV head, query).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import int2_rotated_paged_gb300 as K
from gpu_util import check_int2_bytes, make_cache, oracle_rk, rel_l2

pytestmark = pytest.mark.gpu

REL_L2 = 1e-3
MAX_ABS = 2e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    from int2_rotated_paged_gb300 import build
    build.build()
    oracle.build()
    assert torch.cuda.is_available()
    K.oscar_set_decode_path(K.PATH_WARP_MMA)


def _prefill_case(hq, hkv, lens0, n_q, seed, q_dtype=torch.float32, out_dtype=torch.float32):
    B = len(lens0)
    cfg = synth.LayerConfig("prefill", B, hq, hkv, lens0, 1, "permuted", "fp32", seed)
    g = hq // hkv
    rk = oracle_rk(seed, hkv, 1024)
    rk_dev = torch.tensor(rk, device="cuda")
    total = [lens0[b] + n_q[b] for b in range(B)]
    cache = make_cache(cfg, max(total))
    # the context, then the chunk (its own append), both through the write path
    k0, v0 = synth.kv_block(seed, lens0, [0] * B, hkv, device="cuda")
    if sum(lens0):
        cache.append(k0, v0, lens0, rk_dev)
    k1, v1 = synth.kv_block(seed, n_q, lens0, hkv, device="cuda")
    cache.append(k1, v1, n_q, rk_dev)
    rows = sum(n_q)
    qg = torch.Generator(device="cpu").manual_seed(seed + 1)
    q = (torch.randn(rows, hq, 128, generator=qg) * 0.7).to(q_dtype).cuda()
    out = torch.full((rows, hq, 128), float("nan"), dtype=out_dtype, device="cuda")
    ws = cache.prefill(q, n_q, rk_dev, out)
    K.oscar_decode_status(cache.handle, ws)          # no bounded wait gave up
    torch.cuda.synchronize()
    got = out.float().cpu().numpy()
    qh = q.float().cpu().numpy()
    assert np.isfinite(got).all()
    bar_abs = MAX_ABS + (2.0 ** -8 if out_dtype == torch.bfloat16 else 0.0)
    bar_rel = REL_L2 + (2.0 ** -8 if out_dtype == torch.bfloat16 else 0.0)
    r0 = 0
    worst = 0.0
    for b in range(B):
        for h in range(hkv):
            oc = oracle.OracleCache(rk[h])
            kk = synth.bf16_bits(synth.keys(seed, b, h, 0, total[b], device="cuda"))
            vv = synth.bf16_bits(synth.values(seed, b, h, 0, total[b], device="cuda"))
            oc.append(kk, vv)
            if h == 0:
                check_int2_bytes(cache, oc, b, h)
            for i in range(n_q[b]):
                ref, _ = oc.attend_upto(qh[r0 + i, h * g:(h + 1) * g], lens0[b] + i)
                o = got[r0 + i, h * g:(h + 1) * g]
                r = rel_l2(o, ref)
                worst = max(worst, r)
                assert r <= bar_rel and np.abs(o - ref).max() <= bar_abs * max(1.0, float(np.abs(ref).max())), \
                    f"(b={b}, h={h}, query {i}): rel-L2 {r:.3e}"
        r0 += n_q[b]
    return worst


@pytest.mark.parametrize("hq,hkv", [(16, 2), (8, 2), (24, 2), (6, 2), (2, 2)])
def test_chunks_in_window_into_int2_and_long(hq, hkv):
    # request 0: all BF16 after the chunk; 1: the chunk pushes tokens into INT2; 2: long context;
    # 3: an empty chunk
    _prefill_case(hq, hkv, [100, 300, 3000, 500], [64, 120, 37, 0], 7100 + hq)


@pytest.mark.parametrize("n", [1, 2, 3, 255, 256])
def test_chunk_sizes(n):
    _prefill_case(16, 2, [2000, 700], [n, min(n, 200)], 7200 + n)


def test_chunk_from_an_empty_request_and_bf16_io():
    _prefill_case(16, 2, [0, 900], [256, 5], 7300, q_dtype=torch.bfloat16, out_dtype=torch.bfloat16)


def test_prefill_of_one_token_matches_decode_attention():
    cfg = synth.scaled(synth.config("qwen3_4b"), [1500, 800], batch=2)
    rk = torch.tensor(oracle_rk(cfg.seed, cfg.num_kv_heads, 1024), device="cuda")
    cache = make_cache(cfg, 1600)
    k, v = synth.kv_block(cfg.seed, cfg.ctx, [0, 0], cfg.num_kv_heads, device="cuda")
    cache.append(k, v, cfg.ctx, rk)
    q = synth.queries(cfg.seed, 0, 2, cfg.num_q_heads, cfg.num_kv_heads, device="cuda")
    dec = torch.empty_like(q)
    cache.attend(q, rk, dec)
    pre = torch.empty_like(q)
    cache.prefill(q, [1, 1], rk, pre)
    torch.cuda.synchronize()
    d, p = dec.cpu().numpy(), pre.cpu().numpy()
    assert rel_l2(p, d) <= 1e-3 and np.abs(p - d).max() <= 2e-3


def test_prefill_errors():
    cache = K.Cache(2, 16, 2, 64, 32)
    q = torch.zeros(300, 16, 128, device="cuda")
    out = torch.zeros_like(q)
    rk = torch.eye(128, device="cuda").repeat(2, 1, 1).contiguous()
    ws = torch.empty(K.oscar_prefill_workspace_bytes(cache.handle), dtype=torch.uint8, device="cuda")
    k, v = synth.kv_block(1, [300, 10], [0, 0], 2, device="cuda")
    cache.append(k, v, [300, 10], rk)
    with pytest.raises(K.OscarError) as e:           # more than 256 queries in a chunk
        K.oscar_prefill_attention(cache.handle, q, K.DTYPE_F32, [257, 0], rk, out, K.DTYPE_F32, ws)
    assert e.value.code == K.OSCAR_ERANGE
    with pytest.raises(K.OscarError) as e:           # more queries than tokens held
        K.oscar_prefill_attention(cache.handle, q, K.DTYPE_F32, [1, 11], rk, out, K.DTYPE_F32, ws)
    assert e.value.code == K.OSCAR_ERANGE
    with pytest.raises(K.OscarError) as e:           # workspace too small
        K.oscar_prefill_attention(cache.handle, q, K.DTYPE_F32, [1, 1], rk, out, K.DTYPE_F32, ws[:64])
    assert e.value.code == K.OSCAR_EWORKSPACE
    K.oscar_set_decode_path(K.PATH_SIMT)
    try:
        with pytest.raises(K.OscarError) as e:       # the warp-MMA path only
            K.oscar_prefill_attention(cache.handle, q, K.DTYPE_F32, [1, 1], rk, out, K.DTYPE_F32, ws)
        assert e.value.code == K.OSCAR_EINVAL
    finally:
        K.oscar_set_decode_path(K.PATH_WARP_MMA)
