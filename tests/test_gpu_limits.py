"""GPU parity at the call-size limits: 256 requests in one call (the most a call takes), with
lengths at every region boundary (empty, sink only, the first INT2 token, page edges), through bulk
appends, decode attention and fused decode steps; and a chunked prefill whose request slots
(384 of them) need two launches.  Sampled requests are checked against the oracle (attention,
every stored byte).  Bars: rel-L2 <= 1e-3, max-abs <= 2e-3.
Sources: axbrief.com OSCAR page, sections "attention-statistics rotation + Triton kernels" and
"OSCAR release".
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import int2_rotated_paged_gb300 as K
from gpu_util import check_bf16_bytes, check_int2_bytes, oracle_rk, pages_needed, rel_l2

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


def _oracle(seed, rk, b, h, n):
    oc = oracle.OracleCache(rk[h])
    if n:
        oc.append(synth.bf16_bits(synth.keys(seed, b, h, 0, n, device="cuda")),
                  synth.bf16_bits(synth.values(seed, b, h, 0, n, device="cuda")))
    return oc


def test_256_requests_in_one_call():
    B, hq, hkv, seed = 256, 8, 1, 9100
    edges = [0, 1, 63, 64, 65, 255, 319, 320, 321, 383, 384, 385, 447, 448, 1000, 1500]
    rng = np.random.default_rng(seed)
    lens = [edges[b] if b < len(edges) else int(rng.integers(0, 1500)) for b in range(B)]
    rk = oracle_rk(seed, hkv, 1024)
    rk_dev = torch.tensor(rk, device="cuda")
    steps = 2
    per_seq = pages_needed(1500 + steps) + 1
    cache = K.Cache(B, hq, hkv, per_seq * B, per_seq, page_order=synth.page_order(seed, per_seq * B, "permuted"))
    k, v = synth.kv_block(seed, lens, [0] * B, hkv, device="cuda")
    cache.append(k, v, lens, rk_dev)
    sample = list(range(len(edges))) + [int(x) for x in rng.choice(np.arange(len(edges), B), 8, replace=False)]
    out = torch.empty(B, hq, 128, device="cuda")
    q = synth.queries(seed, 0, B, hq, hkv, device="cuda")
    cache.attend(q, rk_dev, out)
    torch.cuda.synchronize()
    got, qh = out.cpu().numpy(), q.cpu().numpy()
    ocs = {b: _oracle(seed, rk, b, 0, lens[b]) for b in sample}
    for b in sample:
        if lens[b] == 0:
            continue
        ref, _ = ocs[b].attend(qh[b])
        assert rel_l2(got[b], ref) <= REL_L2 and np.abs(got[b] - ref).max() <= MAX_ABS, (b, lens[b])
    # fused decode steps on every request (the empty ones get their first token)
    for s in range(steps):
        q = synth.queries(seed, 1 + s, B, hq, hkv, device="cuda")
        k1, v1 = synth.kv_block(seed, [1] * B, [lens[b] + s for b in range(B)], hkv, device="cuda")
        cache.step(k1, v1, q, rk_dev, out)
        cache.status()
        torch.cuda.synchronize()
        got, qh = out.cpu().numpy(), q.cpu().numpy()
        k16, v16 = synth.bf16_bits(k1), synth.bf16_bits(v1)
        for b in sample:
            ocs[b].append(k16[b, 0][None], v16[b, 0][None])
            ref, _ = ocs[b].attend(qh[b])
            assert rel_l2(got[b], ref) <= REL_L2 and np.abs(got[b] - ref).max() <= MAX_ABS, (s, b, lens[b])
    for b in sample:
        check_int2_bytes(cache, ocs[b], b, 0)
        check_bf16_bytes(cache, ocs[b], b, 0)


def test_prefill_slots_over_two_launches():
    # 3 requests x 256 new tokens, two queries per slot (G = 8): 384 slots, two launches of the kernels
    hq, hkv, seed = 16, 2, 9200
    lens0 = [600, 3000, 1500]
    n_q = [256, 256, 256]
    B = len(lens0)
    g = hq // hkv
    rk = oracle_rk(seed, hkv, 1024)
    rk_dev = torch.tensor(rk, device="cuda")
    total = [lens0[b] + n_q[b] for b in range(B)]
    per_seq = pages_needed(max(total)) + 1
    cache = K.Cache(B, hq, hkv, per_seq * B, per_seq, page_order=synth.page_order(seed, per_seq * B, "permuted"))
    k0, v0 = synth.kv_block(seed, lens0, [0] * B, hkv, device="cuda")
    cache.append(k0, v0, lens0, rk_dev)
    k1, v1 = synth.kv_block(seed, n_q, lens0, hkv, device="cuda")
    cache.append(k1, v1, n_q, rk_dev)
    qg = torch.Generator(device="cpu").manual_seed(seed + 1)
    q = (torch.randn(sum(n_q), hq, 128, generator=qg) * 0.7).cuda()
    out = torch.full_like(q, float("nan"))
    ws = cache.prefill(q, n_q, rk_dev, out)
    K.oscar_decode_status(cache.handle, ws)        # the error word of the workspace the prefill used
    torch.cuda.synchronize()
    got, qh = out.cpu().numpy(), q.cpu().numpy()
    assert np.isfinite(got).all()
    rng = np.random.default_rng(seed)
    r0 = 0
    for b in range(B):
        h = b % hkv
        oc = _oracle(seed, rk, b, h, total[b])
        check_int2_bytes(cache, oc, b, h)
        for i in sorted(set([0, 1, 127, 128, 254, 255] + [int(x) for x in rng.integers(0, 256, 10)])):
            ref, _ = oc.attend_upto(qh[r0 + i, h * g:(h + 1) * g], lens0[b] + i)
            o = got[r0 + i, h * g:(h + 1) * g]
            assert rel_l2(o, ref) <= REL_L2 and np.abs(o - ref).max() <= MAX_ABS, (b, i)
        r0 += n_q[b]
