"""GPU parity at the workloads' full sizes, in the launch configuration the benchmark times.

The whole layer is filled through the write path in 16384-token appends (as bench.py does) and
decoded with the default warp-MMA kernel over every request at once; the CPU oracle then checks a
sample of (request, KV head) pairs one by one: every stored INT2 code and fp16 scale/min and the
BF16 window bytes bit for bit, and the attention output within rel-L2 1e-3 / max-abs 2e-3, for the
filled cache and again after one more decode-step append.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import int2_rotated_paged_gb300 as K
from gpu_util import (append_initial, check_bf16_bytes, check_int2_bytes, decode_query, make_cache,
                      oracle_caches, oracle_rk, rel_l2)

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


def _attend(cache, q, rk_dev):
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    cache.attend(q, rk_dev, out)
    cache.status()
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("name,pairs", [
    ("qwen3_8b", [(0, 0), (31, 7)]),           # B32, 32/8 heads, 32768 tokens
    ("qwen3_32b", [(0, 3), (17, 5)]),          # B32, 64/8 heads, 100000 tokens (the benchmark layer)
    ("ragged_128k", [(0, 0), (15, 7)]),        # B16, 96/8 heads (G = 12), 65536..131072 tokens
])
def test_full_size_sampled_pairs(name, pairs):
    cfg = synth.config(name)
    rk = oracle_rk(cfg.seed, cfg.num_kv_heads, 1024)
    rk_dev = torch.tensor(rk, device="cuda")
    lens = list(cfg.ctx)
    cache = make_cache(cfg, max(lens) + 1)
    append_initial(cache, cfg, lens, rk_dev, chunks=[16384] * (max(lens) // 16384 + 1))
    ocs = oracle_caches(cfg, pairs, lens, rk)
    g = cfg.group
    for step in range(2):
        for (b, h), oc in ocs.items():
            check_int2_bytes(cache, oc, b, h)
            check_bf16_bytes(cache, oc, b, h)
        q = decode_query(cfg, step)
        out = _attend(cache, q, rk_dev)
        assert np.isfinite(out).all()
        for (b, h), oc in ocs.items():
            ref, _ = oc.attend(q[b, h * g:(h + 1) * g].cpu().numpy())
            got = out[b, h * g:(h + 1) * g]
            r, m = rel_l2(got, ref), float(np.abs(got - ref).max())
            assert r <= REL_L2 and m <= MAX_ABS, f"{name} step {step} (b={b}, h={h}): rel-L2 {r:.3e}, max-abs {m:.3e}"
        if step == 0:
            # one decode-step append: every request gains a token, one token per request leaves the
            # window for the INT2 pages
            n = [1] * cfg.batch
            k, v = synth.kv_block(cfg.seed, n, lens, cfg.num_kv_heads, device="cuda")
            cache.append(k, v, n, rk_dev)
            for (b, h), oc in ocs.items():
                oc.append(synth.bf16_bits(k[b, h][None]), synth.bf16_bits(v[b, h][None]))
            lens = [x + 1 for x in lens]
