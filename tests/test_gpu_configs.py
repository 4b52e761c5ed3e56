"""GPU parity on the five synthetic layers as the benchmark runs them: fused decode steps
(oscar_decode_step: append one token per request, then attend) on a cache filled through the
write path in 16384-token appends.

  * Qwen3-4B-shaped layer (B8, 32/8 heads, 8192 tokens): every (request, KV head) pair, all 16
    decode steps, attention against the oracle at every step, every stored byte at the end;
  * Qwen3-8B-shaped layer (B32, 32/8 heads, 32768 tokens): every INT2 code and fp16 scale/min and
    every BF16 byte of all 256 pairs, and attention of all pairs over two fused steps;
  * Qwen3-32B-shaped layer (B32, 64/8 heads, 100000 tokens): 16 fused steps, sampled pairs;
  * ragged 128K layer (B16, 96/8 heads, G = 12, 65536..131072 tokens): 32 fused steps, sampled pairs.
The oracle caches are filled on the host's cores in parallel (its C calls release the interpreter
lock).  Bars: codes and scales bit-exact; attention rel-L2 <= 1e-3 and max-abs <= 2e-3.
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
import synth
import int2_rotated_paged_gb300 as K
from gpu_util import check_bf16_bytes, check_int2_bytes, make_cache, append_initial, oracle_rk, rel_l2

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


def _oracle_caches(cfg, pairs, lens, rk):
    def make(bh):
        b, h = bh
        oc = oracle.OracleCache(rk[h])
        # drawn on the GPU like the cache's own inputs (the CPU and CUDA generators differ)
        oc.append(synth.bf16_bits(synth.keys(cfg.seed, b, h, 0, lens[b], device="cuda")),
                  synth.bf16_bits(synth.values(cfg.seed, b, h, 0, lens[b], device="cuda")))
        return bh, oc
    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        return dict(ex.map(make, pairs))


def _fused_steps(name, pairs, steps, check_every_step=True, q_factor=1.0):
    cfg = synth.config(name)
    rk = oracle_rk(cfg.seed, cfg.num_kv_heads, 1024)
    rk_dev = torch.tensor(rk, device="cuda")
    lens = list(cfg.ctx)
    cache = make_cache(cfg, max(lens) + steps)
    append_initial(cache, cfg, lens, rk_dev, chunks=[16384] * (max(lens) // 16384 + 1))
    pairs = pairs or [(b, h) for b in range(cfg.batch) for h in range(cfg.num_kv_heads)]
    ocs = _oracle_caches(cfg, pairs, lens, rk)
    g = cfg.group
    out = torch.empty(cfg.batch, cfg.num_q_heads, 128, device="cuda")
    worst = 0.0
    with ThreadPoolExecutor(max_workers=os.cpu_count() or 1) as ex:
        for s in range(steps):
            q = synth.queries(cfg.seed, s, cfg.batch, cfg.num_q_heads, cfg.num_kv_heads, dtype=cfg.q_dtype,
                              device="cuda") * q_factor
            k, v = synth.kv_block(cfg.seed, [1] * cfg.batch, [lens[b] + s for b in range(cfg.batch)],
                                  cfg.num_kv_heads, device="cuda")
            cache.step(k, v, q, rk_dev, out)
            cache.status()
            torch.cuda.synchronize()
            got = out.cpu().numpy()
            qh = q.float().cpu().numpy()
            k16, v16 = synth.bf16_bits(k), synth.bf16_bits(v)
            for (b, h), oc in ocs.items():
                oc.append(k16[b, h][None], v16[b, h][None])
            if not (check_every_step or s == steps - 1):
                continue

            def one(item):
                (b, h), oc = item
                ref, _ = oc.attend(qh[b, h * g:(h + 1) * g])
                r = rel_l2(got[b, h * g:(h + 1) * g], ref)
                m = float(np.abs(got[b, h * g:(h + 1) * g] - ref).max())
                return (b, h), r, m
            for (b, h), r, m in ex.map(one, list(ocs.items())):
                worst = max(worst, r)
                assert r <= REL_L2 and m <= MAX_ABS, f"{name} step {s} (b={b}, h={h}): rel-L2 {r:.3e}, max-abs {m:.3e}"
    for (b, h), oc in ocs.items():
        check_int2_bytes(cache, oc, b, h)
        check_bf16_bytes(cache, oc, b, h)
    return worst


def test_qwen3_4b_every_pair_16_fused_steps():
    _fused_steps("qwen3_4b", None, 16)


def test_qwen3_8b_every_token():
    _fused_steps("qwen3_8b", None, 2)


def test_qwen3_32b_16_fused_steps_sampled_pairs():
    _fused_steps("qwen3_32b", [(0, 0), (9, 3), (31, 7)], 16)


def test_ragged_128k_32_fused_steps_sampled_pairs():
    _fused_steps("ragged_128k", [(0, 1), (7, 4), (15, 7)], 32)


@pytest.mark.parametrize("q_factor", [0.0, 1e-3])
def test_qwen3_32b_nearly_flat_attention(q_factor):
    # zero (or tiny) queries: attention spreads evenly over all 100000 tokens, so the output, a mean
    # of zero-mean values, is ~300x smaller than the sums of P' code and p m_V the tensor-core kernel
    # adds up over each warp's run of about 200 pages: the hardest case for its accumulation
    _fused_steps("qwen3_32b", [(0, 0), (31, 7)], 2, q_factor=q_factor)
