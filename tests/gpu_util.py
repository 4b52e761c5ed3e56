"""Helpers shared by the GPU parity tests: build a cache for a workload, fill it, run
decode steps through the C ABI and mirror the same tokens in the CPU oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth
import int2_rotated_paged_gb300 as K

D = 128


def pages_needed(length: int) -> int:
    return max(0, (length - 320 + 63) // 64)


def oracle_rk(seed: int, hkv: int, n: int = 4096) -> np.ndarray:
    """R_K of every KV head from the oracle (an input of both sides)."""
    return np.stack([oracle.build_rk(synth.calibration_queries(seed, h, n).numpy())[0] for h in range(hkv)])


def make_cache(cfg: synth.LayerConfig, max_len: int, table: str | None = None, group_k: int = 64,
               group_v: int = 64) -> K.Cache:
    per_seq = pages_needed(max_len) + 1
    total = per_seq * cfg.batch + 3
    order = synth.page_order(cfg.seed, total, table or cfg.table)
    return K.Cache(cfg.batch, cfg.num_q_heads, cfg.num_kv_heads, total, per_seq, page_order=order,
                   group_k=group_k, group_v=group_v)


def append_initial(cache: K.Cache, cfg: synth.LayerConfig, lens, rk_dev, chunks=None):
    """Append lens[b] tokens per request (positions 0 ..); `chunks` splits the append."""
    lens = list(lens)
    done = [0] * len(lens)
    plan = chunks or [max(lens) if lens else 0]
    for step in plan:
        n = [min(step, lens[b] - done[b]) for b in range(len(lens))]
        if sum(n) == 0:
            continue
        k, v = synth.kv_block(cfg.seed, n, done, cfg.num_kv_heads, device="cuda")
        cache.append(k, v, n, rk_dev)
        done = [done[b] + n[b] for b in range(len(lens))]
    while any(done[b] < lens[b] for b in range(len(lens))):
        n = [lens[b] - done[b] for b in range(len(lens))]
        k, v = synth.kv_block(cfg.seed, n, done, cfg.num_kv_heads, device="cuda")
        cache.append(k, v, n, rk_dev)
        done = list(lens)


def oracle_caches(cfg: synth.LayerConfig, pairs, lens, rk: np.ndarray, group_k: int = 64, group_v: int = 64):
    """OracleCache per (b, h) in `pairs`, filled with the same tokens (drawn like the cache's)."""
    out = {}
    for (b, h) in pairs:
        oc = oracle.OracleCache(rk[h], group_k=group_k, group_v=group_v)
        if lens[b]:
            k16 = synth.bf16_bits(synth.keys(cfg.seed, b, h, 0, lens[b], device="cuda"))
            v16 = synth.bf16_bits(synth.values(cfg.seed, b, h, 0, lens[b], device="cuda"))
            oc.append(k16, v16)
        out[(b, h)] = oc
    return out


def rel_l2(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def check_int2_bytes(cache: K.Cache, oc: oracle.OracleCache, b: int, h: int):
    n = oc.kc.shape[0]
    if n == 0:
        return
    kc, ks, vc, vs = cache.read_int2(b, h, 64, n)
    for name, got, ref in (("k codes", kc, oc.kc), ("k scale/min", ks, oc.ks),
                           ("v codes", vc, oc.vc), ("v scale/min", vs, oc.vs)):
        if not np.array_equal(got, ref):
            bad = np.argwhere(got != ref)
            raise AssertionError(f"{name} differ at (b={b}, h={h}): first {bad[:5].tolist()} of {len(bad)}")


def check_bf16_bytes(cache: K.Cache, oc: oracle.OracleCache, b: int, h: int):
    (s0, s1), _, (w0, w1), _ = oracle.regions(oc.length)
    kb, vb = oc.bf16_tokens()
    got_k, got_v = [], []
    if s1 > s0:
        k, v = K.oscar_read_bf16(cache.handle, b, h, s0, s1 - s0)
        got_k.append(k)
        got_v.append(v)
    if w1 > w0:
        k, v = K.oscar_read_bf16(cache.handle, b, h, w0, w1 - w0)
        got_k.append(k)
        got_v.append(v)
    if got_k:
        assert np.array_equal(np.concatenate(got_k), kb)
        assert np.array_equal(np.concatenate(got_v), vb)


def decode_query(cfg: synth.LayerConfig, step: int, device="cuda") -> torch.Tensor:
    return synth.queries(cfg.seed, step, cfg.batch, cfg.num_q_heads, cfg.num_kv_heads,
                         dtype=cfg.q_dtype, device=device)
