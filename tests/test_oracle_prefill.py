"""Pins of the oracle's causal view of the mixed-precision cache (chunked prefill): query i of a chunk
appended as a whole attends to positions 0 .. L + i, each at the precision the cache holds it in.

  * the last query of the chunk sees the whole cache: the same result as the pinned decode
    attention (attend);
  * a cache that is all sink + window (no INT2 token) gives plain causal attention over the BF16
    tokens (torch SDPA with a causal mask, in fp64);
  * the tokens a query cannot see do not matter: changing them leaves its output unchanged.
"""
import numpy as np
import pytest
import torch

import oracle

D = 128


def _bf16(x):
    return torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _cache(L, seed, rk=None):
    rng = np.random.default_rng(seed)
    oc = oracle.OracleCache(rk)
    k = _bf16(rng.standard_normal((L, D)))
    v = _bf16(rng.standard_normal((L, D)))
    oc.append(k, v)
    return oc, k, v


def test_last_query_of_a_chunk_sees_the_whole_cache():
    rng = np.random.default_rng(3)
    r, _ = np.linalg.qr(rng.standard_normal((D, D)))
    oc, _, _ = _cache(1000, 4, r.astype(np.float32))
    q = rng.standard_normal((4, D)).astype(np.float32)
    a, _ = oc.attend(q)
    b, _ = oc.attend_upto(q, oc.length - 1)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("L,last", [(300, 250), (320, 100), (200, 0), (320, 319)])
def test_bf16_only_cache_is_plain_causal_attention(L, last):
    oc, k, v = _cache(L, 5)
    rng = np.random.default_rng(6)
    q = rng.standard_normal((3, D)).astype(np.float32)
    got, _ = oc.attend_upto(q, last)
    kf = torch.tensor(k.view(np.int16)).view(torch.bfloat16).double()[: last + 1]
    vf = torch.tensor(v.view(np.int16)).view(torch.bfloat16).double()[: last + 1]
    ref = torch.nn.functional.scaled_dot_product_attention(torch.tensor(q).double()[None], kf[None], vf[None])[0]
    assert np.abs(got - ref.numpy()).max() < 1e-12


def test_positions_after_the_query_do_not_matter():
    rng = np.random.default_rng(8)
    r, _ = np.linalg.qr(rng.standard_normal((D, D)))
    oc1, k, v = _cache(900, 9, r.astype(np.float32))
    k2, v2 = k.copy(), v.copy()
    k2[800:] = _bf16(rng.standard_normal((100, D)) * 5)       # positions after 799 differ
    v2[800:] = _bf16(rng.standard_normal((100, D)) * 5)
    oc2 = oracle.OracleCache(r.astype(np.float32))
    oc2.append(k2, v2)
    q = rng.standard_normal((2, D)).astype(np.float32)
    a, _ = oc1.attend_upto(q, 799)
    b, _ = oc2.attend_upto(q, 799)
    assert np.array_equal(a, b)
