"""oscar_decode_attention_noalloc: decode attention for callers that cannot allocate.

Some callers run attention where no device allocation is possible: inside an inference
engine's plugin hook that forbids allocation, in a real-time loop that must not touch the
allocator, or next to another runtime that has already reserved all device memory.  For them
the library offers a variant that takes no workspace and uses one fixed scratch array built
into the library.  These tests check, through the C ABI, that it returns what the regular
entry point returns (same tolerance as the other parity tests) on two calls in a row, that a
warm call changes neither torch's allocator nor the device's free memory, that a bounded
in-kernel wait that runs out is reported by oscar_decode_status_noalloc (and the next call is
correct again), and that a call too large for the fixed scratch is refused before anything is
enqueued.
"""
import numpy as np
import pytest
import torch

import synth
import int2_rotated_paged_gb300 as K
from gpu_util import append_initial, decode_query, make_cache, oracle_rk, rel_l2

pytestmark = pytest.mark.gpu

REL_L2 = 1e-3
MAX_ABS = 2e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    from int2_rotated_paged_gb300 import build
    build.build()
    assert torch.cuda.is_available()
    K.oscar_set_decode_path(K.PATH_WARP_MMA)     # the path the fixed-scratch variant always uses


def test_noalloc_matches_regular_entry_point_twice():
    cfg = synth.scaled(synth.config("qwen3_4b"), [2500, 900, 4000], batch=3)
    rk = torch.tensor(oracle_rk(cfg.seed, cfg.num_kv_heads, 1024), device="cuda")
    cache = make_cache(cfg, max(cfg.ctx) + 2)
    append_initial(cache, cfg, cfg.ctx, rk)
    for step in range(2):                                   # two calls in a row, different queries
        q = decode_query(cfg, step)
        ref = torch.empty_like(q)
        got = torch.full_like(q, float("nan"))
        cache.attend(q, rk, ref)
        K.oscar_decode_attention_noalloc(cache.handle, q, K.DTYPE_F32, rk, got, K.DTYPE_F32)
        torch.cuda.synchronize()
        r, g = ref.cpu().numpy(), got.cpu().numpy()
        assert np.isfinite(g).all()
        assert rel_l2(g, r) <= REL_L2 and np.abs(g - r).max() <= MAX_ABS


def test_noalloc_allocates_nothing():
    cfg = synth.scaled(synth.config("qwen3_4b"), [3000, 1200], batch=2)
    rk = torch.tensor(oracle_rk(cfg.seed, cfg.num_kv_heads, 1024), device="cuda")
    cache = make_cache(cfg, max(cfg.ctx) + 2)
    append_initial(cache, cfg, cfg.ctx, rk)
    q = decode_query(cfg, 0)
    out = torch.empty_like(q)
    K.oscar_decode_attention_noalloc(cache.handle, q, K.DTYPE_F32, rk, out, K.DTYPE_F32)   # warm
    torch.cuda.synchronize()
    alloc0 = torch.cuda.memory_allocated()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        K.oscar_decode_attention_noalloc(cache.handle, q, K.DTYPE_F32, rk, out, K.DTYPE_F32)
    torch.cuda.synchronize()                 # raises if the calls left a CUDA error behind
    K.oscar_decode_status_noalloc()
    assert torch.cuda.memory_allocated() == alloc0
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0


def test_noalloc_reports_a_wait_that_ran_out():
    # the probe makes the call's first kernel wait on a barrier nothing arrives at, with a short
    # limit (5 tests of up to 1 ms): the wait runs out, the call must report OSCAR_ETIMEOUT through
    # the status query, and the next call, without the probe, must be correct again
    cfg = synth.scaled(synth.config("qwen3_4b"), [2500, 900], batch=2)
    rk = torch.tensor(oracle_rk(cfg.seed, cfg.num_kv_heads, 1024), device="cuda")
    cache = make_cache(cfg, max(cfg.ctx) + 2)
    append_initial(cache, cfg, cfg.ctx, rk)
    q = decode_query(cfg, 0)
    ref = torch.empty_like(q)
    cache.attend(q, rk, ref)
    got = torch.empty_like(q)
    K.oscar_set_wait_limit(5)
    K.oscar_set_wait_probe(True)
    try:
        K.oscar_decode_attention_noalloc(cache.handle, q, K.DTYPE_F32, rk, got, K.DTYPE_F32)
        with pytest.raises(K.OscarError) as e:
            K.oscar_decode_status_noalloc()
        assert e.value.code == K.OSCAR_ETIMEOUT
    finally:
        K.oscar_set_wait_probe(False)
        K.oscar_set_wait_limit(-1)
    torch.cuda.synchronize()
    K.oscar_decode_attention_noalloc(cache.handle, q, K.DTYPE_F32, rk, got, K.DTYPE_F32)
    K.oscar_decode_status_noalloc()
    r, g = ref.cpu().numpy(), got.cpu().numpy()
    assert rel_l2(g, r) <= REL_L2 and np.abs(g - r).max() <= MAX_ABS


def test_noalloc_refuses_calls_beyond_its_scratch():
    # 256 requests x 128 query heads need 16 MiB for the rotated queries alone
    cache = K.Cache(256, 128, 8, 256 * 2, 2)
    k, v = synth.kv_block(3, [400] * 256, [0] * 256, 8, device="cuda")
    rk = torch.eye(128, device="cuda").repeat(8, 1, 1).contiguous()
    cache.append(k, v, [400] * 256, rk)
    q = torch.zeros(256, 128, 128, device="cuda")
    out = torch.zeros_like(q)
    with pytest.raises(K.OscarError) as e:
        K.oscar_decode_attention_noalloc(cache.handle, q, K.DTYPE_F32, rk, out, K.DTYPE_F32)
    assert e.value.code == K.OSCAR_ESCRATCH
