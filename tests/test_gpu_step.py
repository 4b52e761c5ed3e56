"""The fused decode step (oscar_decode_step) against the two calls it stands for: over enough
steps that every request evicts tokens and crosses an INT2 page boundary, the outputs, the INT2
pool and the BF16 region must be identical, byte for byte, to those of kv_quant_append followed by
oscar_decode_attention on a second cache fed the same tokens.  The two-call path is itself checked
against the oracle by the parity tests, so equality here carries that check over."""
import pytest
import torch

import synth
import int2_rotated_paged_gb300 as K
from gpu_util import append_initial, make_cache, oracle_rk

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("path", [K.PATH_WARP_MMA, K.PATH_SIMT])
@pytest.mark.parametrize("hq,hkv,lens", [
    (32, 8, [700, 321, 64, 1000]),        # G = 4: no eviction yet, first eviction, sink only, long
    (24, 2, [1500, 319]),                 # G = 12 (transposed tile layout of the MMA path)
    (16, 2, [320, 2000, 383]),            # G = 8
])
def test_fused_step_matches_append_then_attend(path, hq, hkv, lens):
    steps = 70
    cfg = synth.LayerConfig("step", len(lens), hq, hkv, lens, steps, "permuted", "bf16", 4711)
    rk = torch.tensor(oracle_rk(cfg.seed, hkv), device="cuda")
    K.oscar_set_decode_path(path)
    try:
        two = make_cache(cfg, max(lens) + steps + 64)
        one = make_cache(cfg, max(lens) + steps + 64)
        for c in (two, one):
            c.pool.zero_()
            append_initial(c, cfg, lens, rk)
        B = len(lens)
        out_two = torch.empty(B, hq, 128, device="cuda")
        out_one = torch.empty_like(out_two)
        for s in range(steps):
            q = synth.queries(cfg.seed, s, B, hq, hkv, dtype=cfg.q_dtype, device="cuda")
            k, v = synth.kv_block(cfg.seed, [1] * B, [lens[b] + s for b in range(B)], hkv, device="cuda")
            two.append(k, v, [1] * B, rk)
            two.attend(q, rk, out_two)
            one.step(k, v, q, rk, out_one)
            assert torch.equal(out_two, out_one), f"step {s}"
        torch.cuda.synchronize()
        assert [two.length(b) for b in range(B)] == [one.length(b) for b in range(B)] == [n + steps for n in lens]
        assert torch.equal(two.seq_lens, one.seq_lens)
        assert torch.equal(two.page_table, one.page_table)
        assert torch.equal(two.pool, one.pool)
        assert torch.equal(two.bf16, one.bf16)
        one.status()
    finally:
        K.oscar_set_decode_path(K.PATH_WARP_MMA)


@pytest.mark.parametrize("pinned", [True, False])
def test_host_buffer_step_matches_device_step(pinned):
    # oscar_decode_step_host: the step's q, k, v and output in host memory (page-locked or pageable);
    # outputs and cache bytes must equal those of oscar_decode_step on device copies
    hq, hkv, lens, steps = 16, 2, [900, 330, 2000], 12
    cfg = synth.LayerConfig("host", len(lens), hq, hkv, lens, steps, "permuted", "bf16", 4712)
    rk = torch.tensor(oracle_rk(cfg.seed, hkv, 1024), device="cuda")
    dev_c = make_cache(cfg, max(lens) + steps + 64)
    host_c = make_cache(cfg, max(lens) + steps + 64)
    for c in (dev_c, host_c):
        c.pool.zero_()
        append_initial(c, cfg, lens, rk)
    B = len(lens)
    out_dev = torch.empty(B, hq, 128, device="cuda")
    out_host = torch.empty(B, hq, 128, pin_memory=pinned)
    staging = None
    for s in range(steps):
        q = synth.queries(cfg.seed, s, B, hq, hkv, dtype="bf16", device="cuda").to(torch.bfloat16)
        k, v = synth.kv_block(cfg.seed, [1] * B, [lens[b] + s for b in range(B)], hkv, device="cuda")
        dev_c.step(k, v, q, rk, out_dev)
        if staging is None:
            staging = torch.empty(K.oscar_decode_step_host_staging_bytes(host_c.handle, K.DTYPE_BF16, K.DTYPE_F32),
                                  dtype=torch.uint8, device="cuda")
        qh, kh, vh = (t.contiguous().cpu() for t in (q, k, v))
        if pinned:
            qh, kh, vh = qh.pin_memory(), kh.pin_memory(), vh.pin_memory()
        assert qh.dtype == torch.bfloat16 and kh.dtype == torch.bfloat16
        K.oscar_decode_step_host(host_c.handle, kh, vh, qh, K.DTYPE_BF16, rk, out_host, K.DTYPE_F32, staging,
                                 host_c.workspace)
        torch.cuda.synchronize()
        assert torch.equal(out_dev.cpu(), out_host), f"step {s}"
    for name in ("seq_lens", "page_table", "pool", "bf16"):
        assert torch.equal(getattr(dev_c, name), getattr(host_c, name)), name
    host_c.status()
    # argument errors before anything is enqueued: a short staging buffer, a missing host buffer
    qh = torch.zeros(B, hq, 128, dtype=torch.bfloat16)
    kh = torch.zeros(B, hkv, 128, dtype=torch.bfloat16)
    with pytest.raises(K.OscarError) as e:
        K.oscar_decode_step_host(host_c.handle, kh, kh, qh, K.DTYPE_BF16, rk, out_host, K.DTYPE_F32, staging[:256],
                                 host_c.workspace)
    assert e.value.code == K.OSCAR_EWORKSPACE
    with pytest.raises(K.OscarError) as e:
        K.oscar_decode_step_host(host_c.handle, kh, None, qh, K.DTYPE_BF16, rk, out_host, K.DTYPE_F32, staging,
                                 host_c.workspace)
    assert e.value.code == K.OSCAR_EINVAL
    assert [host_c.length(b) for b in range(B)] == [n + steps for n in lens]
