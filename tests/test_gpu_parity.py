"""GPU parity: the CUDA write path is bit-exact against the CPU oracle (codes and fp16
scale/min of every INT2 token, BF16 sink/window bytes), and decode attention is within
relative L2 1e-3 and max-abs 2e-3 of the oracle's fp64 attention on the same cache.
Everything is called through the C ABI."""
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


PATHS = {"mma": K.PATH_WARP_MMA, "simt": K.PATH_SIMT}


@pytest.fixture(params=list(PATHS), autouse=True)
def decode_path(request):
    """Every test runs against each decode kernel: warp-level MMA and the SIMT baseline."""
    K.oscar_set_decode_path(PATHS[request.param])
    yield request.param
    K.oscar_set_decode_path(K.PATH_WARP_MMA)


def _attend(cache, q, rk_dev, out_dtype=torch.float32):
    out = torch.empty(q.shape, dtype=out_dtype, device="cuda")
    cache.attend(q, rk_dev, out)
    cache.status()          # raises if a bounded in-kernel wait gave up
    torch.cuda.synchronize()
    return out.float().cpu().numpy()


def _check_attention(out, q, ocs, cfg):
    g = cfg.group
    worst = 0.0
    for (b, h), oc in ocs.items():
        ref, _ = oc.attend(q[b, h * g:(h + 1) * g].cpu().numpy())
        got = out[b, h * g:(h + 1) * g]
        r = rel_l2(got, ref)
        m = float(np.abs(got - ref).max())
        worst = max(worst, r)
        assert r <= REL_L2 and m <= MAX_ABS, f"(b={b}, h={h}): rel-L2 {r:.3e}, max-abs {m:.3e}"
    return worst


def _run(cfg, lens, pairs=None, steps=2, chunks=None, table=None, check_bytes=True, out_dtype=torch.float32,
         groups=(64, 64), fused=False):
    rk = oracle_rk(cfg.seed, cfg.num_kv_heads, 1024)
    rk_dev = torch.tensor(rk, device="cuda")
    cache = make_cache(cfg, max(lens) + steps, table, *groups)
    append_initial(cache, cfg, lens, rk_dev, chunks)
    pairs = pairs or [(b, h) for b in range(cfg.batch) for h in range(cfg.num_kv_heads)]
    ocs = oracle_caches(cfg, pairs, lens, rk, *groups)
    cur = list(lens)
    for step in range(steps):
        if check_bytes:
            for (b, h), oc in ocs.items():
                check_int2_bytes(cache, oc, b, h)
                check_bf16_bytes(cache, oc, b, h)
        q = decode_query(cfg, step)
        if fused and step > 0:
            out = step_out
        else:
            out = _attend(cache, q, rk_dev, out_dtype)
        if out_dtype == torch.float32:
            _check_attention(out, q, ocs, cfg)
        else:
            g = cfg.group
            for (b, h), oc in ocs.items():
                ref, _ = oc.attend(q[b, h * g:(h + 1) * g].cpu().numpy())
                got = out[b, h * g:(h + 1) * g]
                # bf16 output = fp32-mode result rounded once more to 8 significant bits: its
                # error budget is the fp32-mode bar plus the bf16 unit roundoff 2^-8 per element
                r = rel_l2(got, ref)
                assert r <= REL_L2 + 2.0 ** -8, f"(b={b}, h={h}): rel-L2 {r:.3e}"
                assert (np.abs(got - ref) <= MAX_ABS + 2.0 ** -8 * np.abs(ref)).all()
        # one decode token per request, then the next step attends over it too
        n = [1] * cfg.batch
        k, v = synth.kv_block(cfg.seed, n, cur, cfg.num_kv_heads, device="cuda")
        if fused:
            # the next step's append and attention in one call (oscar_decode_step)
            qn = decode_query(cfg, step + 1)
            o = torch.empty(qn.shape, dtype=out_dtype, device="cuda")
            cache.step(k, v, qn, rk_dev, o)
            cache.status()
            torch.cuda.synchronize()
            step_out = o.float().cpu().numpy()
        else:
            cache.append(k, v, n, rk_dev)
        for (b, h), oc in ocs.items():
            oc.append(synth.bf16_bits(k[b, h][None]), synth.bf16_bits(v[b, h][None]))
        cur = [c + 1 for c in cur]
    return cache, ocs


def test_tiny_config_bulk_then_decode():
    cfg = synth.config("tiny")
    _run(cfg, cfg.ctx, steps=cfg.decode_steps)


def test_incremental_append_matches_bulk():
    cfg = synth.scaled(synth.config("qwen3_4b"), [700, 333, 321, 1024], batch=4)
    # chunked appends of odd sizes must store exactly what one bulk append stores
    _run(cfg, cfg.ctx, steps=1, chunks=[1, 7, 64, 100, 3, 300, 256])


@pytest.mark.parametrize("lens", [[0, 1, 63, 64], [65, 319, 320, 321], [383, 384, 385, 448],
                                  [320 + 64 * 5 - 1, 320 + 64 * 5, 320 + 64 * 5 + 1, 2]])
def test_lengths_at_region_and_page_edges(lens):
    cfg = synth.scaled(synth.config("qwen3_4b"), lens, batch=4)
    _run(cfg, lens, steps=3)


@pytest.mark.parametrize("hq,hkv", [(2, 2), (4, 2), (6, 2), (8, 2), (16, 2), (24, 2), (32, 2), (12, 2), (14, 2)])
def test_gqa_group_sizes(hq, hkv):
    base = synth.config("qwen3_4b")
    cfg = synth.LayerConfig("gqa", 2, hq, hkv, [1500, 900], 2, "permuted", "bf16", 4242)
    _run(cfg, cfg.ctx, steps=2)


@pytest.mark.parametrize("groups", [(64, 128), (128, 128), (128, 64)])
@pytest.mark.parametrize("hq,hkv", [(16, 2), (24, 2), (8, 2)])
def test_group_size_formats(groups, hq, hkv):
    # keys / values in groups of 64 or 128 channels: codes and scales bit-exact against the oracle's
    # grouped quantiser, attention against its grouped attention, through bulk appends, chunked
    # appends and fused decode steps
    cfg = synth.LayerConfig("groups", 3, hq, hkv, [1700, 383, 960], 4, "permuted", "bf16", 5150)
    _run(cfg, cfg.ctx, steps=4, chunks=[500, 1, 700, 1000], groups=groups, fused=True)


def test_qwen3_4b_shape_sampled_heads():
    cfg = synth.config("qwen3_4b")
    pairs = [(0, 0), (3, 5), (7, 7)]
    _run(cfg, cfg.ctx, pairs=pairs, steps=2)


def test_bf16_output_and_bf16_query():
    cfg = synth.scaled(synth.config("qwen3_8b"), [2000, 700], batch=2)
    _run(cfg, cfg.ctx, steps=1, out_dtype=torch.bfloat16)


def test_page_order_does_not_change_output():
    cfg = synth.scaled(synth.config("qwen3_4b"), [3000, 1400, 2500], batch=3)
    rk = oracle_rk(cfg.seed, cfg.num_kv_heads, 1024)
    rk_dev = torch.tensor(rk, device="cuda")
    outs = []
    for table in ("contiguous", "permuted"):
        cache = make_cache(cfg, max(cfg.ctx), table)
        append_initial(cache, cfg, cfg.ctx, rk_dev)
        q = decode_query(cfg, 0)
        outs.append(_attend(cache, q, rk_dev))
    assert np.array_equal(outs[0], outs[1])


def test_release_and_reuse_pages():
    cfg = synth.scaled(synth.config("qwen3_4b"), [900, 900], batch=2)
    rk = oracle_rk(cfg.seed, cfg.num_kv_heads, 1024)
    rk_dev = torch.tensor(rk, device="cuda")
    cache = make_cache(cfg, 1000)
    append_initial(cache, cfg, [900, 900], rk_dev)
    K.kv_page_table_release(cache.handle, 0)
    assert cache.length(0) == 0
    q = decode_query(cfg, 0)
    out = _attend(cache, q, rk_dev)
    assert np.all(out[0] == 0)                     # an empty request attends to nothing
    # refill request 0 with other tokens: pages come back from the free list
    k, v = synth.kv_block(cfg.seed + 1, [800, 0], [0, 0], cfg.num_kv_heads, device="cuda")
    cache.append(k, v, [800, 0], rk_dev)
    oc = oracle.OracleCache(rk[1])
    oc.append(synth.bf16_bits(k[:, 1]), synth.bf16_bits(v[:, 1]))
    check_int2_bytes(cache, oc, 0, 1)
    out = _attend(cache, q, rk_dev)
    ref, _ = oc.attend(q[0, cfg.group:2 * cfg.group].cpu().numpy())
    assert rel_l2(out[0, cfg.group:2 * cfg.group], ref) <= REL_L2


def test_build_rv_on_gpu_from_score_weighted_values():
    # the value rotation: rows of S V (attention outputs of calibration queries) as the samples
    hkv, n, t = 2, 2048, 600
    ys = []
    for h in range(hkv):
        rng = np.random.default_rng(100 + h)
        qc = rng.standard_normal((n, 128)) * np.linspace(2.0, 0.2, 128)
        kc = rng.standard_normal((t, 128))
        vc = rng.standard_normal((t, 128)) * np.exp(0.5 * rng.standard_normal(128))
        ys.append(oracle.score_weighted_values(qc, kc, vc).astype(np.float32))
    y = torch.tensor(np.stack(ys)).cuda().contiguous()
    rv = torch.empty(hkv, 128, 128, device="cuda")
    ws = torch.empty(K.oscar_build_rk_workspace_bytes(hkv), dtype=torch.uint8, device="cuda")
    K.oscar_build_rk(y, n, hkv, rv, ws)
    torch.cuda.synchronize()
    got = rv.cpu().numpy().astype(np.float64)
    for h in range(hkv):
        _, ref64, ev = oracle.build_rk(ys[h])         # the oracle's builder on the same samples
        assert np.abs(got[h] @ got[h].T - np.eye(128)).max() < 1e-6
        # invariants that hold whatever the eigen-gaps: R_V = U_S H P_br with H P_br known, so
        # U_S = R_V (H P_br)^T must diagonalise C_S with the oracle's eigenvalues, descending
        c = ys[h].astype(np.float64).T @ ys[h].astype(np.float64) / n
        hp = oracle.build_rk(np.eye(128, dtype=np.float32))[1]      # C = I/N: R = H P_br exactly
        u = got[h] @ hp.T
        lam = np.diag(u.T @ c @ u)
        off = u.T @ c @ u - np.diag(lam)
        assert np.abs(off).max() <= 1e-6 * np.abs(ev).max()
        assert np.abs(lam - ev).max() <= 1e-6 * np.abs(ev).max()
        # element-wise agreement with the oracle's vectors, where the eigen-gaps make them unique
        gap = np.minimum(np.r_[np.inf, -np.diff(ev)], np.r_[-np.diff(ev), np.inf])
        unique = gap > 1e-4 * np.abs(ev).max()
        u_ref = ref64 @ hp.T
        assert np.abs(u[:, unique] - u_ref[:, unique]).max() < 1e-5


def test_build_rk_on_gpu_matches_oracle():
    hkv, n = 4, 4096
    q = torch.stack([synth.calibration_queries(77, h, n) for h in range(hkv)]).cuda().contiguous()
    rk = torch.empty(hkv, 128, 128, device="cuda")
    ws = torch.empty(K.oscar_build_rk_workspace_bytes(hkv), dtype=torch.uint8, device="cuda")
    K.oscar_build_rk(q, n, hkv, rk, ws)
    torch.cuda.synchronize()
    got = rk.cpu().numpy().astype(np.float64)
    for h in range(hkv):
        ref32, ref64, _ = oracle.build_rk(q[h].cpu().numpy())
        assert np.abs(got[h] - ref64).max() < 1e-6
        assert np.abs(got[h] @ got[h].T - np.eye(128)).max() < 1e-6


def test_streaming_cq_accumulation_matches_the_oracle():
    # C_Q accumulated over three uneven calls, R_K built, then refreshed with more samples: each R_K
    # equals the oracle's R_K of all the samples seen so far
    hkv, n = 3, 4096
    q = torch.stack([synth.calibration_queries(91, h, 2 * n) for h in range(hkv)]).cuda().contiguous()
    acc = torch.empty(K.oscar_cq_accumulator_bytes(hkv), dtype=torch.uint8, device="cuda")
    ws = torch.empty(K.oscar_build_rk_workspace_bytes(hkv), dtype=torch.uint8, device="cuda")
    rk = torch.empty(hkv, 128, 128, device="cuda")
    K.oscar_cq_reset(acc, hkv)
    for a, b in [(0, 1000), (1000, 1001), (1001, n)]:
        K.oscar_cq_accumulate(q[:, a:b].contiguous(), b - a, hkv, acc)
    K.oscar_cq_accumulate(q[:, :0].contiguous(), 0, hkv, acc)        # an empty call changes nothing
    for upto in (n, 2 * n):
        if upto == 2 * n:
            K.oscar_cq_accumulate(q[:, n:].contiguous(), n, hkv, acc)
        K.oscar_cq_finalize(acc, hkv, rk, ws)
        torch.cuda.synchronize()
        got = rk.cpu().numpy().astype(np.float64)
        for h in range(hkv):
            _, ref64, _ = oracle.build_rk(q[h, :upto].cpu().numpy())
            assert np.abs(got[h] - ref64).max() < 1e-6
            assert np.abs(got[h] @ got[h].T - np.eye(128)).max() < 1e-6


def _calibration_set(seed, hkv, n, t):
    out = []
    for h in range(hkv):
        rng = np.random.default_rng(seed + h)
        qc = (rng.standard_normal((n, 128)) * np.linspace(2.0, 0.2, 128)).astype(np.float32)
        kc = rng.standard_normal((t, 128)).astype(np.float32)
        vc = (rng.standard_normal((t, 128)) * np.exp(0.5 * rng.standard_normal(128))).astype(np.float32)
        out.append((qc, kc, vc))
    return out


def test_score_weighted_values_on_gpu_match_the_oracle():
    hkv, n, t = 2, 1024, 600
    cal = _calibration_set(300, hkv, n, t)
    dq, dk, dv = (torch.tensor(np.stack([c[i] for c in cal])).cuda().contiguous() for i in range(3))
    y = torch.empty(hkv, n, 128, device="cuda")
    K.oscar_score_weighted_values(dq, n, dk, dv, t, hkv, y)
    torch.cuda.synchronize()
    got = y.cpu().numpy().astype(np.float64)
    for h in range(hkv):
        ref = oracle.score_weighted_values(*cal[h])
        assert np.abs(got[h] - ref).max() <= 1e-5 * np.abs(ref).max()


def test_value_rotation_built_on_gpu_and_a_layer_stored_through_it():
    # R_V entirely on the device (S V samples, then the eigen-solver), checked against the oracle's
    # R_V through invariants that hold whatever the eigen-gaps; then a layer whose values are stored
    # rotated (V' = X W_V R_V, the projection with R_V folded in) is checked like any other: codes
    # bit-exact and attention within tolerance against the oracle on the same cache, and the
    # absorbed output out' R_V^T W_O against the unrotated layer's fp64 attention (INT2 error only)
    hkv, n, t, dm = 2, 2048, 800, 256
    cal = _calibration_set(400, hkv, n, t)
    dq, dk, dv = (torch.tensor(np.stack([c[i] for c in cal])).cuda().contiguous() for i in range(3))
    y = torch.empty(hkv, n, 128, device="cuda")
    K.oscar_score_weighted_values(dq, n, dk, dv, t, hkv, y)
    rv = torch.empty(hkv, 128, 128, device="cuda")
    ws = torch.empty(K.oscar_build_rk_workspace_bytes(hkv), dtype=torch.uint8, device="cuda")
    K.oscar_build_rk(y, n, hkv, rv, ws)
    torch.cuda.synchronize()
    rvh = rv.cpu().numpy().astype(np.float64)
    hp = oracle.build_rk(np.eye(128, dtype=np.float32))[1]       # H P_br
    for h in range(hkv):
        cs = oracle.value_covariance(*cal[h])
        _, _, ev = oracle.build_rv(*cal[h])
        u = rvh[h] @ hp.T
        d = u.T @ cs @ u
        assert np.abs(d - np.diag(np.diag(d))).max() <= 1e-5 * ev.max()
        assert np.abs(np.diag(d) - ev).max() <= 1e-5 * ev.max()
    # the layer: hidden states X, projections W_V, W_O (random), R_V folded into W_V
    B, L, hq = 2, 1500, 16
    rng = np.random.default_rng(401)
    wv = rng.standard_normal((hkv, dm, 128)) / np.sqrt(dm)
    wo = rng.standard_normal((hkv, 128, dm)) / np.sqrt(128)
    x = rng.standard_normal((B, L + 1, dm))
    cfg = synth.LayerConfig("rv", B, hq, hkv, [L] * B, 1, "permuted", "fp32", 402)
    rk = oracle_rk(cfg.seed, hkv, 1024)
    rk_dev = torch.tensor(rk, device="cuda")
    cache = make_cache(cfg, L + 1)
    kb = synth.bf16_bits(torch.stack([torch.stack([synth.keys(cfg.seed, b, h, 0, L + 1) for h in range(hkv)], 1)
                                      for b in range(B)]))                       # [B, L + 1, hkv, 128]
    vrot = np.einsum("bld,hdc,hce->blhe", x, wv, rvh)                           # X W_V R_V
    vb = synth.bf16_bits(torch.tensor(vrot, dtype=torch.float32).to(torch.bfloat16))
    tens = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    cache.append(tens(kb[:, :L].reshape(B * L, hkv, 128)), tens(vb[:, :L].reshape(B * L, hkv, 128)), [L] * B, rk_dev)
    q = synth.queries(cfg.seed, 0, B, hq, hkv, device="cuda")
    out = torch.empty(B, hq, 128, device="cuda")
    cache.step(tens(kb[:, L]), tens(vb[:, L]), q, rk_dev, out)
    cache.status()
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    g = hq // hkv
    for b in range(B):
        for h in range(hkv):
            oc = oracle.OracleCache(rk[h])
            oc.append(kb[b, :, h], vb[b, :, h])
            check_int2_bytes(cache, oc, b, h)
            ref, _ = oc.attend(q[b, h * g:(h + 1) * g].cpu().numpy())
            r = rel_l2(got[b, h * g:(h + 1) * g], ref)
            assert r <= REL_L2 and np.abs(got[b, h * g:(h + 1) * g] - ref).max() <= MAX_ABS
            # absorption: out' R_V^T W_O against softmax attention over the unrotated X W_V (fp64,
            # unquantised); the difference is the INT2 quantisation error only
            v_plain = np.einsum("ld,dc->lc", x[b, :, :], wv[h])
            k_plain = synth.keys(cfg.seed, b, h, 0, L + 1).to(torch.bfloat16).float().numpy().astype(np.float64)
            qh = q[b, h * g:(h + 1) * g].cpu().numpy().astype(np.float64)
            logit = qh @ k_plain.T / np.sqrt(128)
            pm = np.exp(logit - logit.max(1, keepdims=True))
            pm /= pm.sum(1, keepdims=True)
            exact = pm @ v_plain @ wo[h]
            absorbed = got[b, h * g:(h + 1) * g].astype(np.float64) @ rvh[h].T @ wo[h]
            # the same layer stored without R_V (oracle): the rotation must not make the INT2 error worse
            vplain16 = synth.bf16_bits(torch.tensor(np.einsum("ld,dc->lc", x[b], wv[h]), dtype=torch.float32)
                                       .to(torch.bfloat16))
            op = oracle.OracleCache(rk[h])
            op.append(kb[b, :, h], vplain16)
            plain, _ = op.attend(q[b, h * g:(h + 1) * g].cpu().numpy())
            err_rot, err_plain = rel_l2(absorbed, exact), rel_l2(plain @ wo[h], exact)
            assert err_rot < 2.0 * err_plain + 0.01, (err_rot, err_plain)


@pytest.mark.parametrize("base", ["qwen3_4b", "qwen3_32b"])
def test_stale_nan_bf16_slots(base, decode_path):
    # The BF16 region starts as NaN bits, as a caller's uninitialised buffer may.  Slots the requests
    # have not reached (the rest of a partly filled sink or window tile) must not reach the attention:
    # the warp-MMA path runs P.V on the tensor cores, where a zero probability times NaN is still NaN.
    # Requests of 5 and 63 tokens end inside the sink, 70 and 300 inside the window; G = 4 and 8.
    lens = [5, 63, 70, 300]
    cfg = synth.scaled(synth.config(base), lens, batch=len(lens))
    rk = oracle_rk(cfg.seed, cfg.num_kv_heads, 1024)
    rk_dev = torch.tensor(rk, device="cuda")
    cache = make_cache(cfg, max(lens) + 2)
    cache.bf16.fill_(float("nan"))
    append_initial(cache, cfg, lens, rk_dev)
    pairs = [(b, h) for b in range(cfg.batch) for h in range(cfg.num_kv_heads)]
    ocs = oracle_caches(cfg, pairs, lens, rk)
    q = decode_query(cfg, 0)
    out = _attend(cache, q, rk_dev)
    assert np.isfinite(out).all()
    _check_attention(out, q, ocs, cfg)
    if decode_path == "mma":
        # chunked prefill over the same cache: the last n_q tokens of each request as the chunk
        n_q = [min(x, 4) for x in lens]
        g = cfg.group
        qg = torch.Generator(device="cpu").manual_seed(cfg.seed + 7)
        qp = (torch.randn(sum(n_q), cfg.num_q_heads, 128, generator=qg) * 0.7).cuda()
        po = torch.full_like(qp, float("nan"))
        ws = cache.prefill(qp, n_q, rk_dev, po)
        K.oscar_decode_status(cache.handle, ws)
        torch.cuda.synchronize()
        got, qh = po.cpu().numpy(), qp.cpu().numpy()
        assert np.isfinite(got).all()
        r0 = 0
        for b in range(cfg.batch):
            for h in range(cfg.num_kv_heads):
                for i in range(n_q[b]):
                    ref, _ = ocs[(b, h)].attend_upto(qh[r0 + i, h * g:(h + 1) * g], lens[b] - n_q[b] + i)
                    o = got[r0 + i, h * g:(h + 1) * g]
                    assert rel_l2(o, ref) <= REL_L2 and np.abs(o - ref).max() <= MAX_ABS, (b, h, i)
            r0 += n_q[b]
