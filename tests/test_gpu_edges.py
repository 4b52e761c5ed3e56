"""GPU parity on the quantiser's edge cases and at the numeric range limits of the read path.

The CUDA path is compared with the CPU oracle element by element on inputs the synthetic layers
never produce:
  * hand-built tokens whose 64-channel groups are constant (scale 0), sit exactly on rounding ties,
    are all positive or all negative, span fp16-extreme ranges (scales near 2^15 and in the fp16
    subnormals), or carry one huge outlier, with clip factors 1.0 and the defaults.  Keys are
    rotated by a signed permutation, an orthogonal R_K whose fp32 rotation is exact, so the rotated
    groups are exactly the hand-built ones;
  * the synthetic layers with keys, values or queries scaled by powers of ten from 1e-5 to 1e4, which
    drive the tensor-core kernel's fp16 operands (query high / low parts, P' = p * s_V) to both ends
    of their range.
Codes and fp16 scale/min are checked bit for bit, the BF16 region byte for byte, and attention
within rel-L2 1e-3 / max-abs 2e-3 against the oracle's fp64 attention on the same cache, on both
decode paths (G = 4 and 12 run the warp-MMA path's transposed-score kernel, G = 8 its query-as-A
kernel), through bulk appends and through fused decode steps (oscar_decode_step).
Source of the quantiser: axbrief.com OSCAR page, section "attention-statistics rotation + Triton
kernels" (per-token asymmetric INT2 in 64-channel groups, clip factors c_K, c_V).
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
D = 128


@pytest.fixture(scope="module", autouse=True)
def _built():
    from int2_rotated_paged_gb300 import build
    build.build()
    oracle.build()
    assert torch.cuda.is_available()


PATHS = {"mma": K.PATH_WARP_MMA, "simt": K.PATH_SIMT}


@pytest.fixture(params=list(PATHS), autouse=True)
def decode_path(request):
    K.oscar_set_decode_path(PATHS[request.param])
    yield request.param
    K.oscar_set_decode_path(K.PATH_WARP_MMA)


def _bf16(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (round to nearest even), through torch."""
    return synth.bf16_bits(torch.tensor(np.asarray(x, np.float32)).to(torch.bfloat16))


def _bits_tensor(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits, np.uint16).view(np.int16)).view(torch.bfloat16)


def signed_permutation(seed: int) -> np.ndarray:
    """R[j][pi(j)] = +-1: orthogonal, and k . R is exact in fp32 (one non-zero term per output)."""
    rng = np.random.default_rng(seed)
    pi = rng.permutation(D)
    r = np.zeros((D, D), np.float32)
    r[np.arange(D), pi] = rng.choice([-1.0, 1.0], D).astype(np.float32)
    return r


KINDS = ("constant", "ties", "positive", "negative", "large", "tiny", "normal", "outlier", "zero")


def edge_group(rng, kind: str) -> np.ndarray:
    """64 bf16-exact values of one quantisation group of the given kind."""
    n = 64
    if kind == "constant":
        return np.full(n, rng.choice([-3.25, 0.5, 17.0, 1024.0]), np.float32)
    if kind == "zero":
        return np.zeros(n, np.float32)
    if kind == "ties":
        # with clip 1: lo = a, hi = a + 3d, s = d exactly; the points a + (k + 1/2) d are rounding ties
        d = float(2.0 ** rng.integers(-6, 6))
        a = float(rng.integers(-8, 8)) * d
        pts = a + d * np.array([0.0, 0.5, 1.0, 1.5, 2.0, 2.5, 3.0])
        x = rng.choice(pts, n)
        x[0], x[1] = pts[0], pts[-1]
        return x.astype(np.float32)
    if kind == "positive":
        return rng.uniform(1.0, 5.0, n).astype(np.float32)
    if kind == "negative":
        return rng.uniform(-5.0, -1.0, n).astype(np.float32)
    if kind == "large":
        x = rng.uniform(-1.0, 1.0, n) * 3.0e4
        return x.astype(np.float32)
    if kind == "tiny":
        return (rng.standard_normal(n) * 2.0e-6).astype(np.float32)
    if kind == "outlier":
        x = rng.standard_normal(n)
        x[rng.integers(n)] = 900.0
        return x.astype(np.float32)
    return rng.standard_normal(n).astype(np.float32)


def edge_tokens(seed: int, n: int) -> np.ndarray:
    """n vectors of 128 channels whose two groups cycle through every edge kind."""
    rng = np.random.default_rng(seed)
    out = np.empty((n, D), np.float32)
    for t in range(n):
        out[t, :64] = edge_group(rng, KINDS[t % len(KINDS)])
        out[t, 64:] = edge_group(rng, KINDS[(t // len(KINDS) + 3 * t) % len(KINDS)])
    return out


def _run(hq, hkv, lens, kfn, vfn, qfn, rk, clip=(0.96, 0.92), steps=3, chunks=None):
    """Fill a cache with lens[b] tokens (bulk, or chunked appends), then `steps` fused decode steps;
    kfn / vfn (b, h, n_total) give bf16 bits [n_total, 128], qfn(step) fp32 queries [B, hq, 128].
    Every (request, KV head) pair is checked against its oracle cache."""
    B = len(lens)
    g = hq // hkv
    total = [L + steps for L in lens]
    kb = {(b, h): kfn(b, h, total[b]) for b in range(B) for h in range(hkv)}
    vb = {(b, h): vfn(b, h, total[b]) for b in range(B) for h in range(hkv)}
    per_seq = pages_needed(max(total)) + 1
    cache = K.Cache(B, hq, hkv, per_seq * B + 2, per_seq, page_order=synth.page_order(7, per_seq * B + 2, "permuted"),
                    clip_k=clip[0], clip_v=clip[1])
    rk_dev = torch.tensor(rk, device="cuda")

    def block(n, start):
        rows = sum(n)
        k = np.zeros((rows, hkv, D), np.uint16)
        v = np.zeros((rows, hkv, D), np.uint16)
        o = 0
        for b in range(B):
            for h in range(hkv):
                k[o:o + n[b], h] = kb[(b, h)][start[b]:start[b] + n[b]]
                v[o:o + n[b], h] = vb[(b, h)][start[b]:start[b] + n[b]]
            o += n[b]
        return _bits_tensor(k).cuda(), _bits_tensor(v).cuda()

    done = [0] * B
    for step in (chunks or [max(lens)]):
        n = [min(step, lens[b] - done[b]) for b in range(B)]
        if sum(n):
            k, v = block(n, done)
            cache.append(k, v, n, rk_dev)
            done = [done[b] + n[b] for b in range(B)]
    assert done == list(lens)
    ocs = {}
    for (b, h) in kb:
        oc = oracle.OracleCache(rk[h], clip_k=clip[0], clip_v=clip[1])
        if lens[b]:
            oc.append(kb[(b, h)][:lens[b]], vb[(b, h)][:lens[b]])
        ocs[(b, h)] = oc
    out = torch.empty(B, hq, D, device="cuda")
    for s in range(steps):
        q = qfn(s)
        k, v = block([1] * B, [lens[b] + s for b in range(B)])
        cache.step(k, v, q, rk_dev, out)
        cache.status()
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        assert np.isfinite(got).all(), f"step {s}: non-finite output"
        for (b, h), oc in ocs.items():
            oc.append(kb[(b, h)][lens[b] + s][None], vb[(b, h)][lens[b] + s][None])
            ref, _ = oc.attend(q[b, h * g:(h + 1) * g].cpu().numpy())
            r = rel_l2(got[b, h * g:(h + 1) * g], ref)
            m = float(np.abs(got[b, h * g:(h + 1) * g] - ref).max())
            scale = max(1.0, float(np.abs(ref).max()))
            assert r <= REL_L2 and m <= MAX_ABS * scale, f"step {s} (b={b}, h={h}): rel-L2 {r:.3e}, max-abs {m:.3e}"
    for (b, h), oc in ocs.items():
        check_int2_bytes(cache, oc, b, h)
        check_bf16_bytes(cache, oc, b, h)
    return cache, ocs


@pytest.mark.parametrize("clip", [(1.0, 1.0), (0.96, 0.92)])
@pytest.mark.parametrize("hq,hkv", [(8, 2), (16, 2), (24, 2)])
def test_edge_groups_bit_exact_and_attention(clip, hq, hkv):
    rk = np.stack([signed_permutation(11 + h) for h in range(hkv)])

    def kfn(b, h, n):
        # the hand-built vectors are the ROTATED keys: the input is y R^T (exact for a signed permutation)
        y = edge_tokens(1000 * b + 10 * h + 1, n)
        return _bf16(y @ rk[h].T)

    def vfn(b, h, n):
        return _bf16(edge_tokens(1000 * b + 10 * h + 2, n))

    rng = np.random.default_rng(5)

    def qfn(s):
        # small queries keep the logits of the 3e4-sized groups near 1, so attention stays spread
        return torch.tensor(rng.standard_normal((2, hq, D)).astype(np.float32) * 1e-4, device="cuda")

    cache, ocs = _run(hq, hkv, [320 + 64 * 6 + 13, 320 + 64 * 3], kfn, vfn, qfn, rk, clip=clip)
    # the edge kinds really were exercised: zero scales, and (clip 1) ties rounded to even
    kc, ks, vc, vs = K.oscar_read_int2(cache.handle, 0, 0, 64, 100)
    assert (vs[:, 0] == 0).any() and (vs[:, 0] != 0).any()
    assert (ks[:, 0] == 0).any()


def test_all_value_groups_constant():
    # every value group constant: s_V = 0 everywhere, the output is the softmax average of m_V
    hq, hkv = 16, 2
    rk = oracle_rk(3, hkv, 1024)

    def kfn(b, h, n):
        return synth.bf16_bits(synth.keys(3, b, h, 0, n))

    def vfn(b, h, n):
        x = np.repeat(np.random.default_rng(b * 7 + h).standard_normal((n, 2)), 64, axis=1)
        return _bf16(x)

    def qfn(s):
        return synth.queries(3, s, 2, hq, hkv, device="cuda")

    _run(hq, hkv, [1200, 700], kfn, vfn, qfn, rk)


SCALES = [("k", 1e-5), ("k", 1e-3), ("k", 1e-1), ("k", 10.0), ("k", 100.0),
          ("v", 1e-5), ("v", 1e-3), ("v", 1e-1), ("v", 10.0), ("v", 100.0), ("v", 1e3), ("v", 1e4),
          ("q", 1e-5), ("q", 1e-3), ("q", 1e-1), ("q", 10.0), ("q", 100.0), ("q", 1e3)]


@pytest.mark.parametrize("hq,hkv", [(8, 2), (16, 2), (24, 2)])
@pytest.mark.parametrize("which,factor", SCALES)
def test_scaled_inputs(which, factor, hq, hkv):
    seed = 4321
    rk = oracle_rk(seed, hkv, 1024)
    fk = factor if which == "k" else 1.0
    fv = factor if which == "v" else 1.0
    fq = factor if which == "q" else 1.0

    def kfn(b, h, n):
        return _bf16(synth.keys(seed, b, h, 0, n).float().numpy() * fk)

    def vfn(b, h, n):
        return _bf16(synth.values(seed, b, h, 0, n).float().numpy() * fv)

    def qfn(s):
        return synth.queries(seed, s, 2, hq, hkv, device="cuda") * fq

    _run(hq, hkv, [1500, 900], kfn, vfn, qfn, rk, steps=2, chunks=[700, 1000])


def test_value_scale_rising_across_pages():
    # value scales growing by 2^2 every page within one request (2^-9 .. 2^13): the kernel must keep
    # lowering its reference slack so that P' = p * s_V stays inside fp16
    hq, hkv = 16, 1
    rk = oracle_rk(9, hkv, 1024)
    L = 320 + 64 * 12

    def kfn(b, h, n):
        return synth.bf16_bits(synth.keys(9, b, h, 0, n))

    def vfn(b, h, n):
        x = synth.values(9, b, h, 0, n).float().numpy()
        page = np.clip((np.arange(n) - 64) // 64, 0, 11)
        return _bf16(x * (2.0 ** (2 * page - 9))[:, None].astype(np.float32))

    def qfn(s):
        return synth.queries(9, s, 1, hq, hkv, device="cuda")

    _run(hq, hkv, [L], kfn, vfn, qfn, rk, steps=2)


def _recorded_vmax(cache, B, hkv):
    """The largest-value-scale words the write path keeps after the lengths (fp16 bits)."""
    off = 4 * ((B + 3) // 4)                                   # int32 index of the first word
    return cache.seq_lens[off:off + B * hkv].cpu().numpy().view(np.uint32).reshape(B, hkv)


def _stored_vmax(cache, b, h, n_int2):
    """The largest fp16 value scale stored in the request's INT2 pages (bits), read back."""
    if n_int2 == 0:
        return 0
    _, _, _, vs = K.oscar_read_int2(cache.handle, b, h, 64, n_int2)
    return int(np.asarray(vs, np.uint16)[:, 0::2].max())


def test_recorded_value_scale_maxima_follow_appends_steps_and_release():
    # the read path takes its fp16 range limit for P' = p * s_V from these words, so each must be the
    # largest value scale of its (request, KV head) INT2 pages, grown by appends and fused decode steps,
    # and zeroed when the request is released
    hq, hkv, B = 16, 2, 3
    seed = 77
    rk = oracle_rk(seed, hkv, 1024)
    rk_dev = torch.tensor(rk, device="cuda")
    cache = K.Cache(B, hq, hkv, 3 * 40, 40)
    lens = [2500, 900, 330]
    k, v = synth.kv_block(seed, lens, [0] * B, hkv, device="cuda")
    v[:lens[0]] *= 100.0                      # request 0's values 100x larger than the others'
    cache.append(k, v, lens, rk_dev)
    torch.cuda.synchronize()
    rec = _recorded_vmax(cache, B, hkv)
    for b in range(B):
        for h in range(hkv):
            assert rec[b, h] == _stored_vmax(cache, b, h, max(0, lens[b] - 320)), (b, h)
    assert rec[2].max() > 0 and rec[0].min() > rec[1].max()
    # fused decode steps quantise the token leaving the window: one with 1000x larger values
    out = torch.empty(B, hq, 128, device="cuda")
    for s in range(3):
        k1, v1 = synth.kv_block(seed, [1] * B, [lens[b] + s for b in range(B)], hkv, device="cuda")
        q = synth.queries(seed, s, B, hq, hkv, device="cuda")
        if s == 0:
            v1 *= 1000.0   # enters the window now, leaves it 256 steps later: not quantised yet
        cache.step(k1, v1, q, rk_dev, out)
    torch.cuda.synchronize()
    lens = [L + 3 for L in lens]
    rec = _recorded_vmax(cache, B, hkv)
    for b in range(B):
        for h in range(hkv):
            assert rec[b, h] == _stored_vmax(cache, b, h, max(0, lens[b] - 320)), (b, h)
    # release request 1: its words are zeroed at the next sync, the others stay
    K.kv_page_table_release(cache.handle, 1)
    K.kv_page_table_sync(cache.handle)
    torch.cuda.synchronize()
    rec2 = _recorded_vmax(cache, B, hkv)
    assert (rec2[1] == 0).all() and (rec2[0] == rec[0]).all() and (rec2[2] == rec[2]).all()
    # refilled with small values, request 1 records only those
    k, v = synth.kv_block(seed + 1, [0, 700, 0], [0, 0, 0], hkv, device="cuda")
    cache.append(k, v * 0.01, [0, 700, 0], rk_dev)
    torch.cuda.synchronize()
    rec3 = _recorded_vmax(cache, B, hkv)
    for h in range(hkv):
        assert rec3[1, h] == _stored_vmax(cache, 1, h, 700 - 320)
    assert rec3[1].max() < rec[1].min()
