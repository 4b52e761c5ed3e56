"""Pins of the CPU oracle to facts outside itself (CPU only).

Each test checks the oracle against a library routine, a closed form, an
invariant, a hand-derived example or brute force, so that a dropped term, a
wrong sign or index, or a transposed operand in the oracle fails here.
"""
import os

import numpy as np
import pytest
import scipy.linalg
import scipy.special
import torch

import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
D = 128


def _golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, *v = line.split()
            out[k] = v
    return out


def _bf16(x):
    return synth.bf16_bits(torch.as_tensor(np.asarray(x, np.float32)).to(torch.bfloat16))


# ------------------------------------------------------------------ number formats

def test_f32_to_f16_matches_numpy(orc):
    rng = np.random.default_rng(1)
    mags = rng.integers(-30, 18, 6000)
    x = (rng.standard_normal(6000) * np.exp2(mags)).astype(np.float32)
    # exact ties between two fp16 neighbours, subnormals, and the overflow edge
    ties = (np.arange(1024, 1100) + 0.5) * 2.0 ** -10
    sub = (np.arange(0, 64) + 0.5) * 2.0 ** -24
    edge = np.array([65504.0, 65519.99, 65520.0, 65536.0, 6.1035156e-05, 5.96e-08, 2.98e-08, 0.0, -0.0])
    x = np.concatenate([x, ties, -ties, sub, edge]).astype(np.float32)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    mine = np.array([orc.f32_to_f16_bits(v) for v in x], np.uint16)
    assert np.array_equal(mine, ref)


def test_f16_to_f32_all_patterns(orc):
    bits = np.arange(0, 65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    mine = np.array([orc.f16_bits_to_f32(int(b)) for b in bits[::7]], np.float32)
    r = ref[::7]
    ok = np.isnan(r) & np.isnan(mine) | (mine == r)
    assert ok.all()


# ------------------------------------------------------------------ rotation pieces

def test_hadamard_closed_form(orc):
    h = orc.hadamard128()
    assert np.array_equal(h, scipy.linalg.hadamard(128).astype(np.float64) / np.sqrt(128.0))
    # Sylvester recursion H_2n = [[H, H], [H, -H]], built independently
    s = np.array([[1.0]])
    while s.shape[0] < 128:
        s = np.block([[s, s], [s, -s]])
    assert np.allclose(h, s / np.sqrt(128.0), atol=0, rtol=0)
    assert np.abs(h @ h.T - np.eye(128)).max() < 1e-14


def test_bitrev7(orc):
    table = [int(format(i, "07b")[::-1], 2) for i in range(128)]
    assert [orc.bitrev7(i) for i in range(128)] == table
    assert orc.bitrev7(1) == 64 and orc.bitrev7(3) == 96 and orc.bitrev7(127) == 127
    assert all(orc.bitrev7(orc.bitrev7(i)) == i for i in range(128))


def test_query_covariance_vs_matmul(orc):
    q = synth.calibration_queries(7, 0, 512).numpy()
    c = orc.query_covariance(q)
    ref = q.astype(np.float64).T @ q.astype(np.float64) / q.shape[0]
    assert np.abs(c - ref).max() < 1e-12 * np.abs(ref).max()


def test_jacobi_vs_lapack(orc):
    rng = np.random.default_rng(3)
    a = rng.standard_normal((128, 128))
    a = a @ a.T / 128.0
    ev, v, sweeps = orc.jacobi_eigh(a)
    assert sweeps < 30
    w, u = np.linalg.eigh(a)
    w, u = w[::-1], u[:, ::-1]
    assert np.abs(ev - w).max() < 1e-12 * w.max()
    assert np.all(np.diff(ev) <= 0)
    assert np.abs(v.T @ v - np.eye(128)).max() < 1e-12
    assert np.abs(a @ v - v * ev).max() < 1e-10 * np.abs(a).max()
    # same eigenvectors up to sign; the oracle's sign makes the largest entry positive
    for j in range(128):
        col = u[:, j] * np.sign(u[np.argmax(np.abs(u[:, j])), j])
        assert np.abs(col - v[:, j]).max() < 1e-8
        assert v[np.argmax(np.abs(v[:, j])), j] > 0


def test_rk_orthogonal_and_eigenbasis(orc):
    q = synth.calibration_queries(11, 0, 4096).numpy()
    r32, r64, ev = orc.build_rk(q)
    assert np.abs(r32.astype(np.float64) @ r32.astype(np.float64).T - np.eye(128)).max() < 1e-6
    # undo P_br and H: U = R P_br^T H^T must diagonalise C_Q with the returned spectrum
    h = scipy.linalg.hadamard(128) / np.sqrt(128.0)
    perm = [int(format(i, "07b")[::-1], 2) for i in range(128)]
    p = np.zeros((128, 128))
    p[np.arange(128), perm] = 1.0
    u = r64 @ p.T @ h.T
    c = q.astype(np.float64).T @ q.astype(np.float64) / q.shape[0]
    assert np.abs(c @ u - u * ev).max() < 1e-9 * ev[0]
    assert np.allclose(ev, np.linalg.eigvalsh(c)[::-1], rtol=1e-10, atol=1e-12)


def test_rk_special_case_diagonal_covariance(orc):
    # Queries along the coordinate axes with decreasing energy: C_Q is diagonal and
    # descending, so U_Q = I and R_K = H P_br, i.e. R[r][c] = H[r][bitrev7(c)].
    lam = np.linspace(4.0, 1.0, 128)
    q = np.diag(np.sqrt(lam * 128)).astype(np.float32)          # (1/128) sum q^T q = diag(lam)
    r32, r64, ev = orc.build_rk(q)
    h = scipy.linalg.hadamard(128) / np.sqrt(128.0)
    perm = [int(format(i, "07b")[::-1], 2) for i in range(128)]
    assert np.abs(r64 - h[:, perm]).max() < 1e-12
    # a permuted diagonal: U_Q is that permutation (the axis with the largest energy first)
    order = np.random.default_rng(5).permutation(128)
    q2 = np.zeros((128, 128), np.float32)
    q2[np.arange(128), order] = np.sqrt(lam * 128)
    _, r64b, _ = orc.build_rk(q2)
    u = np.zeros((128, 128))
    u[order, np.arange(128)] = 1.0
    assert np.abs(r64b - (u @ h)[:, perm]).max() < 1e-12


def test_rotate_is_row_vector_times_rk(orc):
    q = synth.calibration_queries(13, 0, 1024).numpy()
    r32, _, _ = orc.build_rk(q)
    x = synth.keys(13, 0, 0, 0, 16).float().numpy()
    for t in range(16):
        y = orc.rotate_f32(x[t], r32)
        ref = x[t].astype(np.float64) @ r32.astype(np.float64)
        assert np.abs(y - ref).max() <= 1e-5 * np.abs(ref).max()
    # R_K is not symmetric, so the transposed product is far away
    assert np.abs(x[0] @ r32 - r32 @ x[0]).max() > 1.0


def test_rotate_is_the_serial_fused_chain_from_plus_zero(orc):
    """Closed-form cases of the write contract: each rotated channel is acc = fma(x_j, R[j][c], acc)
    over j = 0..127 in ascending order, from acc = +0, rounding once per step (fp32, nearest-even).
    Column 0 pins the order: x = (1, 2^-24 x 127) against a column of ones adds 2^-24 to 1 at every
    step, an exact tie that rounds back to 1, so the result is exactly 1; any other order (or a wider
    accumulator) adds the small terms first and gives 1 + 2^-17.  Column 1 pins the fusion:
    acc = -(1 + 2^-11) after j = 0, then x_1 R_11 = (1 + 2^-12)^2 = 1 + 2^-11 + 2^-24, so the fused
    step gives 2^-24 exactly while a rounded product first gives 0.  Column 2 pins the start value:
    a chain of -1 x +0 products ends at +0 only if it starts from +0."""
    x = np.zeros(128, np.float32)
    r = np.zeros((128, 128), np.float32)
    # column 0: order
    x0 = np.full(128, 2.0 ** -24, np.float32)
    x0[0] = 1.0
    r[:, 0] = 1.0
    y = orc.rotate_f32(x0, r)
    assert y[0] == np.float32(1.0)
    assert np.float32(np.sum(x0.astype(np.float64))) != np.float32(1.0)   # what a wider sum gives
    # column 1: fused multiply-add
    x1 = np.zeros(128, np.float32)
    x1[0], x1[1] = -(1.0 + 2.0 ** -11), 1.0 + 2.0 ** -12
    r1 = np.zeros((128, 128), np.float32)
    r1[0, 1], r1[1, 1] = 1.0, 1.0 + 2.0 ** -12
    y1 = orc.rotate_f32(x1, r1)
    assert y1[1] == np.float32(2.0 ** -24)
    assert np.float32(x1[1]) * np.float32(r1[1, 1]) + np.float32(x1[0]) == np.float32(0.0)   # split
    # column 2: the chain starts from +0 (every product is -1 x +0 = -0; -0 + -0 stays -0, so only a
    # +0 start ends at +0)
    x2 = np.full(128, -1.0, np.float32)
    y2 = orc.rotate_f32(x2, np.zeros((128, 128), np.float32))
    assert y2[2] == 0.0 and not np.signbit(y2[2])


# ------------------------------------------------------------------ quantiser

def test_golden_grid_example(orc):
    g = _golden("int2_grid_example.txt")
    c = np.arange(128)
    x = np.where(c < 64, -1.0 + 0.5 * (c % 4), 2.0 - 0.25 * (c % 4))
    codes, sm = orc.quant_tokens(_bf16(x)[None, :], None, 1.0)
    assert list(codes[0, :16]) == [int(g["group0_byte"][0], 16)] * 16
    assert list(codes[0, 16:]) == [int(g["group1_byte"][0], 16)] * 16
    assert list(sm[0]) == [int(v, 16) for v in g["sm"]]
    assert np.array_equal(orc.dequant_tokens(codes, sm)[0], x)


def _grid_group(rng, n):
    """Vectors whose groups sit exactly on a 4-level grid with fp16-exact m and s."""
    out = np.empty((n, 128), np.float32)
    codes = rng.integers(0, 4, (n, 128))
    codes[:, 0] = 0
    codes[:, 1] = 3
    codes[:, 64] = 0
    codes[:, 65] = 3
    for t in range(n):
        for g in range(2):
            s = float(2.0 ** rng.integers(-6, 3)) * (1, 3)[rng.integers(0, 2)]
            m = float(rng.integers(-8, 9)) * s      # (j + code) * s has at most 6 significant bits
            out[t, 64 * g:64 * g + 64] = m + codes[t, 64 * g:64 * g + 64] * s
    return out, codes


def test_round_trip_exact_on_grid(orc):
    rng = np.random.default_rng(17)
    x, codes = _grid_group(rng, 200)
    x16 = _bf16(x)
    xb = (x16.astype(np.uint32) << 16).view(np.float32)
    assert np.array_equal(xb, x), "grid must be bf16-exact"
    pc, sm = orc.quant_tokens(x16, None, 1.0)
    assert np.array_equal(orc.dequant_tokens(pc, sm), x.astype(np.float64))
    unpacked = (pc[:, :, None] >> (2 * np.arange(4))[None, None, :]) & 3
    assert np.array_equal(unpacked.reshape(-1, 128), codes)


def _quant_cases(rng, n):
    sig = np.exp(0.5 * rng.standard_normal(128))
    x = rng.standard_normal((n, 128)) * sig * 2.0 ** rng.integers(-8, 8, (n, 1))
    return _bf16(x)


@pytest.mark.parametrize("clip", [1.0, 0.96, 0.92])
def test_brute_force_nearest_level(orc, clip):
    rng = np.random.default_rng(23)
    x16 = _quant_cases(rng, 400)
    codes, sm = orc.quant_tokens(x16, None, clip)
    x = (x16.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    code = ((codes[:, :, None] >> (2 * np.arange(4))) & 3).reshape(-1, 128)
    assert code.min() >= 0 and code.max() <= 3
    n_ties = 0
    for g in range(2):
        sl = slice(64 * g, 64 * g + 64)
        xs = x[:, sl]
        cf = np.float32(clip)
        lo = (cf * xs.min(1).astype(np.float32)).astype(np.float64)
        hi = (cf * xs.max(1).astype(np.float32)).astype(np.float64)
        s = sm[:, 2 * g].view(np.float16).astype(np.float64)
        m = sm[:, 2 * g + 1].view(np.float16).astype(np.float64)
        # stored values are the fp16 rounding of the clipped range and its low end
        assert np.array_equal(sm[:, 2 * g + 1], lo.astype(np.float16).view(np.uint16))
        assert np.array_equal(sm[:, 2 * g], (np.float32(hi - lo) / np.float32(3.0)).astype(np.float32)
                              .astype(np.float16).view(np.uint16))
        xc = np.clip(xs, lo[:, None], hi[:, None])
        levels = m[:, None, None] + np.arange(4)[None, None, :] * s[:, None, None]
        dist = np.abs(xc[:, :, None] - levels)
        best = dist.argmin(-1)
        t = (xc - m[:, None]) / s[:, None]
        near_tie = np.abs(t - np.floor(t) - 0.5) < 1e-5
        n_ties += near_tie.sum()
        # exact ties go to the even level (round half to even)
        exact_tie = (t - np.floor(t)) == 0.5
        assert (code[:, sl][exact_tie] % 2 == 0).all()
        mismatch = (best != code[:, sl]) & ~near_tie
        assert not mismatch.any()
        # reconstruction error: at most half a step plus the fp16 rounding of s and m
        err = np.abs(m[:, None] + code[:, sl] * s[:, None] - xc)
        bound = s[:, None] / 2 + np.abs(lo - m)[:, None] + 3 * np.abs((hi - lo) / 3 - s)[:, None]
        assert (err <= bound * (1 + 1e-6) + 1e-30).all()
    assert n_ties < 0.002 * code.size


def test_clip_scales_group_extremes(orc):
    # min -1 and max 2 in group 0: lo = -0.96, hi = 1.92 for c_K; extremes get codes 0 and 3
    x = np.zeros(128, np.float32)
    x[:64] = np.linspace(-1.0, 2.0, 64)
    x[64:] = np.linspace(0.5, 1.5, 64)              # all positive: c * min < min, nothing clipped below
    codes, sm = orc.quant_tokens(_bf16(x)[None], None, 0.96)
    lo = np.float32(0.96) * np.float32(-1.0)
    assert sm[0, 1] == np.float16(lo).view(np.uint16)
    assert sm[0, 0] == np.float16((np.float32(0.96) * np.float32(2.0) - lo) / np.float32(3)).view(np.uint16)
    c = ((codes[0, :, None] >> (2 * np.arange(4))) & 3).reshape(128)
    assert c[0] == 0 and c[63] == 3 and c[64] == 0 and c[127] == 3
    assert sm[0, 3] == np.float16(np.float32(0.96) * np.float32(0.5)).view(np.uint16)


def test_constant_group_gives_zero_scale(orc):
    x = np.full(128, 0.75, np.float32)
    x[64:] = -3.0
    codes, sm = orc.quant_tokens(_bf16(x)[None], None, 0.92)
    assert sm[0, 0] == 0 and sm[0, 2] == 0
    assert (codes == 0).all()
    deq = orc.dequant_tokens(codes, sm)[0]
    assert np.array_equal(deq[:64], np.full(64, np.float16(np.float32(0.92) * np.float32(0.75)), np.float64))


# ------------------------------------------------------------------ attention

def _sdpa(q, k, v):
    """fp64 reference through torch's scaled_dot_product_attention (library routine)."""
    qt = torch.as_tensor(q, dtype=torch.float64)[None, :, None, :]        # [1, G, 1, D]
    kt = torch.as_tensor(k, dtype=torch.float64)[None, None].expand(1, q.shape[0], -1, -1)
    vt = torch.as_tensor(v, dtype=torch.float64)[None, None].expand(1, q.shape[0], -1, -1)
    return torch.nn.functional.scaled_dot_product_attention(qt, kt, vt)[0, :, 0].numpy()


def _f(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _rand_cache(orc, seed, n_int2, n_bf16, g=4, rk=True):
    rng_seed = seed
    q = synth.queries(rng_seed, 0, 1, g, 1)[0].numpy()
    r32 = orc.build_rk(synth.calibration_queries(rng_seed, 0, 2048).numpy())[0] if rk else None
    k_all = synth.keys(rng_seed, 0, 0, 0, n_int2 + n_bf16)
    v_all = synth.values(rng_seed, 0, 0, 0, n_int2 + n_bf16)
    k16 = synth.bf16_bits(k_all)
    v16 = synth.bf16_bits(v_all)
    kc, ks = orc.quant_tokens(k16[:n_int2], r32, 0.96)
    vc, vs = orc.quant_tokens(v16[:n_int2], None, 0.92)
    return q, r32, kc, ks, vc, vs, k16[n_int2:], v16[n_int2:]


def test_bf16_only_cache_is_plain_attention(orc):
    q, r32, kc, ks, vc, vs, k16, v16 = _rand_cache(orc, 31, 0, 320)
    out, lse = orc.attention(q, r32, kc, ks, vc, vs, k16, v16)
    ref = _sdpa(q, _f(k16), _f(v16))
    assert np.abs(out - ref).max() < 1e-12
    logits = q.astype(np.float64) @ _f(k16).T / np.sqrt(128.0)
    assert np.abs(lse - scipy.special.logsumexp(logits, axis=1)).max() < 1e-10


def test_int2_attention_rotated_domain(orc):
    q, r32, kc, ks, vc, vs, k16, v16 = _rand_cache(orc, 37, 200, 40)
    out, _ = orc.attention(q, r32, kc, ks, vc, vs, k16, v16)
    kh = orc.dequant_tokens(kc, ks)
    vh = orc.dequant_tokens(vc, vs)
    r = r32.astype(np.float64)
    # bf16 tokens in the rotated domain too: q.k = (qR).(kR) because R is orthogonal
    keys = np.concatenate([kh, _f(k16) @ r])
    vals = np.concatenate([vh, _f(v16)])
    ref = _sdpa(q.astype(np.float64) @ r, keys, vals)
    assert np.abs(out - ref).max() < 1e-6 * np.abs(ref).max()


def test_int2_attention_identity_rotation(orc):
    q, _, kc, ks, vc, vs, k16, v16 = _rand_cache(orc, 41, 150, 0, rk=False)
    out, _ = orc.attention(q, None, kc, ks, vc, vs, k16, v16)
    ref = _sdpa(q.astype(np.float64), orc.dequant_tokens(kc, ks), orc.dequant_tokens(vc, vs))
    assert np.abs(out - ref).max() < 1e-12


def test_attention_degenerate_cases(orc):
    q, r32, kc, ks, vc, vs, k16, v16 = _rand_cache(orc, 43, 1, 0)
    out, lse = orc.attention(q, r32, kc, ks, vc, vs, k16, v16)
    assert np.allclose(out, np.broadcast_to(orc.dequant_tokens(vc, vs)[0], out.shape), rtol=0, atol=1e-15)
    # q = 0: uniform weights, the output is the mean of all values
    q, r32, kc, ks, vc, vs, k16, v16 = _rand_cache(orc, 47, 30, 20)
    out, lse = orc.attention(np.zeros_like(q), r32, kc, ks, vc, vs, k16, v16)
    mean = np.concatenate([orc.dequant_tokens(vc, vs), _f(v16)]).mean(0)
    assert np.abs(out - mean).max() < 1e-12
    assert np.allclose(lse, np.log(50.0))
    # heads are independent: G = 3 equals three G = 1 calls
    q3 = synth.queries(49, 0, 1, 3, 1)[0].numpy()
    out3, _ = orc.attention(q3, r32, kc, ks, vc, vs, k16, v16)
    for i in range(3):
        o1, _ = orc.attention(q3[i:i + 1], r32, kc, ks, vc, vs, k16, v16)
        assert np.array_equal(o1[0], out3[i])


# ------------------------------------------------------------------ cache bookkeeping

def test_bf16_share_at_128k_matches_pages(orc):
    g = _golden("bf16_share_128k.txt")
    ctx = int(g["context"][0])
    (s0, s1), (i0, i1), (w0, w1), n_win = orc.regions(ctx)
    share = 100.0 * ((s1 - s0) + (w1 - w0)) / ctx
    assert round(share, 2) == float(g["percent_printed"][0])
    assert (s1 - s0, i1 - i0, w1 - w0) == (64, ctx - 320, 256)


def test_regions_small_lengths(orc):
    for L in [0, 1, 63, 64, 65, 319, 320, 321, 1000]:
        (s0, s1), (i0, i1), (w0, w1), n_win = orc.regions(L)
        assert (s0, s1) == (0, min(L, 64))
        assert i1 - i0 == max(0, L - 320) and i0 == 64
        assert n_win == min(256, max(0, L - 64)) == w1 - w0
        if L > 64:
            assert w1 == L and w0 == i1


def test_incremental_equals_bulk(orc):
    seed = 53
    r32 = orc.build_rk(synth.calibration_queries(seed, 0, 2048).numpy())[0]
    n = 700
    k16 = synth.bf16_bits(synth.keys(seed, 0, 0, 0, n))
    v16 = synth.bf16_bits(synth.values(seed, 0, 0, 0, n))
    inc = orc.OracleCache(r32)
    for t in range(0, n, 37):
        inc.append(k16[t:t + 37], v16[t:t + 37])
    assert inc.length == n
    kc, ks = orc.quant_tokens(k16[64:n - 256], r32, 0.96)
    vc, vs = orc.quant_tokens(v16[64:n - 256], None, 0.92)
    assert np.array_equal(inc.kc, kc) and np.array_equal(inc.ks, ks)
    assert np.array_equal(inc.vc, vc) and np.array_equal(inc.vs, vs)
    kb, vb = inc.bf16_tokens()
    assert np.array_equal(kb, np.concatenate([k16[:64], k16[n - 256:]]))
    assert np.array_equal(vb, np.concatenate([v16[:64], v16[n - 256:]]))
