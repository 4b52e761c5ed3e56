"""Pins of the oracle's group-size parameter (keys and values quantised in groups of 64 or 128
channels), checked against facts outside the oracle: a reduction to the 64-channel case, exact
grids, brute-force nearest levels, attention computed by hand from the dequantised tensors, and
the effective bit counts the pages print."""
import os

import numpy as np
import pytest
import torch

import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
D = 128


def _bf16(x):
    return synth.bf16_bits(torch.as_tensor(np.asarray(x, np.float32)).to(torch.bfloat16))


def _unpack(codes):
    return ((codes[..., :, None] >> (2 * np.arange(4))) & 3).reshape(codes.shape[:-1] + (D,))


def test_group_of_128_reduces_to_64_when_halves_share_their_range(orc):
    rng = np.random.default_rng(5)
    for clip in (1.0, 0.96, 0.92):
        for _ in range(50):
            half = rng.standard_normal(64).astype(np.float32) * np.float32(2.0 ** rng.integers(-6, 6))
            x = np.concatenate([half, rng.permutation(half)])    # same min and max in both halves
            c64, sm64 = orc.quant_vec(x, clip, group=64)
            c128, sm128 = orc.quant_vec(x, clip, group=128)
            assert sm128.shape == (2,) and sm64.shape == (4,)
            assert np.array_equal(c64, c128)
            assert np.array_equal(sm128, sm64[:2]) and np.array_equal(sm128, sm64[2:])


def test_group_of_128_round_trip_exact_on_grid(orc):
    rng = np.random.default_rng(29)
    for _ in range(100):
        s = np.float32(2.0 ** rng.integers(-6, 3)) * np.float32(rng.choice([1.0, 3.0]))
        m = np.float32(rng.integers(-8, 9)) * s       # (j + code) * s: at most 6 significant bits
        codes = rng.integers(0, 4, D)
        codes[rng.integers(0, D)] = 0
        codes[rng.integers(0, D)] = 3                         # both ends of the one group present
        x = (m + codes * s).astype(np.float32)
        x16 = _bf16(x)
        assert np.array_equal((x16.astype(np.uint32) << 16).view(np.float32), x), "grid must be bf16-exact"
        pc, sm = orc.quant_tokens(x16[None], None, 1.0, group=128)
        assert np.array_equal(_unpack(pc[0]), codes)
        assert np.array_equal(orc.dequant_tokens(pc, sm, group=128)[0], x.astype(np.float64))


@pytest.mark.parametrize("clip", [1.0, 0.92])
def test_group_of_128_brute_force_nearest_level(orc, clip):
    rng = np.random.default_rng(31)
    sig = np.exp(0.5 * rng.standard_normal(D))
    x16 = _bf16(rng.standard_normal((300, D)) * sig)
    codes, sm = orc.quant_tokens(x16, None, clip, group=128)
    x = (x16.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    cf = np.float32(clip)
    lo = (cf * x.min(1).astype(np.float32)).astype(np.float64)      # one group: the whole vector
    hi = (cf * x.max(1).astype(np.float32)).astype(np.float64)
    assert np.array_equal(sm[:, 1], lo.astype(np.float16).view(np.uint16))
    assert np.array_equal(sm[:, 0], (np.float32(hi - lo) / np.float32(3.0)).astype(np.float32)
                          .astype(np.float16).view(np.uint16))
    s = sm[:, 0].view(np.float16).astype(np.float64)
    m = sm[:, 1].view(np.float16).astype(np.float64)
    xc = np.clip(x, lo[:, None], hi[:, None])
    levels = m[:, None, None] + np.arange(4) * s[:, None, None]
    best = np.abs(xc[:, :, None] - levels).argmin(-1)
    t = (xc - m[:, None]) / s[:, None]
    near_tie = np.abs(t - np.floor(t) - 0.5) < 1e-5
    assert not ((best != _unpack(codes)) & ~near_tie).any()


def test_attention_takes_each_tensors_group_size(orc):
    rng = np.random.default_rng(37)
    n_int2, n_bf16, g = 150, 20, 3
    kx = _bf16(rng.standard_normal((n_int2, D)) * np.exp(0.5 * rng.standard_normal(D)))
    vx = _bf16(rng.standard_normal((n_int2, D)))
    kc, ks = orc.quant_tokens(kx, None, 0.96, group=64)
    vc, vs = orc.quant_tokens(vx, None, 0.92, group=128)
    k16 = _bf16(rng.standard_normal((n_bf16, D)))
    v16 = _bf16(rng.standard_normal((n_bf16, D)))
    q = rng.standard_normal((g, D)).astype(np.float32)
    out, lse = orc.attention(q, None, kc, ks, vc, vs, k16, v16, group_k=64, group_v=128)
    # by hand: dequantise each tensor with its own groups, then fp64 softmax attention
    kh = np.concatenate([orc.dequant_tokens(kc, ks, group=64), (k16.astype(np.uint32) << 16).view(np.float32)])
    vh = np.concatenate([orc.dequant_tokens(vc, vs, group=128), (v16.astype(np.uint32) << 16).view(np.float32)])
    logit = q.astype(np.float64) @ kh.T / np.sqrt(D)
    p = np.exp(logit - logit.max(1, keepdims=True))
    ref = (p @ vh) / p.sum(1, keepdims=True)
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12)
    assert np.allclose(lse, logit.max(1) + np.log(p.sum(1)), rtol=1e-12)
    # and a value group of 64 is a different cache
    vc64, vs64 = orc.quant_tokens(vx, None, 0.92, group=64)
    assert not np.array_equal(orc.dequant_tokens(vc64, vs64, group=64), orc.dequant_tokens(vc, vs, group=128))


def test_bad_group_sizes_rejected(orc):
    with pytest.raises(ValueError):
        orc.quant_vec(np.zeros(D, np.float32), 1.0, group=48)
    with pytest.raises(ValueError):
        orc.dequant_tokens(np.zeros((1, 32), np.uint8), np.zeros((1, 4), np.uint16), group=0)


def _golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = line.split()
                out[k] = v
    return out


def _bits_per_element(orc, group_k, group_v, ctx, with_bf16):
    """Average stored bits per key / value element of one request, from the formats: an INT2
    token stores 2 bits per channel plus one fp16 (scale, minimum) pair per group."""
    (s0, s1), (i0, i1), (w0, w1), _ = orc.regions(ctx)
    n_int2, n_bf16 = i1 - i0, (s1 - s0) + (w1 - w0)
    int2_bits = D * 4 + 2 * 16 * (D // group_k + D // group_v)     # K and V of one token
    if not with_bf16:
        return int2_bits / (2 * D)
    return (n_int2 * int2_bits + n_bf16 * 2 * D * 16) / (ctx * 2 * D)


def test_effective_bits_match_the_pages(orc):
    g = _golden("effective_bits.txt")
    ctx = int(g["context"])
    assert round(_bits_per_element(orc, 128, 128, ctx, True), 2) == float(g["bits_g128_with_bf16"])
    assert round(_bits_per_element(orc, 64, 128, ctx, False), 2) == float(g["bits_k64_v128_int2"])
    # the library's format today: groups of 64 for both, 2.5 bits per element in the INT2 part
    assert _bits_per_element(orc, 64, 64, ctx, False) == 2.5
