"""Seeded synthetic workloads for the INT2 rotated paged KV cache.

This module only draws inputs: key / value / query vectors with the
distributions of the OSCAR pages' workloads, request lengths, and page-order
permutations.  It holds none of the method's arithmetic (no rotation, no
covariance, no quantisation, no attention), so both the CPU oracle and the
CUDA path may take their inputs from it.

Distributions (one synthetic attention layer, head_dim 128):

* keys: per KV head h, channel c has standard deviation
  sigma_c = exp(0.5 * z_c), z_c ~ N(0, 1) (log-normal(0, 0.5)), and 4 distinct
  seed-drawn outlier channels are multiplied by 20; k[t, c] = sigma_c * n_tc.
* queries: anisotropic Gaussian whose covariance eigenvalues are
  lambda_i = kappa * i**-1.5 (i = 1..128, kappa so that sum(lambda) = 128)
  under one random orthogonal basis per KV head (QR of a Gaussian with the
  sign of R's diagonal folded in), shared by the KV head's query heads.
* values: N(0, 1).

All vectors are drawn in fp32 and rounded (round-to-nearest-even) to bf16
where the cache stores bf16.  Every draw is keyed by (seed, stream, KV head,
request, token block) so any slice can be regenerated alone.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import numpy as np
import torch

HEAD_DIM = 128
N_OUTLIERS = 4
OUTLIER_GAIN = 20.0
Q_DECAY = 1.5
BLOCK = 4096  # tokens per independently seeded draw

# stream ids keep the draws of different tensors apart
_S_KSIGMA, _S_KOUT, _S_QBASIS, _S_K, _S_V, _S_Q, _S_QCAL, _S_LEN, _S_PERM = range(9)


def _seed(*parts: int) -> int:
    """Mix integers into one 63-bit seed (splitmix64 finaliser per part)."""
    x = 0x9E3779B97F4A7C15
    mask = (1 << 64) - 1
    for p in parts:
        x = (x + (int(p) & mask) + 0x9E3779B97F4A7C15) & mask
        z = x
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & mask
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & mask
        x = z ^ (z >> 31)
    return x & ((1 << 63) - 1)


def _gen(device, *parts: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(_seed(*parts))
    return g


@dataclasses.dataclass(frozen=True)
class LayerConfig:
    """Shape of one synthetic attention layer and its decode workload."""
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    ctx: Sequence[int]          # initial tokens per request
    decode_steps: int
    table: str                  # "contiguous" | "permuted"
    q_dtype: str                # dtype the queries are rounded to: "fp32" | "bf16"
    seed: int

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads


def _ragged_lengths(seed: int, batch: int, lo: int, hi: int) -> List[int]:
    g = _gen("cpu", seed, _S_LEN)
    return [int(x) for x in torch.randint(lo, hi + 1, (batch,), generator=g)]


def config(name: str) -> LayerConfig:
    """The five workloads: shapes of Qwen3-4B/8B/32B-like and a 12-way GQA layer."""
    if name == "tiny":
        return LayerConfig("tiny", 1, 4, 1, [1024], 16, "contiguous", "fp32", 1001)
    if name == "qwen3_4b":
        return LayerConfig("qwen3_4b", 8, 32, 8, [8192] * 8, 16, "permuted", "bf16", 1002)
    if name == "qwen3_8b":
        return LayerConfig("qwen3_8b", 32, 32, 8, [32768] * 32, 16, "permuted", "bf16", 1003)
    if name == "qwen3_32b":
        return LayerConfig("qwen3_32b", 32, 64, 8, [100000] * 32, 16, "permuted", "bf16", 1004)
    if name == "ragged_128k":
        return LayerConfig("ragged_128k", 16, 96, 8, _ragged_lengths(1005, 16, 65536, 131072),
                           32, "permuted", "bf16", 1005)
    raise KeyError(name)


CONFIG_NAMES = ["tiny", "qwen3_4b", "qwen3_8b", "qwen3_32b", "ragged_128k"]


def scaled(cfg: LayerConfig, ctx: Sequence[int], batch: Optional[int] = None,
           decode_steps: Optional[int] = None) -> LayerConfig:
    """Same heads and distributions at other lengths (for small test cases)."""
    b = cfg.batch if batch is None else batch
    return dataclasses.replace(cfg, batch=b, ctx=list(ctx)[:b] if len(ctx) >= b else list(ctx) * b,
                               decode_steps=cfg.decode_steps if decode_steps is None else decode_steps)


# ----------------------------------------------------------------------------------------------
# per-KV-head statistics (small; always drawn on the CPU in fp64 so every device agrees)

def key_sigma(seed: int, h: int) -> np.ndarray:
    """Per-channel key standard deviation of KV head h, outliers included (fp64 [128])."""
    g = _gen("cpu", seed, _S_KSIGMA, h)
    z = torch.randn(HEAD_DIM, generator=g, dtype=torch.float64).numpy()
    sigma = np.exp(0.5 * z)
    g2 = _gen("cpu", seed, _S_KOUT, h)
    idx = torch.randperm(HEAD_DIM, generator=g2)[:N_OUTLIERS].numpy()
    sigma[idx] *= OUTLIER_GAIN
    return sigma


def outlier_channels(seed: int, h: int) -> np.ndarray:
    g2 = _gen("cpu", seed, _S_KOUT, h)
    return np.sort(torch.randperm(HEAD_DIM, generator=g2)[:N_OUTLIERS].numpy())


def query_basis(seed: int, h: int) -> np.ndarray:
    """Random orthogonal 128x128 basis of KV head h's query distribution (fp64)."""
    g = _gen("cpu", seed, _S_QBASIS, h)
    a = torch.randn(HEAD_DIM, HEAD_DIM, generator=g, dtype=torch.float64)
    qm, r = torch.linalg.qr(a)
    d = torch.sign(torch.diagonal(r))
    d[d == 0] = 1.0
    return (qm * d[None, :]).numpy()


def query_spectrum() -> np.ndarray:
    i = np.arange(1, HEAD_DIM + 1, dtype=np.float64)
    lam = i ** (-Q_DECAY)
    return lam * (HEAD_DIM / lam.sum())


# ----------------------------------------------------------------------------------------------
# bulk draws

def _blocks(pos0: int, n: int):
    p = pos0
    end = pos0 + n
    while p < end:
        blk = p // BLOCK
        hi = min(end, (blk + 1) * BLOCK)
        yield blk, p - blk * BLOCK, hi - p
        p = hi


def _normal_rows(device, stream: int, seed: int, b: int, h: int, pos0: int, n: int) -> torch.Tensor:
    out = torch.empty(n, HEAD_DIM, dtype=torch.float32, device=device)
    o = 0
    for blk, off, cnt in _blocks(pos0, n):
        g = _gen(device, seed, stream, h, b, blk)
        full = torch.randn(off + cnt, HEAD_DIM, generator=g, device=device, dtype=torch.float32)
        out[o:o + cnt] = full[off:off + cnt]
        o += cnt
    return out


def keys(seed: int, b: int, h: int, pos0: int, n: int, device="cpu") -> torch.Tensor:
    """bf16 keys [n, 128] of request b, KV head h, positions pos0 .. pos0+n-1 (unrotated)."""
    sig = torch.tensor(key_sigma(seed, h), dtype=torch.float32, device=device)
    return (_normal_rows(device, _S_K, seed, b, h, pos0, n) * sig).to(torch.bfloat16)


def values(seed: int, b: int, h: int, pos0: int, n: int, device="cpu") -> torch.Tensor:
    """bf16 values [n, 128] of request b, KV head h, positions pos0 .. pos0+n-1."""
    return _normal_rows(device, _S_V, seed, b, h, pos0, n).to(torch.bfloat16)


def kv_block(seed: int, batch_lens: Sequence[int], pos0: Sequence[int], num_kv_heads: int,
             device="cpu"):
    """Keys and values for several requests, packed as [sum(n_b), Hkv, 128] bf16 in request order.

    batch_lens[b] tokens are drawn for request b starting at position pos0[b].
    """
    total = int(sum(batch_lens))
    k = torch.empty(total, num_kv_heads, HEAD_DIM, dtype=torch.bfloat16, device=device)
    v = torch.empty_like(k)
    o = 0
    for b, n in enumerate(batch_lens):
        if n == 0:
            continue
        for h in range(num_kv_heads):
            k[o:o + n, h] = keys(seed, b, h, pos0[b], n, device)
            v[o:o + n, h] = values(seed, b, h, pos0[b], n, device)
        o += n
    return k, v


def queries(seed: int, step: int, batch: int, num_q_heads: int, num_kv_heads: int,
            dtype: str = "fp32", device="cpu", stream: int = _S_Q) -> torch.Tensor:
    """Decode queries [batch, Hq, 128] fp32 for one step (values rounded to bf16 if dtype='bf16')."""
    group = num_q_heads // num_kv_heads
    lam = torch.tensor(np.sqrt(query_spectrum()), dtype=torch.float64)
    out = torch.empty(batch, num_q_heads, HEAD_DIM, dtype=torch.float64)
    for h in range(num_kv_heads):
        basis = torch.tensor(query_basis(seed, h))
        g = _gen("cpu", seed, stream, h, step)
        z = torch.randn(batch, group, HEAD_DIM, generator=g, dtype=torch.float64)
        out[:, h * group:(h + 1) * group] = (z * lam) @ basis.T
    out = out.to(torch.float32)
    if dtype == "bf16":
        out = out.to(torch.bfloat16).to(torch.float32)
    return out.to(device)


def calibration_queries(seed: int, h: int, n: int = 4096, device="cpu") -> torch.Tensor:
    """n query samples [n, 128] fp32 of KV head h (pooled over its query heads)."""
    lam = torch.tensor(np.sqrt(query_spectrum()), dtype=torch.float64)
    basis = torch.tensor(query_basis(seed, h))
    g = _gen("cpu", seed, _S_QCAL, h)
    z = torch.randn(n, HEAD_DIM, generator=g, dtype=torch.float64)
    return ((z * lam) @ basis.T).to(torch.float32).to(device)


def page_order(seed: int, num_pages: int, kind: str) -> np.ndarray:
    """Order in which physical page ids are handed out: identity or a seeded permutation."""
    if kind == "contiguous":
        return np.arange(num_pages, dtype=np.int32)
    g = _gen("cpu", seed, _S_PERM)
    return torch.randperm(num_pages, generator=g).numpy().astype(np.int32)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw uint16 bit patterns of a bf16 tensor (host copy)."""
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)
