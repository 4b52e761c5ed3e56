"""CPU oracle of OSCAR-style INT2 KV caching -- TEST INFRASTRUCTURE ONLY.

Only the test-suite, the smoke check and the benchmark's CPU-baseline leg may
import this package.  The product library never loads it and shares no code
with it.  The arithmetic lives in ``oracle.c`` (plain C, fp32 write-path
contract, fp64 everywhere else); this module marshals numpy arrays and keeps
the bookkeeping of the mixed-precision cache (sink, recent window, INT2
history) in plain Python.

Method source: axbrief.com, "Together AI's OSCAR breaks the 2-bit KV cache
accuracy barrier", sections "attention-statistics rotation + Triton kernels"
(R_K = U_Q H_Had P_br; c_K = 0.96, c_V = 0.92; per-token asymmetric INT2 in
64-channel groups; fused read path) and "OSCAR release" (BF16 sink and
recent-window tokens); techllm.github.io, "KV cache compression: TurboQuant,
OSCAR, EpiCache", section "OSCAR" (Hadamard plus bit-reversal permutation to
spread important channels; mixed-precision paged cache).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import List, Optional

import numpy as np

D = 128
GROUP = 64
SINK = 64
WINDOW = 256
CLIP_K = 0.96
CLIP_V = 0.92

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (no fast-math, no floating-point contraction)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
               _SRC, "-o", _LIB_PATH + ".tmp", "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


def _L():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        lib.or_f32_to_f16.restype = ctypes.c_uint16
        lib.or_f32_to_f16.argtypes = [ctypes.c_float]
        lib.or_f16_to_f32.restype = ctypes.c_float
        lib.or_f16_to_f32.argtypes = [ctypes.c_uint16]
        lib.or_hadamard128.argtypes = [P]
        lib.or_bitrev7.restype = ctypes.c_int
        lib.or_bitrev7.argtypes = [ctypes.c_int]
        lib.or_query_covariance.argtypes = [P, ctypes.c_long, P]
        lib.or_jacobi_eigh.restype = ctypes.c_int
        lib.or_jacobi_eigh.argtypes = [P, ctypes.c_int, P, P]
        lib.or_build_rk.argtypes = [P, ctypes.c_long, P, P, P]
        lib.or_rotate_f32.argtypes = [P, P, P]
        lib.or_quant_vec.argtypes = [P, ctypes.c_float, P, P]
        lib.or_quant_vec_g.argtypes = [P, ctypes.c_float, ctypes.c_int, P, P]
        lib.or_quant_tokens.argtypes = [P, ctypes.c_long, P, ctypes.c_float, P, P, P]
        lib.or_quant_tokens_g.argtypes = [P, ctypes.c_long, P, ctypes.c_float, ctypes.c_int, P, P, P]
        lib.or_dequant_tokens.argtypes = [P, P, ctypes.c_long, P]
        lib.or_dequant_tokens_g.argtypes = [P, P, ctypes.c_long, ctypes.c_int, P]
        lib.or_attention.argtypes = [ctypes.c_int, P, P, ctypes.c_long, P, P, P, P, ctypes.c_long,
                                     P, P, P, P]
        lib.or_attention_g.argtypes = [ctypes.c_int, P, P, ctypes.c_long, ctypes.c_int, ctypes.c_int,
                                       P, P, P, P, ctypes.c_long, P, P, P, P]
        _lib = lib
    return _lib


def _p(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


# ------------------------------------------------------------------ number formats

def f32_to_f16_bits(x: float) -> int:
    return int(_L().or_f32_to_f16(float(x)))


def f16_bits_to_f32(h: int) -> float:
    return float(_L().or_f16_to_f32(int(h)))


# ------------------------------------------------------------------ rotation

def hadamard128() -> np.ndarray:
    h = np.empty((D, D), np.float64)
    _L().or_hadamard128(_p(h))
    return h


def bitrev7(i: int) -> int:
    return int(_L().or_bitrev7(int(i)))


def query_covariance(q: np.ndarray) -> np.ndarray:
    q = _c(q, np.float32)
    c = np.empty((D, D), np.float64)
    _L().or_query_covariance(_p(q), q.shape[0], _p(c))
    return c


def jacobi_eigh(a: np.ndarray):
    """(eigenvalues descending, eigenvector columns, sweeps) of a symmetric matrix."""
    a = _c(a, np.float64).copy()
    n = a.shape[0]
    ev = np.empty(n, np.float64)
    v = np.empty((n, n), np.float64)
    sweeps = _L().or_jacobi_eigh(_p(a), n, _p(ev), _p(v))
    return ev, v, sweeps


def build_rk(q: np.ndarray):
    """R_K = U_Q H P_br from query samples; returns (fp32 R_K, fp64 R_K, eigenvalues)."""
    q = _c(q, np.float32)
    r32 = np.empty((D, D), np.float32)
    r64 = np.empty((D, D), np.float64)
    ev = np.empty(D, np.float64)
    _L().or_build_rk(_p(q), q.shape[0], _p(r64), _p(r32), _p(ev))
    return r32, r64, ev


def score_weighted_values(q: np.ndarray, k: np.ndarray, v: np.ndarray) -> np.ndarray:
    """Rows of S V (fp64) for calibration queries q [N, 128] against keys k [T, 128] and values
    v [T, 128]: S = row-wise softmax(q k^T / sqrt(128)).  These are the samples whose covariance
    is the score-weighted value covariance C_S of the OSCAR page (axbrief.com, section
    "attention-statistics rotation + Triton kernels")."""
    q64, k64, v64 = (np.asarray(a, np.float64) for a in (q, k, v))
    logit = q64 @ k64.T / np.sqrt(D)
    s = np.exp(logit - logit.max(axis=1, keepdims=True))
    s /= s.sum(axis=1, keepdims=True)
    return s @ v64


def value_covariance(q: np.ndarray, k: np.ndarray, v: np.ndarray) -> np.ndarray:
    """C_S = (1/N) V^T S^T S V as the page writes it (fp64), S as in score_weighted_values."""
    q64, k64, v64 = (np.asarray(a, np.float64) for a in (q, k, v))
    logit = q64 @ k64.T / np.sqrt(D)
    s = np.exp(logit - logit.max(axis=1, keepdims=True))
    s /= s.sum(axis=1, keepdims=True)
    return v64.T @ (s.T @ s) @ v64 / q64.shape[0]


def build_rv(q: np.ndarray, k: np.ndarray, v: np.ndarray):
    """R_V = U_S H P_br from calibration queries, keys and values (same page and section): U_S the
    eigenvectors of C_S by the oracle's Jacobi solver (descending, same sign rule as R_K).  Returns
    (fp32 R_V, fp64 R_V, eigenvalues)."""
    ev, u, _ = jacobi_eigh(value_covariance(q, k, v))
    pbr = np.zeros((D, D))
    pbr[np.arange(D), [bitrev7(i) for i in range(D)]] = 1.0
    r64 = u @ hadamard128() @ pbr
    return r64.astype(np.float32), r64, ev


# ------------------------------------------------------------------ write path

def rotate_f32(x: np.ndarray, r: np.ndarray) -> np.ndarray:
    x = _c(x, np.float32)
    r = _c(r, np.float32)
    y = np.empty(D, np.float32)
    _L().or_rotate_f32(_p(x), _p(r), _p(y))
    return y


def _group_ok(group: int) -> int:
    if group <= 0 or D % group:
        raise ValueError(f"group size {group} does not divide {D}")
    return int(group)


def quant_vec(y: np.ndarray, clip: float, group: int = GROUP):
    """One 128-channel vector -> (codes [32] u8, sm [2 * 128 / group] u16: s, m per group)."""
    y = _c(y, np.float32)
    group = _group_ok(group)
    codes = np.empty(D // 4, np.uint8)
    sm = np.empty(2 * D // group, np.uint16)
    _L().or_quant_vec_g(_p(y), float(clip), group, _p(codes), _p(sm))
    return codes, sm


def quant_tokens(x16: np.ndarray, r: Optional[np.ndarray], clip: float, want_y: bool = False,
                 group: int = GROUP):
    """bf16 bit patterns [n, 128] -> (codes [n, 32] u8, sm [n, 2 * 128 / group] u16[, rotated fp32
    [n, 128]])."""
    x16 = _c(x16, np.uint16).reshape(-1, D)
    group = _group_ok(group)
    n = x16.shape[0]
    codes = np.empty((n, D // 4), np.uint8)
    sm = np.empty((n, 2 * D // group), np.uint16)
    y = np.empty((n, D), np.float32) if want_y else None
    rr = None if r is None else _c(r, np.float32)
    _L().or_quant_tokens_g(_p(x16), n, _p(rr), float(clip), group, _p(codes), _p(sm), _p(y))
    return (codes, sm, y) if want_y else (codes, sm)


def dequant_tokens(codes: np.ndarray, sm: np.ndarray, group: int = GROUP) -> np.ndarray:
    group = _group_ok(group)
    codes = _c(codes, np.uint8).reshape(-1, D // 4)
    sm = _c(sm, np.uint16).reshape(-1, 2 * D // group)
    out = np.empty((codes.shape[0], D), np.float64)
    _L().or_dequant_tokens_g(_p(codes), _p(sm), codes.shape[0], group, _p(out))
    return out


# ------------------------------------------------------------------ read path

def attention(q: np.ndarray, r: Optional[np.ndarray], k_codes, k_sm, v_codes, v_sm, k16, v16,
              group_k: int = GROUP, group_v: int = GROUP):
    """Decode attention of G heads over one KV head (fp64).  Returns (out [G,128], lse [G])."""
    q = _c(q, np.float32).reshape(-1, D)
    g = q.shape[0]
    group_k, group_v = _group_ok(group_k), _group_ok(group_v)
    kc = _c(k_codes, np.uint8).reshape(-1, D // 4)
    ks = _c(k_sm, np.uint16).reshape(-1, 2 * D // group_k)
    vc = _c(v_codes, np.uint8).reshape(-1, D // 4)
    vs = _c(v_sm, np.uint16).reshape(-1, 2 * D // group_v)
    k16 = _c(k16, np.uint16).reshape(-1, D)
    v16 = _c(v16, np.uint16).reshape(-1, D)
    out = np.empty((g, D), np.float64)
    lse = np.empty(g, np.float64)
    rr = None if r is None else _c(r, np.float32)
    _L().or_attention_g(g, _p(q), _p(rr), kc.shape[0], group_k, group_v, _p(kc), _p(ks), _p(vc), _p(vs),
                        k16.shape[0], _p(k16), _p(v16), _p(out), _p(lse))
    return out, lse


# ------------------------------------------------------------------ the mixed-precision cache

def regions(length: int, sink: int = SINK, window: int = WINDOW):
    """Positions held in each region of a request of `length` tokens.

    sink: [0, min(L, S)); INT2 history: [S, L - W) when L > S + W; window: the
    last min(W, L - S) positions at or after S.
    """
    n_sink = min(length, sink)
    n_int2 = max(0, length - sink - window)
    n_win = max(0, length - sink) - n_int2
    w0 = min(length, sink + n_int2)
    return (0, n_sink), (sink, sink + n_int2), (w0, length), n_win


class OracleCache:
    """Token-by-token model of one request's cache for one KV head.

    Appending a token at position p stores it (bf16) in the sink when p < S,
    otherwise in the window; when the window already holds W tokens, its oldest
    token (position p - W) leaves it and is quantised to INT2 from its bf16 copy.
    Keys are rotated by R_K before quantisation; values are not.
    """

    def __init__(self, rk: Optional[np.ndarray], clip_k: float = CLIP_K, clip_v: float = CLIP_V,
                 sink: int = SINK, window: int = WINDOW, group_k: int = GROUP, group_v: int = GROUP):
        self.rk = rk
        self.clip_k = clip_k
        self.clip_v = clip_v
        self.sink = sink
        self.window = window
        self.group_k = _group_ok(group_k)
        self.group_v = _group_ok(group_v)
        self.k16: List[np.ndarray] = []   # bf16 bits of every position (kept for the bf16 regions)
        self.v16: List[np.ndarray] = []
        self.kc = np.zeros((0, D // 4), np.uint8)
        self.ks = np.zeros((0, 2 * D // self.group_k), np.uint16)
        self.vc = np.zeros((0, D // 4), np.uint8)
        self.vs = np.zeros((0, 2 * D // self.group_v), np.uint16)

    @property
    def length(self) -> int:
        return len(self.k16)

    def append(self, k16: np.ndarray, v16: np.ndarray):
        """Append tokens one by one (k16, v16: [n, 128] bf16 bit patterns)."""
        k16 = _c(k16, np.uint16).reshape(-1, D)
        v16 = _c(v16, np.uint16).reshape(-1, D)
        evict_k, evict_v = [], []
        for t in range(k16.shape[0]):
            p = self.length
            self.k16.append(k16[t])
            self.v16.append(v16[t])
            if p >= self.sink + self.window:
                q = p - self.window            # leaves the window now
                evict_k.append(self.k16[q])
                evict_v.append(self.v16[q])
        if evict_k:
            kc, ks = quant_tokens(np.stack(evict_k), self.rk, self.clip_k, group=self.group_k)
            vc, vs = quant_tokens(np.stack(evict_v), None, self.clip_v, group=self.group_v)
            self.kc = np.concatenate([self.kc, kc])
            self.ks = np.concatenate([self.ks, ks])
            self.vc = np.concatenate([self.vc, vc])
            self.vs = np.concatenate([self.vs, vs])

    def bf16_tokens(self):
        """(k16, v16) of the sink and window positions, in position order."""
        (s0, s1), _, (w0, w1), _ = regions(self.length, self.sink, self.window)
        pos = list(range(s0, s1)) + list(range(w0, w1))
        if not pos:
            z = np.zeros((0, D), np.uint16)
            return z, z
        return np.stack([self.k16[p] for p in pos]), np.stack([self.v16[p] for p in pos])

    def attend(self, q: np.ndarray):
        k16, v16 = self.bf16_tokens()
        return attention(q, self.rk, self.kc, self.ks, self.vc, self.vs, k16, v16, self.group_k, self.group_v)

    def attend_upto(self, q: np.ndarray, last: int):
        """Attention of G heads over the cached positions 0 .. last only, each at the precision the
        cache holds it in now (the causal view of one query of a chunk appended as a whole; reading
        of the mixed-precision cache for chunked prefill)."""
        (s0, s1), (i0, i1), (w0, w1), _ = regions(self.length, self.sink, self.window)
        pos = [p for p in list(range(s0, s1)) + list(range(w0, w1)) if p <= last]
        n_int2 = max(0, min(i1, last + 1) - i0)
        if pos:
            k16 = np.stack([self.k16[p] for p in pos])
            v16 = np.stack([self.v16[p] for p in pos])
        else:
            k16 = v16 = np.zeros((0, D), np.uint16)
        return attention(q, self.rk, self.kc[:n_int2], self.ks[:n_int2], self.vc[:n_int2], self.vs[:n_int2],
                         k16, v16, self.group_k, self.group_v)
