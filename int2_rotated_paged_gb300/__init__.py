"""Python binding of liboscar_kv.so, the GB300 INT2 rotated paged KV cache.

Argument marshalling only: every step of the write path, the read path and the
calibration runs in the CUDA kernels of the shared library (C ABI in
include/oscar_kv.h).  PyTorch tensors serve as device memory and streams.  The
library must have been built (``int2_rotated_paged_gb300.build.build()``); there is no
fallback of any kind, and every call raises if the library or a GPU is missing.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "liboscar_kv.so")

OSCAR_OK = 0
OSCAR_EINVAL = -1
OSCAR_ENOPAGES = -2
OSCAR_EWORKSPACE = -3
OSCAR_ECUDA = -4
OSCAR_EALIGN = -5
OSCAR_ERANGE = -6
DTYPE_F32 = 0
DTYPE_BF16 = 1
PAGE_HEAD_BYTES = 5120

# every entry point declared in include/oscar_kv.h
EXPORTS = [
    "oscar_default_desc", "oscar_pool_bytes", "oscar_bf16_bytes", "oscar_page_table_bytes",
    "oscar_seq_lens_bytes", "oscar_cache_create", "oscar_cache_destroy", "oscar_cache_length",
    "kv_page_table_init", "kv_page_table_reserve", "kv_page_table_release", "kv_page_table_sync",
    "kv_page_table_read",
    "kv_page_table_free_pages", "kv_quant_append", "kv_quant_append_layers_workspace_bytes",
    "kv_quant_append_layers", "oscar_decode_workspace_bytes", "oscar_decode_step_host_staging_bytes",
    "oscar_decode_step_host",
    "oscar_decode_attention", "oscar_build_rk_workspace_bytes", "oscar_build_rk", "oscar_read_int2",
    "oscar_read_bf16", "oscar_strerror", "oscar_last_cuda_error", "oscar_launch_count",
    "oscar_set_decode_path", "oscar_decode_status", "oscar_decode_attention_noalloc", "oscar_decode_step",
    "oscar_kernel_timing", "oscar_kernel_timing_read", "oscar_set_wait_limit", "oscar_decode_status_noalloc",
    "oscar_set_wait_probe", "oscar_page_head_bytes", "oscar_cq_accumulator_bytes", "oscar_cq_reset",
    "oscar_cq_accumulate", "oscar_cq_finalize", "oscar_score_weighted_values", "oscar_prefill_workspace_bytes",
    "oscar_prefill_attention",
]
OSCAR_ESCRATCH = -8
OSCAR_ETIMEOUT = -7
PATH_SIMT = 1
PATH_WARP_MMA = 2


class OscarError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {code} ({strerror(code)})"
                         + (f", cuda error {lib().oscar_last_cuda_error()}" if code == OSCAR_ECUDA else ""))
        self.code = code


class CacheDesc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "batch", "num_kv_heads", "num_q_heads", "head_dim", "page_size", "group_size", "sink",
        "window", "max_pages_total", "max_pages_per_seq")] + [("clip_k", ctypes.c_float),
                                                              ("clip_v", ctypes.c_float),
                                                              ("group_size_v", ctypes.c_int32)]


_lib = None


def lib() -> ctypes.CDLL:
    """Load liboscar_kv.so (raises if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build the CUDA library first "
                           "(python -m int2_rotated_paged_gb300.build)")
    L = ctypes.CDLL(LIB_PATH)
    P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    DP = ctypes.POINTER(CacheDesc)
    sig = {
        "oscar_default_desc": (None, [DP]),
        "oscar_pool_bytes": (SZ, [DP]),
        "oscar_page_head_bytes": (SZ, [DP]),
        "oscar_bf16_bytes": (SZ, [DP]),
        "oscar_page_table_bytes": (SZ, [DP]),
        "oscar_seq_lens_bytes": (SZ, [DP]),
        "oscar_cache_create": (ctypes.c_int, [DP, P, P, P, P, ctypes.POINTER(P)]),
        "oscar_cache_destroy": (ctypes.c_int, [P]),
        "oscar_cache_length": (I64, [P, I32]),
        "kv_page_table_init": (ctypes.c_int, [P, P]),
        "kv_page_table_reserve": (ctypes.c_int, [P, I32, I64]),
        "kv_page_table_release": (ctypes.c_int, [P, I32]),
        "kv_page_table_sync": (ctypes.c_int, [P, P]),
        "kv_page_table_read": (ctypes.c_int, [P, I32, P, I32]),
        "kv_page_table_free_pages": (I32, [P]),
        "kv_quant_append": (ctypes.c_int, [P, P, P, P, P, P]),
        "kv_quant_append_layers_workspace_bytes": (SZ, [I32]),
        "kv_quant_append_layers": (ctypes.c_int, [P, I32, P, P, P, P, P, SZ, P]),
        "oscar_decode_step_host_staging_bytes": (SZ, [P, I32, I32]),
        "oscar_decode_step_host": (ctypes.c_int, [P, P, P, P, I32, P, P, I32, P, SZ, P, SZ, P]),
        "oscar_decode_workspace_bytes": (SZ, [P]),
        "oscar_decode_attention": (ctypes.c_int, [P, P, I32, P, P, I32, P, SZ, P]),
        "oscar_build_rk_workspace_bytes": (SZ, [I32]),
        "oscar_build_rk": (ctypes.c_int, [P, I64, I32, P, P, SZ, P]),
        "oscar_read_int2": (ctypes.c_int, [P, I32, I32, I64, I64, P, P, P, P, P]),
        "oscar_read_bf16": (ctypes.c_int, [P, I32, I32, I64, I64, P, P, P]),
        "oscar_strerror": (ctypes.c_char_p, [ctypes.c_int]),
        "oscar_last_cuda_error": (ctypes.c_int, []),
        "oscar_launch_count": (I64, []),
        "oscar_set_decode_path": (ctypes.c_int, [I32]),
        "oscar_decode_status": (ctypes.c_int, [P, SZ, P, P]),
        "oscar_decode_attention_noalloc": (ctypes.c_int, [P, P, I32, P, P, I32, P]),
        "oscar_decode_step": (ctypes.c_int, [P, P, P, P, I32, P, P, I32, P, SZ, P]),
        "oscar_kernel_timing": (ctypes.c_int, [P, I32]),
        "oscar_kernel_timing_read": (ctypes.c_int, [P, P, I32, P]),
        "oscar_set_wait_limit": (ctypes.c_int, [I32]),
        "oscar_set_wait_probe": (ctypes.c_int, [I32]),
        "oscar_cq_accumulator_bytes": (SZ, [I32]),
        "oscar_prefill_workspace_bytes": (SZ, [P]),
        "oscar_prefill_attention": (ctypes.c_int, [P, P, I32, P, P, P, I32, P, SZ, P]),
        "oscar_cq_reset": (ctypes.c_int, [P, I32, P]),
        "oscar_cq_accumulate": (ctypes.c_int, [P, I64, I32, P, P]),
        "oscar_cq_finalize": (ctypes.c_int, [P, I32, P, P, SZ, P]),
        "oscar_score_weighted_values": (ctypes.c_int, [P, I64, P, P, I32, I32, P, P]),
        "oscar_decode_status_noalloc": (ctypes.c_int, [P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _lib = L
    return L


def strerror(code: int) -> str:
    return lib().oscar_strerror(code).decode()


def _check(fn: str, rc: int) -> int:
    if rc < 0:
        raise OscarError(fn, rc)
    return rc


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _host_i32(values: Sequence[int]):
    arr = (ctypes.c_int32 * len(values))(*[int(v) for v in values])
    return arr


def default_desc() -> CacheDesc:
    d = CacheDesc()
    lib().oscar_default_desc(ctypes.byref(d))
    return d


# ------------------------------------------------------------------ thin wrappers (same names)

def oscar_cache_create(desc: CacheDesc, pool, bf16, page_table, seq_lens) -> ctypes.c_void_p:
    h = ctypes.c_void_p()
    _check("oscar_cache_create", lib().oscar_cache_create(ctypes.byref(desc), _ptr(pool), _ptr(bf16),
                                                          _ptr(page_table), _ptr(seq_lens), ctypes.byref(h)))
    return h


def kv_page_table_init(cache, page_order: Optional[Sequence[int]] = None):
    arr = None if page_order is None else _host_i32(page_order)
    _check("kv_page_table_init", lib().kv_page_table_init(cache, arr))


def kv_page_table_reserve(cache, b: int, new_len: int):
    _check("kv_page_table_reserve", lib().kv_page_table_reserve(cache, b, new_len))


def kv_page_table_release(cache, b: int):
    _check("kv_page_table_release", lib().kv_page_table_release(cache, b))


def kv_page_table_sync(cache, stream=None):
    _check("kv_page_table_sync", lib().kv_page_table_sync(cache, _stream(stream)))


def kv_page_table_free_pages(cache) -> int:
    return _check("kv_page_table_free_pages", lib().kv_page_table_free_pages(cache))


def kv_page_table_read(cache, b: int, max_out: int = 1 << 20):
    n = _check("kv_page_table_read", lib().kv_page_table_read(cache, b, None, 0))
    arr = (ctypes.c_int32 * max(n, 1))()
    lib().kv_page_table_read(cache, b, arr, n)
    return list(arr[:n])


def kv_quant_append(cache, k, v, new_tokens: Sequence[int], rk, stream=None):
    _check("kv_quant_append", lib().kv_quant_append(cache, _ptr(k), _ptr(v), _host_i32(new_tokens),
                                                    _ptr(rk), _stream(stream)))


def kv_quant_append_layers_workspace_bytes(n_layers: int) -> int:
    return int(lib().kv_quant_append_layers_workspace_bytes(n_layers))


def kv_quant_append_layers(caches, ks, vs, new_tokens: Sequence[int], rks, workspace, stream=None):
    """One append of new_tokens per request to every layer's cache (kv_quant_append_layers): caches,
    ks, vs, rks are per-layer sequences (cache handles, bf16 keys, bf16 values, fp32 R_K)."""
    n = len(caches)
    if not (len(ks) == len(vs) == len(rks) == n):
        raise ValueError("one key, value and R_K tensor per layer")
    arr = lambda xs: (ctypes.c_void_p * n)(*[_ptr(x) for x in xs])
    nbytes = workspace.numel() * workspace.element_size()
    def handle(c):   # a Cache, a handle from oscar_cache_create, or its address
        c = getattr(c, "handle", c)
        return c if isinstance(c, int) else c.value
    _check("kv_quant_append_layers", lib().kv_quant_append_layers(
        (ctypes.c_void_p * n)(*[handle(c) for c in caches]), n,
        arr(ks), arr(vs), _host_i32(new_tokens), arr(rks), _ptr(workspace), nbytes, _stream(stream)))


def oscar_decode_step_host_staging_bytes(cache, q_dtype: int, out_dtype: int) -> int:
    return int(lib().oscar_decode_step_host_staging_bytes(cache, q_dtype, out_dtype))


def oscar_decode_step_host(cache, k_host, v_host, q_host, q_dtype: int, rk, out_host, out_dtype: int, staging, workspace,
                           stream=None):
    """oscar_decode_step on host buffers (pinned tensors or host addresses): copies in, step, copy out,
    all enqueued; the output is in out_host once the stream has passed the call."""
    sbytes = staging.numel() * staging.element_size()
    wbytes = workspace.numel() * workspace.element_size()
    _check("oscar_decode_step_host", lib().oscar_decode_step_host(
        cache, _ptr(k_host), _ptr(v_host), _ptr(q_host), q_dtype, _ptr(rk), _ptr(out_host), out_dtype,
        _ptr(staging), sbytes, _ptr(workspace), wbytes, _stream(stream)))


def oscar_decode_workspace_bytes(cache) -> int:
    return int(lib().oscar_decode_workspace_bytes(cache))


def oscar_decode_attention(cache, q, q_dtype: int, rk, out, out_dtype: int, workspace, stream=None):
    nbytes = workspace.numel() * workspace.element_size()
    _check("oscar_decode_attention", lib().oscar_decode_attention(
        cache, _ptr(q), q_dtype, _ptr(rk), _ptr(out), out_dtype, _ptr(workspace), nbytes, _stream(stream)))


def oscar_decode_step(cache, k, v, q, q_dtype: int, rk, out, out_dtype: int, workspace, stream=None):
    """Append one token per request (k, v: [batch, Hkv, 128] bf16) and attend with q, in one call."""
    nbytes = workspace.numel() * workspace.element_size()
    _check("oscar_decode_step", lib().oscar_decode_step(
        cache, _ptr(k), _ptr(v), _ptr(q), q_dtype, _ptr(rk), _ptr(out), out_dtype, _ptr(workspace), nbytes,
        _stream(stream)))


def oscar_decode_attention_noalloc(cache, q, q_dtype: int, rk, out, out_dtype: int, stream=None):
    """Decode attention with the library's fixed device scratch (for callers that cannot allocate)."""
    _check("oscar_decode_attention_noalloc", lib().oscar_decode_attention_noalloc(
        cache, _ptr(q), q_dtype, _ptr(rk), _ptr(out), out_dtype, _stream(stream)))


def oscar_build_rk_workspace_bytes(num_kv_heads: int) -> int:
    return int(lib().oscar_build_rk_workspace_bytes(num_kv_heads))


def oscar_build_rk(q, n: int, num_kv_heads: int, rk, workspace, stream=None):
    nbytes = workspace.numel() * workspace.element_size()
    _check("oscar_build_rk", lib().oscar_build_rk(_ptr(q), n, num_kv_heads, _ptr(rk), _ptr(workspace),
                                                  nbytes, _stream(stream)))


def oscar_prefill_workspace_bytes(cache) -> int:
    return int(lib().oscar_prefill_workspace_bytes(cache))


def oscar_prefill_attention(cache, q, q_dtype: int, n_q: Sequence[int], rk, out, out_dtype: int, workspace,
                            stream=None):
    """Causal attention of the queries of the chunk each request just appended (n_q[b] tokens)."""
    nbytes = workspace.numel() * workspace.element_size()
    _check("oscar_prefill_attention", lib().oscar_prefill_attention(
        cache, _ptr(q), q_dtype, _host_i32(n_q), _ptr(rk), _ptr(out), out_dtype, _ptr(workspace), nbytes,
        _stream(stream)))


def oscar_cq_accumulator_bytes(num_kv_heads: int) -> int:
    return int(lib().oscar_cq_accumulator_bytes(num_kv_heads))


def oscar_cq_reset(acc, num_kv_heads: int, stream=None):
    _check("oscar_cq_reset", lib().oscar_cq_reset(_ptr(acc), num_kv_heads, _stream(stream)))


def oscar_cq_accumulate(q, n: int, num_kv_heads: int, acc, stream=None):
    _check("oscar_cq_accumulate", lib().oscar_cq_accumulate(_ptr(q), n, num_kv_heads, _ptr(acc), _stream(stream)))


def oscar_cq_finalize(acc, num_kv_heads: int, rk, workspace, stream=None):
    nbytes = workspace.numel() * workspace.element_size()
    _check("oscar_cq_finalize", lib().oscar_cq_finalize(_ptr(acc), num_kv_heads, _ptr(rk), _ptr(workspace), nbytes,
                                                        _stream(stream)))


def oscar_score_weighted_values(q, n: int, k, v, t_keys: int, num_kv_heads: int, y, stream=None):
    _check("oscar_score_weighted_values", lib().oscar_score_weighted_values(
        _ptr(q), n, _ptr(k), _ptr(v), t_keys, num_kv_heads, _ptr(y), _stream(stream)))


def oscar_read_int2(cache, b: int, h: int, pos0: int, n: int, stream=None, group_k: int = 64, group_v: int = 64):
    """(k_codes [n,32] u8, k_sm [n, 2*128/group_k] u16, v_codes, v_sm [n, 2*128/group_v]) as numpy
    arrays, logical per-token format (the group sizes must be the cache's)."""
    import numpy as np
    kc = np.zeros((n, 32), np.uint8)
    ks = np.zeros((n, 256 // group_k), np.uint16)
    vc = np.zeros((n, 32), np.uint8)
    vs = np.zeros((n, 256 // group_v), np.uint16)
    p = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    _check("oscar_read_int2", lib().oscar_read_int2(cache, b, h, pos0, n, p(kc), p(ks), p(vc), p(vs),
                                                    _stream(stream)))
    return kc, ks, vc, vs


def oscar_read_bf16(cache, b: int, h: int, pos0: int, n: int, stream=None):
    import numpy as np
    k = np.zeros((n, 128), np.uint16)
    v = np.zeros((n, 128), np.uint16)
    p = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    _check("oscar_read_bf16", lib().oscar_read_bf16(cache, b, h, pos0, n, p(k), p(v), _stream(stream)))
    return k, v


def oscar_cache_length(cache, b: int) -> int:
    return _check("oscar_cache_length", lib().oscar_cache_length(cache, b))


def oscar_set_decode_path(path: int):
    _check("oscar_set_decode_path", lib().oscar_set_decode_path(path))


def oscar_decode_status(cache, workspace, stream=None):
    nbytes = workspace.numel() * workspace.element_size()
    _check("oscar_decode_status", lib().oscar_decode_status(_ptr(workspace), nbytes, cache, _stream(stream)))


def oscar_set_wait_limit(iters: int):
    """Bounded in-kernel waits give up after `iters` tests of up to 1 ms (< 0: the default)."""
    _check("oscar_set_wait_limit", lib().oscar_set_wait_limit(iters))


def oscar_set_wait_probe(on: bool):
    """Timeout-path check: decode calls also wait, bounded, on a barrier nothing arrives at."""
    _check("oscar_set_wait_probe", lib().oscar_set_wait_probe(1 if on else 0))


def oscar_decode_status_noalloc(stream=None):
    """Raise OscarError(OSCAR_ETIMEOUT) if the last fixed-scratch decode hit a bounded wait."""
    _check("oscar_decode_status_noalloc", lib().oscar_decode_status_noalloc(_stream(stream)))


def oscar_kernel_timing(cache, capacity: int):
    _check("oscar_kernel_timing", lib().oscar_kernel_timing(cache, capacity))


def oscar_kernel_timing_read(cache, max_n: int):
    """Durations (ms) of the decode kernel launches recorded since oscar_kernel_timing."""
    buf = (ctypes.c_float * max(1, max_n))()
    got = ctypes.c_int32(0)
    _check("oscar_kernel_timing_read", lib().oscar_kernel_timing_read(cache, buf, max_n, ctypes.byref(got)))
    return [float(buf[i]) for i in range(got.value)]


def oscar_launch_count() -> int:
    return int(lib().oscar_launch_count())


# ------------------------------------------------------------------ convenience owner of the buffers

class Cache:
    """Allocates the caller-owned device buffers with torch and holds the C handle."""

    def __init__(self, batch: int, num_q_heads: int, num_kv_heads: int, max_pages_total: int,
                 max_pages_per_seq: int, page_order: Optional[Sequence[int]] = None,
                 clip_k: float = 0.96, clip_v: float = 0.92, device="cuda", group_k: int = 64, group_v: int = 64):
        import torch
        d = default_desc()
        d.batch, d.num_q_heads, d.num_kv_heads = batch, num_q_heads, num_kv_heads
        d.max_pages_total, d.max_pages_per_seq = max_pages_total, max_pages_per_seq
        d.clip_k, d.clip_v = clip_k, clip_v
        d.group_size, d.group_size_v = group_k, group_v
        self.desc = d
        self.group_k, self.group_v = group_k, group_v
        L = lib()
        sizes = [L.oscar_pool_bytes(ctypes.byref(d)), L.oscar_bf16_bytes(ctypes.byref(d)),
                 L.oscar_page_table_bytes(ctypes.byref(d)), L.oscar_seq_lens_bytes(ctypes.byref(d))]
        if min(sizes) == 0:
            raise OscarError("cache descriptor", OSCAR_EINVAL)
        self.pool = torch.empty(sizes[0], dtype=torch.uint8, device=device)
        self.bf16 = torch.zeros(sizes[1] // 2, dtype=torch.bfloat16, device=device)
        self.page_table = torch.zeros(sizes[2] // 4, dtype=torch.int32, device=device)
        self.seq_lens = torch.zeros(sizes[3] // 4, dtype=torch.int32, device=device)
        self.handle = oscar_cache_create(d, self.pool, self.bf16, self.page_table, self.seq_lens)
        kv_page_table_init(self.handle, page_order)
        # zeroed once, so that status() before the first decode call reads a clear error word
        self.workspace = torch.zeros(oscar_decode_workspace_bytes(self.handle), dtype=torch.uint8,
                                     device=device)

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None and _lib is not None:
            _lib.oscar_cache_destroy(h)
            self.handle = None

    def append(self, k, v, new_tokens: Sequence[int], rk, stream=None):
        kv_quant_append(self.handle, k, v, new_tokens, rk, stream)

    def attend(self, q, rk, out, stream=None):
        qd = DTYPE_BF16 if str(q.dtype) == "torch.bfloat16" else DTYPE_F32
        od = DTYPE_BF16 if str(out.dtype) == "torch.bfloat16" else DTYPE_F32
        oscar_decode_attention(self.handle, q, qd, rk, out, od, self.workspace, stream)

    def step(self, k, v, q, rk, out, stream=None):
        """One decode step: append one token per request and attend (oscar_decode_step)."""
        qd = DTYPE_BF16 if str(q.dtype) == "torch.bfloat16" else DTYPE_F32
        od = DTYPE_BF16 if str(out.dtype) == "torch.bfloat16" else DTYPE_F32
        oscar_decode_step(self.handle, k, v, q, qd, rk, out, od, self.workspace, stream)

    def prefill(self, q, n_q: Sequence[int], rk, out, workspace=None, stream=None):
        """Chunked-prefill attention of the n_q[b] tokens each request just appended (queries q)."""
        import torch
        if workspace is None:
            workspace = torch.empty(oscar_prefill_workspace_bytes(self.handle), dtype=torch.uint8, device=q.device)
        qd = DTYPE_BF16 if str(q.dtype) == "torch.bfloat16" else DTYPE_F32
        od = DTYPE_BF16 if str(out.dtype) == "torch.bfloat16" else DTYPE_F32
        oscar_prefill_attention(self.handle, q, qd, n_q, rk, out, od, workspace, stream)
        return workspace

    def status(self, stream=None):
        """Raise if the last decode on this cache's workspace hit a bounded in-kernel wait."""
        oscar_decode_status(self.handle, self.workspace, stream)

    def length(self, b: int) -> int:
        return oscar_cache_length(self.handle, b)

    def read_int2(self, b: int, h: int, pos0: int, n: int):
        """INT2 codes and scale/min of n tokens in the logical per-token format (oscar_read_int2)."""
        return oscar_read_int2(self.handle, b, h, pos0, n, group_k=self.group_k, group_v=self.group_v)

    def page_head_bytes(self) -> int:
        return int(lib().oscar_page_head_bytes(ctypes.byref(self.desc)))
