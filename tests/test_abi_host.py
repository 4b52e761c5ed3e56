"""C-ABI checks that need no GPU: the library loads, exports every entry point that
include/oscar_kv.h declares, validates descriptors, and its page-table free list
behaves (host mirror only; nothing here enqueues GPU work)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def K():
    from int2_rotated_paged_gb300 import build
    build.build()
    import int2_rotated_paged_gb300 as k
    return k


def _declared():
    src = open(os.path.join(ROOT, "include", "oscar_kv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b([a-z_0-9]+)\s*\([^;{]*\)\s*;", src)))


def test_every_declared_symbol_is_exported(K):
    names = _declared()
    assert "kv_quant_append" in names and "oscar_decode_attention" in names and "kv_page_table_init" in names
    L = ctypes.CDLL(K.LIB_PATH)
    for n in names:
        assert hasattr(L, n), n
    assert sorted(K.EXPORTS) == names
    out = subprocess.run(["nm", "-D", "--defined-only", K.LIB_PATH], capture_output=True, text=True).stdout
    for n in names:
        assert re.search(rf"\bT {n}$", out, re.M), n


def _desc(K, **kw):
    d = K.default_desc()
    d.batch, d.num_q_heads, d.num_kv_heads = 4, 32, 8
    d.max_pages_total, d.max_pages_per_seq = 20, 8
    for k, v in kw.items():
        setattr(d, k, v)
    return d


FAKE = [0x10000, 0x20000, 0x30000, 0x40000]   # never dereferenced by host-only calls


def _create(K, d):
    return K.oscar_cache_create(d, *FAKE)


def test_descriptor_defaults_and_sizes(K):
    d = _desc(K)
    assert (d.head_dim, d.page_size, d.group_size, d.sink, d.window) == (128, 64, 64, 64, 256)
    assert abs(d.clip_k - 0.96) < 1e-7 and abs(d.clip_v - 0.92) < 1e-7
    L = K.lib()
    assert L.oscar_pool_bytes(ctypes.byref(d)) == 20 * 8 * 5120
    assert d.group_size_v == 64 and L.oscar_page_head_bytes(ctypes.byref(d)) == 5120
    assert L.oscar_bf16_bytes(ctypes.byref(d)) == 4 * 8 * 2 * 320 * 128 * 2
    assert L.oscar_page_table_bytes(ctypes.byref(d)) == 4 * 8 * 4
    # 4 lengths (16 bytes), then 4 x 8 value-scale maxima
    assert L.oscar_seq_lens_bytes(ctypes.byref(d)) == 16 + 4 * 8 * 4


@pytest.mark.parametrize("field,value", [("head_dim", 64), ("page_size", 32), ("group_size", 32),
                                         ("group_size", 96), ("group_size_v", 32), ("group_size_v", 256),
                                         ("sink", 0), ("window", 128), ("num_q_heads", 36),
                                         ("num_q_heads", 80), ("batch", 0), ("clip_k", 0.0),
                                         ("clip_v", 1.5), ("max_pages_total", 0)])
def test_bad_descriptors_rejected(K, field, value):
    d = _desc(K, **{field: value})
    assert K.lib().oscar_pool_bytes(ctypes.byref(d)) == 0
    with pytest.raises(K.OscarError) as e:
        _create(K, d)
    assert e.value.code == K.OSCAR_EINVAL


def test_alignment_checked(K):
    d = _desc(K)
    with pytest.raises(K.OscarError) as e:
        K.oscar_cache_create(d, FAKE[0] + 4, *FAKE[1:])
    assert e.value.code == K.OSCAR_EALIGN


def test_free_list_order_and_reuse(K):
    d = _desc(K)
    c = _create(K, d)
    order = [7, 3, 19, 0, 11, 5, 2, 13, 1, 4, 6, 8, 9, 10, 12, 14, 15, 16, 17, 18]
    K.kv_page_table_init(c, order)
    assert K.kv_page_table_free_pages(c) == 20
    # 320 tokens fit in sink + window: no page; 321 needs one; 320 + 64*3 + 1 needs four
    K.kv_page_table_reserve(c, 0, 320)
    assert K.kv_page_table_read(c, 0) == []
    K.kv_page_table_reserve(c, 0, 321)
    assert K.kv_page_table_read(c, 0) == [7]
    K.kv_page_table_reserve(c, 1, 320 + 64 * 3 + 1)
    assert K.kv_page_table_read(c, 1) == [3, 19, 0, 11]
    K.kv_page_table_reserve(c, 0, 320 + 128)      # grows by one page only
    assert K.kv_page_table_read(c, 0) == [7, 5]
    assert K.kv_page_table_free_pages(c) == 14
    K.kv_page_table_release(c, 1)
    assert K.kv_page_table_free_pages(c) == 18 and K.kv_page_table_read(c, 1) == []
    K.kv_page_table_reserve(c, 2, 320 + 64 * 2)    # released pages come back first, in order
    assert K.kv_page_table_read(c, 2) == [3, 19]
    K.lib().oscar_cache_destroy(c)


def test_capacity_errors_leave_state_unchanged(K):
    d = _desc(K, max_pages_total=6, max_pages_per_seq=4)
    c = _create(K, d)
    K.kv_page_table_init(c, None)
    with pytest.raises(K.OscarError) as e:          # row limit: 5 pages > 4
        K.kv_page_table_reserve(c, 0, 320 + 64 * 5)
    assert e.value.code == K.OSCAR_ENOPAGES and K.kv_page_table_free_pages(c) == 6
    K.kv_page_table_reserve(c, 0, 320 + 64 * 4)
    with pytest.raises(K.OscarError) as e:          # pool limit: 3 pages > 2 left
        K.kv_page_table_reserve(c, 1, 320 + 64 * 3)
    assert e.value.code == K.OSCAR_ENOPAGES
    assert K.kv_page_table_free_pages(c) == 2 and K.kv_page_table_read(c, 1) == []
    with pytest.raises(K.OscarError) as e:
        K.kv_page_table_reserve(c, 4, 10)
    assert e.value.code == K.OSCAR_ERANGE
    with pytest.raises(K.OscarError) as e:
        K.kv_page_table_init(c, [0, 1, 2, 3, 4, 4])  # not a permutation
    assert e.value.code == K.OSCAR_EINVAL
    assert K.kv_page_table_read(c, 0) == [0, 1, 2, 3]   # unchanged by the failed init
    K.lib().oscar_cache_destroy(c)


def test_append_argument_errors_before_any_launch(K):
    d = _desc(K, max_pages_total=4, max_pages_per_seq=4)
    c = _create(K, d)
    L = K.lib()
    arr = (ctypes.c_int32 * 4)(1, 1, 1, 1)
    # no key / value pointers
    assert L.kv_quant_append(c, None, None, arr, None, None) == K.OSCAR_EINVAL
    neg = (ctypes.c_int32 * 4)(1, -1, 0, 0)
    assert L.kv_quant_append(c, FAKE[0], FAKE[1], neg, FAKE[2], None) == K.OSCAR_EINVAL
    big = (ctypes.c_int32 * 4)(320 + 64 * 5, 0, 0, 0)
    assert L.kv_quant_append(c, FAKE[0], FAKE[1], big, FAKE[2], None) == K.OSCAR_ENOPAGES
    assert L.kv_quant_append(c, FAKE[0] + 2, FAKE[1], arr, FAKE[2], None) == K.OSCAR_EALIGN
    assert L.oscar_cache_length(c, 0) == 0 and L.kv_page_table_free_pages(c) == 4
    # decode: workspace too small, bad dtype
    assert L.oscar_decode_attention(c, FAKE[0], 0, FAKE[1], FAKE[2], 0, FAKE[3], 16, None) == K.OSCAR_EWORKSPACE
    assert L.oscar_decode_attention(c, FAKE[0], 7, FAKE[1], FAKE[2], 0, FAKE[3], 1 << 40, None) == K.OSCAR_EINVAL
    assert L.oscar_build_rk(FAKE[0], 0, 8, FAKE[1], FAKE[2], 1 << 30, None) == K.OSCAR_EINVAL
    assert L.oscar_build_rk(FAKE[0], 10, 8, FAKE[1], FAKE[2], 8, None) == K.OSCAR_EWORKSPACE
    assert K.strerror(K.OSCAR_ENOPAGES) == "out of INT2 pages"
    # fused decode step: the decode checks, then the append checks, all before anything changes
    big_ws = ctypes.c_size_t(1 << 40)
    assert L.oscar_decode_step(c, FAKE[0], FAKE[1], FAKE[2], 0, FAKE[3], FAKE[0], 0, FAKE[1], 16,
                               None) == K.OSCAR_EWORKSPACE
    assert L.oscar_decode_step(c, FAKE[0], FAKE[1], FAKE[2], 7, FAKE[3], FAKE[0], 0, FAKE[1], big_ws,
                               None) == K.OSCAR_EINVAL
    assert L.oscar_decode_step(c, FAKE[0] + 2, FAKE[1], FAKE[2], 0, FAKE[3], FAKE[0], 0, FAKE[1], big_ws,
                               None) == K.OSCAR_EALIGN
    assert L.oscar_decode_step(c, None, FAKE[1], FAKE[2], 0, FAKE[3], FAKE[0], 0, FAKE[1], big_ws,
                               None) == K.OSCAR_EINVAL
    assert L.oscar_cache_length(c, 0) == 0 and L.kv_page_table_free_pages(c) == 4
    L.oscar_cache_destroy(c)


def test_decode_path_and_timing_arguments(K):
    L = K.lib()
    assert L.oscar_set_decode_path(0) == K.OSCAR_EINVAL          # no tensor-memory path any more
    assert L.oscar_set_decode_path(3) == K.OSCAR_EINVAL
    assert L.oscar_set_decode_path(K.PATH_SIMT) == 0
    assert L.oscar_set_decode_path(K.PATH_WARP_MMA) == 0
    c = _create(K, _desc(K))
    assert L.oscar_kernel_timing(c, -1) == K.OSCAR_EINVAL
    assert L.oscar_kernel_timing(c, 0) == 0                      # nothing recorded, nothing to free
    got = ctypes.c_int32(5)
    assert L.oscar_kernel_timing_read(c, None, 0, ctypes.byref(got)) == 0 and got.value == 0
    assert L.oscar_kernel_timing_read(c, None, 4, ctypes.byref(got)) == K.OSCAR_EINVAL
    assert L.oscar_kernel_timing_read(c, None, 0, None) == K.OSCAR_EINVAL
    L.oscar_cache_destroy(c)


@pytest.mark.parametrize("gk,gv,page", [(64, 64, 5120), (64, 128, 4864), (128, 128, 4608), (128, 64, 4864),
                                        (128, 0, 4608)])
def test_page_format_per_group_sizes(K, gk, gv, page):
    # one fp16 (scale, minimum) pair per group and token: 64 tokens x 4 B x (128 / group) per tensor
    d = _desc(K, group_size=gk, group_size_v=gv)
    L = K.lib()
    assert L.oscar_page_head_bytes(ctypes.byref(d)) == page
    assert L.oscar_pool_bytes(ctypes.byref(d)) == d.max_pages_total * d.num_kv_heads * page
    # bits per stored INT2 value: codes (2 bits) plus the scale/min pairs
    assert page * 8 / (64 * 256) == (2 * 128 + 32 * 128 / gk + 2 * 128 + 32 * 128 / (gv or gk)) / 256
