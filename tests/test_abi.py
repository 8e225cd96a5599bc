"""C-ABI checks that need no GPU: the library loads, exports every entry
point include/ibp.h declares, and rejects bad arguments on the host before
touching the device."""
import ctypes

import pytest

from lossless_invariant_bit_gb300 import ibp
from lossless_invariant_bit_gb300 import build as libbuild


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return ibp._lib_handle()


def test_exports_every_declared_symbol(lib):
    names = ibp.declared_symbols()
    assert len(names) >= 17
    for n in names:
        assert hasattr(lib, n), n
    # and the binding wraps each of them under the same name
    for n in names:
        assert callable(getattr(ibp, n)), n


def test_status_strings(lib):
    for code, name in enumerate(ibp.STATUS_NAMES):
        assert ibp.ibp_status_str(code).startswith(name)
    assert "unknown" in ibp.ibp_status_str(99)


def test_host_side_argument_checks(lib):
    out = ctypes.c_void_p()
    # geometry outside the limits is rejected before any device call
    assert lib.ibp_store_create(ctypes.byref(out), 0, 256, 10, 0) == ibp.IBP_EINVAL
    assert lib.ibp_store_create(ctypes.byref(out), 1000, 256, 10, 0) == ibp.IBP_EINVAL  # R % 16
    assert lib.ibp_store_create(ctypes.byref(out), 65536, 256, 10, 0) == ibp.IBP_EINVAL  # > max
    assert lib.ibp_store_create(ctypes.byref(out), 1024, 6, 10, 0) == ibp.IBP_EINVAL  # C % 4
    assert lib.ibp_store_create(ctypes.byref(out), 8192, 4, 10, 0) == ibp.IBP_EINVAL  # nch > max
    assert lib.ibp_store_create(ctypes.byref(out), 1024, 256, 0, 0) == ibp.IBP_EINVAL  # no rows
    assert lib.ibp_store_create(ctypes.byref(out), 1024, 256, 10, 1000) == ibp.IBP_EALIGN
    assert lib.ibp_store_create(ctypes.byref(out), 1024, 256, 10, 512) == ibp.IBP_EALIGN
    assert lib.ibp_store_create(None, 1024, 256, 10, 0) == ibp.IBP_EINVAL
    # NULL store
    assert lib.ibp_build_meta(None, 16, 16, None, 1, 95, 100, None) == ibp.IBP_EINVAL
    assert lib.ibp_compress(None, 16, 16, 16, None, 1, None, None) == ibp.IBP_EINVAL
    assert lib.ibp_decompress(None, 16, 16, None, 1, None) == ibp.IBP_EINVAL
    assert lib.ibp_gather_decompress(None, 16, 16, None, 16, 1, None) == ibp.IBP_EINVAL
    assert lib.ibp_gather_decompress_strided(None, 16, 16, 16, None, 16, 1, None) == ibp.IBP_EINVAL
    assert lib.ibp_gather_decompress_cached(None, 16, 16, 16, 16, 1, 16, 16, 1, None) == ibp.IBP_EINVAL
    assert lib.ibp_gather_decompress_split(None, 16, 1, 0, 16, 256, 16, None, 16, 1,
                                           None) == ibp.IBP_EINVAL
    assert lib.ibp_gather_decompress_ordered(None, 16, 16, 16, None, 16, 1, 16, 4112,
                                             None) == ibp.IBP_EINVAL
    assert ibp.order_workspace_bytes(10) == 20 * 10 + 65536
    assert lib.ibp_store_set_lengths(None, 16) == ibp.IBP_EINVAL
    # a cache front needs both its map and its cache, the cache 16-byte aligned
    assert lib.ibp_gather_decompress_cached(None, 16, 16, 16, 16, 1, None, 16, 1, None) == ibp.IBP_EINVAL
    assert lib.ibp_gather_decompress_cached(None, 16, 16, 16, None, 1, 16, 16, 1, None) == ibp.IBP_EINVAL
    assert lib.ibp_gather_decompress_cached(None, 16, 16, 16, 17, 1, 16, 16, 1, None) == ibp.IBP_EALIGN
    assert lib.ibp_pack(None, None, 16, None, None, 0, None) == ibp.IBP_EINVAL
    assert lib.ibp_meta_get(None, 16, 16) == ibp.IBP_EINVAL
    assert lib.ibp_meta_set(None, 16, 16) == ibp.IBP_EINVAL
    assert lib.ibp_bitmap_get(None, 16) == ibp.IBP_EINVAL
    assert lib.ibp_bitmap_set(None, 16) == ibp.IBP_EINVAL
    assert lib.ibp_store_get_info(None, None) == ibp.IBP_EINVAL
    st = ctypes.c_int()
    assert lib.ibp_stream_status(None, None, ctypes.byref(st), 0) == ibp.IBP_EINVAL
    assert lib.ibp_store_destroy(None) == ibp.IBP_OK
    grp = ctypes.c_void_p()
    assert lib.ibp_group_create(ctypes.byref(grp), None, None, 1) == ibp.IBP_EINVAL
    assert lib.ibp_group_create(None, 16, 16, 1) == ibp.IBP_EINVAL
    assert lib.ibp_group_gather_decompress(None, 16, 512, 16, 1, None) == ibp.IBP_EINVAL
    assert lib.ibp_group_order_plan(None, 16, 1, 16, 65556, None) == ibp.IBP_EINVAL
    assert lib.ibp_group_gather_decompress_planned(None, 16, 512, 16, 1, 16, 65556,
                                                   None) == ibp.IBP_EINVAL
    assert lib.ibp_group_destroy(None) == ibp.IBP_OK
    num = (ctypes.c_uint32 * 1)(95)
    den = (ctypes.c_uint32 * 1)(100)
    assert lib.ibp_build_meta_tuned(None, 16, 16, None, 1, num, den, 1, None, None,
                                    None) == ibp.IBP_EINVAL
    # copies: alignment and size checked on the host
    assert lib.ibp_link_copy(16, 16, 0, None) == ibp.IBP_OK
    assert lib.ibp_link_copy(None, 16, 16, None) == ibp.IBP_EINVAL
    assert lib.ibp_link_copy(17, 16, 16, None) == ibp.IBP_EALIGN
    assert lib.ibp_link_copy(16, 16, 24, None) == ibp.IBP_EALIGN
    assert lib.ibp_gather_copy(16, 16, 512, 500, 16, 4, 10, None) == ibp.IBP_EALIGN
    assert lib.ibp_gather_copy(16, 16, 512, 512, None, 4, 10, None) == ibp.IBP_EINVAL


def test_binding_raises_on_error(lib):
    with pytest.raises(ibp.IbpError) as ei:
        ibp.ibp_store_create(1000, 256, 10)
    assert ei.value.status == ibp.IBP_EINVAL


def test_project_compress_host_checks(lib):
    """The fused projection rejects a missing store on the host, and its
    workspace size is the header's formula: a 4-byte participation flag per
    (row, tile), up to four tiles per 256-byte chunk (rounded to 256 bytes),
    then R bytes of staged kept bits per row."""
    assert lib.ibp_project_compress(None, 16, 20, 4096, 16, None, 0, 16, 16, None, None, 16,
                                    1 << 20, None) == ibp.IBP_EINVAL
    # m = 20 rows of 8 KB (32 chunks, up to 128 tiles): 20*128*4 = 10240 + 20*8192
    assert ibp.project_workspace_bytes(20, 8192) == 10240 + 163840
    # m = 300: 300*512 = 153600 bytes of flags (a multiple of 256)
    assert ibp.project_workspace_bytes(300, 8192) == 153600 + 300 * 8192
    assert ibp.project_workspace_bytes(3, 256) == 256 + 768
