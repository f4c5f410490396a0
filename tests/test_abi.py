"""The C-ABI library builds, loads and exports every entry point include/hsa.h declares. Only host
paths run here, with no compute calls: version, status strings, workspace sizing, and argument
validation that returns before any CUDA call."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from hierarchical_sparse_attention_index_gb300 import build
    try:
        build.nvcc()
    except RuntimeError as e:
        pytest.skip(str(e))
    build.build()
    import hierarchical_sparse_attention_index_gb300 as H
    return H.load_library()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "hsa.h"), encoding="utf-8").read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(hsa_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    import hierarchical_sparse_attention_index_gb300 as H
    assert sorted(H.EXPORTS) == names


def test_version_and_status_strings(lib):
    import hierarchical_sparse_attention_index_gb300 as H
    assert H.hsa_abi_version() == 3
    for code, name in H.STATUS.items():
        assert H.hsa_status_string(code).startswith(name)
    assert H.hsa_status_string(99) == "HSA_ERR_UNKNOWN"


def test_workspace_sizing(lib):
    import hierarchical_sparse_attention_index_gb300 as H
    assert H.hsa_workspace_bytes(0, 1, 100) == 0
    assert H.hsa_workspace_bytes(1, 0, 100) == 0
    assert H.hsa_workspace_bytes(1, 9, 100) == 0
    assert H.hsa_workspace_bytes(1, 1, (1 << 20) + 1) == 0
    a = H.hsa_workspace_bytes(32, 1, 131072)
    b = H.hsa_workspace_bytes(32, 1, 1 << 20)
    assert 0 < a < b
    # scores, block maxima and candidate lists dominate: ~ rows * ld_s * 4 * 2.25
    assert a > 32 * 131072 * 4 * 2


def test_host_validation_without_gpu(lib):
    import hierarchical_sparse_attention_index_gb300 as H
    null = None
    # NULL cache descriptor
    assert lib.hsa_index_full(null, null, null, null, 1, 10, null, null, null, 0, null) == 1
    assert lib.hsa_index_reindex(null, null, null, null, 1, 10, null, null, null, 0, null) == 1
    assert lib.hsa_sparse_attn_decode(null, null, null, null, null, 1, 10, 1.0, null, null, 0, null) == 1
    assert lib.hsa_cache_write_compress(null, null, null, null, 4, null, null) == 1
    assert lib.hsa_schedule_step(null, null, null, 0, null) == 1
    # shape and alignment errors with fake (never dereferenced) pointers
    c = H.hsa_cache(1, 1, 1004, 0, 0, 0x1000, 0x2000, 0x3000, 0x4000)   # capacity not a multiple of 8
    assert lib.hsa_index_full(ctypes.byref(c), 0x10, 0x20, 0x30, 1, 10, 0x40, 0x50, 0x60, 1 << 30, null) == 2
    c.capacity = 1024
    assert lib.hsa_index_full(ctypes.byref(c), 0x10, 0x20, 0x30, 9, 10, 0x40, 0x50, 0x60, 1 << 30, null) == 2
    assert lib.hsa_index_full(ctypes.byref(c), 0x10, 0x20, 0x30, 1, 2000, 0x40, 0x50, 0x60, 1 << 30, null) == 2
    assert lib.hsa_index_full(ctypes.byref(c), 0x11, 0x20, 0x30, 1, 10, 0x40, 0x50, 0x60, 1 << 30, null) == 3
    assert lib.hsa_index_full(ctypes.byref(c), 0x10, 0x20, 0x30, 1, 10, 0x40, 0x50, 0x60, 16, null) == 4
    # attention: the workspace carries the partial outputs, so a missing or short one is refused
    assert lib.hsa_sparse_attn_decode(ctypes.byref(c), 0x10, 0x20, 0x30, 0x40, 1, 10, 1.0, 0x50, null, 0,
                                      null) == 4
    assert lib.hsa_sparse_attn_decode(ctypes.byref(c), 0x10, 0x20, 0x30, 0x40, 1, 10, 1.0, 0x50, 0x60, 16,
                                      null) == 4
    assert lib.hsa_sparse_attn_decode(ctypes.byref(c), 0x10, 0x20, 0x30, 0x40, 1, 10, 1.0, 0x58, 0x60, 1 << 30,
                                      null) == 3
    c.ratio = 3
    assert lib.hsa_index_full(ctypes.byref(c), 0x10, 0x20, 0x30, 1, 10, 0x40, 0x50, 0x60, 1 << 30, null) == 1
    c.ratio = 2
    # ratio 2 without wgate
    assert lib.hsa_cache_write_compress(ctypes.byref(c), 0x10, null, 0x20, 4, null, null) == 1
    flags = ctypes.c_uint32(0)
    assert lib.hsa_get_device_status(null, None) == 1


def test_wait_limit_and_stall_hook_are_host_only(lib):
    """The wait limit and the stall hook only set host state (no CUDA call, no device needed)."""
    import hierarchical_sparse_attention_index_gb300 as H
    assert lib.hsa_set_wait_limit(1000) == 0
    assert lib.hsa_set_wait_limit(0) == 0
    assert H.STATUS_CODES["HSA_ERR_TIMEOUT"] == 6


def test_schedule_step_checks_every_slot_cache_without_gpu(lib):
    """hsa_schedule_step takes one cache per layer slot and refuses, before any launch, slots
    whose caches disagree on batch, ratio or the pool-tail flag, or hold fewer than max_vis
    entries (fake, never dereferenced pointers)."""
    import hierarchical_sparse_attention_index_gb300 as H
    n = 2
    modes = (ctypes.c_int32 * n)(H.HSA_MODE_FULL, H.HSA_MODE_REUSE)
    ptrs = lambda *v: (ctypes.c_void_p * n)(*v)  # noqa: E731
    keep = [ptrs(0x100, None), ptrs(0x200, None), ptrs(0x300, 0x310), ptrs(0x400, 0x410), ptrs(0x500, 0x510),
            ptrs(0x600, None)]
    vp = ctypes.POINTER(ctypes.c_void_p)
    args = H.hsa_step_args(n, 1, ctypes.cast(modes, ctypes.POINTER(ctypes.c_int32)),
                           *[ctypes.cast(k, vp) for k in keep], 0x700, 0x800, 1000, 1.0)

    def caches(*specs):
        return (H.hsa_cache * n)(*[H.hsa_cache(b, 1, cap, 0, fl, 0x1000, 0x2000, 0x3000, 0x4000)
                                   for b, cap, fl in specs])

    step = lambda cs: lib.hsa_schedule_step(cs, ctypes.byref(args), 0x900, 1 << 30, None)  # noqa: E731
    assert step(caches((2, 1024, 0), (1, 1024, 0))) == 2                          # batch differs
    assert step(caches((2, 1024, 0), (2, 1024, H.HSA_CACHE_POOL_TAIL))) == 2      # pool-tail flag differs
    assert step(caches((2, 1024, 0), (2, 512, 0))) == 2                           # slot 1 holds < max_vis
    assert step(caches((2, 1024, 0), (2, 1020, 0))) == 2                          # slot 1 capacity invalid
    assert step(None) == 1
