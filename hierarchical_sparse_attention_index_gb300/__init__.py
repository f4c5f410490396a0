"""Python binding of libhsa, the GB300 (sm_103a) CSA2 hierarchical sparse indexer and sparse
attention (DeepSeek-V4.1-Flash decode hot path).

The functions keep the C ABI's names (``hsa_index_full`` and so on; see include/hsa.h). They
only marshal arguments. Tensors are passed as raw device pointers, and every step of the path
runs in the library's CUDA kernels. The library is built in-tree by ``build.py``. Loading it
when it is missing raises, because there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libhsa.so")

HSA_D_LATENT, HSA_D_INDEX, HSA_H_INDEX, HSA_H_ATTN = 512, 128, 16, 64
HSA_TOPK, HSA_CAND_BLOCKS, HSA_BLOCK, HSA_POOL_SLOTS, HSA_SWA_W = 512, 2048, 8, 16384, 128
HSA_MAX_NQ, HSA_MAX_VIS = 8, 1 << 20
HSA_NOALLOC_SCRATCH_BYTES = 64 << 20
HSA_SCALE_E8M0, HSA_SCALE_E4M3 = 0, 1
HSA_MODE_FULL, HSA_MODE_REINDEX, HSA_MODE_REUSE = 0, 1, 2
HSA_FLAG_INDEX_RANGE, HSA_FLAG_WRITE_RANGE, HSA_FLAG_TIMEOUT = 1, 2, 4
HSA_CACHE_ROPE, HSA_CACHE_POOL_TAIL = 1, 2
HSA_POOL_TAIL_SLOTS = 160
HSA_ROPE_DIMS, HSA_ROPE_THETA = 64, 160000.0

STATUS = {0: "HSA_OK", 1: "HSA_ERR_INVALID_ARG", 2: "HSA_ERR_SHAPE", 3: "HSA_ERR_ALIGN",
          4: "HSA_ERR_WORKSPACE", 5: "HSA_ERR_CUDA", 6: "HSA_ERR_TIMEOUT", 7: "HSA_ERR_UNSUPPORTED"}
STATUS_CODES = {v: k for k, v in STATUS.items()}

EXPORTS = ("hsa_abi_version", "hsa_status_string", "hsa_workspace_bytes", "hsa_workspace_init",
           "hsa_cache_write_compress", "hsa_index_full", "hsa_index_reindex", "hsa_sparse_attn_decode",
           "hsa_schedule_step", "hsa_get_device_status", "hsa_index_full_noalloc", "hsa_set_wait_limit",
           "hsa_debug_stall_next_scan")


class HsaError(RuntimeError):
    def __init__(self, fn, code, text):
        super().__init__(f"{fn} failed: {text} ({code})")
        self.code = code


class hsa_cache(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("ratio", ctypes.c_int32), ("capacity", ctypes.c_int64),
                ("kv_scale_fmt", ctypes.c_int32), ("flags", ctypes.c_int32),
                ("kv_q", ctypes.c_void_p), ("kv_s", ctypes.c_void_p), ("ik_q", ctypes.c_void_p),
                ("ik_s", ctypes.c_void_p)]


class hsa_step_args(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("nq", ctypes.c_int32),
                ("modes", ctypes.POINTER(ctypes.c_int32)), ("q_idx", ctypes.POINTER(ctypes.c_void_p)),
                ("w_idx", ctypes.POINTER(ctypes.c_void_p)), ("q_attn", ctypes.POINTER(ctypes.c_void_p)),
                ("swa", ctypes.POINTER(ctypes.c_void_p)), ("out", ctypes.POINTER(ctypes.c_void_p)),
                ("topk", ctypes.POINTER(ctypes.c_void_p)), ("pool", ctypes.c_void_p),
                ("vis", ctypes.c_void_p), ("max_vis", ctypes.c_int64), ("sm_scale", ctypes.c_float)]


_lib = None


def load_library(path: str = LIB_PATH):
    """Load libhsa.so (build it first with build.build()); raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libhsa.so not found at {path}: build it with "
                           "`python -m hierarchical_sparse_attention_index_gb300.build`")
    lib = ctypes.CDLL(path)
    P, I32, I64, SZ, F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
    C = ctypes.POINTER(hsa_cache)
    sig = {
        "hsa_abi_version": (I32, []),
        "hsa_status_string": (ctypes.c_char_p, [I32]),
        "hsa_workspace_bytes": (SZ, [I32, I32, I64]),
        "hsa_workspace_init": (I32, [P, SZ, P]),
        "hsa_cache_write_compress": (I32, [C, P, P, P, I64, P, P]),
        "hsa_index_full": (I32, [C, P, P, P, I32, I64, P, P, P, SZ, P]),
        "hsa_index_reindex": (I32, [C, P, P, P, I32, I64, P, P, P, SZ, P]),
        "hsa_sparse_attn_decode": (I32, [C, P, P, P, P, I32, I64, F, P, P, SZ, P]),
        "hsa_schedule_step": (I32, [C, ctypes.POINTER(hsa_step_args), P, SZ, P]),
        "hsa_get_device_status": (I32, [P, ctypes.POINTER(ctypes.c_uint32)]),
        "hsa_index_full_noalloc": (I32, [C, P, P, P, I32, I64, P, P, P]),
        "hsa_set_wait_limit": (I32, [ctypes.c_uint64]),
        "hsa_debug_stall_next_scan": (I32, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _ptr(t):
    """Device (or host) address of a tensor, None stays NULL, ints pass through."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn, code):
    if code != 0:
        text = load_library().hsa_status_string(code).decode()
        raise HsaError(fn, code, text)


class Cache:
    """Caller-owned FP4 cache of one KV-source layer: four uint8 device tensors
    (kv_q [B][cap][256], kv_s [B][cap][32], ik_q [B][cap][64], ik_s [B][cap][4]); `flags` holds
    HSA_CACHE_* bits (HSA_CACHE_ROPE: the writer applies RoPE to the main-KV latent)."""

    def __init__(self, batch, capacity, ratio=1, kv_scale_fmt=HSA_SCALE_E8M0, device="cuda", tensors=None, flags=0):
        import torch
        self.batch, self.capacity, self.ratio, self.kv_scale_fmt = batch, capacity, ratio, kv_scale_fmt
        self.flags = flags
        if tensors is None:
            z = dict(dtype=torch.uint8, device=device)
            tensors = (torch.zeros(batch, capacity, 256, **z), torch.zeros(batch, capacity, 32, **z),
                       torch.zeros(batch, capacity, 64, **z), torch.zeros(batch, capacity, 4, **z))
        self.kv_q, self.kv_s, self.ik_q, self.ik_s = tensors
        self.desc = hsa_cache(batch, ratio, capacity, kv_scale_fmt, flags, _ptr(self.kv_q), _ptr(self.kv_s),
                              _ptr(self.ik_q), _ptr(self.ik_s))

    @property
    def ref(self):
        return ctypes.byref(self.desc)


def hsa_abi_version():
    return load_library().hsa_abi_version()


def hsa_status_string(code):
    return load_library().hsa_status_string(code).decode()


def hsa_workspace_bytes(batch, nq, max_vis):
    return load_library().hsa_workspace_bytes(batch, nq, max_vis)


def hsa_workspace_init(ws, stream=None):
    _check("hsa_workspace_init", load_library().hsa_workspace_init(_ptr(ws), ws.numel() * ws.element_size(),
                                                                   _stream(stream)))


def new_workspace(batch, nq, max_vis, device="cuda", stream=None):
    """Allocate (torch) and zero-fill a workspace for the given sizes."""
    import torch
    n = hsa_workspace_bytes(batch, nq, max_vis)
    if n == 0:
        raise ValueError("invalid workspace sizes")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    hsa_workspace_init(ws, stream)
    return ws


def hsa_cache_write_compress(cache: Cache, wkv, wgate, w_idx, n_tokens, start_entry=None, stream=None):
    _check("hsa_cache_write_compress", load_library().hsa_cache_write_compress(
        cache.ref, _ptr(wkv), _ptr(wgate), _ptr(w_idx), n_tokens, _ptr(start_entry), _stream(stream)))


def hsa_index_full(cache: Cache, q, w, vis, nq, max_vis, topk_out, pool_out, ws, stream=None):
    _check("hsa_index_full", load_library().hsa_index_full(
        cache.ref, _ptr(q), _ptr(w), _ptr(vis), nq, max_vis, _ptr(topk_out), _ptr(pool_out), _ptr(ws),
        ws.numel() * ws.element_size(), _stream(stream)))


def hsa_index_reindex(cache: Cache, q, w, vis, nq, max_vis, pool, topk_out, ws, stream=None):
    _check("hsa_index_reindex", load_library().hsa_index_reindex(
        cache.ref, _ptr(q), _ptr(w), _ptr(vis), nq, max_vis, _ptr(pool), _ptr(topk_out), _ptr(ws),
        ws.numel() * ws.element_size(), _stream(stream)))


def hsa_index_full_noalloc(cache: Cache, q, w, vis, nq, max_vis, topk_out, pool_out, stream=None):
    """hsa_index_full for callers that cannot allocate device memory: its scratch is a fixed
    array inside the library (HSA_NOALLOC_SCRATCH_BYTES), shared by every call, so calls that
    overlap on the GPU race. The first call on a device looks up the array's address there and
    should come before any stream capture."""
    _check("hsa_index_full_noalloc", load_library().hsa_index_full_noalloc(
        cache.ref, _ptr(q), _ptr(w), _ptr(vis), nq, max_vis, _ptr(topk_out), _ptr(pool_out), _stream(stream)))


def hsa_sparse_attn_decode(cache: Cache, q, topk, swa, vis, nq, max_vis, sm_scale, out, ws, stream=None):
    _check("hsa_sparse_attn_decode", load_library().hsa_sparse_attn_decode(
        cache.ref, _ptr(q), _ptr(topk), _ptr(swa), _ptr(vis), nq, max_vis, float(sm_scale), _ptr(out),
        _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


class StepArgs:
    """Builds hsa_step_args from per-layer tensor lists (None for unused slots)."""

    def __init__(self, modes, q_idx, w_idx, q_attn, swa, out, topk, pool, vis, nq, max_vis, sm_scale):
        n = len(modes)
        arr = lambda xs: (ctypes.c_void_p * n)(*[_ptr(x) for x in xs])  # noqa: E731
        self._keep = [arr(q_idx), arr(w_idx), arr(q_attn), arr(swa), arr(out), arr(topk),
                      (ctypes.c_int32 * n)(*modes)]
        self.tensors = (q_idx, w_idx, q_attn, swa, out, topk, pool, vis)
        vp = ctypes.POINTER(ctypes.c_void_p)
        self.args = hsa_step_args(n, nq, ctypes.cast(self._keep[6], ctypes.POINTER(ctypes.c_int32)),
                                  ctypes.cast(self._keep[0], vp), ctypes.cast(self._keep[1], vp),
                                  ctypes.cast(self._keep[2], vp), ctypes.cast(self._keep[3], vp),
                                  ctypes.cast(self._keep[4], vp), ctypes.cast(self._keep[5], vp),
                                  _ptr(pool), _ptr(vis), max_vis, float(sm_scale))


def hsa_schedule_step(caches, step: StepArgs, ws, stream=None):
    """`caches`: one Cache per layer slot (a list), or one Cache that every slot uses."""
    n = step.args.n_layers
    if isinstance(caches, Cache):
        caches = [caches] * n
    if len(caches) != n:
        raise ValueError(f"{len(caches)} caches for {n} layer slots")
    descs = (hsa_cache * n)(*[c.desc for c in caches])
    _check("hsa_schedule_step", load_library().hsa_schedule_step(
        descs, ctypes.byref(step.args), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def hsa_set_wait_limit(ns):
    """Limit of the kernels' bounded waits for later launches, in ns (0: the default, 2 s)."""
    _check("hsa_set_wait_limit", load_library().hsa_set_wait_limit(int(ns)))


def hsa_debug_stall_next_scan():
    """Test hook: the next hsa_index_full withholds one copy of its scan, so a bounded wait runs
    out (HSA_FLAG_TIMEOUT); that call's outputs are invalid, later calls are unaffected."""
    _check("hsa_debug_stall_next_scan", load_library().hsa_debug_stall_next_scan())


def hsa_get_device_status(stream=None):
    """Synchronise the stream and return (status code, flags); the flags are cleared."""
    flags = ctypes.c_uint32(0)
    code = load_library().hsa_get_device_status(_stream(stream), ctypes.byref(flags))
    return code, flags.value
