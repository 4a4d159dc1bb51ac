"""Python binding of libhs, the HiSparse decode hot path for GB300 (sm_103a).

Argument marshalling only: every step of the path runs in libhs's CUDA
kernels.  Function names match the C ABI in include/hs.h.  Device buffers are
passed as torch CUDA tensors (or raw integer addresses); streams and events as
torch.cuda.Stream / torch.cuda.Event (or raw handles).  If libhs.so cannot be
loaded an ImportError-style RuntimeError is raised -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import _build

LIB_PATH = _build.LIB

HS_OK = 0
HS_ERR_INVALID = -1
HS_ERR_CUDA = -2
HS_ERR_OOM = -3
HS_ERR_CAPACITY = -4
HS_ERR_DEVICE = -5
HS_ERR_TIMEOUT = -6

HS_KV_BF16 = 0
HS_KV_FP8 = 1
FP8_ROW_BYTES = 656

DEV_ERR_RANGE = 1
DEV_ERR_DUPLICATE = 2
DEV_ERR_CAPACITY = 4
DEV_ERR_BLOCK = 8
HS_OFFLOAD_MAX_PAGES = 256  # pages one hs_offload_pages call takes
DEV_ERR_WAIT = 16
DEV_ERR_INTERNAL = 32
DEV_ERR_VALUE = 64

EXPORTED = (
    "hs_pool_create", "hs_pool_destroy", "hs_pool_get_views", "hs_pool_reset",
    "hs_set_request", "hs_map_page", "hs_load_page", "hs_resolve", "hs_gather",
    "hs_sparse_mla_decode", "hs_offload_prefix", "hs_offload_pages", "hs_commit_offload",
    "hs_step_advance", "hs_check_errors", "hs_status_string", "hs_version", "hs_host_read",
    "hs_sparse_mla_decode_noalloc", "hs_decode_step", "hs_decode_step_tokens", "hs_resolve_tokens",
    "hs_selftest_bounded_waits",
    "hs_sparse_mla_decode_tokens", "hs_noalloc_check_errors", "hs_wait_offload",
    "hs_pool_host_numa_node", "hs_pool_touch_host",
)


class HsError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)}")


class hs_pool_desc(ctypes.Structure):
    _fields_ = [("num_requests", ctypes.c_int32), ("num_layers", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("hot_slots", ctypes.c_int32),
                ("page_tokens", ctypes.c_int32), ("row_elems", ctypes.c_int32),
                ("max_pages", ctypes.c_int32), ("kv_format", ctypes.c_int32),
                ("host_tokens", ctypes.c_int64), ("resident_blocks", ctypes.c_int64)]


class hs_pool_views(ctypes.Structure):
    _fields_ = [("kv_pool", ctypes.c_void_p), ("host_pool", ctypes.c_void_p),
                ("host_pool_device", ctypes.c_void_p), ("page_table", ctypes.c_void_p),
                ("ctx_len", ctypes.c_void_p), ("host_off", ctypes.c_void_p),
                ("hot_block", ctypes.c_void_p), ("slot_pos", ctypes.c_void_p),
                ("slot_stamp", ctypes.c_void_p), ("lru_order", ctypes.c_void_p),
                ("step", ctypes.c_void_p), ("error_word", ctypes.c_void_p),
                ("blocks_per_layer", ctypes.c_int64), ("kv_pool_bytes", ctypes.c_int64),
                ("host_pool_bytes", ctypes.c_int64)]


_lib = None


def load(build: bool = True) -> ctypes.CDLL:
    """Load libhs.so (building it first if sources are newer)."""
    global _lib
    if _lib is not None:
        return _lib
    if build:
        try:
            _build.build()
        except Exception as e:  # no toolkit: only a pre-built library can serve
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libhs.so is missing and cannot be built: {e}") from e
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libhs.so not found at {LIB_PATH}")
    lib = ctypes.CDLL(LIB_PATH)
    i32, i64, p, f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_float
    sig = {
        "hs_pool_create": [ctypes.POINTER(hs_pool_desc), ctypes.POINTER(p)],
        "hs_pool_destroy": [p],
        "hs_pool_get_views": [p, ctypes.POINTER(hs_pool_views)],
        "hs_pool_reset": [p, p],
        "hs_set_request": [p, i32, i32, i64, p],
        "hs_map_page": [p, i32, i32, i32, p],
        "hs_load_page": [p, i32, i32, i32, p],
        "hs_resolve": [p, i32, i32, p, p, p, p, p, p],
        "hs_gather": [p, i32, p, i64, p, p],
        "hs_sparse_mla_decode": [p, i32, p, p, i32, i32, f32, p, p, p],
        "hs_offload_prefix": [p, i32, i32, p, p, p],
        "hs_offload_pages": [p, i32, p, p, p, p, p],
        "hs_selftest_bounded_waits": [i64, p, p],
        "hs_commit_offload": [p, i32, i32, p, p],
        "hs_step_advance": [p, p],
        "hs_check_errors": [p, ctypes.POINTER(i32)],
        "hs_host_read": [p, i64, p, p],
        "hs_sparse_mla_decode_noalloc": [p, i64, p, p, i32, i32, i32, i32, f32, p, p, p],
        "hs_decode_step": [p, i32, i32, p, p, i32, i32, f32, p, p, p, p, p, p, p],
        "hs_decode_step_tokens": [p, i32, i32, i32, p, p, i32, i32, f32, p, p, p, p, p, p, p],
        "hs_resolve_tokens": [p, i32, i32, i32, p, p, p, p, p, p],
        "hs_sparse_mla_decode_tokens": [p, i32, i32, p, p, i32, i32, f32, p, p, p],
        "hs_noalloc_check_errors": [ctypes.POINTER(i32)],
        "hs_wait_offload": [p, i64],
        "hs_pool_host_numa_node": [p, ctypes.POINTER(i32)],
        "hs_pool_touch_host": [p, p],
    }
    for name, args in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = ctypes.c_int
    lib.hs_status_string.argtypes = [ctypes.c_int]
    lib.hs_status_string.restype = ctypes.c_char_p
    lib.hs_version.argtypes = []
    lib.hs_version.restype = ctypes.c_char_p
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().hs_status_string(int(status)).decode()


def _addr(x) -> int | None:
    """Device/host address of a tensor-like or an int; None stays None (NULL)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    raise TypeError(f"cannot take the address of {type(x)}")


def _stream(s) -> int | None:
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    if hasattr(s, "cuda_stream"):
        return s.cuda_stream
    raise TypeError(f"not a stream: {type(s)}")


def _event(e) -> int:
    if isinstance(e, int):
        return e
    if hasattr(e, "cuda_event"):
        if e.cuda_event == 0:  # torch creates events lazily
            e.record()
            e.synchronize()
        return e.cuda_event
    raise TypeError(f"not an event: {type(e)}")


def _check(status: int, what: str) -> int:
    if status != HS_OK:
        raise HsError(status, what)
    return status


# ---------------------------------------------------------------- C ABI names

def hs_pool_create(desc: hs_pool_desc) -> int:
    h = ctypes.c_void_p()
    _check(load().hs_pool_create(ctypes.byref(desc), ctypes.byref(h)), "hs_pool_create")
    return h.value


def hs_pool_destroy(pool: int) -> None:
    _check(load().hs_pool_destroy(pool), "hs_pool_destroy")


def hs_pool_get_views(pool: int) -> hs_pool_views:
    v = hs_pool_views()
    _check(load().hs_pool_get_views(pool, ctypes.byref(v)), "hs_pool_get_views")
    return v


def hs_pool_reset(pool: int, stream=None) -> None:
    _check(load().hs_pool_reset(pool, _stream(stream)), "hs_pool_reset")


def hs_set_request(pool: int, req: int, ctx_len: int, host_off: int, stream=None) -> None:
    _check(load().hs_set_request(pool, req, ctx_len, host_off, _stream(stream)), "hs_set_request")


def hs_map_page(pool: int, req: int, page: int, block: int, stream=None) -> None:
    _check(load().hs_map_page(pool, req, page, block, _stream(stream)), "hs_map_page")


def hs_load_page(pool: int, req: int, page: int, block: int, stream=None) -> None:
    _check(load().hs_load_page(pool, req, page, block, _stream(stream)), "hs_load_page")


def hs_resolve(pool: int, layer_begin: int, num_layers: int, topk_idx, d_step, out_row_ids,
               miss_count=None, miss_log=None, stream=None) -> None:
    _check(load().hs_resolve(pool, layer_begin, num_layers, _addr(topk_idx), _addr(d_step),
                             _addr(out_row_ids), _addr(miss_count), _addr(miss_log),
                             _stream(stream)), "hs_resolve")


def hs_resolve_tokens(pool: int, layer_begin: int, num_layers: int, num_tokens: int, topk_idx,
                      d_step, out_row_ids, miss_count=None, miss_log=None, stream=None) -> None:
    """RESOLVE of the T verify tokens of a speculative-decoding step, as one
    list per unit (topk_idx / out_row_ids [num_layers][R][T][K])."""
    _check(load().hs_resolve_tokens(pool, layer_begin, num_layers, num_tokens, _addr(topk_idx),
                                    _addr(d_step), _addr(out_row_ids), _addr(miss_count),
                                    _addr(miss_log), _stream(stream)), "hs_resolve_tokens")


def hs_sparse_mla_decode_tokens(pool: int, layer: int, num_tokens: int, q, row_ids,
                                num_heads: int, v_dim: int, scale: float, out, lse=None,
                                stream=None) -> None:
    """Decode attention of the T verify tokens of each request (q [R][T][H][576],
    row_ids [R][T][K], out [R][T][H][512])."""
    _check(load().hs_sparse_mla_decode_tokens(pool, layer, num_tokens, _addr(q), _addr(row_ids),
                                              num_heads, v_dim, scale, _addr(out), _addr(lse),
                                              _stream(stream)), "hs_sparse_mla_decode_tokens")


def hs_gather(pool: int, layer: int, row_ids, n_rows: int, out_rows, stream=None) -> None:
    _check(load().hs_gather(pool, layer, _addr(row_ids), n_rows, _addr(out_rows),
                            _stream(stream)), "hs_gather")


def hs_sparse_mla_decode(pool: int, layer: int, q, row_ids, num_heads: int, v_dim: int,
                         scale: float, out, lse=None, stream=None) -> None:
    _check(load().hs_sparse_mla_decode(pool, layer, _addr(q), _addr(row_ids), num_heads, v_dim,
                                       scale, _addr(out), _addr(lse), _stream(stream)),
           "hs_sparse_mla_decode")


def hs_sparse_mla_decode_noalloc(kv_rows, num_rows: int, q, row_ids, num_requests: int,
                                 top_k: int, num_heads: int, v_dim: int, scale: float, out,
                                 lse=None, stream=None) -> None:
    """Decode attention without any device allocation (scratch is a fixed
    library array); for callers that cannot allocate when they decode."""
    _check(load().hs_sparse_mla_decode_noalloc(_addr(kv_rows), num_rows, _addr(q), _addr(row_ids),
                                               num_requests, top_k, num_heads, v_dim, scale,
                                               _addr(out), _addr(lse), _stream(stream)),
           "hs_sparse_mla_decode_noalloc")


def hs_noalloc_check_errors() -> int:
    """Synchronise, read and clear the allocation-free call's device error
    word on the current device; returns its bits."""
    code = ctypes.c_int32(0)
    st = load().hs_noalloc_check_errors(ctypes.byref(code))
    if st not in (HS_OK, HS_ERR_DEVICE):
        raise HsError(st, "hs_noalloc_check_errors")
    return code.value


def hs_decode_step(pool: int, layer_begin: int, num_layers: int, topk_idx, q, num_heads: int,
                   v_dim: int, scale: float, d_step, out_row_ids, out, lse=None, miss_count=None,
                   stream=None, copy_stream=None) -> None:
    """RESOLVE + attention for each layer of one decode step; the later layers'
    RESOLVE runs on `copy_stream` beside layer 0's RESOLVE or the attention."""
    _check(load().hs_decode_step(pool, layer_begin, num_layers, _addr(topk_idx), _addr(q),
                                 num_heads, v_dim, scale, _addr(d_step), _addr(out_row_ids),
                                 _addr(out), _addr(lse), _addr(miss_count), _stream(stream),
                                 _stream(copy_stream)), "hs_decode_step")


def hs_decode_step_tokens(pool: int, layer_begin: int, num_layers: int, num_tokens: int, topk_idx,
                          q, num_heads: int, v_dim: int, scale: float, d_step, out_row_ids, out,
                          lse=None, miss_count=None, stream=None, copy_stream=None) -> None:
    """hs_decode_step over num_tokens verify tokens per request."""
    _check(load().hs_decode_step_tokens(pool, layer_begin, num_layers, num_tokens,
                                        _addr(topk_idx), _addr(q), num_heads, v_dim, scale,
                                        _addr(d_step), _addr(out_row_ids), _addr(out), _addr(lse),
                                        _addr(miss_count), _stream(stream), _stream(copy_stream)),
           "hs_decode_step_tokens")


def hs_offload_prefix(pool: int, req: int, page: int, main_stream, side_stream, done_event) -> None:
    _check(load().hs_offload_prefix(pool, req, page, _stream(main_stream), _stream(side_stream),
                                    _event(done_event)), "hs_offload_prefix")


def hs_selftest_bounded_waits(timeout_ns: int, result, stream=None) -> None:
    """Run the bounded-wait self-test; `result` a device int32[2] tensor."""
    _check(load().hs_selftest_bounded_waits(int(timeout_ns), _addr(result), _stream(stream)),
           "hs_selftest_bounded_waits")


def hs_offload_pages(pool: int, reqs, pages, main_stream, side_stream, done_event) -> None:
    """One launch copying every (reqs[i], pages[i]) page; host sequences."""
    n = len(reqs)
    if len(pages) != n:
        raise HsError(HS_ERR_INVALID, "hs_offload_pages: reqs and pages differ in length")
    r = (ctypes.c_int32 * max(n, 1))(*[int(x) for x in reqs])
    g = (ctypes.c_int32 * max(n, 1))(*[int(x) for x in pages])
    _check(load().hs_offload_pages(pool, n, ctypes.addressof(r), ctypes.addressof(g),
                                   _stream(main_stream), _stream(side_stream), _event(done_event)),
           "hs_offload_pages")


def hs_commit_offload(pool: int, req: int, page: int, main_stream, done_event) -> None:
    _check(load().hs_commit_offload(pool, req, page, _stream(main_stream), _event(done_event)),
           "hs_commit_offload")


def hs_wait_offload(done_event, timeout_ns: int) -> int:
    """Bounded host-side wait for an offload's copy event: HS_OK once it has
    completed, HS_ERR_TIMEOUT if not within timeout_ns (other statuses raise)."""
    st = load().hs_wait_offload(_event(done_event), int(timeout_ns))
    if st not in (HS_OK, HS_ERR_TIMEOUT):
        raise HsError(st, "hs_wait_offload")
    return st


def hs_pool_touch_host(pool: int, stream=None) -> None:
    _check(load().hs_pool_touch_host(pool, _stream(stream)), "hs_pool_touch_host")


def hs_pool_host_numa_node(pool: int) -> int:
    """Host NUMA node the pool's pinned host pool was placed on (-1: not placed)."""
    node = ctypes.c_int32(-1)
    _check(load().hs_pool_host_numa_node(pool, ctypes.byref(node)), "hs_pool_host_numa_node")
    return node.value


def hs_step_advance(d_step, stream=None) -> None:
    _check(load().hs_step_advance(_addr(d_step), _stream(stream)), "hs_step_advance")


def hs_check_errors(pool: int) -> int:
    """Synchronise, read and clear the device error word; returns its bits."""
    code = ctypes.c_int32(0)
    st = load().hs_check_errors(pool, ctypes.byref(code))
    if st not in (HS_OK, HS_ERR_DEVICE):
        raise HsError(st, "hs_check_errors")
    return code.value


def hs_host_read(host_device_ptr: int, nbytes: int, dst, stream=None) -> None:
    _check(load().hs_host_read(host_device_ptr, nbytes, _addr(dst), _stream(stream)),
           "hs_host_read")


def hs_version() -> str:
    return load().hs_version().decode()


from .pool import Pool  # noqa: E402  (convenience wrapper over the calls above)
