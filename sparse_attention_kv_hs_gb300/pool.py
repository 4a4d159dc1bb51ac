"""Convenience wrapper: one libhs pool with torch / numpy views of its buffers.

Views only alias the library-owned memory (no copies); the library keeps
ownership until ``close()``.
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import (hs_pool_create, hs_pool_destroy, hs_pool_desc, hs_pool_get_views)


class _CudaArray:
    """Minimal __cuda_array_interface__ holder so torch can alias device memory."""

    def __init__(self, ptr: int, shape, typestr: str):
        self.__cuda_array_interface__ = {
            "shape": tuple(int(s) for s in shape), "typestr": typestr,
            "data": (int(ptr), False), "version": 3, "strides": None}


def device_tensor(ptr: int, shape, typestr: str = "<i4"):
    import torch
    return torch.as_tensor(_CudaArray(ptr, shape, typestr), device="cuda")


class Pool:
    """A libhs pool (R requests x L sparse layers, top-K, B hot slots/unit)."""

    def __init__(self, num_requests: int, num_layers: int, top_k: int, hot_slots: int,
                 page_tokens: int, row_elems: int, max_pages: int, host_tokens: int,
                 resident_blocks: int, kv_format: int = 0):
        self.R, self.L, self.K, self.B, self.P = (num_requests, num_layers, top_k, hot_slots,
                                                  page_tokens)
        self.row_elems, self.max_pages = row_elems, max_pages
        self.host_tokens, self.resident_blocks = host_tokens, resident_blocks
        self.kv_format = kv_format
        # a row's width in 2-byte units: row_elems bf16 values, or 656 FP8-row bytes
        self.row_units = 656 // 2 if kv_format == 1 else row_elems
        desc = hs_pool_desc(num_requests, num_layers, top_k, hot_slots, page_tokens, row_elems,
                            max_pages, kv_format, host_tokens, resident_blocks)
        self.handle = hs_pool_create(desc)
        v = hs_pool_get_views(self.handle)
        self.raw = v
        self.blocks_per_layer = int(v.blocks_per_layer)
        self.hot_blocks = num_requests * (hot_slots // page_tokens)
        rows = self.blocks_per_layer * page_tokens
        # device views
        self.kv_pool = device_tensor(v.kv_pool, (num_layers, rows, self.row_units), "<i2")
        self.page_table = device_tensor(v.page_table, (num_requests, max_pages))
        self.ctx_len = device_tensor(v.ctx_len, (num_requests,))
        self.host_off = device_tensor(v.host_off, (num_requests,), "<i8")
        self.hot_block = device_tensor(v.hot_block, (num_requests, hot_slots // page_tokens))
        self.slot_pos = device_tensor(v.slot_pos, (num_layers, num_requests, hot_slots))
        self.slot_stamp = device_tensor(v.slot_stamp, (num_layers, num_requests, hot_slots))
        self.lru_order = device_tensor(v.lru_order, (num_layers, num_requests, hot_slots))
        self.step = device_tensor(v.step, (1,))
        self.error_word = device_tensor(v.error_word, (1,))
        # host view of the pinned pool (raw row bits in 2-byte units)
        n = num_layers * host_tokens * self.row_units
        buf = (ctypes.c_uint16 * n).from_address(v.host_pool)
        self.host_pool = np.ctypeslib.as_array(buf).reshape(num_layers, host_tokens,
                                                             self.row_units)
        self.host_pool_addr = int(v.host_pool)

    def hot_row(self, req: int, slot: int) -> int:
        """Pool row id of hot slot `slot` of request `req` (blocks leased at create)."""
        return (req * (self.B // self.P) + slot // self.P) * self.P + slot % self.P

    def close(self):
        if getattr(self, "handle", None):
            # drop aliases before the memory goes away
            for name in ("kv_pool", "page_table", "ctx_len", "host_off", "hot_block", "slot_pos",
                         "slot_stamp", "lru_order", "step", "error_word", "host_pool"):
                setattr(self, name, None)
            hs_pool_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
