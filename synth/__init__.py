"""Seeded synthetic inputs for the HiSparse decode path (ctypes wrapper).

Input generation only: KV rows, decode queries and top-K selection traces, as
pure functions of a seed and coordinates.  Both the CUDA path's tests/bench and
the CPU oracle draw their inputs from here; nothing in this package computes
any step of the method itself.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_HDR = os.path.join(_HERE, "synth.h")
_LIB = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None

ROW_ELEMS = 576  # bf16 values per KV row (512 latent + 64 rope)


def build(force: bool = False) -> str:
    """Compile libsynth.so in place (gcc, plain C, no target-specific flags)."""
    stale = force or not os.path.exists(_LIB) or max(
        os.path.getmtime(_SRC), os.path.getmtime(_HDR)) > os.path.getmtime(_LIB)
    if stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call([
            "gcc", "-O2", "-std=gnu11", "-fPIC", "-shared", "-pthread",
            "-ffp-contract=off", "-Wall", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            u64, i32, i64 = ctypes.c_uint64, ctypes.c_int32, ctypes.c_int64
            p = ctypes.c_void_p
            lib.sy_mix.restype = u64
            lib.sy_mix.argtypes = [u64]
            lib.sy_key.restype = u64
            lib.sy_key.argtypes = [u64, u64, u64, u64, u64]
            lib.sy_draw.restype = u64
            lib.sy_draw.argtypes = [u64, u64]
            lib.sy_normal_bf16.restype = ctypes.c_uint16
            lib.sy_normal_bf16.argtypes = [u64]
            lib.sy_fill_rows.restype = None
            lib.sy_fill_rows.argtypes = [u64, i32, i32, i64, i64, i32, p, i32]
            lib.sy_fill_rows_at.restype = None
            lib.sy_fill_rows_at.argtypes = [u64, i32, i32, p, i64, i32, p]
            lib.sy_fill_rows_fp8.restype = None
            lib.sy_fill_rows_fp8.argtypes = [u64, i32, i32, i64, i64, p, i32]
            lib.sy_fill_rows_fp8_at.restype = None
            lib.sy_fill_rows_fp8_at.argtypes = [u64, i32, i32, p, i64, p]
            lib.sy_e4m3_encode.restype = ctypes.c_uint8
            lib.sy_e4m3_encode.argtypes = [ctypes.c_float]
            lib.sy_fill_q.restype = None
            lib.sy_fill_q.argtypes = [u64, i32, i32, i32, i32, i32, p]
            lib.sy_trace_request.restype = i32
            lib.sy_trace_request.argtypes = [p, i32, p, p]
            lib.sy_permute.restype = i64
            lib.sy_permute.argtypes = [u64, i32, i64, i64]
            _lib = lib
    return _lib


class TraceParams(ctypes.Structure):
    _fields_ = [("seed", ctypes.c_uint64), ("k", ctypes.c_int32),
                ("layers", ctypes.c_int32), ("steps", ctypes.c_int32),
                ("reuse", ctypes.c_double), ("zipf_frac", ctypes.c_double),
                ("zipf_s", ctypes.c_double), ("layer_share", ctypes.c_double)]


def mix(x: int) -> int:
    return _load().sy_mix(x & (2**64 - 1))


def key(seed: int, tag: int, a: int = 0, b: int = 0, c: int = 0) -> int:
    m = 2**64 - 1
    return _load().sy_key(seed & m, tag & m, a & m, b & m, c & m)


def draw(k: int, i: int) -> int:
    return _load().sy_draw(k & (2**64 - 1), i & (2**64 - 1))


def uniform(k: int, i: int) -> float:
    """A double in [0, 1) from the i-th draw of stream k."""
    return (draw(k, i) >> 11) * 2.0**-53


def normal_bf16(d: int) -> int:
    return _load().sy_normal_bf16(d & (2**64 - 1))


def rows(seed: int, req: int, layer: int, pos0: int, n: int,
         width: int = ROW_ELEMS, threads: int = 1, out: np.ndarray | None = None) -> np.ndarray:
    """KV rows for positions pos0..pos0+n-1 as raw bf16 bits, shape [n, width]."""
    if out is None:
        out = np.empty((n, width), dtype=np.uint16)
    assert out.dtype == np.uint16 and out.flags.c_contiguous and out.size >= n * width
    _load().sy_fill_rows(seed, req, layer, pos0, n, width, out.ctypes.data, threads)
    return out


def rows_into(seed: int, req: int, layer: int, pos0: int, n: int, width: int,
              addr: int, threads: int) -> None:
    """Write rows straight to a raw host address (e.g. a pinned pool)."""
    _load().sy_fill_rows(seed, req, layer, pos0, n, width, ctypes.c_void_p(addr), threads)


def rows_at(seed: int, req: int, layer: int, pos, width: int = ROW_ELEMS) -> np.ndarray:
    """KV rows for an explicit position list (negative position -> zero row)."""
    pos = np.ascontiguousarray(pos, dtype=np.int32).reshape(-1)
    out = np.empty((pos.size, width), dtype=np.uint16)
    _load().sy_fill_rows_at(seed, req, layer, pos.ctypes.data, pos.size, width, out.ctypes.data)
    return out


FP8_ROW_BYTES = 656


def rows_fp8(seed: int, req: int, layer: int, pos0: int, n: int, threads: int = 1,
             out: np.ndarray | None = None) -> np.ndarray:
    """The KV rows of rows(...) stored as 656-byte FP8 rows (synth.h), [n, 656] uint8."""
    if out is None:
        out = np.empty((n, FP8_ROW_BYTES), dtype=np.uint8)
    assert out.dtype == np.uint8 and out.flags.c_contiguous and out.size >= n * FP8_ROW_BYTES
    _load().sy_fill_rows_fp8(seed, req, layer, pos0, n, out.ctypes.data, threads)
    return out


def rows_fp8_into(seed: int, req: int, layer: int, pos0: int, n: int, addr: int,
                  threads: int) -> None:
    """FP8 rows straight to a raw host address (e.g. a pinned pool)."""
    _load().sy_fill_rows_fp8(seed, req, layer, pos0, n, ctypes.c_void_p(addr), threads)


def rows_fp8_at(seed: int, req: int, layer: int, pos) -> np.ndarray:
    """FP8 rows for an explicit position list (negative position -> zero row)."""
    pos = np.ascontiguousarray(pos, dtype=np.int32).reshape(-1)
    out = np.empty((pos.size, FP8_ROW_BYTES), dtype=np.uint8)
    _load().sy_fill_rows_fp8_at(seed, req, layer, pos.ctypes.data, pos.size, out.ctypes.data)
    return out


def e4m3_encode(v: float) -> int:
    """The generator's fp32 -> E4M3 rounding (for its own tests)."""
    return int(_load().sy_e4m3_encode(float(v)))


def q(seed: int, req: int, layer: int, step: int, heads: int,
      width: int = ROW_ELEMS) -> np.ndarray:
    """Decode query of one (request, layer, step) as raw bf16 bits [heads, width]."""
    out = np.empty((heads, width), dtype=np.uint16)
    _load().sy_fill_q(seed, req, layer, step, heads, width, out.ctypes.data)
    return out


def trace(seed: int, req: int, k: int, layers: int, steps: int, ctx_per_step,
          reuse: float, zipf_frac: float, zipf_s: float = 1.1,
          layer_share: float = 0.0) -> np.ndarray:
    """Top-K selection trace of one request: int32 [steps, layers, k]."""
    ctx = np.ascontiguousarray(np.broadcast_to(
        np.asarray(ctx_per_step, dtype=np.int32), (steps,)))
    prm = TraceParams(seed, k, layers, steps, reuse, zipf_frac, zipf_s, layer_share)
    out = np.empty((steps, layers, k), dtype=np.int32)
    rc = _load().sy_trace_request(ctypes.byref(prm), req, ctx.ctypes.data, out.ctypes.data)
    if rc != 0:
        raise ValueError(f"trace generation failed ({rc}): top-K larger than the context?")
    return out


def permute(seed: int, req: int, rank: int, n: int) -> int:
    return _load().sy_permute(seed, req, rank, n)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Decode raw bf16 bits to float32 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
