"""CPU ORACLE for the HiSparse decode path -- TEST INFRASTRUCTURE ONLY.

Plain, slow, obviously-correct restatements of what the decode path computes,
used to check the CUDA library.  Only tests/, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of bench.py may import this package.  It shares no code
with the CUDA library (``sparse_attention_kv_hs_gb300``) and never imports it.

* ``ResolveOracle`` -- the page table + per-(request, layer) LRU hot buffer +
  miss copies of RESOLVE, one unit and one step at a time (C, resolve_oracle.c).
  Follows page "59188saintaubert.com ... HiSparse" section 02 and page
  "GLM 5.3 Optimizations, Part 1: Hybrid HiSparse Offloading in vLLM",
  section "How it works"; the readings for points the pages leave open are
  listed in resolve_oracle.c.
* ``policy_misses`` -- misses of one hot buffer under LRU, FIFO, random or
  Belady replacement with RESOLVE's step structure (C, policy_sim.c), for the
  replacement-policy comparison of page "59188saintaubert.com ... HiSparse",
  section 04.
* ``fp8_rows_to_f64`` -- the rows an FP8 KV row (656 bytes: E4M3 latent codes,
  per-128 fp32 scales, bf16 rope) stands for, decoded from the E4M3
  definition.
* ``sparse_mla_decode`` -- attention of one decode query over exactly the K
  selected rows, in fp64 (softmax(scale * q k^T) v with v = the first 512
  columns of each 576-wide latent row).  The pages state the method is exact:
  only placement changes, so the output equals attention over the same
  positions read from full KV (page "59188saintaubert.com ... HiSparse",
  end of section 02).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "resolve_oracle.c")
_POLICY_SRC = os.path.join(_HERE, "policy_sim.c")
_HDR = os.path.join(_HERE, "resolve_oracle.h")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

ERR_RANGE, ERR_DUPLICATE, ERR_CAPACITY, ERR_BLOCK = 1, 2, 4, 8


def build(force: bool = False) -> str:
    """Compile the C part of the oracle in place (plain C, gcc)."""
    stale = force or not os.path.exists(_LIB) or max(
        os.path.getmtime(_SRC), os.path.getmtime(_HDR),
        os.path.getmtime(_POLICY_SRC)) > os.path.getmtime(_LIB)
    if stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared",
                               "-ffp-contract=off", "-Wall", "-o", tmp, _SRC, _POLICY_SRC])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            i32, i64, p = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p
            lib.or_create.restype = p
            lib.or_create.argtypes = [i32, i32, i32, i32, i32, i32, i64, p]
            lib.or_destroy.restype = None
            lib.or_destroy.argtypes = [p]
            lib.or_set_ctx.restype = i32
            lib.or_set_ctx.argtypes = [p, i32, i32]
            for name in ("or_set_page", "or_set_hot_block"):
                f = getattr(lib, name)
                f.restype = i32
                f.argtypes = [p, i32, i32, i32]
            lib.or_resolve.restype = i32
            lib.or_resolve.argtypes = [p, i32, i32, p, i32, p, p, p]
            lib.or_resolve_tokens.restype = i32
            lib.or_resolve_tokens.argtypes = [p, i32, i32, i32, p, i32, p, p, p]
            lib.or_get_unit.restype = i32
            lib.or_get_unit.argtypes = [p, i32, i32, p, p]
            lib.or_row_content.restype = i32
            lib.or_row_content.argtypes = [p, i32, i32, i32, p]
            lib.ps_simulate.restype = i32
            lib.ps_simulate.argtypes = [i32, i32, i32, i32, i32, p, ctypes.c_uint64, p]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags.c_contiguous
    return a.ctypes.data


class ResolveOracle:
    """Sequential simulation of RESOLVE state for R requests x L layers."""

    def __init__(self, num_requests: int, num_layers: int, top_k: int,
                 hot_slots: int, page_tokens: int, ctx_cap, blocks_per_layer: int):
        self.R, self.L, self.K, self.B, self.P = (num_requests, num_layers, top_k,
                                                  hot_slots, page_tokens)
        cap = np.ascontiguousarray(np.broadcast_to(
            np.asarray(ctx_cap, dtype=np.int32), (num_requests,)))
        self.max_pages = int((int(cap.max()) + page_tokens - 1) // page_tokens)
        self._lib = _load()
        self._h = self._lib.or_create(num_requests, num_layers, top_k, hot_slots,
                                      page_tokens, self.max_pages,
                                      int(blocks_per_layer), _ptr(cap))
        if not self._h:
            raise MemoryError("oracle state allocation failed or bad shape")

    def close(self):
        if self._h:
            self._lib.or_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_ctx(self, req: int, ctx: int):
        if self._lib.or_set_ctx(self._h, req, ctx) != 0:
            raise ValueError("bad ctx")

    def set_page(self, req: int, page: int, block: int):
        if self._lib.or_set_page(self._h, req, page, block) != 0:
            raise ValueError("bad page")

    def set_hot_block(self, req: int, index: int, block: int):
        if self._lib.or_set_hot_block(self._h, req, index, block) != 0:
            raise ValueError("bad hot block")

    def resolve(self, layer: int, req: int, topk, step: int):
        """One step of one unit -> (row_ids[K], miss_log[n][3], err_bits)."""
        topk = np.ascontiguousarray(topk, dtype=np.int32)
        assert topk.shape == (self.K,)
        out = np.empty(self.K, dtype=np.int32)
        log = np.empty((self.K, 3), dtype=np.int32)
        n = ctypes.c_int32(0)
        err = self._lib.or_resolve(self._h, layer, req, _ptr(topk), step, _ptr(out),
                                   _ptr(log), ctypes.addressof(n))
        if err < 0:
            raise ValueError("bad unit")
        return out, log[: n.value].copy(), err

    def resolve_tokens(self, layer: int, req: int, topk, step: int):
        """One speculative-decoding step of one unit: topk[T][K] (T verify
        tokens) -> (row_ids[T][K], miss_log[n][3] with j indexing the
        flattened [T*K] list, err_bits)."""
        topk = np.ascontiguousarray(topk, dtype=np.int32)
        T = topk.shape[0]
        assert topk.shape == (T, self.K)
        out = np.empty((T, self.K), dtype=np.int32)
        log = np.empty((T * self.K, 3), dtype=np.int32)
        n = ctypes.c_int32(0)
        err = self._lib.or_resolve_tokens(self._h, layer, req, T, _ptr(topk), step, _ptr(out),
                                          _ptr(log), ctypes.addressof(n))
        if err < 0:
            raise ValueError("bad unit")
        return out, log[: n.value].copy(), err

    def unit_state(self, layer: int, req: int):
        """(slot_pos[B], slot_stamp[B]) of one unit."""
        pos = np.empty(self.B, dtype=np.int32)
        stamp = np.empty(self.B, dtype=np.int32)
        self._lib.or_get_unit(self._h, layer, req, _ptr(pos), _ptr(stamp))
        return pos, stamp

    def row_content(self, layer: int, req: int, row: int) -> int:
        """Logical position held by a pool row for this request, or -1."""
        p = ctypes.c_int32(-1)
        self._lib.or_row_content(self._h, layer, req, int(row), ctypes.addressof(p))
        return p.value


POLICIES = {"lru": 0, "fifo": 1, "random": 2, "belady": 3}


def policy_misses(policy: str, trace, hot_slots: int, ctx: int, seed: int = 0) -> np.ndarray:
    """Misses per step of one hot buffer of `hot_slots` slots over `trace`
    ([steps][K] positions, -1 = skipped) under the named replacement policy
    (page "59188saintaubert.com ... HiSparse", section 04 compares these)."""
    tr = np.ascontiguousarray(trace, dtype=np.int32)
    steps, K = tr.shape
    out = np.zeros(steps, dtype=np.int32)
    rc = _load().ps_simulate(POLICIES[policy], K, hot_slots, steps, ctx, _ptr(tr), seed,
                             _ptr(out))
    if rc != 0:
        raise ValueError("ps_simulate: bad arguments")
    return out


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact bf16 -> float64 decoding (bf16 bits are the top half of an fp32)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def e4m3_value(code: int) -> float:
    """Value of an OCP FP8 E4M3 code: 1 sign bit, 4 exponent bits (bias 7), 3
    mantissa bits; exponent field 0 is subnormal (m/8 * 2^-6); S.1111.111 is
    NaN and there are no infinities (largest finite 448)."""
    sign = -1.0 if code & 0x80 else 1.0
    e, m = (code >> 3) & 0xF, code & 0x7
    if e == 15 and m == 7:
        return float("nan")
    if e == 0:
        return sign * (m / 8.0) * 2.0 ** -6
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


E4M3_TABLE = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)


def fp8_rows_to_f64(raw: np.ndarray) -> np.ndarray:
    """FP8 KV rows ([n, 656] bytes: 512 E4M3 latent codes, 4 fp32 group scales,
    64 bf16 rope values) -> the 576-wide rows they stand for, exactly, in fp64:
    latent value i = E4M3(code i) * scale[i // 128]."""
    raw = np.ascontiguousarray(raw, dtype=np.uint8).reshape(-1, 656)
    lat = E4M3_TABLE[raw[:, :512]]
    scales = raw[:, 512:528].copy().view(np.float32).astype(np.float64)   # [n, 4]
    lat = lat * np.repeat(scales, 128, axis=1)
    rope = bf16_bits_to_f64(raw[:, 528:656].copy().view(np.uint16))
    return np.concatenate([lat, rope], axis=1)


def sparse_mla_decode(q: np.ndarray, rows: np.ndarray, valid: np.ndarray | None,
                      scale: float, v_dim: int = 512):
    """Attention of one decode query over exactly the given rows, in fp64.

    q:     [H, D] query (absorbed MLA: D = 576), float or raw bf16 bits (uint16)
    rows:  [K, D] the selected latent rows, float or raw bf16 bits
    valid: [K] bool (padding rows excluded), or None for all valid
    Returns (out [H, v_dim] float64, lse [H] float64, natural log).

        s[h, j] = scale * sum_d q[h, d] * rows[j, d]
        out[h]  = sum_j exp(s[h, j] - m[h]) rows[j, :v_dim] / sum_j exp(s[h, j] - m[h])
        lse[h]  = m[h] + log(sum_j exp(s[h, j] - m[h])),  m[h] = max_j s[h, j]
    With no valid row the output is zero and lse is -inf.
    """
    qf = bf16_bits_to_f64(q) if q.dtype == np.uint16 else np.asarray(q, dtype=np.float64)
    kf = bf16_bits_to_f64(rows) if rows.dtype == np.uint16 else np.asarray(rows, dtype=np.float64)
    if valid is not None:
        kf = kf[np.asarray(valid, dtype=bool)]
    H = qf.shape[0]
    if kf.shape[0] == 0:
        return np.zeros((H, v_dim)), np.full(H, -np.inf)
    s = scale * (qf @ kf.T)                    # [H, K]
    m = s.max(axis=1, keepdims=True)
    p = np.exp(s - m)
    denom = p.sum(axis=1, keepdims=True)
    out = (p @ kf[:, :v_dim]) / denom
    lse = (m + np.log(denom))[:, 0]
    return out, lse
