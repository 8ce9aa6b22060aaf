"""Float64 CPU oracle for paged GQA decode attention and the KV append.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package.  It shares
no code with the CUDA library (``paged_kv_decode_16_gb300``) and never imports
it.  The arithmetic lives in ``pkv_oracle.c``; this module only marshals numpy
arrays into it.

Inputs are passed as raw 16-bit patterns (``numpy.uint16`` arrays) together
with a dtype name, ``"f16"`` (IEEE binary16) or ``"bf16"`` (bfloat16); the C
code decodes them from their bit fields into double.

Sources (page title, section): CacheIR "Compiler Example" and "Boundaries"
(paged_attention_decode; multi-batch page-table decode attention with GQA
mapping); TorchInferno "Runtime Scaffolds" (runtime.paged materialization,
runtime.paged_attention reference) and "Custom Kernels"
(paged_decode_attention, batched_paged_decode_attention).

Parity pins: every function here is checked in ``tests/test_oracle.py``
against hand-derived worked examples (``tests/golden/``), closed forms,
invariants, library routines (numpy / torch dtype conversion, torch
scaled_dot_product_attention in float64) and brute force; none is unpinned.
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import build as _build

DTYPES = {"f16": 0, "bf16": 1}
ERRORS = {0: "ok", 1: "invalid argument", 2: "page id outside the pool",
          3: "context length beyond the page-table row"}


class OracleError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {ERRORS.get(code, code)}")
        self.code = code


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        a = a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError(f"expected 16-bit patterns (uint16 or float16), got {a.dtype}")
    return a


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str):
    if rc != 0:
        raise OracleError(rc, what)


class Oracle:
    """One loaded build of pkv_oracle.c (the default build, or a test variant)."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i32 = ctypes.c_int
        lib.pkv_oracle_decode_array.argtypes = [P, ctypes.c_int64, i32, P]
        lib.pkv_oracle_paged_decode.argtypes = [P, P, P, i32, P, i32, P, i32, i32, i32, i32, i32,
                                                i32, ctypes.c_double, P]
        lib.pkv_oracle_paged_decode_rows.argtypes = [P, P, P, i32, P, i32, P, i32, i32, i32, i32,
                                                     i32, i32, ctypes.c_double, P, i32, P]
        lib.pkv_oracle_kv_append.argtypes = [P, P, P, P, P, i32, P, i32, i32, i32, i32, i32]
        lib.pkv_oracle_gather.argtypes = [P, P, i32, P, i32, i32, i32, i32, i32, i32, P]
        lib.pkv_oracle_set_threads.argtypes = [i32]
        lib.pkv_oracle_encode_array.argtypes = [P, ctypes.c_int64, i32, P]
        lib.pkv_oracle_paged_decode_multi.argtypes = [P, P, P, i32, P, i32, P, i32, i32, i32, i32,
                                                      i32, i32, i32, ctypes.c_double, P]
        lib.pkv_oracle_paged_decode_multi.restype = ctypes.c_int
        lib.pkv_oracle_rope.argtypes = [P, P, i32, i32, i32, ctypes.c_double, i32, P, P]
        lib.pkv_oracle_norm_rope.argtypes = [P, P, i32, i32, i32, P, ctypes.c_double,
                                             ctypes.c_double, i32, P, P]
        for name in ("pkv_oracle_encode_array", "pkv_oracle_rope", "pkv_oracle_norm_rope"):
            getattr(lib, name).restype = ctypes.c_int
        for name in ("pkv_oracle_decode_array", "pkv_oracle_paged_decode",
                     "pkv_oracle_paged_decode_rows", "pkv_oracle_kv_append",
                     "pkv_oracle_gather", "pkv_oracle_set_threads", "pkv_oracle_max_threads"):
            getattr(lib, name).restype = ctypes.c_int
        self.lib = lib
        self.path = path

    def set_threads(self, n: int) -> int:
        """Set the OpenMP thread count (n <= 0 keeps it); returns the count in use."""
        return self.lib.pkv_oracle_set_threads(int(n))

    def max_threads(self) -> int:
        return self.lib.pkv_oracle_max_threads()

    def decode_bits(self, bits, dtype: str) -> np.ndarray:
        """Decode 16-bit float patterns to float64 from their sign/exponent/fraction."""
        b = _u16(bits)
        out = np.empty(b.shape, dtype=np.float64)
        _check(self.lib.pkv_oracle_decode_array(_ptr(b), b.size, DTYPES[dtype], _ptr(out)),
               "decode")
        return out

    def paged_decode(self, q, k_pool, v_pool, page_table, context_lens, scale: float,
                     dtype: str) -> np.ndarray:
        """out[b, hq, :] = softmax(scale * q[b,hq] . K_b^T) V_b over the first
        context_lens[b] tokens of sequence b, K_b/V_b read through page_table[b].

        q [B, Hq, D]; k_pool, v_pool [NP, Hkv, P, D] (uint16 patterns);
        page_table int32 [B, MP]; context_lens int32 [B].  Returns float64 [B, Hq, D].
        """
        q, k_pool, v_pool = _u16(q), _u16(k_pool), _u16(v_pool)
        table, lens = _i32(page_table), _i32(context_lens)
        B, Hq, D = q.shape
        NP, Hkv, P, D2 = k_pool.shape
        if D2 != D or v_pool.shape != k_pool.shape or table.ndim != 2 or table.shape[0] != B:
            raise ValueError("shape mismatch")
        out = np.zeros((B, Hq, D), dtype=np.float64)
        rc = self.lib.pkv_oracle_paged_decode(_ptr(q), _ptr(k_pool), _ptr(v_pool), DTYPES[dtype],
                                              _ptr(table), table.shape[1], _ptr(lens), B, Hq, Hkv,
                                              D, P, NP, float(scale), _ptr(out))
        _check(rc, "paged_decode")
        return out

    def paged_decode_multi(self, q, k_pool, v_pool, page_table, context_lens, scale: float,
                           dtype: str) -> np.ndarray:
        """Several query tokens per sequence: q [B, Qn, Hq, D]; query j of sequence
        b stands at position L_b - Qn + j and attends causally to tokens
        0 .. L_b - Qn + j.  Returns float64 [B, Qn, Hq, D]."""
        q, k_pool, v_pool = _u16(q), _u16(k_pool), _u16(v_pool)
        table, lens = _i32(page_table), _i32(context_lens)
        B, Qn, Hq, D = q.shape
        NP, Hkv, P, D2 = k_pool.shape
        if D2 != D or v_pool.shape != k_pool.shape or table.ndim != 2 or table.shape[0] != B:
            raise ValueError("shape mismatch")
        out = np.zeros((B, Qn, Hq, D), dtype=np.float64)
        rc = self.lib.pkv_oracle_paged_decode_multi(_ptr(q), _ptr(k_pool), _ptr(v_pool),
                                                    DTYPES[dtype], _ptr(table), table.shape[1],
                                                    _ptr(lens), B, Qn, Hq, Hkv, D, P, NP,
                                                    float(scale), _ptr(out))
        _check(rc, "paged_decode_multi")
        return out

    def paged_decode_rows(self, q, k_pool, v_pool, page_table, context_lens, scale: float,
                          dtype: str, rows) -> np.ndarray:
        """Selected outputs only: rows is an int array [n, 2] of (b, hq); returns [n, D]."""
        q, k_pool, v_pool = _u16(q), _u16(k_pool), _u16(v_pool)
        table, lens = _i32(page_table), _i32(context_lens)
        rows = _i32(rows).reshape(-1, 2)
        B, Hq, D = q.shape
        NP, Hkv, P, _ = k_pool.shape
        out = np.zeros((rows.shape[0], D), dtype=np.float64)
        rc = self.lib.pkv_oracle_paged_decode_rows(_ptr(q), _ptr(k_pool), _ptr(v_pool),
                                                   DTYPES[dtype], _ptr(table), table.shape[1],
                                                   _ptr(lens), B, Hq, Hkv, D, P, NP, float(scale),
                                                   _ptr(rows), rows.shape[0], _ptr(out))
        _check(rc, "paged_decode_rows")
        return out

    def encode(self, values, dtype: str) -> np.ndarray:
        """Round float64 values to 16-bit patterns (to nearest, ties to even)."""
        x = np.ascontiguousarray(values, dtype=np.float64)
        out = np.empty(x.shape, dtype=np.uint16)
        _check(self.lib.pkv_oracle_encode_array(_ptr(x), x.size, DTYPES[dtype], _ptr(out)),
               "encode")
        return out

    def rope(self, x, positions, theta: float, dtype: str, with_f64: bool = False):
        """Rotary embedding of rows x [B, H, D] (16-bit patterns) at positions[b].

        Returns the rotated rows as 16-bit patterns, plus the float64 values
        before rounding when with_f64."""
        xb = _u16(x)
        pos = _i32(positions)
        B, H, D = xb.shape
        out = np.empty(xb.shape, dtype=np.uint16)
        f64 = np.empty(xb.shape, dtype=np.float64) if with_f64 else None
        _check(self.lib.pkv_oracle_rope(_ptr(xb), _ptr(pos), B, H, D, float(theta), DTYPES[dtype],
                                        _ptr(out), _ptr(f64) if with_f64 else None), "rope")
        return (out, f64) if with_f64 else out

    def norm_rope(self, x, positions, weight, eps: float, theta: float, dtype: str,
                  with_f64: bool = False):
        """Per-head RMS norm (weight [D], 16-bit patterns) then the rotary
        embedding of rows x [B, H, D] at positions[b]; one rounding at the end.
        Returns the rows as 16-bit patterns, plus the float64 values when
        with_f64."""
        xb = _u16(x)
        pos = _i32(positions)
        wb = _u16(weight)
        B, H, D = xb.shape
        if wb.shape != (D,):
            raise ValueError("weight must hold head_dim values")
        out = np.empty(xb.shape, dtype=np.uint16)
        f64 = np.empty(xb.shape, dtype=np.float64) if with_f64 else None
        _check(self.lib.pkv_oracle_norm_rope(_ptr(xb), _ptr(pos), B, H, D, _ptr(wb), float(eps),
                                             float(theta), DTYPES[dtype], _ptr(out),
                                             _ptr(f64) if with_f64 else None), "norm_rope")
        return (out, f64) if with_f64 else out

    def kv_append(self, k_pool, v_pool, k_new, v_new, page_table, positions):
        """Return copies of (k_pool, v_pool) with the new rows written in.

        k_new, v_new [B, Hkv, D]; positions int32 [B] (negative: skip)."""
        kp, vp = _u16(k_pool).copy(), _u16(v_pool).copy()
        kn, vn = _u16(k_new), _u16(v_new)
        table, pos = _i32(page_table), _i32(positions)
        NP, Hkv, P, D = kp.shape
        B = pos.shape[0]
        rc = self.lib.pkv_oracle_kv_append(_ptr(kp), _ptr(vp), _ptr(kn), _ptr(vn), _ptr(table),
                                           table.shape[1], _ptr(pos), B, Hkv, D, P, NP)
        _check(rc, "kv_append")
        return kp, vp

    def gather(self, pool, page_table, context_lens, max_len: int | None = None,
               fill: int = 0) -> np.ndarray:
        """Dense [B, Hkv, max_len, D] uint16 copy of each sequence's cached rows."""
        pool, table, lens = _u16(pool), _i32(page_table), _i32(context_lens)
        NP, Hkv, P, D = pool.shape
        B = lens.shape[0]
        if max_len is None:
            max_len = int(lens.max()) if B else 0
        dense = np.full((B, Hkv, max_len, D), fill, dtype=np.uint16)
        rc = self.lib.pkv_oracle_gather(_ptr(pool), _ptr(table), table.shape[1], _ptr(lens), B,
                                        Hkv, D, P, NP, max_len, _ptr(dense))
        _check(rc, "gather")
        return dense


_default: Oracle | None = None


def get() -> Oracle:
    """The oracle built from oracle/pkv_oracle.c (compiled on first use)."""
    global _default
    if _default is None:
        _default = Oracle(_build.build())
    return _default


def set_threads(n: int) -> int:
    return get().set_threads(n)


def max_threads() -> int:
    return get().max_threads()


def decode_bits(bits, dtype: str) -> np.ndarray:
    return get().decode_bits(bits, dtype)


def paged_decode(*a, **k) -> np.ndarray:
    return get().paged_decode(*a, **k)


def paged_decode_rows(*a, **k) -> np.ndarray:
    return get().paged_decode_rows(*a, **k)


def kv_append(*a, **k):
    return get().kv_append(*a, **k)


def paged_decode_multi(*a, **k) -> np.ndarray:
    return get().paged_decode_multi(*a, **k)


def encode(*a, **k) -> np.ndarray:
    return get().encode(*a, **k)


def rope(*a, **k):
    return get().rope(*a, **k)


def norm_rope(*a, **k):
    return get().norm_rope(*a, **k)


def gather(*a, **k) -> np.ndarray:
    return get().gather(*a, **k)
