"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
and the oracle on host copies of the same inputs, and compare.

Tolerance (decode outputs, fp16/bf16 inputs, fp32 accumulation, output
rounded to the input dtype):
  * every element: |gpu - ref| <= ATOL + RTOL * |ref|      (ATOL 2e-3, RTOL 1e-2)
  * every element, when the output is a 16-bit tensor: |gpu - ref| <= ATOL +
    one ulp of the output format at |ref| (the fp32 result within ATOL, then
    one rounding to the format; for fp16 this is much tighter than RTOL)
  * strict form, also required on the five named workloads (their outputs are
    small, |out| < 1, so output rounding stays below ATOL):
      max |gpu - ref| <= ATOL  and  max |gpu - ref| / max(|ref|, ATOL/RTOL) <= RTOL
    The strict form cannot hold for bf16 outputs of magnitude >= 1 (half an
    ulp of bf16 in [1, 2) is 2^-8 = 0.0039 > ATOL), which short contexts
    produce; those cases use the per-element forms only.
Append, gather and page-table indexing are compared bit for bit.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import paged_kv_decode_16_gb300 as pkv
from paged_kv_decode_16_gb300 import workloads as wl

ATOL = 2e-3
RTOL = 1e-2


def to_dev(w: wl.Workload, dev="cuda"):
    table = torch.from_numpy(np.ascontiguousarray(w.page_table)).to(dev)
    lens = torch.from_numpy(np.ascontiguousarray(w.context_lens)).to(dev)
    pos = torch.from_numpy(np.ascontiguousarray(w.positions)).to(dev)
    return table, lens, pos


VARIANTS = (pkv.VARIANT_CUDA_CORES, pkv.VARIANT_TENSOR_CORES)
VARIANT_IDS = ("cuda_cores", "tensor_cores")


def run_gpu(w: wl.Workload, num_workers: int = 0, append: bool | None = None,
            variant: int = pkv.VARIANT_AUTO):
    """kv_append (when the workload has one) then paged_decode_attention.
    Returns (out tensor, workspace, host status)."""
    dev = w.q.device
    table, lens, pos = to_dev(w, dev)
    if append if append is not None else w.append:
        pool = pkv.kv_pool_create(w.num_pages, w.page_size, w.n_kv_heads, w.head_dim, w.dtype,
                                  w.k_pool, w.v_pool)
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        pkv.kv_append(pool, w.k_new, w.v_new, table, pos, dev_status=st)
        assert int(st.item()) == 0
    out = torch.empty_like(w.q)
    ws = pkv.alloc_workspace(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, num_workers,
                             device=dev, variant=variant)
    pkv.paged_decode_attention(w.q, w.k_pool, w.v_pool, table, lens, w.scale, out, ws,
                               num_workers=num_workers, variant=variant)
    torch.cuda.synchronize()
    return out, ws, pkv.pkv_read_device_status(ws)


def oracle_inputs(w: wl.Workload, pools_before=None, append: bool | None = None):
    """Host bit patterns for the oracle; applies the append on the host copy
    of the pre-append pools when the workload has one."""
    kp, vp = pools_before if pools_before is not None else (wl.to_bits(w.k_pool),
                                                            wl.to_bits(w.v_pool))
    if append if append is not None else w.append:
        kp, vp = oracle.kv_append(kp, vp, wl.to_bits(w.k_new), wl.to_bits(w.v_new),
                                  w.page_table, w.positions)
    return wl.to_bits(w.q), kp, vp


def oracle_full(w: wl.Workload, pools_before=None, append=None) -> np.ndarray:
    q, kp, vp = oracle_inputs(w, pools_before, append)
    return oracle.paged_decode(q, kp, vp, w.page_table, w.context_lens, w.scale, w.dtype_name)


def oracle_rows(w: wl.Workload, rows, pools_before=None, append=None) -> np.ndarray:
    q, kp, vp = oracle_inputs(w, pools_before, append)
    return oracle.paged_decode_rows(q, kp, vp, w.page_table, w.context_lens, w.scale,
                                    w.dtype_name, rows)


def errors(got: np.ndarray, ref: np.ndarray):
    err = np.abs(got - ref)
    rel = err / np.maximum(np.abs(ref), ATOL / RTOL)
    return float(err.max(initial=0.0)), float(rel.max(initial=0.0))


# significant bits and smallest normal exponent of the 16-bit output formats
_FORMATS = {torch.bfloat16: (8, -126), torch.float16: (11, -14)}


def ulp(ref: np.ndarray, dtype) -> np.ndarray:
    """Spacing of the 16-bit format `dtype` at |ref| (subnormal spacing below
    the smallest normal)."""
    p, emin = _FORMATS[dtype]
    a = np.abs(ref)
    _, k = np.frexp(a)  # |ref| = m 2^k, m in [0.5, 1): exponent k - 1
    e = np.where(a > 0, np.maximum(k - 1, emin), emin)
    return np.ldexp(1.0, e - (p - 1))


def assert_close(got, ref: np.ndarray, strict: bool = False, what: str = ""):
    fmt = None
    if isinstance(got, torch.Tensor):
        fmt = got.dtype if got.dtype in _FORMATS else None
        got = got.float().cpu().numpy().astype(np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bad = err > ATOL + RTOL * np.abs(ref)
    if bad.any():
        i = np.unravel_index(np.argmax(err - (ATOL + RTOL * np.abs(ref))), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} elements out of tolerance; worst at {i}: "
                             f"gpu {got[i]!r} ref {ref[i]!r}")
    if fmt is not None:
        lim = ATOL + ulp(ref, fmt)
        bad = err > lim
        if bad.any():
            i = np.unravel_index(np.argmax(err - lim), err.shape)
            raise AssertionError(f"{what}: {int(bad.sum())} elements beyond ATOL + 1 ulp; worst "
                                 f"at {i}: gpu {got[i]!r} ref {ref[i]!r}")
    if strict:
        mx, rel = errors(got, ref)
        assert mx <= ATOL, f"{what}: max abs err {mx:.3g} > {ATOL}"
        assert rel <= RTOL, f"{what}: max rel err {rel:.3g} > {RTOL}"
