"""GB300-native paged GQA decode attention: thin Python binding of libpagedkv.so.

Every function here has the name of the C-ABI entry point it calls
(``include/pagedkv.h``) and only marshals arguments: torch tensors are
checked for device, dtype and contiguity and passed as raw device pointers;
the current torch CUDA stream is passed as the stream.  All computation runs
in the library's CUDA kernels.  There is no fallback: if the library was not
built, or a call fails, an exception is raised.

PyTorch is used only to own device memory and streams.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

from . import build as _build

__all__ = [
    "PagedKVError", "load_library", "library_path", "pkv_status_string", "pkv_version",
    "Pool", "kv_pool_create", "PrefixCache", "kv_append", "kv_append_rope", "kv_gather",
    "paged_decode_workspace_size", "paged_decode_step_rope", "paged_decode_attention_prefix",
    "paged_decode_prefix_workspace_size", "alloc_prefix_workspace", "DEV_BAD_PREFIX",
    "paged_decode_attention_multi", "paged_decode_multi_workspace_size", "alloc_multi_workspace",
    "check_bounded_wait",
    "paged_decode_plan", "paged_decode_run", "paged_decode_combine", "paged_decode_attention",
    "paged_decode_step", "paged_decode_attention_no_alloc", "NO_ALLOC_SCRATCH_BYTES",
    "paged_decode_step_host", "paged_decode_step_host_workspace_size", "alloc_step_host_workspace",
    "pkv_read_device_status", "pkv_read_no_alloc_status", "alloc_workspace", "DEV_BAD_PAGE", "DEV_BAD_LEN", "DEV_TIMEOUT",
    "VARIANT_AUTO", "VARIANT_CUDA_CORES", "VARIANT_TENSOR_CORES", "VARIANT_TCGEN05",
]

PKV_OK = 0
STATUS_NAMES = {0: "PKV_OK", 1: "PKV_ERR_INVALID_ARG", 2: "PKV_ERR_UNSUPPORTED",
                3: "PKV_ERR_ALIAS", 4: "PKV_ERR_OUT_OF_PAGES", 5: "PKV_ERR_WORKSPACE",
                6: "PKV_ERR_CUDA", 7: "PKV_ERR_DEVICE_CHECK", 8: "PKV_ERR_REFCOUNT"}
DEV_BAD_PAGE, DEV_BAD_LEN, DEV_TIMEOUT, DEV_BAD_PREFIX = 0x1, 0x2, 0x4, 0x8
# decode kernels (pkv_decode_variant)
VARIANT_AUTO, VARIANT_CUDA_CORES, VARIANT_TENSOR_CORES, VARIANT_TCGEN05 = 0, 1, 2, 3
# size of the library's fixed device scratch (PKV_NO_ALLOC_SCRATCH_BYTES)
NO_ALLOC_SCRATCH_BYTES = 32 << 20
_DT = {torch.float16: 0, torch.bfloat16: 1}

# fields of pkv_prefix_cache_stats, in order (all uint64)
PREFIX_STATS_FIELDS = ("lookups", "hits", "misses", "pages_hit", "pages_missed",
                       "pages_inserted", "pages_evicted")

_lib = None


class PagedKVError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        self.name = STATUS_NAMES.get(code, str(code))
        super().__init__(f"{where}: {self.name} ({pkv_status_string(code)})")


def library_path() -> str:
    return _build.LIB


def load_library(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libpagedkv.so (building it first when missing and nvcc is present)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if not os.path.exists(path):
        if not build_if_missing:
            raise RuntimeError(f"CUDA library not built: {path}")
        _build.build()
    lib = ctypes.CDLL(path)
    V, I, Z, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
    sig = {
        "pkv_status_string": ([I], ctypes.c_char_p),
        "pkv_version": ([], I),
        "kv_pool_create": ([I, I, I, I, I, V, V, ctypes.POINTER(V)], I),
        "kv_pool_destroy": ([V], I),
        "kv_pool_k": ([V], V),
        "kv_pool_v": ([V], V),
        "kv_pool_alloc_pages": ([V, I, V], I),
        "kv_pool_retain_pages": ([V, V, I], I),
        "kv_pool_release_pages": ([V, V, I], I),
        "kv_pool_free_count": ([V], I),
        "kv_pool_refcount": ([V, ctypes.c_int32], I),
        "kv_pool_info": ([V, V, V, V, V, V], I),
        "kv_append": ([V, V, V, V, I, V, I, V, V], I),
        "pkv_prefix_cache_create": ([V, ctypes.POINTER(V)], I),
        "pkv_prefix_cache_destroy": ([V], I),
        "pkv_prefix_cache_insert": ([V, V, I, V, ctypes.POINTER(I)], I),
        "pkv_prefix_cache_match": ([V, V, I, V, I, ctypes.POINTER(I)], I),
        "pkv_prefix_cache_evict": ([V, I, ctypes.POINTER(I)], I),
        "pkv_prefix_cache_pages": ([V], I),
        "pkv_prefix_cache_get_stats": ([V, I, V], I),
        "kv_append_rope": ([V, V, V, V, V, I, V, I, I, ctypes.c_double, V, V, F, V, V, V], I),
        "paged_decode_prefix_workspace_size": ([I, I, I, I, I, I, ctypes.POINTER(Z)], I),
        "paged_decode_multi_workspace_size": ([I, I, I, I, I, I, I, ctypes.POINTER(Z)], I),
        "pkv_check_bounded_wait": ([ctypes.c_uint32, V, V, V], I),
        "paged_decode_attention_multi": ([V, V, V, V, I, V, I, I, I, I, I, I, I, I, F, V, V, Z, I,
                                          I, V], I),
        "paged_decode_attention_prefix": ([V, V, V, V, I, V, I, I, I, I, I, I, I, F, I, V, V, Z,
                                           I, I, V], I),
        "paged_decode_step_rope": ([V, V, V, V, V, V, V, I, V, I, I, I, I, I, I, I, F,
                                    ctypes.c_double, V, V, F, V, V, Z, I, I, V], I),
        "kv_gather": ([V, V, I, V, I, I, V, V, V, V], I),
        "paged_decode_workspace_size": ([I, I, I, I, I, I, ctypes.POINTER(Z)], I),
        "paged_decode_plan": ([V, I, I, I, I, I, I, I, I, V, Z, V], I),
        "paged_decode_run": ([V, V, V, V, I, I, I, I, I, I, I, I, F, V, V, Z, I, I, I, V], I),
        "paged_decode_combine": ([I, I, I, I, I, V, V, Z, I, I, V], I),
        "paged_decode_attention": ([V, V, V, V, I, V, I, I, I, I, I, I, I, F, V, V, Z, I, I, V],
                                   I),
        "paged_decode_step": ([V, V, V, V, V, V, V, I, V, I, I, I, I, I, I, I, F, V, V, Z, I, I,
                               V], I),
        "paged_decode_attention_no_alloc": ([V, V, V, V, I, V, I, I, I, I, I, I, I, F, V, I, I,
                                             V], I),
        "paged_decode_step_host": ([V, V, V, V, V, V, V, I, V, I, I, I, I, I, I, I, F, V, V, Z, I,
                                    I, V], I),
        "paged_decode_step_host_workspace_size": ([I, I, I, I, I, I, I, ctypes.POINTER(Z)], I),
        "pkv_read_device_status": ([V, ctypes.POINTER(ctypes.c_uint32)], I),
        "pkv_read_no_alloc_status": ([ctypes.POINTER(ctypes.c_uint32)], I),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def pkv_status_string(code: int) -> str:
    return load_library().pkv_status_string(int(code)).decode()


def pkv_version() -> int:
    return load_library().pkv_version()


def _check(code: int, where: str):
    if code != PKV_OK:
        raise PagedKVError(code, where)


def _ptr(t: torch.Tensor | None):
    # ctypes converts a plain int for a c_void_p argument
    return None if t is None else t.data_ptr()


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream):
    if stream is not None:
        return stream.cuda_stream
    if _raw_stream is not None:
        return _raw_stream(torch.cuda.current_device())
    return torch.cuda.current_stream().cuda_stream


def _on_current_device(t) -> bool:
    # the library launches on the current device's stream and, for the
    # allocation-free call, uses that device's scratch: operands elsewhere
    # would be read by the wrong GPU
    idx = t.device.index
    return idx is None or idx == torch.cuda.current_device()


def _dev(t: torch.Tensor, name: str, dtype=None, ndim=None):
    """A contiguous CUDA tensor on the current device (of dtype / ndim when
    given), else raise."""
    try:
        ok = (t.is_cuda and t.is_contiguous() and (dtype is None or t.dtype == dtype)
              and (ndim is None or t.dim() == ndim) and _on_current_device(t))
    except AttributeError:
        raise TypeError(f"{name} must be a torch tensor") from None
    if ok:
        return t
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device")
    if not _on_current_device(t):
        raise ValueError(f"{name} is on {t.device} but the current device is "
                         f"cuda:{torch.cuda.current_device()}: call inside "
                         f"torch.cuda.device({t.device})")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    raise ValueError(f"{name} must have {ndim} dims, got {t.dim()}")


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype not in _DT:
        raise ValueError(f"dtype {t.dtype} not supported (float16 or bfloat16)")
    return _DT[t.dtype]


# ---------------------------------------------------------------------------
class Pool:
    """Handle of a page pool (kv_pool_create).  Borrowed torch tensors are kept
    alive by the handle."""

    def __init__(self, handle: int, k: torch.Tensor | None, v: torch.Tensor | None,
                 num_pages: int, page_size: int, n_kv_heads: int, head_dim: int, dtype):
        self._h = ctypes.c_void_p(handle)
        self._keep = (k, v)
        self.num_pages, self.page_size = num_pages, page_size
        self.n_kv_heads, self.head_dim, self.dtype = n_kv_heads, head_dim, dtype

    @property
    def handle(self):
        if not self._h:
            raise ValueError("pool destroyed")
        return self._h

    def k_ptr(self) -> int:
        return load_library().kv_pool_k(self.handle) or 0

    def v_ptr(self) -> int:
        return load_library().kv_pool_v(self.handle) or 0

    def alloc_pages(self, n: int) -> list[int]:
        ids = (ctypes.c_int32 * max(n, 1))()
        _check(load_library().kv_pool_alloc_pages(self.handle, n, ids), "kv_pool_alloc_pages")
        return list(ids[:n])

    def retain_pages(self, ids) -> None:
        arr = (ctypes.c_int32 * max(len(ids), 1))(*ids)
        _check(load_library().kv_pool_retain_pages(self.handle, arr, len(ids)),
               "kv_pool_retain_pages")

    def release_pages(self, ids) -> None:
        arr = (ctypes.c_int32 * max(len(ids), 1))(*ids)
        _check(load_library().kv_pool_release_pages(self.handle, arr, len(ids)),
               "kv_pool_release_pages")

    def free_count(self) -> int:
        return load_library().kv_pool_free_count(self.handle)

    def refcount(self, page_id: int) -> int:
        return load_library().kv_pool_refcount(self.handle, int(page_id))

    def destroy(self) -> None:
        if self._h:
            code = load_library().kv_pool_destroy(self._h)
            self._h = ctypes.c_void_p(None)
            self._keep = (None, None)
            _check(code, "kv_pool_destroy")

    def __del__(self):
        try:
            if self._h:
                load_library().kv_pool_destroy(self._h)
        except Exception:
            pass


def kv_pool_create(num_pages: int, page_size: int, n_kv_heads: int, head_dim: int,
                   dtype=torch.bfloat16, k_pool: torch.Tensor | None = None,
                   v_pool: torch.Tensor | None = None) -> Pool:
    """Create a pool; with k_pool/v_pool given ([NP, Hkv, P, D] device tensors)
    the pool borrows them, otherwise it allocates device memory itself."""
    if (k_pool is None) != (v_pool is None):
        raise ValueError("give both k_pool and v_pool or neither")
    code_dt = _DT.get(dtype)
    if code_dt is None:
        raise ValueError(f"dtype {dtype} not supported")
    if k_pool is not None:
        shape = (num_pages, n_kv_heads, page_size, head_dim)
        for name, t in (("k_pool", k_pool), ("v_pool", v_pool)):
            _dev(t, name, dtype, 4)
            if tuple(t.shape) != shape:
                raise ValueError(f"{name} shape {tuple(t.shape)} != {shape}")
    h = ctypes.c_void_p()
    _check(load_library().kv_pool_create(num_pages, page_size, n_kv_heads, head_dim, code_dt,
                                         _ptr(k_pool), _ptr(v_pool), ctypes.byref(h)),
           "kv_pool_create")
    return Pool(h.value, k_pool, v_pool, num_pages, page_size, n_kv_heads, head_dim, dtype)


class PrefixCache:
    """Host radix tree of cached prompt prefixes over a pool (whole pages of
    token ids -> pool pages).  `pool` is a Pool or a raw pool handle; it must
    outlive the cache.  match() hands the caller one reference per returned
    page (release them through the pool when the sequence ends)."""

    def __init__(self, pool):
        self._pool = pool
        h = pool.handle if isinstance(pool, Pool) else pool
        self._h = ctypes.c_void_p()
        _check(load_library().pkv_prefix_cache_create(h, ctypes.byref(self._h)),
               "pkv_prefix_cache_create")
        ps = ctypes.c_int()
        _check(load_library().kv_pool_info(h, None, ctypes.byref(ps), None, None, None),
               "kv_pool_info")
        self._page_size = ps.value

    @staticmethod
    def _i32(xs):
        # contiguous int32 numpy arrays are passed without a copy
        if isinstance(xs, np.ndarray) and xs.dtype == np.int32 and xs.flags.c_contiguous:
            return xs.ctypes.data if xs.size else None
        return (ctypes.c_int32 * max(len(xs), 1))(*[int(x) for x in xs])

    def insert(self, tokens, pages) -> int:
        """Cache the full pages of `tokens` stored in `pages`; returns how many
        pages were new to the cache."""
        n = ctypes.c_int()
        _check(load_library().pkv_prefix_cache_insert(self._h, self._i32(tokens), len(tokens),
                                                      self._i32(pages), ctypes.byref(n)),
               "pkv_prefix_cache_insert")
        return n.value

    def match(self, tokens, max_pages: int | None = None) -> list[int]:
        """Pages of the longest cached whole-page prefix of `tokens` (retained
        for the caller)."""
        cap = len(tokens) // self._page_size if max_pages is None else int(max_pages)
        out = (ctypes.c_int32 * max(cap, 1))()
        n = ctypes.c_int()
        _check(load_library().pkv_prefix_cache_match(self._h, self._i32(tokens), len(tokens), out,
                                                     cap, ctypes.byref(n)),
               "pkv_prefix_cache_match")
        return out[:n.value]

    def evict(self, n_pages: int) -> int:
        n = ctypes.c_int()
        _check(load_library().pkv_prefix_cache_evict(self._h, int(n_pages), ctypes.byref(n)),
               "pkv_prefix_cache_evict")
        return n.value

    def pages(self) -> int:
        return load_library().pkv_prefix_cache_pages(self._h)

    def stats(self, reset: bool = False) -> dict:
        """Lookup, hit and miss counters and pages inserted / evicted
        (pkv_prefix_cache_get_stats); reset zeroes them after reading."""
        buf = (ctypes.c_uint64 * len(PREFIX_STATS_FIELDS))()
        _check(load_library().pkv_prefix_cache_get_stats(self._h, int(bool(reset)), buf),
               "pkv_prefix_cache_get_stats")
        return dict(zip(PREFIX_STATS_FIELDS, (int(x) for x in buf)))

    def destroy(self) -> None:
        if self._h:
            h, self._h = self._h, ctypes.c_void_p(None)
            _check(load_library().pkv_prefix_cache_destroy(h), "pkv_prefix_cache_destroy")

    def __del__(self):
        try:
            if self._h:
                load_library().pkv_prefix_cache_destroy(self._h)
        except Exception:
            pass


def kv_append(pool: Pool, k_new: torch.Tensor, v_new: torch.Tensor, page_table: torch.Tensor,
              positions: torch.Tensor, dev_status: torch.Tensor | None = None,
              stream=None) -> None:
    """Write k_new/v_new [B, Hkv, D] into slot positions[b] of each sequence."""
    _dev(k_new, "k_new", pool.dtype, 3)
    _dev(v_new, "v_new", pool.dtype, 3)
    _dev(page_table, "page_table", torch.int32, 2)
    _dev(positions, "positions", torch.int32, 1)
    B = positions.shape[0]
    if k_new.shape != v_new.shape or k_new.shape != (B, pool.n_kv_heads, pool.head_dim):
        raise ValueError("k_new/v_new must be [B, Hkv, D] matching the pool")
    if page_table.shape[0] != B:
        raise ValueError("page_table rows != batch")
    if dev_status is not None:
        _dev(dev_status, "dev_status", torch.int32)
    _check(load_library().kv_append(pool.handle, _ptr(k_new), _ptr(v_new), _ptr(page_table),
                                    page_table.shape[1], _ptr(positions), B, _ptr(dev_status),
                                    _stream(stream)), "kv_append")


def _norm_weights(q_norm_weight, k_norm_weight, dtype, head_dim: int):
    for name, w in (("q_norm_weight", q_norm_weight), ("k_norm_weight", k_norm_weight)):
        if w is not None:
            _dev(w, name, dtype, 1)
            if w.shape[0] != head_dim:
                raise ValueError(f"{name} must hold head_dim values")


def kv_append_rope(pool: Pool, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                   page_table: torch.Tensor, positions: torch.Tensor, rope_theta: float,
                   q_out: torch.Tensor, dev_status: torch.Tensor | None = None,
                   stream=None, q_norm_weight: torch.Tensor | None = None,
                   k_norm_weight: torch.Tensor | None = None,
                   norm_eps: float = 1e-6) -> torch.Tensor:
    """Rotary embedding of q [B, Hq, D] (into q_out) and k_new at positions[b],
    then the append of the rotated k_new and v_new into the pool; with a norm
    weight [D], the per-head RMS norm of that side comes first."""
    _dev(q, "q", pool.dtype, 3)
    _dev(q_out, "q_out", pool.dtype, 3)
    _dev(k_new, "k_new", pool.dtype, 3)
    _dev(v_new, "v_new", pool.dtype, 3)
    _dev(page_table, "page_table", torch.int32, 2)
    _dev(positions, "positions", torch.int32, 1)
    B = positions.shape[0]
    if k_new.shape != v_new.shape or k_new.shape != (B, pool.n_kv_heads, pool.head_dim):
        raise ValueError("k_new/v_new must be [B, Hkv, D] matching the pool")
    if q.shape[0] != B or q.shape[2] != pool.head_dim or q_out.shape != q.shape:
        raise ValueError("q/q_out must be [B, Hq, D] matching the pool")
    if page_table.shape[0] != B:
        raise ValueError("page_table rows != batch")
    if dev_status is not None:
        _dev(dev_status, "dev_status", torch.int32)
    _norm_weights(q_norm_weight, k_norm_weight, pool.dtype, pool.head_dim)
    _check(load_library().kv_append_rope(
        pool.handle, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(page_table), page_table.shape[1],
        _ptr(positions), B, q.shape[1], float(rope_theta), _ptr(q_norm_weight),
        _ptr(k_norm_weight), float(norm_eps), _ptr(q_out), _ptr(dev_status), _stream(stream)),
        "kv_append_rope")
    return q_out


def kv_gather(pool: Pool, page_table: torch.Tensor, context_lens: torch.Tensor, max_len: int,
              k_out: torch.Tensor, v_out: torch.Tensor, dev_status: torch.Tensor | None = None,
              stream=None) -> None:
    """Dense [B, Hkv, max_len, D] copy of each sequence's cached rows."""
    _dev(page_table, "page_table", torch.int32, 2)
    _dev(context_lens, "context_lens", torch.int32, 1)
    B = context_lens.shape[0]
    for name, t in (("k_out", k_out), ("v_out", v_out)):
        _dev(t, name, pool.dtype, 4)
        if tuple(t.shape) != (B, pool.n_kv_heads, max_len, pool.head_dim):
            raise ValueError(f"{name} must be [B, Hkv, max_len, D]")
    if dev_status is not None:
        _dev(dev_status, "dev_status", torch.int32)
    _check(load_library().kv_gather(pool.handle, _ptr(page_table), page_table.shape[1],
                                    _ptr(context_lens), B, max_len, _ptr(k_out), _ptr(v_out),
                                    _ptr(dev_status), _stream(stream)), "kv_gather")


def paged_decode_workspace_size(batch: int, n_q_heads: int, n_kv_heads: int, head_dim: int,
                                num_workers: int = 0, variant: int = VARIANT_AUTO) -> int:
    n = ctypes.c_size_t()
    _check(load_library().paged_decode_workspace_size(batch, n_q_heads, n_kv_heads, head_dim,
                                                      num_workers, variant, ctypes.byref(n)),
           "paged_decode_workspace_size")
    return n.value


def alloc_workspace(batch: int, n_q_heads: int, n_kv_heads: int, head_dim: int,
                    num_workers: int = 0, device=None, variant: int = VARIANT_AUTO) -> torch.Tensor:
    """A torch uint8 buffer of the size paged_decode_attention needs (256-B aligned)."""
    n = paged_decode_workspace_size(batch, n_q_heads, n_kv_heads, head_dim, num_workers, variant)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device or "cuda")


def _decode_shapes(q, k_pool, v_pool, page_table, out):
    _dev(q, "q", None, 3)
    dt = _dtype_code(q)
    _dev(k_pool, "k_pool", q.dtype, 4)
    _dev(v_pool, "v_pool", q.dtype, 4)
    _dev(out, "out", q.dtype, 3)
    _dev(page_table, "page_table", torch.int32, 2)
    B, Hq, D = q.shape
    NP, Hkv, P, D2 = k_pool.shape
    if D2 != D or v_pool.shape != k_pool.shape or out.shape != q.shape:
        raise ValueError("q/out [B, Hq, D] and pools [NP, Hkv, P, D] disagree")
    if page_table.shape[0] != B:
        raise ValueError("page_table rows != batch")
    return B, Hq, Hkv, D, P, NP, dt


def paged_decode_attention(q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                           page_table: torch.Tensor, context_lens: torch.Tensor, scale: float,
                           out: torch.Tensor, workspace: torch.Tensor, num_workers: int = 0,
                           stream=None, variant: int = VARIANT_AUTO) -> torch.Tensor:
    """out[b, hq] = softmax(scale * q[b, hq] . K_b^T) V_b over context_lens[b]
    tokens read through page_table[b] (plan + decode + combine kernels)."""
    B, Hq, Hkv, D, P, NP, dt = _decode_shapes(q, k_pool, v_pool, page_table, out)
    _dev(context_lens, "context_lens", torch.int32, 1)
    _dev(workspace, "workspace", torch.uint8)
    _check(load_library().paged_decode_attention(
        _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(page_table), page_table.shape[1],
        _ptr(context_lens), B, Hq, Hkv, D, P, NP, dt, float(scale), _ptr(out), _ptr(workspace),
        workspace.numel(), int(num_workers), int(variant), _stream(stream)),
        "paged_decode_attention")
    return out


def paged_decode_attention_no_alloc(q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                                    page_table: torch.Tensor, context_lens: torch.Tensor,
                                    scale: float, out: torch.Tensor, num_workers: int = 0,
                                    stream=None, variant: int = VARIANT_AUTO) -> torch.Tensor:
    """paged_decode_attention without a workspace argument: the library uses its
    own fixed device scratch of NO_ALLOC_SCRATCH_BYTES bytes and allocates
    nothing.  For callers that must not allocate device memory at decode time.
    Calls share that scratch, so calls that overlap on the GPU race; make the
    first call on a device before any stream capture (it looks the scratch up)."""
    B, Hq, Hkv, D, P, NP, dt = _decode_shapes(q, k_pool, v_pool, page_table, out)
    _dev(context_lens, "context_lens", torch.int32, 1)
    _check(load_library().paged_decode_attention_no_alloc(
        _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(page_table), page_table.shape[1],
        _ptr(context_lens), B, Hq, Hkv, D, P, NP, dt, float(scale), _ptr(out), int(num_workers),
        int(variant), _stream(stream)),
        "paged_decode_attention_no_alloc")
    return out


def check_bounded_wait(tries: int, stream=None) -> tuple[int, int]:
    """One bounded wait that never succeeds (pkv_check_bounded_wait): returns
    (device status bits, wait duration in ns) once it has given up."""
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ns = torch.zeros(1, dtype=torch.int64, device="cuda")
    _check(load_library().pkv_check_bounded_wait(int(tries), _ptr(st), _ptr(ns), _stream(stream)),
           "pkv_check_bounded_wait")
    torch.cuda.synchronize()
    return int(st.item()) & 0xFFFFFFFF, int(ns.item())


def paged_decode_multi_workspace_size(batch: int, n_queries: int, n_q_heads: int,
                                      n_kv_heads: int, head_dim: int, num_workers: int = 0,
                                      variant: int = VARIANT_AUTO) -> int:
    n = ctypes.c_size_t()
    _check(load_library().paged_decode_multi_workspace_size(
        batch, n_queries, n_q_heads, n_kv_heads, head_dim, int(num_workers), int(variant),
        ctypes.byref(n)), "paged_decode_multi_workspace_size")
    return n.value


def alloc_multi_workspace(batch: int, n_queries: int, n_q_heads: int, n_kv_heads: int,
                          head_dim: int, num_workers: int = 0, device=None,
                          variant: int = VARIANT_AUTO) -> torch.Tensor:
    n = paged_decode_multi_workspace_size(batch, n_queries, n_q_heads, n_kv_heads, head_dim,
                                          num_workers, variant)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device or "cuda")


def paged_decode_attention_multi(q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                                 page_table: torch.Tensor, context_lens: torch.Tensor,
                                 scale: float, out: torch.Tensor, workspace: torch.Tensor,
                                 num_workers: int = 0, stream=None,
                                 variant: int = VARIANT_AUTO) -> torch.Tensor:
    """q, out [B, Qn, Hq, D]: query j of sequence b attends causally to tokens
    0 .. context_lens[b] - Qn + j."""
    _dev(q, "q", None, 4)
    dt = _dtype_code(q)
    _dev(out, "out", q.dtype, 4)
    _dev(k_pool, "k_pool", q.dtype, 4)
    _dev(v_pool, "v_pool", q.dtype, 4)
    _dev(page_table, "page_table", torch.int32, 2)
    _dev(context_lens, "context_lens", torch.int32, 1)
    _dev(workspace, "workspace", torch.uint8)
    B, Qn, Hq, D = q.shape
    NP, Hkv, P, D2 = k_pool.shape
    if D2 != D or v_pool.shape != k_pool.shape or out.shape != q.shape or page_table.shape[0] != B:
        raise ValueError("q/out [B, Qn, Hq, D], pools [NP, Hkv, P, D] and table disagree")
    _check(load_library().paged_decode_attention_multi(
        _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(page_table), page_table.shape[1],
        _ptr(context_lens), B, Qn, Hq, Hkv, D, P, NP, dt, float(scale), _ptr(out),
        _ptr(workspace), workspace.numel(), int(num_workers), int(variant), _stream(stream)),
        "paged_decode_attention_multi")
    return out


def paged_decode_prefix_workspace_size(batch: int, n_q_heads: int, n_kv_heads: int,
                                       head_dim: int, num_workers: int = 0,
                                       variant: int = VARIANT_AUTO) -> int:
    n = ctypes.c_size_t()
    _check(load_library().paged_decode_prefix_workspace_size(
        batch, n_q_heads, n_kv_heads, head_dim, int(num_workers), int(variant), ctypes.byref(n)),
        "paged_decode_prefix_workspace_size")
    return n.value


def alloc_prefix_workspace(batch: int, n_q_heads: int, n_kv_heads: int, head_dim: int,
                           num_workers: int = 0, device=None,
                           variant: int = VARIANT_AUTO) -> torch.Tensor:
    """A torch uint8 buffer of the size paged_decode_attention_prefix needs."""
    n = paged_decode_prefix_workspace_size(batch, n_q_heads, n_kv_heads, head_dim, num_workers,
                                           variant)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device or "cuda")


def paged_decode_attention_prefix(q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                                  page_table: torch.Tensor, context_lens: torch.Tensor,
                                  scale: float, prefix_tokens: int, out: torch.Tensor,
                                  workspace: torch.Tensor, num_workers: int = 0, stream=None,
                                  variant: int = VARIANT_AUTO) -> torch.Tensor:
    """Decode attention for a batch whose rows share their first prefix_tokens
    tokens (the same pages): the prefix is attended once for all queries."""
    B, Hq, Hkv, D, P, NP, dt = _decode_shapes(q, k_pool, v_pool, page_table, out)
    _dev(context_lens, "context_lens", torch.int32, 1)
    _dev(workspace, "workspace", torch.uint8)
    _check(load_library().paged_decode_attention_prefix(
        _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(page_table), page_table.shape[1],
        _ptr(context_lens), B, Hq, Hkv, D, P, NP, dt, float(scale), int(prefix_tokens), _ptr(out),
        _ptr(workspace), workspace.numel(), int(num_workers), int(variant), _stream(stream)),
        "paged_decode_attention_prefix")
    return out


def paged_decode_step(k_new: torch.Tensor, v_new: torch.Tensor, positions: torch.Tensor,
                      q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                      page_table: torch.Tensor, context_lens: torch.Tensor, scale: float,
                      out: torch.Tensor, workspace: torch.Tensor, num_workers: int = 0,
                      stream=None, variant: int = VARIANT_AUTO) -> torch.Tensor:
    """One decode step: append k_new/v_new [B, Hkv, D] at positions[b] (fused
    into the plan launch), then decode attention into out."""
    B, Hq, Hkv, D, P, NP, dt = _decode_shapes(q, k_pool, v_pool, page_table, out)
    _dev(context_lens, "context_lens", torch.int32, 1)
    _dev(workspace, "workspace", torch.uint8)
    _dev(k_new, "k_new", q.dtype, 3)
    _dev(v_new, "v_new", q.dtype, 3)
    _dev(positions, "positions", torch.int32, 1)
    if k_new.shape != (B, Hkv, D) or v_new.shape != (B, Hkv, D):
        raise ValueError("k_new/v_new must be [B, Hkv, D]")
    _check(load_library().paged_decode_step(
        _ptr(k_new), _ptr(v_new), _ptr(positions), _ptr(q), _ptr(k_pool), _ptr(v_pool),
        _ptr(page_table), page_table.shape[1], _ptr(context_lens), B, Hq, Hkv, D, P, NP, dt,
        float(scale), _ptr(out), _ptr(workspace), workspace.numel(), int(num_workers),
        int(variant), _stream(stream)), "paged_decode_step")
    return out


def _host(t: torch.Tensor, name: str, dtype=None, ndim=None):
    """A contiguous pinned (page-locked) CPU tensor (of dtype / ndim when
    given), else raise.  The library checks the pages themselves again."""
    try:
        ok = (not t.is_cuda and t.is_contiguous() and t.is_pinned()
              and (dtype is None or t.dtype == dtype) and (ndim is None or t.dim() == ndim))
    except AttributeError:
        raise TypeError(f"{name} must be a torch tensor") from None
    if ok:
        return t
    if t.is_cuda or not t.is_pinned():
        raise ValueError(f"{name} must be a pinned host tensor (tensor.pin_memory())")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    raise ValueError(f"{name} must have {ndim} dims, got {t.dim()}")


def paged_decode_step_host_workspace_size(batch: int, n_q_heads: int, n_kv_heads: int,
                                          head_dim: int, table_stride: int, num_workers: int = 0,
                                          variant: int = VARIANT_AUTO) -> int:
    n = ctypes.c_size_t()
    _check(load_library().paged_decode_step_host_workspace_size(
        batch, n_q_heads, n_kv_heads, head_dim, table_stride, num_workers, variant,
        ctypes.byref(n)), "paged_decode_step_host_workspace_size")
    return n.value


def alloc_step_host_workspace(batch: int, n_q_heads: int, n_kv_heads: int, head_dim: int,
                              table_stride: int, num_workers: int = 0, device=None,
                              variant: int = VARIANT_AUTO) -> torch.Tensor:
    """A torch uint8 device buffer of the size paged_decode_step_host needs."""
    n = paged_decode_step_host_workspace_size(batch, n_q_heads, n_kv_heads, head_dim,
                                              table_stride, num_workers, variant)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device or "cuda")


def paged_decode_step_host(k_new: torch.Tensor, v_new: torch.Tensor, positions: torch.Tensor,
                           q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                           page_table: torch.Tensor, context_lens: torch.Tensor, scale: float,
                           out: torch.Tensor, workspace: torch.Tensor, num_workers: int = 0,
                           stream=None, variant: int = VARIANT_AUTO) -> torch.Tensor:
    """paged_decode_step with k_new, v_new, positions, q, page_table,
    context_lens and out in pinned host memory (the pools and the workspace on
    the device): the kernels read the inputs and write out across the
    host-device link themselves.  out holds the result once the stream has
    finished the step."""
    _host(q, "q", None, 3)
    dt = _dtype_code(q)
    _dev(k_pool, "k_pool", q.dtype, 4)
    _dev(v_pool, "v_pool", q.dtype, 4)
    _dev(workspace, "workspace", torch.uint8)
    _host(out, "out", q.dtype, 3)
    _host(page_table, "page_table", torch.int32, 2)
    _host(context_lens, "context_lens", torch.int32, 1)
    _host(k_new, "k_new", q.dtype, 3)
    _host(v_new, "v_new", q.dtype, 3)
    _host(positions, "positions", torch.int32, 1)
    B, Hq, D = q.shape
    NP, Hkv, P, D2 = k_pool.shape
    if D2 != D or v_pool.shape != k_pool.shape or out.shape != q.shape:
        raise ValueError("q/out [B, Hq, D] and pools [NP, Hkv, P, D] disagree")
    if page_table.shape[0] != B:
        raise ValueError("page_table rows != batch")
    if k_new.shape != (B, Hkv, D) or v_new.shape != (B, Hkv, D):
        raise ValueError("k_new/v_new must be [B, Hkv, D]")
    _check(load_library().paged_decode_step_host(
        _ptr(k_new), _ptr(v_new), _ptr(positions), _ptr(q), _ptr(k_pool), _ptr(v_pool),
        _ptr(page_table), page_table.shape[1], _ptr(context_lens), B, Hq, Hkv, D, P, NP, dt,
        float(scale), _ptr(out), _ptr(workspace), workspace.numel(), int(num_workers),
        int(variant), _stream(stream)), "paged_decode_step_host")
    return out


def paged_decode_step_rope(k_new: torch.Tensor, v_new: torch.Tensor, positions: torch.Tensor,
                           q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                           page_table: torch.Tensor, context_lens: torch.Tensor, scale: float,
                           rope_theta: float, out: torch.Tensor, workspace: torch.Tensor,
                           num_workers: int = 0, stream=None,
                           variant: int = VARIANT_AUTO,
                           q_norm_weight: torch.Tensor | None = None,
                           k_norm_weight: torch.Tensor | None = None,
                           norm_eps: float = 1e-6) -> torch.Tensor:
    """paged_decode_step with the rotary embedding of q and k_new at positions[b]
    (angle base rope_theta) fused into the append, after the optional per-head
    RMS norm of either side; q stays as given, the rotated queries pass through
    out before the result overwrites them."""
    B, Hq, Hkv, D, P, NP, dt = _decode_shapes(q, k_pool, v_pool, page_table, out)
    _dev(context_lens, "context_lens", torch.int32, 1)
    _dev(workspace, "workspace", torch.uint8)
    _dev(k_new, "k_new", q.dtype, 3)
    _dev(v_new, "v_new", q.dtype, 3)
    _dev(positions, "positions", torch.int32, 1)
    if k_new.shape != (B, Hkv, D) or v_new.shape != (B, Hkv, D):
        raise ValueError("k_new/v_new must be [B, Hkv, D]")
    _norm_weights(q_norm_weight, k_norm_weight, q.dtype, D)
    _check(load_library().paged_decode_step_rope(
        _ptr(k_new), _ptr(v_new), _ptr(positions), _ptr(q), _ptr(k_pool), _ptr(v_pool),
        _ptr(page_table), page_table.shape[1], _ptr(context_lens), B, Hq, Hkv, D, P, NP, dt,
        float(scale), float(rope_theta), _ptr(q_norm_weight), _ptr(k_norm_weight),
        float(norm_eps), _ptr(out), _ptr(workspace), workspace.numel(), int(num_workers),
        int(variant), _stream(stream)), "paged_decode_step_rope")
    return out


def paged_decode_plan(context_lens: torch.Tensor, n_q_heads: int, n_kv_heads: int,
                      head_dim: int, page_size: int, table_stride: int, workspace: torch.Tensor,
                      num_workers: int = 0, stream=None, variant: int = VARIANT_AUTO) -> None:
    _dev(context_lens, "context_lens", torch.int32, 1)
    _dev(workspace, "workspace", torch.uint8)
    _check(load_library().paged_decode_plan(
        _ptr(context_lens), context_lens.shape[0], n_q_heads, n_kv_heads, head_dim, page_size,
        table_stride, int(num_workers), int(variant), _ptr(workspace), workspace.numel(),
        _stream(stream)), "paged_decode_plan")


def paged_decode_run(q, k_pool, v_pool, page_table, scale: float, out, workspace,
                     num_workers: int = 0, stream=None, variant: int = VARIANT_AUTO,
                     merge: bool = False) -> None:
    """The decode kernel; merge=True also merges split units (no combine needed)."""
    B, Hq, Hkv, D, P, NP, dt = _decode_shapes(q, k_pool, v_pool, page_table, out)
    _dev(workspace, "workspace", torch.uint8)
    _check(load_library().paged_decode_run(
        _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(page_table), page_table.shape[1], B, Hq, Hkv,
        D, P, NP, dt, float(scale), _ptr(out), _ptr(workspace), workspace.numel(),
        int(num_workers), int(variant), int(bool(merge)), _stream(stream)), "paged_decode_run")


def paged_decode_combine(out: torch.Tensor, n_kv_heads: int, workspace: torch.Tensor,
                         num_workers: int = 0, stream=None, variant: int = VARIANT_AUTO) -> None:
    _dev(out, "out", None, 3)
    _dev(workspace, "workspace", torch.uint8)
    B, Hq, D = out.shape
    _check(load_library().paged_decode_combine(
        B, Hq, n_kv_heads, D, _dtype_code(out), _ptr(out), _ptr(workspace), workspace.numel(),
        int(num_workers), int(variant), _stream(stream)), "paged_decode_combine")


def pkv_read_device_status(workspace: torch.Tensor) -> int:
    """The status word of the last decode on this workspace (synchronises)."""
    _dev(workspace, "workspace", torch.uint8)
    v = ctypes.c_uint32()
    code = load_library().pkv_read_device_status(_ptr(workspace), ctypes.byref(v))
    if code not in (0, 7):
        _check(code, "pkv_read_device_status")
    return v.value


def pkv_read_no_alloc_status() -> int:
    """The status word of the last paged_decode_attention_no_alloc call on the
    current device (synchronises)."""
    v = ctypes.c_uint32()
    code = load_library().pkv_read_no_alloc_status(ctypes.byref(v))
    if code not in (0, 7):
        _check(code, "pkv_read_no_alloc_status")
    return v.value
