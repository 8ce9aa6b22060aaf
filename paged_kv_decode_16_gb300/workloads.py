"""Seeded synthetic decode-step workloads (inputs only, no attention arithmetic).

This module builds the inputs that both the CUDA path and the float64 oracle
consume: context lengths, a physical page permutation, page tables (optionally
with a shared prefix), and random Q / K / V / new-token rows.  It contains none
of the method's arithmetic, so the tests, the benchmark and the oracle checks
can all draw from it without sharing computation.

Recipe (fixed, so that every run with the same seed sees the same inputs):

* ``numpy.random.default_rng(seed)`` draws, in this order, the context lengths
  and then the permutation of physical page ids ``[0, num_pages)``.
* Sequence b takes the next ``ceil(L_b / P)`` ids of the permutation (after the
  shared-prefix ids, if any); unused table entries are -1.
* Q, K-pool, V-pool, K-new, V-new are drawn in that order from
  ``torch.randn(..., generator=torch.Generator(device).manual_seed(seed))`` in
  float32 and rounded to the storage dtype (round to nearest even).
* ``positions[b]`` is the slot written by the per-step append: the last
  attended token ``L_b - 1`` (the new token of this step).

Named workloads follow the five shapes the method is exercised on (a tiny
correctness case, a Llama-3-8B-shaped step, a long-context step, a Mistral-7B
shape sharing a 2048-token prefix, and a Qwen2-7B-shaped mixed batch with the
append).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass
class Workload:
    name: str
    batch: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    page_size: int
    dtype: torch.dtype
    scale: float
    context_lens: np.ndarray          # int32 [B], tokens attended (incl. the new one)
    page_table: np.ndarray            # int32 [B, MP], -1 where unused
    num_pages: int
    positions: np.ndarray             # int32 [B], append slot (L_b - 1), or -1
    q: torch.Tensor                   # [B, Hq, D]
    k_pool: torch.Tensor              # [NP, Hkv, P, D]
    v_pool: torch.Tensor
    k_new: torch.Tensor               # [B, Hkv, D]
    v_new: torch.Tensor
    prefix_len: int = 0
    append: bool = False              # whether the named workload includes the append
    meta: dict = field(default_factory=dict)

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def dtype_name(self) -> str:
        return "bf16" if self.dtype == torch.bfloat16 else "f16"

    def kv_bytes_unique(self) -> int:
        """Bytes of K and V that one decode step must read (each distinct page
        slot once): distinct physical (page, slot) pairs in use x Hkv x D x 2 x 2."""
        P = self.page_size
        used = set()
        for b in range(self.batch):
            L = int(self.context_lens[b])
            for p in range((L + P - 1) // P):
                pg = int(self.page_table[b, p])
                n = min(P, L - p * P)
                used.add((pg, n))
        # a page shared by several sequences counts once, with its largest fill
        best: dict[int, int] = {}
        for pg, n in used:
            best[pg] = max(best.get(pg, 0), n)
        tokens = sum(best.values())
        return tokens * self.n_kv_heads * self.head_dim * 2 * 2

    def kv_bytes_logical(self) -> int:
        """Bytes of K and V summed per sequence (shared pages counted per reader)."""
        return int(self.context_lens.astype(np.int64).sum()) * self.n_kv_heads * self.head_dim * 4

    def qo_bytes(self) -> int:
        return 2 * self.batch * self.n_q_heads * self.head_dim * 2

    def append_bytes(self) -> int:
        """Read of k_new/v_new plus the write of the same rows into the pool."""
        n = int((self.positions >= 0).sum())
        return 2 * 2 * n * self.n_kv_heads * self.head_dim * 2

    def to(self, device) -> "Workload":
        w = Workload(**{k: getattr(self, k) for k in self.__dataclass_fields__})
        for k in ("q", "k_pool", "v_pool", "k_new", "v_new"):
            setattr(w, k, getattr(self, k).to(device))
        return w


def _randn(shape, gen, device, dtype):
    return torch.randn(*shape, generator=gen, device=device, dtype=torch.float32).to(dtype)


def build(name: str, *, batch: int, n_q_heads: int, n_kv_heads: int, head_dim: int,
          page_size: int, dtype: torch.dtype, context_lens, rng: np.random.Generator,
          seed: int, device="cpu", num_pages: int | None = None, prefix_len: int = 0,
          scale: float | None = None, append: bool = False, positions=None,
          poison: bool = False) -> Workload:
    """Assemble a workload from already-drawn lengths; draws the page permutation
    from ``rng`` next, then the tensors from a torch generator seeded ``seed``."""
    P = page_size
    lens = np.asarray(context_lens, dtype=np.int64)
    B = batch
    assert lens.shape == (B,)
    if prefix_len % P:
        raise ValueError("the shared prefix must fill whole pages")
    n_prefix = prefix_len // P
    if prefix_len and (lens < prefix_len).any():
        raise ValueError("every sequence must contain the shared prefix")
    pages_per_seq = [(int(L) + P - 1) // P for L in lens]
    private = [n - n_prefix for n in pages_per_seq]
    needed = n_prefix + sum(private)
    NP = needed if num_pages is None else int(num_pages)
    if NP < needed:
        raise ValueError("pool too small")
    perm = rng.permutation(NP).astype(np.int32)
    MP = max([1] + pages_per_seq)
    table = np.full((B, MP), -1, dtype=np.int32)
    cur = n_prefix
    for b in range(B):
        table[b, :n_prefix] = perm[:n_prefix]
        table[b, n_prefix:pages_per_seq[b]] = perm[cur:cur + private[b]]
        cur += private[b]

    gen = torch.Generator(device=device).manual_seed(seed)
    q = _randn((B, n_q_heads, head_dim), gen, device, dtype)
    k_pool = _randn((NP, n_kv_heads, P, head_dim), gen, device, dtype)
    v_pool = _randn((NP, n_kv_heads, P, head_dim), gen, device, dtype)
    k_new = _randn((B, n_kv_heads, head_dim), gen, device, dtype)
    v_new = _randn((B, n_kv_heads, head_dim), gen, device, dtype)
    if positions is None:
        pos = np.where(lens > 0, lens - 1, -1).astype(np.int32)
    else:
        pos = np.asarray(positions, dtype=np.int32)
    if scale is None:
        scale = 1.0 / math.sqrt(head_dim)
    w = Workload(name=name, batch=B, n_q_heads=n_q_heads, n_kv_heads=n_kv_heads,
                 head_dim=head_dim, page_size=P, dtype=dtype, scale=float(scale),
                 context_lens=lens.astype(np.int32), page_table=table, num_pages=NP,
                 positions=pos, q=q, k_pool=k_pool, v_pool=v_pool, k_new=k_new,
                 v_new=v_new, prefix_len=prefix_len, append=append)
    if poison:
        poison_unused(w)
    return w


def poison_unused(w: Workload) -> None:
    """Write NaN into every pool row no sequence attends to: unused pages and the
    tail slots of each sequence's last page.  A kernel that reads one of them into
    its result shows NaN there."""
    P = w.page_size
    nan = float("nan")
    live = torch.zeros((w.num_pages, P), dtype=torch.bool)
    for b in range(w.batch):
        L = int(w.context_lens[b])
        for p in range((L + P - 1) // P):
            pg = int(w.page_table[b, p])
            live[pg, :min(P, L - p * P)] = True
    dead = (~live).to(w.k_pool.device)
    # [NP, Hkv, P, D] viewed as [NP, P, Hkv, D] so that the [NP, P] mask applies
    w.k_pool.permute(0, 2, 1, 3)[dead] = nan
    w.v_pool.permute(0, 2, 1, 3)[dead] = nan


# ---------------------------------------------------------------------------
# the five named shapes
# ---------------------------------------------------------------------------
NAMES = ("tiny", "llama3_8b", "long_context", "prefix_sharing", "mixed_append")


def make(name: str, seed: int = 0, device="cpu", poison: bool = False,
         batch: int | None = None) -> Workload:
    """Build one of the named workloads.  ``batch`` overrides the batch size (the
    other parameters and the recipe stay the same) for reduced-size checks."""
    rng = np.random.default_rng(seed)
    if name == "tiny":
        # batch 2, 4 q heads / 2 kv heads, head_dim 64, pages of 16, lens {37, 100},
        # pool of 32 pages randomly permuted, fp16, scale 1/sqrt(64)
        B = batch or 2
        lens = np.array([37, 100][:B] + [100] * max(0, B - 2))
        return build(name, batch=B, n_q_heads=4, n_kv_heads=2, head_dim=64, page_size=16,
                     dtype=torch.float16, context_lens=lens, rng=rng, seed=seed, device=device,
                     num_pages=max(32, int(sum((lens + 15) // 16))), scale=1.0 / 8.0,
                     poison=poison)
    if name == "llama3_8b":
        B = batch or 32
        lens = rng.integers(512, 4096, size=B, endpoint=True)
        return build(name, batch=B, n_q_heads=32, n_kv_heads=8, head_dim=128, page_size=16,
                     dtype=torch.bfloat16, context_lens=lens, rng=rng, seed=seed, device=device,
                     poison=poison)
    if name == "long_context":
        B = batch or 8
        lens = np.full(B, 32768)
        return build(name, batch=B, n_q_heads=32, n_kv_heads=8, head_dim=128, page_size=16,
                     dtype=torch.bfloat16, context_lens=lens, rng=rng, seed=seed, device=device,
                     poison=poison)
    if name == "prefix_sharing":
        B = batch or 64
        suffix = rng.integers(64, 512, size=B, endpoint=True)
        lens = 2048 + suffix
        return build(name, batch=B, n_q_heads=32, n_kv_heads=8, head_dim=128, page_size=16,
                     dtype=torch.bfloat16, context_lens=lens, rng=rng, seed=seed, device=device,
                     prefix_len=2048, poison=poison)
    if name == "mixed_append":
        B = batch or 256
        before = np.floor(np.exp(rng.uniform(math.log(16), math.log(8192), size=B))).astype(np.int64)
        # the append writes position L (the length before this step); attention
        # then covers L + 1 tokens
        return build(name, batch=B, n_q_heads=28, n_kv_heads=4, head_dim=128, page_size=32,
                     dtype=torch.float16, context_lens=before + 1, rng=rng, seed=seed,
                     device=device, append=True, positions=before, poison=poison)
    raise KeyError(name)


def make_random(seed: int, *, batch: int, n_q_heads: int, n_kv_heads: int, head_dim: int,
                page_size: int, dtype: torch.dtype, lens, extra_pages: int = 3,
                device="cpu", poison: bool = False, scale: float | None = None) -> Workload:
    """A small random case with given lengths and a few unused pages in the pool."""
    rng = np.random.default_rng(seed)
    lens = np.asarray(lens, dtype=np.int64)
    needed = int(sum((int(L) + page_size - 1) // page_size for L in lens))
    return build("random", batch=batch, n_q_heads=n_q_heads, n_kv_heads=n_kv_heads,
                 head_dim=head_dim, page_size=page_size, dtype=dtype, context_lens=lens, rng=rng,
                 seed=seed, device=device, num_pages=needed + extra_pages, poison=poison,
                 scale=scale)


def scatter_dense(k_dense: np.ndarray, v_dense: np.ndarray, lens, page_size: int,
                  rng: np.random.Generator, extra_pages: int = 0, fill: int = 0):
    """Place dense per-sequence K/V ([B, Hkv, Lmax, D] uint16 patterns) into a
    randomly permuted page pool.  Returns (k_pool, v_pool, table).  Used to build
    oracle checks from a known dense cache."""
    B, Hkv, Lmax, D = k_dense.shape
    P = page_size
    lens = np.asarray(lens, dtype=np.int64)
    n_pages = [(int(L) + P - 1) // P for L in lens]
    NP = sum(n_pages) + extra_pages
    perm = rng.permutation(NP)
    MP = max([1] + n_pages)
    table = np.full((B, MP), -1, dtype=np.int32)
    k_pool = np.full((NP, Hkv, P, D), fill, dtype=np.uint16)
    v_pool = np.full((NP, Hkv, P, D), fill, dtype=np.uint16)
    cur = 0
    for b in range(B):
        for p in range(n_pages[b]):
            pg = int(perm[cur])
            cur += 1
            table[b, p] = pg
            lo, hi = p * P, min(int(lens[b]), (p + 1) * P)
            k_pool[pg, :, :hi - lo, :] = k_dense[b, :, lo:hi, :]
            v_pool[pg, :, :hi - lo, :] = v_dense[b, :, lo:hi, :]
    return k_pool, v_pool, table


def to_bits(t: torch.Tensor) -> np.ndarray:
    """16-bit patterns of a half/bfloat16 tensor as a host numpy uint16 array."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
