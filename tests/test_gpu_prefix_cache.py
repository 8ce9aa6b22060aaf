"""The host prefix cache feeding the GPU path: a stream of requests that share a
system prompt goes through pkv_prefix_cache_match (cached pages retained for
the request), kv_pool_alloc_pages (the rest of the prompt), a prefill that
writes only the freshly allocated pages, and pkv_prefix_cache_insert.  The
batch's page tables are the rows the cache and the allocator handed back.
Checked: every row, gathered through its table, holds exactly the K/V that
its own tokens produce (bitwise, so a matched page is the right page); then
one decode step appends each sequence's new token (bitwise against the
oracle's append) and both paged_decode_attention and the shared-prefix
paged_decode_attention_prefix match the float64 oracle element by element;
the cache's hit/miss counters agree with the request stream."""
import hashlib

import numpy as np
import pytest
import torch

import oracle
import paged_kv_decode_16_gb300 as pkv
from paged_kv_decode_16_gb300 import workloads as wl

from gpu_helpers import VARIANT_IDS, VARIANTS, assert_close

pytestmark = pytest.mark.gpu

P, HKV, HQ, D = 16, 2, 8, 128
DT = torch.bfloat16


def _kv_of_prefix(tokens, t):
    """K and V rows [Hkv, D] of position t: a function of tokens 0..t only, as
    a model's K/V are (seeded by a digest of the prefix)."""
    h = hashlib.sha256(np.asarray(tokens[:t + 1], dtype=np.int32).tobytes()).digest()
    rng = np.random.default_rng(int.from_bytes(h[:8], "little"))
    kv = torch.from_numpy(rng.standard_normal((2, HKV, D)).astype(np.float32)).to(DT)
    return kv[0], kv[1]


def _request_stream(rng):
    system = rng.integers(0, 32000, size=4 * P).tolist()  # 64 shared tokens, 4 pages
    reqs = []
    for i in range(8):
        reqs.append(system + rng.integers(0, 32000, size=int(rng.integers(5, 150))).tolist())
    # a follow-up turn: request 2's whole prompt plus more (matches its pages too)
    reqs.append(reqs[2] + rng.integers(0, 32000, size=40).tolist())
    return reqs


@pytest.mark.parametrize("variant", VARIANTS, ids=VARIANT_IDS)
def test_cache_rows_decode_like_the_oracle(variant):
    rng = np.random.default_rng(2024)
    NP = 256
    k_pool = torch.randn(NP, HKV, P, D, generator=torch.Generator().manual_seed(1)).to(DT).cuda()
    v_pool = torch.randn(NP, HKV, P, D, generator=torch.Generator().manual_seed(2)).to(DT).cuda()
    pool = pkv.kv_pool_create(NP, P, HKV, D, DT, k_pool, v_pool)
    cache = pkv.PrefixCache(pool)
    reqs = _request_stream(rng)
    rows, matched_counts = [], []
    for toks in reqs:
        got = cache.match(toks)
        matched_counts.append(len(got))
        fresh = pool.alloc_pages(-(-len(toks) // P) - len(got))
        row = list(got) + fresh
        # prefill: only the pages this request allocated are written
        for t in range(len(got) * P, len(toks)):
            k, v = _kv_of_prefix(toks, t)
            k_pool[row[t // P], :, t % P] = k.cuda()
            v_pool[row[t // P], :, t % P] = v.cuda()
        cache.insert(toks, row)
        rows.append(row)
    # the system prompt's pages are shared by every row; the follow-up turn
    # reuses all of request 2's whole pages
    assert matched_counts[0] == 0 and all(m >= 4 for m in matched_counts[1:])
    assert matched_counts[-1] == len(reqs[2]) // P
    assert all(r[:4] == rows[0][:4] for r in rows)
    st = cache.stats()
    assert st["lookups"] == len(reqs) and st["misses"] == 1 and st["hits"] == len(reqs) - 1
    assert st["pages_hit"] == sum(matched_counts)

    # the decode step: one new token per sequence at position len(toks)
    B = len(reqs)
    lens_before = np.array([len(t) for t in reqs], dtype=np.int32)
    for b, toks in enumerate(reqs):
        if len(toks) % P == 0:
            rows[b] += pool.alloc_pages(1)
    MP = max(len(r) for r in rows)
    table = np.full((B, MP), -1, dtype=np.int32)
    for b, r in enumerate(rows):
        table[b, :len(r)] = r

    # every row gathered through its table holds its own tokens' K/V
    kb, vb = wl.to_bits(k_pool), wl.to_bits(v_pool)
    for b, toks in enumerate(reqs):
        for t in range(len(toks)):
            k, v = _kv_of_prefix(toks, t)
            page, slot = table[b, t // P], t % P
            assert np.array_equal(kb[page, :, slot], wl.to_bits(k)), (b, t)
            assert np.array_equal(vb[page, :, slot], wl.to_bits(v)), (b, t)

    g = torch.Generator(device="cuda").manual_seed(7)
    q = torch.randn(B, HQ, D, generator=g, device="cuda").to(DT)
    k_new = torch.randn(B, HKV, D, generator=g, device="cuda").to(DT)
    v_new = torch.randn(B, HKV, D, generator=g, device="cuda").to(DT)
    table_d = torch.from_numpy(table).cuda()
    pos = torch.from_numpy(lens_before).cuda()
    lens = torch.from_numpy(lens_before + 1).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.kv_append(pool, k_new, v_new, table_d, pos, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    kp, vp = oracle.kv_append(kb, vb, wl.to_bits(k_new), wl.to_bits(v_new), table, lens_before)
    assert np.array_equal(kp, wl.to_bits(k_pool)) and np.array_equal(vp, wl.to_bits(v_pool))

    scale = D ** -0.5
    ref = oracle.paged_decode(wl.to_bits(q), kp, vp, table, lens_before + 1, scale, "bf16")
    out = torch.full_like(q, float("nan"))
    ws = pkv.alloc_workspace(B, HQ, HKV, D, variant=variant)
    pkv.paged_decode_attention(q, k_pool, v_pool, table_d, lens, scale, out, ws, variant=variant)
    torch.cuda.synchronize()
    assert pkv.pkv_read_device_status(ws) == 0
    assert_close(out, ref, strict=True, what="plain decode over cache rows")

    out2 = torch.full_like(q, float("nan"))
    wsp = pkv.alloc_prefix_workspace(B, HQ, HKV, D, variant=variant)
    pkv.paged_decode_attention_prefix(q, k_pool, v_pool, table_d, lens, scale, 4 * P, out2, wsp,
                                      variant=variant)
    torch.cuda.synchronize()
    assert pkv.pkv_read_device_status(wsp) == 0
    assert_close(out2, ref, strict=True, what="shared-prefix decode over cache rows")

    for r in rows:
        pool.release_pages(r)
    cache.destroy()
    assert pool.free_count() == NP
    pool.destroy()
