"""Parity of the several-queries-per-sequence decode (paged_decode_attention_multi)
with the float64 oracle: query j of sequence b attends causally to tokens
0 .. L_b - Qn + j.  Covers queries that see no token (L_b < Qn - j), whole
chunks hidden from some queries by the causal limit (the online softmax must
keep those rows at weight 0), several query tiles per sequence (up to 64
tokens, the last tile shorter), splits of one sequence over many workers (the
partial states of those rows reach the merge with m = -inf), poisoned unused
page slots, and the argument checks.  Tolerance: that of the other decode
parity tests."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_decode_16_gb300 as pkv
from paged_kv_decode_16_gb300 import workloads as wl

from gpu_helpers import assert_close, to_dev

pytestmark = pytest.mark.gpu


def _case(seed, *, B, Qn, Hq, Hkv, D, P, dtype, lens, poison=True):
    w = wl.make_random(seed, batch=B, n_q_heads=Hq, n_kv_heads=Hkv, head_dim=D, page_size=P,
                       dtype=dtype, lens=lens, device="cuda", poison=poison)
    gen = torch.Generator(device="cuda").manual_seed(seed + 7919)
    q = torch.randn(B, Qn, Hq, D, generator=gen, device="cuda", dtype=torch.float32).to(dtype)
    return w, q


def _run(w, q, num_workers=0, variant=pkv.VARIANT_AUTO):
    table, lens, _ = to_dev(w)
    B, Qn, Hq, D = q.shape
    ws = pkv.alloc_multi_workspace(B, Qn, Hq, w.n_kv_heads, D, num_workers, variant=variant)
    out = torch.full_like(q, float("nan"))
    pkv.paged_decode_attention_multi(q, w.k_pool, w.v_pool, table, lens, w.scale, out, ws,
                                     num_workers=num_workers, variant=variant)
    torch.cuda.synchronize()
    return out, ws


def _oracle(w, q):
    return oracle.paged_decode_multi(wl.to_bits(q), wl.to_bits(w.k_pool), wl.to_bits(w.v_pool),
                                     w.page_table, w.context_lens, w.scale, w.dtype_name)


CASES = [
    # B, Qn, Hq, Hkv, D, P, dtype, lens
    (4, 4, 32, 8, 128, 16, torch.bfloat16, [300, 17, 64, 1029]),     # 4 x 4 rows per unit
    (5, 2, 32, 8, 128, 16, torch.float16, [2, 1, 0, 33, 700]),       # L < Qn, L = 0
    (3, 3, 12, 4, 64, 32, torch.bfloat16, [3, 47, 2048]),           # group 3: 3 x 3 rows
    (6, 8, 28, 4, 128, 16, torch.float16, [8, 9, 15, 16, 17, 500]),  # group 7: 8 x 1 rows
    (2, 16, 8, 8, 64, 16, torch.bfloat16, [16, 5000]),               # 16 queries, group 1
    (3, 5, 16, 2, 128, 32, torch.bfloat16, [4, 37, 1100]),          # 5 x 2 rows, one L < Qn
    (2, 7, 8, 1, 64, 16, torch.float16, [31, 260]),                  # MQA: 7 x 2 rows
    # more than one tile of queries: tiles of equal size but the last
    (3, 17, 8, 2, 128, 16, torch.bfloat16, [5, 17, 400]),           # tiles 9 + 8, one head each
    (2, 32, 16, 2, 64, 16, torch.float16, [40, 777]),               # 2 tiles of 16
    (2, 33, 4, 4, 128, 32, torch.bfloat16, [20, 300]),              # 3 tiles of 11, group 1
    (2, 64, 8, 1, 128, 16, torch.bfloat16, [64, 1000]),             # 4 tiles of 16, MQA
    (2, 48, 12, 4, 64, 16, torch.float16, [3, 129]),                # 3 tiles of 16, group 3
    (2, 23, 24, 2, 128, 16, torch.bfloat16, [30, 90]),              # 2 tiles of 12, group 12
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_multi_query_matches_oracle(case):
    B, Qn, Hq, Hkv, D, P, dtype, lens = CASES[case]
    w, q = _case(200 + case, B=B, Qn=Qn, Hq=Hq, Hkv=Hkv, D=D, P=P, dtype=dtype, lens=lens)
    ref = _oracle(w, q)
    # automatic split, a few workers (long segments), many (one chunk each)
    for nw in (0, 3, 1000):
        out, ws = _run(w, q, num_workers=nw)
        assert pkv.pkv_read_device_status(ws) == 0
        assert_close(out, ref, what=f"case {case} workers {nw}")


def test_queries_without_tokens_give_zeros():
    w, q = _case(230, B=3, Qn=6, Hq=8, Hkv=2, D=128, P=16, dtype=torch.bfloat16, lens=[0, 2, 5])
    out, _ = _run(w, q, num_workers=5)
    o = out.float().cpu()
    assert torch.all(o[0] == 0)
    assert torch.all(o[1, :4] == 0) and torch.all(o[2, :1] == 0)
    assert torch.isfinite(o).all()
    assert_close(out, _oracle(w, q), what="short sequences")


def test_last_query_equals_single_query_decode():
    """Query Qn - 1 sees every token: its output is paged_decode_attention's
    of that query within tolerance, and with Qn = 1 the bits are the same."""
    w, q = _case(231, B=8, Qn=4, Hq=32, Hkv=8, D=128, P=16, dtype=torch.bfloat16,
                 lens=[100, 257, 1024, 33, 4, 700, 1500, 90])
    table, lens, _ = to_dev(w)
    out, _ = _run(w, q)
    last = q[:, -1].contiguous()
    single = torch.empty_like(last)
    pkv.paged_decode_attention(last, w.k_pool, w.v_pool, table, lens, w.scale, single,
                               pkv.alloc_workspace(w.batch, w.n_q_heads, w.n_kv_heads,
                                                   w.head_dim))
    torch.cuda.synchronize()
    assert_close(out[:, -1], single.float().cpu().numpy().astype(np.float64), what="last query")
    one, _ = _run(w, last.unsqueeze(1))
    assert torch.equal(one[:, 0].view(torch.int16), single.view(torch.int16))


def test_bigger_batch_at_the_decode_shape():
    """Llama-3-8B heads (32 / 8, D 128, bf16), four draft tokens, ragged lengths."""
    rng = np.random.default_rng(232)
    lens = rng.integers(4, 3000, size=24)
    w, q = _case(232, B=24, Qn=4, Hq=32, Hkv=8, D=128, P=16, dtype=torch.bfloat16, lens=lens)
    out, ws = _run(w, q)
    assert pkv.pkv_read_device_status(ws) == 0
    assert_close(out, _oracle(w, q), what="llama3-8b heads, 4 queries")


def test_multi_argument_checks():
    w, q = _case(233, B=2, Qn=4, Hq=8, Hkv=2, D=128, P=16, dtype=torch.bfloat16, lens=[40, 50])
    table, lens, _ = to_dev(w)
    with pytest.raises(pkv.PagedKVError) as e:   # CUDA-core kernel: one query row per head
        pkv.alloc_multi_workspace(2, 4, 8, 2, 128, variant=pkv.VARIANT_CUDA_CORES)
    assert e.value.name == "PKV_ERR_UNSUPPORTED"
    with pytest.raises(pkv.PagedKVError) as e:   # beyond 64 query tokens
        pkv.alloc_multi_workspace(2, 65, 8, 2, 128)
    assert e.value.name == "PKV_ERR_UNSUPPORTED"
    with pytest.raises(pkv.PagedKVError) as e:
        pkv.alloc_multi_workspace(2, 0, 8, 2, 128)
    assert e.value.name == "PKV_ERR_INVALID_ARG"
    ws = pkv.alloc_multi_workspace(2, 4, 8, 2, 128)
    with pytest.raises(pkv.PagedKVError) as e:
        pkv.paged_decode_attention_multi(q, w.k_pool, w.v_pool, table, lens, w.scale,
                                         torch.empty_like(q), ws[:256])
    assert e.value.name == "PKV_ERR_WORKSPACE"
    with pytest.raises(pkv.PagedKVError) as e:   # out overlapping q
        pkv.paged_decode_attention_multi(q, w.k_pool, w.v_pool, table, lens, w.scale, q, ws)
    assert e.value.name == "PKV_ERR_ALIAS"


def test_multi_captured_in_cuda_graph_equals_eager():
    """paged_decode_attention_multi recorded into a CUDA graph and replayed
    gives the eager call's bits, and a replay sees new lengths and queries
    written into the same buffers."""
    w, q = _case(234, B=6, Qn=5, Hq=16, Hkv=4, D=128, P=16, dtype=torch.bfloat16,
                 lens=[900, 7, 33, 0, 2048, 160])
    table, lens, _ = to_dev(w)
    eager, ws = _run(w, q)
    out = torch.full_like(q, float("nan"))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            pkv.paged_decode_attention_multi(q, w.k_pool, w.v_pool, table, lens, w.scale, out, ws)
    torch.cuda.current_stream().wait_stream(s)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
    # new lengths no longer than the old ones (slots past those hold NaN)
    lens.copy_(torch.tensor([899, 7, 20, 0, 1500, 150], dtype=torch.int32))
    q.mul_(-0.5)
    g.replay()
    torch.cuda.synchronize()
    w.context_lens[:] = lens.cpu().numpy()
    assert pkv.pkv_read_device_status(ws) == 0
    assert_close(out, _oracle(w, q), what="replay with new lengths")


# ---- the tcgen05 kernel (PKV_VARIANT_TCGEN05): units of up to 64 rows, the
# products transposed (128 tokens of a block as the tile's rows) ----

UMMA_CASES = [c for c in range(len(CASES)) if CASES[c][4] == 128]


@pytest.mark.parametrize("case", UMMA_CASES)
def test_tcgen05_multi_query_matches_oracle(case):
    B, Qn, Hq, Hkv, D, P, dtype, lens = CASES[case]
    w, q = _case(200 + case, B=B, Qn=Qn, Hq=Hq, Hkv=Hkv, D=D, P=P, dtype=dtype, lens=lens)
    ref = _oracle(w, q)
    for nw in (0, 3, 1000):
        out, ws = _run(w, q, num_workers=nw, variant=pkv.VARIANT_TCGEN05)
        assert pkv.pkv_read_device_status(ws) == 0
        assert_close(out, ref, what=f"tcgen05 case {case} workers {nw}")


@pytest.mark.parametrize("qn", [2, 4, 8, 16])
def test_tcgen05_on_the_llama3_8b_cache(qn):
    """Llama-3-8B heads (32 / 8, D 128, bf16), the named workload's cache
    (contexts 512-4096, poisoned unused slots), qn draft tokens per sequence:
    units of qn x 4 rows (8..64), every output element against the oracle."""
    w = wl.make("llama3_8b", seed=0, device="cuda", poison=True)
    gen = torch.Generator(device="cuda").manual_seed(240 + qn)
    q = torch.randn(w.batch, qn, w.n_q_heads, w.head_dim, generator=gen, device="cuda",
                    dtype=torch.float32).to(w.dtype)
    out, ws = _run(w, q, variant=pkv.VARIANT_TCGEN05)
    assert pkv.pkv_read_device_status(ws) == 0
    assert_close(out, _oracle(w, q), strict=True, what=f"llama3_8b cache, {qn} queries")


def test_tcgen05_equals_warp_kernel_within_tolerance_and_is_deterministic():
    rng = np.random.default_rng(241)
    lens = rng.integers(1, 2500, size=12)
    w, q = _case(241, B=12, Qn=8, Hq=32, Hkv=8, D=128, P=16, dtype=torch.bfloat16, lens=lens)
    a, _ = _run(w, q, variant=pkv.VARIANT_TCGEN05)
    b, _ = _run(w, q, variant=pkv.VARIANT_TCGEN05)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    c, _ = _run(w, q, variant=pkv.VARIANT_TENSOR_CORES)
    assert_close(a, c.float().cpu().numpy().astype(np.float64), what="tcgen05 vs warp MMA")


def test_tcgen05_bad_page_is_skipped_and_reported():
    """A page id outside the pool: its chunk is skipped (not copied, not
    attended) and PKV_DEV_BAD_PAGE is set, as in the warp kernel, whose
    output it then matches."""
    w, q = _case(242, B=3, Qn=4, Hq=16, Hkv=4, D=128, P=16, dtype=torch.bfloat16,
                 lens=[200, 500, 64])
    w.page_table[1, 3] = w.num_pages + 5
    out, ws = _run(w, q, variant=pkv.VARIANT_TCGEN05)
    assert pkv.pkv_read_device_status(ws) & pkv.DEV_BAD_PAGE
    ref, ws2 = _run(w, q, variant=pkv.VARIANT_TENSOR_CORES)
    assert pkv.pkv_read_device_status(ws2) & pkv.DEV_BAD_PAGE
    assert torch.isfinite(out.float()).all()
    assert_close(out, ref.float().cpu().numpy().astype(np.float64), what="bad page")


def test_tcgen05_unsupported_shapes():
    with pytest.raises(pkv.PagedKVError) as e:   # head_dim 64
        pkv.alloc_multi_workspace(2, 4, 8, 2, 64, variant=pkv.VARIANT_TCGEN05)
    assert e.value.name == "PKV_ERR_UNSUPPORTED"
    with pytest.raises(pkv.PagedKVError) as e:   # one query per sequence
        pkv.alloc_workspace(2, 8, 2, 128, variant=pkv.VARIANT_TCGEN05)
    assert e.value.name == "PKV_ERR_UNSUPPORTED"
