"""paged_decode_attention_no_alloc: the decode entry point that takes its
workspace from the library's fixed device scratch instead of the caller.

It is for callers that cannot allocate device memory when they decode (a
serving loop that forbids cudaMalloc after warm-up, a plugin whose host
framework owns all device memory).  It runs the same plan, decode and
combine kernels with the same split as paged_decode_attention, so its output
must equal that call's bit for bit, and both must match the float64 oracle
within the parity tolerance; this holds on calls made back to back that
reuse the same scratch.  Bad page ids are flagged in the scratch's status
word, read with pkv_read_no_alloc_status; shapes whose workspace does not fit
the scratch are refused before anything runs.  The file's name keeps it last
in collection order, and it also passes alone in a fresh process (the first
call on the device sets the scratch address up)."""
import pytest
import torch

import paged_kv_decode_16_gb300 as pkv
from paged_kv_decode_16_gb300 import workloads as wl

from gpu_helpers import assert_close, oracle_full, to_dev

pytestmark = pytest.mark.gpu


def _with_workspace(w, table, lens, variant):
    out = torch.empty_like(w.q)
    ws = pkv.alloc_workspace(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, 0,
                             device=w.q.device, variant=variant)
    pkv.paged_decode_attention(w.q, w.k_pool, w.v_pool, table, lens, w.scale, out, ws,
                               variant=variant)
    return out


def _same_bits(a, b, what):
    assert torch.equal(a.view(torch.int16), b.view(torch.int16)), f"{what}: bits differ"


@pytest.mark.parametrize("variant", [pkv.VARIANT_TENSOR_CORES, pkv.VARIANT_CUDA_CORES],
                         ids=["tensor_cores", "cuda_cores"])
def test_two_calls_in_a_row_match_workspace_entry_point(variant):
    dev = "cuda"
    # two different problems, decoded back to back through the shared scratch:
    # the second must not see anything the first left behind
    first = wl.make("llama3_8b", seed=11, device=dev)
    second = wl.make_random(12, batch=5, n_q_heads=12, n_kv_heads=2, head_dim=64, page_size=32,
                            dtype=torch.float16, lens=[1, 700, 0, 33, 2100], device=dev)
    runs = []
    for w in (first, second):
        table, lens, _ = to_dev(w, dev)
        out = torch.full_like(w.q, float("nan"))
        pkv.paged_decode_attention_no_alloc(w.q, w.k_pool, w.v_pool, table, lens, w.scale, out,
                                            variant=variant)
        runs.append((w, table, lens, out))
    torch.cuda.synchronize()
    assert pkv.pkv_read_no_alloc_status() == 0
    for i, (w, table, lens, out) in enumerate(runs):
        ref = _with_workspace(w, table, lens, variant)
        torch.cuda.synchronize()
        _same_bits(out, ref, f"call {i + 1}")
        assert_close(out, oracle_full(w, append=False), strict=(i == 0), what=f"call {i + 1}")


def test_repeated_call_is_stable():
    w = wl.make("mixed_append", seed=3, device="cuda")
    table, lens, _ = to_dev(w, "cuda")
    a = torch.empty_like(w.q)
    b = torch.empty_like(w.q)
    pkv.paged_decode_attention_no_alloc(w.q, w.k_pool, w.v_pool, table, lens, w.scale, a)
    pkv.paged_decode_attention_no_alloc(w.q, w.k_pool, w.v_pool, table, lens, w.scale, b)
    ref = _with_workspace(w, table, lens, pkv.VARIANT_AUTO)
    torch.cuda.synchronize()
    _same_bits(a, ref, "call 1")
    _same_bits(b, ref, "call 2")
    assert_close(a, oracle_full(w, append=False), strict=True, what="mixed_append")


def test_bad_page_id_is_flagged_in_the_scratch_status():
    w = wl.make_random(21, batch=3, n_q_heads=8, n_kv_heads=2, head_dim=128, page_size=16,
                       dtype=torch.bfloat16, lens=[40, 17, 64], device="cuda")
    table, lens, _ = to_dev(w, "cuda")
    out = torch.empty_like(w.q)
    # a clean call first: the status word starts fresh on every call
    pkv.paged_decode_attention_no_alloc(w.q, w.k_pool, w.v_pool, table, lens, w.scale, out)
    assert pkv.pkv_read_no_alloc_status() == 0
    bad = table.clone()
    bad[1, 0] = w.num_pages + 5  # outside the pool: skipped by the kernels and flagged
    pkv.paged_decode_attention_no_alloc(w.q, w.k_pool, w.v_pool, bad, lens, w.scale, out)
    assert pkv.pkv_read_no_alloc_status() & pkv.DEV_BAD_PAGE
    pkv.paged_decode_attention_no_alloc(w.q, w.k_pool, w.v_pool, table, lens, w.scale, out)
    assert pkv.pkv_read_no_alloc_status() == 0


def test_rejects_shapes_beyond_the_scratch():
    B, Hq, Hkv, D = 65536, 32, 8, 128
    need = pkv.paged_decode_workspace_size(B, Hq, Hkv, D, 0, pkv.VARIANT_AUTO)
    assert need > pkv.NO_ALLOC_SCRATCH_BYTES
    q = torch.zeros(B, Hq, D, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros_like(q)
    pool_k = torch.zeros(1, Hkv, 16, D, dtype=torch.bfloat16, device="cuda")
    pool_v = torch.zeros_like(pool_k)
    table = torch.zeros(B, 1, dtype=torch.int32, device="cuda")
    lens = torch.zeros(B, dtype=torch.int32, device="cuda")
    with pytest.raises(pkv.PagedKVError) as e:
        pkv.paged_decode_attention_no_alloc(q, pool_k, pool_v, table, lens, 0.1, out)
    assert e.value.name == "PKV_ERR_WORKSPACE"
    torch.cuda.synchronize()
    assert int(out.abs().max().item()) == 0  # nothing ran
