"""paged_decode_attention_no_alloc: the decode entry point that takes its
workspace from the library's fixed device scratch instead of the caller.

Its outputs must match those of paged_decode_attention (caller-provided
workspace) within the parity tolerance of the other GPU tests, on calls made
back to back that reuse the same scratch; shapes whose workspace does not fit
the scratch are refused before anything runs.  The file's name keeps it last
in collection order, and it also passes alone in a fresh process (the first
call on the device sets the scratch address up)."""
import numpy as np
import pytest
import torch

import paged_kv_decode_16_gb300 as pkv
from paged_kv_decode_16_gb300 import workloads as wl

from gpu_helpers import ATOL, RTOL, to_dev

pytestmark = pytest.mark.gpu


def _with_workspace(w, table, lens, variant):
    out = torch.empty_like(w.q)
    ws = pkv.alloc_workspace(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, 0,
                             device=w.q.device, variant=variant)
    pkv.paged_decode_attention(w.q, w.k_pool, w.v_pool, table, lens, w.scale, out, ws,
                               variant=variant)
    return out


def _close(got, ref, what):
    g = got.float().cpu().numpy()
    r = ref.float().cpu().numpy()
    assert np.isfinite(g).all(), what
    err = np.abs(g - r)
    bad = err > ATOL + RTOL * np.abs(r)
    assert not bad.any(), f"{what}: {int(bad.sum())} elements off, max err {err.max():.3g}"


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
    for i, (w, table, lens, out) in enumerate(runs):
        ref = _with_workspace(w, table, lens, variant)
        torch.cuda.synchronize()
        _close(out, ref, f"call {i + 1}")


def test_repeated_call_is_stable():
    w = wl.make("mixed_append", seed=3, device="cuda")
    table, lens, _ = to_dev(w, "cuda")
    a = torch.empty_like(w.q)
    b = torch.empty_like(w.q)
    pkv.paged_decode_attention_no_alloc(w.q, w.k_pool, w.v_pool, table, lens, w.scale, a)
    pkv.paged_decode_attention_no_alloc(w.q, w.k_pool, w.v_pool, table, lens, w.scale, b)
    ref = _with_workspace(w, table, lens, pkv.VARIANT_AUTO)
    torch.cuda.synchronize()
    _close(a, ref, "call 1")
    _close(b, ref, "call 2")


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
