"""Parity of the shared-prefix decode (paged_decode_attention_prefix) with the
float64 oracle, which attends every sequence over all of its tokens the plain
way: the cascade (prefix once for all queries, then each suffix, then the merge
of the two partial states) must give the same attention within the decode
tolerance.  Also its device checks: rows that do not start with the shared
pages, lengths shorter than the prefix, and bad arguments."""
import numpy as np
import pytest
import torch

import paged_kv_decode_16_gb300 as pkv
from paged_kv_decode_16_gb300 import workloads as wl

from gpu_helpers import VARIANT_IDS, VARIANTS, assert_close, oracle_full, to_dev

pytestmark = pytest.mark.gpu


def _shared(seed, *, B, Hq, Hkv, D, P, dtype, prefix, suffix_max, poison=False):
    rng = np.random.default_rng(seed)
    lens = prefix + rng.integers(0, suffix_max + 1, size=B)
    return wl.build("shared", batch=B, n_q_heads=Hq, n_kv_heads=Hkv, head_dim=D, page_size=P,
                    dtype=dtype, context_lens=lens, rng=rng, seed=seed, device="cuda",
                    prefix_len=prefix, num_pages=None, poison=poison)


def _run(w, prefix, variant, num_workers=0):
    table, lens, _ = to_dev(w)
    ws = pkv.alloc_prefix_workspace(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, num_workers,
                                    variant=variant)
    out = torch.full_like(w.q, float("nan"))
    pkv.paged_decode_attention_prefix(w.q, w.k_pool, w.v_pool, table, lens, w.scale, prefix,
                                      out, ws, num_workers=num_workers, variant=variant)
    torch.cuda.synchronize()
    return out, ws


@pytest.mark.parametrize("variant", VARIANTS, ids=VARIANT_IDS)
def test_prefix_sharing_workload_matches_oracle(variant):
    w = wl.make("prefix_sharing", seed=0, device="cuda", poison=True)
    out, ws = _run(w, w.prefix_len, variant)
    assert pkv.pkv_read_device_status(ws) == 0
    assert_close(out, oracle_full(w), strict=True, what="prefix_sharing")


CASES = [
    # B, Hq, Hkv, D, P, dtype, prefix, suffix_max
    (1, 8, 2, 128, 16, torch.bfloat16, 160, 40),
    (3, 12, 3, 128, 16, torch.bfloat16, 512, 300),     # odd batch
    (5, 28, 4, 128, 32, torch.float16, 256, 700),      # group 7
    (6, 16, 16, 64, 16, torch.float16, 96, 0),         # no suffixes at all, group 1
    (9, 32, 8, 64, 32, torch.bfloat16, 1024, 2000),
    (7, 28, 1, 128, 16, torch.float16, 64, 100),       # group 28: tiles of 4 sequences
    (40, 28, 4, 128, 32, torch.bfloat16, 96, 33),      # group 7: three tiles, the last partial
]


@pytest.mark.parametrize("variant", VARIANTS, ids=VARIANT_IDS)
@pytest.mark.parametrize("case", range(len(CASES)))
def test_random_shared_prefixes_match_oracle(case, variant):
    B, Hq, Hkv, D, P, dtype, prefix, suffix_max = CASES[case]
    w = _shared(100 + case, B=B, Hq=Hq, Hkv=Hkv, D=D, P=P, dtype=dtype, prefix=prefix,
                suffix_max=suffix_max, poison=True)
    for nw in (0, 7):
        out, ws = _run(w, prefix, variant, num_workers=nw)
        assert pkv.pkv_read_device_status(ws) == 0
        assert_close(out, oracle_full(w), what=f"case {case} workers {nw}")


def test_prefix_equals_plain_decode_within_tolerance():
    """The same batch through paged_decode_attention (prefix re-read per row)."""
    w = _shared(7, B=16, Hq=32, Hkv=8, D=128, P=16, dtype=torch.bfloat16, prefix=1024,
                suffix_max=256)
    out, _ = _run(w, 1024, pkv.VARIANT_AUTO)
    table, lens, _ = to_dev(w)
    plain = torch.empty_like(w.q)
    pkv.paged_decode_attention(w.q, w.k_pool, w.v_pool, table, lens, w.scale, plain,
                               pkv.alloc_workspace(w.batch, w.n_q_heads, w.n_kv_heads,
                                                   w.head_dim))
    torch.cuda.synchronize()
    assert_close(out, plain.float().cpu().numpy().astype(np.float64), what="prefix vs plain")


def test_row_without_the_shared_pages_is_reported():
    w = _shared(8, B=4, Hq=8, Hkv=2, D=128, P=16, dtype=torch.bfloat16, prefix=64,
                suffix_max=50)
    w.page_table[2, 1] = w.page_table[2, 3] if w.page_table.shape[1] > 3 else 0
    _, ws = _run(w, 64, pkv.VARIANT_AUTO)
    assert pkv.pkv_read_device_status(ws) & pkv.DEV_BAD_PREFIX


@pytest.mark.parametrize("variant", VARIANTS, ids=VARIANT_IDS)
def test_bad_prefix_page_is_skipped_and_reported(variant):
    """A page id outside the pool inside the shared prefix (the same in every
    row, so the rows still share it): the prefix pass skips that chunk and
    flags PKV_DEV_BAD_PAGE, like the plain decode, whose output it then
    matches (both attend every token but those 16)."""
    w = _shared(31, B=4, Hq=8, Hkv=2, D=128, P=16, dtype=torch.bfloat16, prefix=64,
                suffix_max=40)
    w.page_table[:, 1] = w.num_pages + 3
    out, ws = _run(w, 64, variant)
    assert pkv.pkv_read_device_status(ws) & pkv.DEV_BAD_PAGE
    table, lens, _ = to_dev(w)
    plain = torch.full_like(w.q, float("nan"))
    wsp = pkv.alloc_workspace(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, variant=variant)
    pkv.paged_decode_attention(w.q, w.k_pool, w.v_pool, table, lens, w.scale, plain, wsp,
                               variant=variant)
    torch.cuda.synchronize()
    assert pkv.pkv_read_device_status(wsp) & pkv.DEV_BAD_PAGE
    assert_close(out, plain.float().cpu().numpy().astype(np.float64), what="bad prefix page")


def test_length_shorter_than_prefix_is_reported():
    w = _shared(9, B=3, Hq=8, Hkv=2, D=128, P=16, dtype=torch.bfloat16, prefix=64,
                suffix_max=50)
    table, lens, _ = to_dev(w)
    lens[1] = 32
    ws = pkv.alloc_prefix_workspace(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim)
    pkv.paged_decode_attention_prefix(w.q, w.k_pool, w.v_pool, table, lens, w.scale, 64,
                                      torch.empty_like(w.q), ws)
    torch.cuda.synchronize()
    assert pkv.pkv_read_device_status(ws) & pkv.DEV_BAD_LEN


def test_prefix_argument_checks():
    w = _shared(10, B=2, Hq=8, Hkv=2, D=128, P=16, dtype=torch.bfloat16, prefix=64,
                suffix_max=20)
    table, lens, _ = to_dev(w)
    ws = pkv.alloc_prefix_workspace(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim)
    for bad in (0, 24, -16, 16 * (table.shape[1] + 1)):
        with pytest.raises(pkv.PagedKVError) as e:
            pkv.paged_decode_attention_prefix(w.q, w.k_pool, w.v_pool, table, lens, w.scale, bad,
                                              torch.empty_like(w.q), ws)
        assert e.value.name == "PKV_ERR_INVALID_ARG"
    with pytest.raises(pkv.PagedKVError) as e:
        pkv.paged_decode_attention_prefix(w.q, w.k_pool, w.v_pool, table, lens, w.scale, 64,
                                          torch.empty_like(w.q), ws[:1024])
    assert e.value.name == "PKV_ERR_WORKSPACE"


def test_prefix_captured_in_cuda_graph_equals_eager():
    """paged_decode_attention_prefix (four launches) recorded into a CUDA graph
    and replayed gives the eager call's bits."""
    w = _shared(11, B=12, Hq=32, Hkv=8, D=128, P=16, dtype=torch.bfloat16, prefix=512,
                suffix_max=300)
    eager, ws = _run(w, 512, pkv.VARIANT_AUTO)
    table, lens, _ = to_dev(w)
    out = torch.full_like(w.q, float("nan"))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            pkv.paged_decode_attention_prefix(w.q, w.k_pool, w.v_pool, table, lens, w.scale, 512,
                                              out, ws)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(2):
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
    assert pkv.pkv_read_device_status(ws) == 0
