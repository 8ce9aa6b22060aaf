"""Parity of the CUDA path (through the C ABI) with the float64 oracle."""
import itertools
import zlib

import numpy as np
import pytest
import torch

import oracle
import paged_kv_decode_16_gb300 as pkv
from paged_kv_decode_16_gb300 import workloads as wl
from gpu_helpers import VARIANT_IDS, VARIANTS, assert_close, oracle_full, run_gpu, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("variant", VARIANTS, ids=VARIANT_IDS)
@pytest.mark.parametrize("name", wl.NAMES)
def test_named_workload_matches_oracle(name, variant):
    w = wl.make(name, seed=0, device="cuda")
    before = (wl.to_bits(w.k_pool), wl.to_bits(w.v_pool))
    out, ws, status = run_gpu(w, variant=variant)
    assert status == 0
    # every output element against the oracle (under a second of oracle time
    # per workload on the host cores)
    ref = oracle_full(w, before)
    assert_close(out, ref, strict=True, what=name)
    if w.append:
        # the append itself is bit-exact against the oracle's
        kp, vp = oracle.kv_append(*before, wl.to_bits(w.k_new), wl.to_bits(w.v_new),
                                  w.page_table, w.positions)
        assert np.array_equal(kp, wl.to_bits(w.k_pool))
        assert np.array_equal(vp, wl.to_bits(w.v_pool))


GROUPS = [(4, 4), (4, 2), (12, 4), (8, 2), (14, 2), (16, 2), (32, 2), (9, 1), (20, 2), (6, 1)]
LENS = {
    "one": [1],
    "around_chunk": [15, 16, 17, 1, 31, 33],
    "around_page": [31, 32, 33, 64, 65, 2],
    "ragged": None,  # random in [1, 300], batch 13
}


def _sweep_cases():
    cases = []
    rng = np.random.default_rng(123)
    for dt, D, P in itertools.product((torch.bfloat16, torch.float16), (64, 128), (16, 32)):
        for (hq, hkv) in GROUPS:
            lens_name = list(LENS)[int(rng.integers(len(LENS)))]
            workers = [0, 1, 2, 3, 7, 1000][int(rng.integers(6))]
            cases.append((dt, D, P, hq, hkv, lens_name, workers))
    return cases


@pytest.mark.parametrize("variant", VARIANTS, ids=VARIANT_IDS)
@pytest.mark.parametrize("dt,D,P,hq,hkv,lens_name,workers", _sweep_cases())
def test_random_sweep(dt, D, P, hq, hkv, lens_name, workers, variant):
    seed = zlib.crc32(repr((str(dt), D, P, hq, hkv, lens_name, workers)).encode())
    lens = LENS[lens_name]
    if lens is None:
        lens = np.random.default_rng(seed).integers(1, 301, size=13)
    w = wl.make_random(seed, batch=len(lens), n_q_heads=hq, n_kv_heads=hkv, head_dim=D,
                       page_size=P, dtype=dt, lens=lens, device="cuda", poison=True)
    out, ws, status = run_gpu(w, num_workers=workers, append=False, variant=variant)
    assert status == 0
    ref = oracle_full(w, append=False)
    assert_close(out, ref, what=f"{dt} D{D} P{P} G{hq}/{hkv} {lens_name} w{workers} v{variant}")


@pytest.mark.parametrize("variant", VARIANTS, ids=VARIANT_IDS)
@pytest.mark.parametrize("workers", [1, 2, 3, 5, 64, 0])
def test_forced_worker_counts_agree(workers, variant):
    """Every split of the same batch matches the oracle (partials + combine)."""
    w = wl.make_random(7, batch=9, n_q_heads=32, n_kv_heads=8, head_dim=128, page_size=16,
                       dtype=torch.bfloat16, lens=[1, 16, 17, 100, 257, 600, 33, 48, 1000],
                       device="cuda", poison=True)
    out, ws, status = run_gpu(w, num_workers=workers, append=False, variant=variant)
    assert status == 0
    assert_close(out, oracle_full(w, append=False), what=f"workers={workers}")


@pytest.mark.parametrize("variant", VARIANTS, ids=VARIANT_IDS)
def test_long_sequence_split_many_ways(variant):
    w = wl.make_random(8, batch=2, n_q_heads=28, n_kv_heads=4, head_dim=128, page_size=32,
                       dtype=torch.float16, lens=[20000, 3], device="cuda", poison=True)
    ref = oracle_full(w, append=False)
    for workers in (0, 97, 500):
        out, _, status = run_gpu(w, num_workers=workers, append=False, variant=variant)
        assert status == 0
        assert_close(out, ref, what=f"workers={workers}")


@pytest.mark.parametrize("variant", VARIANTS, ids=VARIANT_IDS)
def test_page_permutation_is_bitwise_invariant(variant):
    """Same dense cache under two page permutations -> identical bits."""
    rng = np.random.default_rng(5)
    B, Hq, Hkv, D, P = 6, 16, 4, 128, 16
    lens = np.array([40, 1, 300, 17, 64, 129])
    dense_k = wl.to_bits(torch.randn(B, Hkv, 300, D).to(torch.bfloat16))
    dense_v = wl.to_bits(torch.randn(B, Hkv, 300, D).to(torch.bfloat16))
    q = torch.randn(B, Hq, D).to(torch.bfloat16).cuda()
    outs = []
    for seed in (1, 2):
        kp, vp, table = wl.scatter_dense(dense_k, dense_v, lens, P, np.random.default_rng(seed),
                                         extra_pages=5, fill=0x7FC0)
        kt = torch.from_numpy(kp.view(np.int16)).view(torch.bfloat16).cuda()
        vt = torch.from_numpy(vp.view(np.int16)).view(torch.bfloat16).cuda()
        out = torch.empty_like(q)
        ws = pkv.alloc_workspace(B, Hq, Hkv, D, 37, variant=variant)
        pkv.paged_decode_attention(q, kt, vt, torch.from_numpy(table).cuda(),
                                   torch.from_numpy(lens.astype(np.int32)).cuda(), 0.088, out, ws,
                                   num_workers=37, variant=variant)
        outs.append(out.cpu())
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    del rng


def test_shared_prefix_equals_private_copies_bitwise():
    w = wl.make("prefix_sharing", seed=3, device="cuda", batch=6)
    table, lens, _ = to_dev(w)
    n_prefix = w.prefix_len // w.page_size
    # give every sequence private copies of the prefix pages
    extra = w.batch * n_prefix
    kp = torch.cat([w.k_pool, w.k_pool.new_empty((extra,) + tuple(w.k_pool.shape[1:]))])
    vp = torch.cat([w.v_pool, w.v_pool.new_empty((extra,) + tuple(w.v_pool.shape[1:]))])
    priv = w.page_table.copy()
    for b in range(w.batch):
        for j in range(n_prefix):
            new_id = w.num_pages + b * n_prefix + j
            kp[new_id] = w.k_pool[w.page_table[b, j]]
            vp[new_id] = w.v_pool[w.page_table[b, j]]
            priv[b, j] = new_id
    out_shared = torch.empty_like(w.q)
    out_priv = torch.empty_like(w.q)
    ws = pkv.alloc_workspace(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim)
    pkv.paged_decode_attention(w.q, w.k_pool, w.v_pool, table, lens, w.scale, out_shared, ws)
    pkv.paged_decode_attention(w.q, kp, vp, torch.from_numpy(priv).cuda(), lens, w.scale,
                               out_priv, ws)
    assert torch.equal(out_shared.view(torch.int16), out_priv.view(torch.int16))


@pytest.mark.parametrize("variant", VARIANTS, ids=VARIANT_IDS)
def test_rerun_is_bitwise_deterministic(variant):
    w = wl.make("mixed_append", seed=2, device="cuda", batch=40)
    a, _, _ = run_gpu(w, append=False, variant=variant)
    b, _, _ = run_gpu(w, append=False, variant=variant)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_variants_agree_with_each_other():
    """The two decode kernels differ only by rounding (P in the input dtype on
    the tensor-core path): on the same inputs they agree within the tolerance."""
    w = wl.make("llama3_8b", seed=9, device="cuda", batch=12)
    a, _, sa = run_gpu(w, append=False, variant=pkv.VARIANT_CUDA_CORES)
    b, _, sb = run_gpu(w, append=False, variant=pkv.VARIANT_TENSOR_CORES)
    assert sa == 0 and sb == 0
    assert_close(a, b.float().cpu().numpy().astype(np.float64), strict=True)


def test_append_then_gather_is_bit_exact():
    for dt, D, P in ((torch.float16, 128, 32), (torch.bfloat16, 64, 16)):
        w = wl.make_random(11, batch=7, n_q_heads=8, n_kv_heads=2, head_dim=D, page_size=P,
                           dtype=dt, lens=[1, 16, 17, 33, 64, 100, 2], device="cuda")
        w.positions[3] = -1  # padded slot: must not write
        table, lens, pos = to_dev(w)
        before = (wl.to_bits(w.k_pool), wl.to_bits(w.v_pool))
        pool = pkv.kv_pool_create(w.num_pages, P, 2, D, dt, w.k_pool, w.v_pool)
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        pkv.kv_append(pool, w.k_new, w.v_new, table, pos, dev_status=st)
        kp, vp = oracle.kv_append(*before, wl.to_bits(w.k_new), wl.to_bits(w.v_new), w.page_table,
                                  w.positions)
        assert np.array_equal(wl.to_bits(w.k_pool), kp)
        assert np.array_equal(wl.to_bits(w.v_pool), vp)
        Lmax = int(w.context_lens.max())
        ko = torch.zeros(7, 2, Lmax, D, dtype=dt, device="cuda")
        vo = torch.zeros_like(ko)
        pkv.kv_gather(pool, table, lens, Lmax, ko, vo, dev_status=st)
        assert int(st.item()) == 0
        gk = oracle.gather(kp, w.page_table, w.context_lens, Lmax)
        gv = oracle.gather(vp, w.page_table, w.context_lens, Lmax)
        assert np.array_equal(wl.to_bits(ko), gk)
        assert np.array_equal(wl.to_bits(vo), gv)
        pool.destroy()


@pytest.mark.parametrize("variant", VARIANTS, ids=VARIANT_IDS)
def test_empty_sequences_give_zeros(variant):
    w = wl.make_random(13, batch=4, n_q_heads=8, n_kv_heads=2, head_dim=128, page_size=16,
                       dtype=torch.bfloat16, lens=[0, 5, 0, 40], device="cuda", poison=True)
    for workers in (0, 1, 3):
        out, _, status = run_gpu(w, num_workers=workers, append=False, variant=variant)
        assert status == 0
        assert_close(out, oracle_full(w, append=False))
        assert (out[0] == 0).all() and (out[2] == 0).all()


@pytest.mark.parametrize("variant", VARIANTS, ids=VARIANT_IDS)
def test_bad_page_id_is_flagged_and_skipped(variant):
    w = wl.make_random(17, batch=3, n_q_heads=8, n_kv_heads=2, head_dim=128, page_size=16,
                       dtype=torch.bfloat16, lens=[40, 20, 33], device="cuda")
    good = oracle_full(w, append=False)
    w.page_table[1, 0] = w.num_pages + 5  # outside the pool
    w.page_table[2, 1] = -3
    out, ws, status = run_gpu(w, append=False, variant=variant)
    assert status & pkv.DEV_BAD_PAGE
    got = out.float().cpu().numpy().astype(np.float64)
    assert_close(got[0], good[0], what="untouched sequence")
    assert np.isfinite(got).all()


def test_length_beyond_table_is_flagged_and_clamped():
    w = wl.make_random(19, batch=2, n_q_heads=4, n_kv_heads=4, head_dim=64, page_size=16,
                       dtype=torch.float16, lens=[20, 32], device="cuda")
    ref = oracle_full(w, append=False)
    w.context_lens[0] = 10_000  # table row holds 2 pages -> clamped to 32 tokens
    out, ws, status = run_gpu(w, append=False)
    assert status & pkv.DEV_BAD_LEN
    assert_close(out[1:], ref[1:])
    assert np.isfinite(out.float().cpu().numpy()).all()


@pytest.mark.parametrize("variant", VARIANTS, ids=VARIANT_IDS)
def test_guard_bands_untouched(variant):
    """Canaries around out and past the end of the workspace stay intact."""
    w = wl.make("tiny", seed=1, device="cuda")
    table, lens, _ = to_dev(w)
    n = w.q.numel()
    big = torch.full((n + 2048,), 7.0, dtype=w.dtype, device="cuda")
    out = big[1024:1024 + n].view_as(w.q)
    need = pkv.paged_decode_workspace_size(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, 3,
                                           variant)
    wsbig = torch.full((need + 4096,), 0xA5, dtype=torch.uint8, device="cuda")
    ws = wsbig[:need]
    pkv.paged_decode_attention(w.q, w.k_pool, w.v_pool, table, lens, w.scale, out, ws,
                               num_workers=3, variant=variant)
    torch.cuda.synchronize()
    assert (big[:1024] == 7.0).all() and (big[1024 + n:] == 7.0).all()
    assert (wsbig[need:] == 0xA5).all()
    assert_close(out, oracle_full(w, append=False), strict=True)


def test_workspace_too_small_is_rejected():
    w = wl.make("tiny", seed=1, device="cuda")
    table, lens, _ = to_dev(w)
    need = pkv.paged_decode_workspace_size(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim)
    ws = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(pkv.PagedKVError) as e:
        pkv.paged_decode_attention(w.q, w.k_pool, w.v_pool, table, lens, w.scale,
                                   torch.empty_like(w.q), ws)
    assert e.value.name == "PKV_ERR_WORKSPACE"


@pytest.mark.parametrize("variant", VARIANTS, ids=VARIANT_IDS)
@pytest.mark.parametrize("case", ["llama3_8b", "mixed_append", "with_empty", "long_split"])
def test_split_steps_equal_fused_call(case, variant):
    """plan + run (merge in the decode kernel) and plan + run + combine, called
    one by one, both equal paged_decode_attention bit for bit; rows of empty
    sequences are zeros either way."""
    if case == "with_empty":
        w = wl.make_random(21, batch=7, n_q_heads=16, n_kv_heads=4, head_dim=128, page_size=16,
                           dtype=torch.bfloat16, lens=[0, 3000, 0, 17, 900, 0, 4500],
                           device="cuda")
    elif case == "long_split":  # one unit over many workers: more than 32 segments
        w = wl.make_random(22, batch=1, n_q_heads=16, n_kv_heads=1, head_dim=128, page_size=16,
                           dtype=torch.bfloat16, lens=[60000], device="cuda")
    else:
        w = wl.make(case, seed=4, device="cuda", batch=8 if case == "llama3_8b" else 40)
    table, lens, _ = to_dev(w)
    ws = pkv.alloc_workspace(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, variant=variant)
    a = torch.full_like(w.q, float("nan"))
    pkv.paged_decode_attention(w.q, w.k_pool, w.v_pool, table, lens, w.scale, a, ws,
                               variant=variant)
    outs = []
    for merge in (True, False):
        b = torch.full_like(w.q, float("nan"))
        pkv.paged_decode_plan(lens, w.n_q_heads, w.n_kv_heads, w.head_dim, w.page_size,
                              table.shape[1], ws, variant=variant)
        pkv.paged_decode_run(w.q, w.k_pool, w.v_pool, table, w.scale, b, ws, variant=variant,
                             merge=merge)
        if not merge:
            pkv.paged_decode_combine(b, w.n_kv_heads, ws, variant=variant)
        outs.append(b)
    torch.cuda.synchronize()
    for b in outs:
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    empty = torch.from_numpy(np.asarray(w.context_lens) == 0)
    if empty.any():
        assert torch.count_nonzero(a[empty.cuda()].float()) == 0
    assert pkv.pkv_read_device_status(ws) == 0
    if case == "long_split":
        assert_close(a, oracle_full(w), what="one sequence over many workers")


def test_pool_owned_memory_roundtrip():
    pool = pkv.kv_pool_create(64, 16, 2, 128, torch.bfloat16)
    assert pool.k_ptr() and pool.v_ptr() and pool.k_ptr() != pool.v_ptr()
    ids = pool.alloc_pages(10)
    assert len(set(ids)) == 10 and pool.free_count() == 54
    pool.release_pages(ids)
    assert pool.free_count() == 64
    pool.destroy()


def test_fused_step_equals_append_then_attention():
    """paged_decode_step == kv_append + paged_decode_attention, bit for bit
    (output and both pools), and matches the oracle."""
    w1 = wl.make("mixed_append", seed=6, device="cuda", batch=48)
    w2 = wl.make("mixed_append", seed=6, device="cuda", batch=48)
    before = (wl.to_bits(w1.k_pool), wl.to_bits(w1.v_pool))
    out1, _, st1 = run_gpu(w1)  # separate calls
    assert st1 == 0
    table, lens, pos = to_dev(w2)
    out2 = torch.empty_like(w2.q)
    ws = pkv.alloc_workspace(w2.batch, w2.n_q_heads, w2.n_kv_heads, w2.head_dim)
    pkv.paged_decode_step(w2.k_new, w2.v_new, pos, w2.q, w2.k_pool, w2.v_pool, table, lens,
                          w2.scale, out2, ws)
    torch.cuda.synchronize()
    assert pkv.pkv_read_device_status(ws) == 0
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(w1.k_pool.view(torch.int16), w2.k_pool.view(torch.int16))
    assert torch.equal(w1.v_pool.view(torch.int16), w2.v_pool.view(torch.int16))
    assert_close(out2, oracle_full(w2, before), strict=True)


def test_fused_step_reports_bad_append_and_skips_padding():
    w = wl.make_random(21, batch=4, n_q_heads=8, n_kv_heads=2, head_dim=128, page_size=16,
                       dtype=torch.bfloat16, lens=[5, 17, 40, 3], device="cuda")
    before = (wl.to_bits(w.k_pool), wl.to_bits(w.v_pool))
    w.positions[1] = -1                        # padded slot: no write
    w.positions[2] = w.page_table.shape[1] * 16 + 3  # beyond the table row: flagged, skipped
    table, lens, pos = to_dev(w)
    out = torch.empty_like(w.q)
    ws = pkv.alloc_workspace(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim)
    pkv.paged_decode_step(w.k_new, w.v_new, pos, w.q, w.k_pool, w.v_pool, table, lens, w.scale,
                          out, ws)
    torch.cuda.synchronize()
    assert pkv.pkv_read_device_status(ws) & pkv.DEV_BAD_LEN
    pos_ok = w.positions.copy()
    pos_ok[2] = -1
    kp, vp = oracle.kv_append(*before, wl.to_bits(w.k_new), wl.to_bits(w.v_new), w.page_table,
                              pos_ok)
    assert np.array_equal(wl.to_bits(w.k_pool), kp) and np.array_equal(wl.to_bits(w.v_pool), vp)
    # a clean call on the same workspace clears the status
    pkv.paged_decode_step(w.k_new, w.v_new, torch.from_numpy(pos_ok).cuda(), w.q, w.k_pool,
                          w.v_pool, table, lens, w.scale, out, ws)
    torch.cuda.synchronize()
    assert pkv.pkv_read_device_status(ws) == 0


@pytest.mark.parametrize("variant", VARIANTS, ids=VARIANT_IDS)
def test_step_captured_in_cuda_graph_equals_eager(variant):
    """paged_decode_step recorded into a CUDA graph (input copy, the three
    launches, output copy) and replayed twice gives the eager call's bits, and
    the replays pick up new inputs written into the same buffers."""
    w = wl.make("mixed_append", seed=8, device="cuda", batch=24)
    table, lens, pos = to_dev(w)
    ws = pkv.alloc_workspace(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, variant=variant)
    k0, v0 = w.k_pool.clone(), w.v_pool.clone()
    q_in = w.q.clone()
    eager = torch.empty_like(w.q)
    pkv.paged_decode_step(w.k_new, w.v_new, pos, q_in, w.k_pool, w.v_pool, table, lens, w.scale,
                          eager, ws, variant=variant)
    torch.cuda.synchronize()
    w.k_pool.copy_(k0)
    w.v_pool.copy_(v0)
    out = torch.full_like(w.q, float("nan"))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            pkv.paged_decode_step(w.k_new, w.v_new, pos, q_in, w.k_pool, w.v_pool, table, lens,
                                  w.scale, out, ws, variant=variant)
    torch.cuda.current_stream().wait_stream(s)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
    # new queries in the same buffer: the replay must see them
    q_in.mul_(-1.0)
    g.replay()
    torch.cuda.synchronize()
    ref = torch.empty_like(w.q)
    pkv.paged_decode_attention(q_in, w.k_pool, w.v_pool, table, lens, w.scale, ref,
                               pkv.alloc_workspace(w.batch, w.n_q_heads, w.n_kv_heads,
                                                   w.head_dim, variant=variant),
                               variant=variant)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert pkv.pkv_read_device_status(ws) == 0


def test_bounded_wait_gives_up_and_the_context_stays_usable():
    """The give-up path of the copy waits: a wait on an mbarrier that nothing
    completes ends after its polls with PKV_DEV_TIMEOUT (no trap, no hang),
    the wait's length grows with the poll count, and decoding right after it
    on the same context is correct."""
    st, ns_short = pkv.check_bounded_wait(1000)
    assert st == pkv.DEV_TIMEOUT
    st, ns_long = pkv.check_bounded_wait(20000)
    assert st == pkv.DEV_TIMEOUT
    assert 0 < ns_short < ns_long < 5_000_000_000
    with pytest.raises(pkv.PagedKVError) as e:
        pkv.check_bounded_wait(0)
    assert e.value.name == "PKV_ERR_INVALID_ARG"
    w = wl.make("tiny", seed=9, device="cuda")
    out, ws, status = run_gpu(w, append=False)
    assert status == 0
    assert_close(out, oracle_full(w, append=False), strict=True, what="after the timeout check")


@pytest.mark.parametrize("variant", VARIANTS, ids=VARIANT_IDS)
def test_batch_beyond_the_plans_shared_memory(variant):
    """5000 sequences (lengths 0..59): the plan's prefix sums no longer fit its
    shared memory (4096 sequences) and are searched in global memory; the
    fused step's append CTAs each take many sequences."""
    rng = np.random.default_rng(55)
    lens = rng.integers(0, 60, size=5000)
    w = wl.make_random(55, batch=5000, n_q_heads=8, n_kv_heads=2, head_dim=64, page_size=16,
                       dtype=torch.float16, lens=lens, device="cuda", poison=True)
    out, ws, status = run_gpu(w, append=False, variant=variant)
    assert status == 0
    assert_close(out, oracle_full(w, append=False), what="B=5000 decode")
    # the fused step: append at L - 1 (sequences with L = 0 skip), then attention
    before = (wl.to_bits(w.k_pool), wl.to_bits(w.v_pool))
    table, lens_d, pos = to_dev(w)
    out2 = torch.full_like(w.q, float("nan"))
    pkv.paged_decode_step(w.k_new, w.v_new, pos, w.q, w.k_pool, w.v_pool, table, lens_d,
                          w.scale, out2, ws, variant=variant)
    torch.cuda.synchronize()
    assert pkv.pkv_read_device_status(ws) == 0
    assert_close(out2, oracle_full(w, before, append=True), what="B=5000 step")


@pytest.mark.parametrize("variant", VARIANTS, ids=VARIANT_IDS)
@pytest.mark.parametrize("P", [64, 256])
def test_large_pages(P, variant):
    """Pages of 64 and 256 tokens (a 16-token chunk is one slice of a page):
    decode and the fused step against the oracle."""
    rng = np.random.default_rng(60 + P)
    lens = rng.integers(1, 2000, size=9)
    w = wl.make_random(60 + P, batch=9, n_q_heads=16, n_kv_heads=4, head_dim=128, page_size=P,
                       dtype=torch.bfloat16, lens=lens, device="cuda", poison=True)
    out, ws, status = run_gpu(w, append=False, variant=variant)
    assert status == 0
    assert_close(out, oracle_full(w, append=False), what=f"P={P} decode")
    before = (wl.to_bits(w.k_pool), wl.to_bits(w.v_pool))
    table, lens_d, pos = to_dev(w)
    out2 = torch.full_like(w.q, float("nan"))
    pkv.paged_decode_step(w.k_new, w.v_new, pos, w.q, w.k_pool, w.v_pool, table, lens_d,
                          w.scale, out2, ws, variant=variant)
    torch.cuda.synchronize()
    assert pkv.pkv_read_device_status(ws) == 0
    assert_close(out2, oracle_full(w, before, append=True), what=f"P={P} step")


@pytest.mark.parametrize("variant", VARIANTS, ids=VARIANT_IDS)
@pytest.mark.parametrize("hq,hkv,d", [(64, 4, 128), (32, 4, 64), (24, 8, 128)],
                         ids=["rows16", "rows8_d64", "rows3"])
def test_kernel_merge_equals_combine_few_segments(hq, hkv, d, variant):
    """The decode kernel's merge (rows of a unit four at a time) and the combine
    kernel give the same bits for units of 3, 8 and 16 rows split over a few
    workers (at most 32 segments each), and both match the oracle."""
    rng = np.random.default_rng(80 + hq + d)
    lens = rng.integers(300, 4000, size=6)
    w = wl.make_random(80 + hq + d, batch=6, n_q_heads=hq, n_kv_heads=hkv, head_dim=d,
                       page_size=16, dtype=torch.bfloat16, lens=lens, device="cuda")
    table, lens_d, _ = to_dev(w)
    nw = 50
    ws = pkv.alloc_workspace(w.batch, hq, hkv, d, num_workers=nw, variant=variant)
    outs = []
    for merge in (True, False):
        o = torch.full_like(w.q, float("nan"))
        pkv.paged_decode_plan(lens_d, hq, hkv, d, w.page_size, table.shape[1], ws,
                              num_workers=nw, variant=variant)
        pkv.paged_decode_run(w.q, w.k_pool, w.v_pool, table, w.scale, o, ws, num_workers=nw,
                             variant=variant, merge=merge)
        if not merge:
            pkv.paged_decode_combine(o, hkv, ws, num_workers=nw, variant=variant)
        torch.cuda.synchronize()
        assert pkv.pkv_read_device_status(ws) == 0
        outs.append(o)
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    assert_close(outs[0], oracle_full(w), what=f"{hq}/{hkv} heads, D={d}, kernel merge")
