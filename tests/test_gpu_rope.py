"""Parity of the rotary embedding + KV append path (kv_append_rope and
paged_decode_step_rope) with the float64 oracle.

The oracle rounds the float64 rotation once to the storage format.  The GPU
forms the same double angle, reduces it exactly, and evaluates cos / sin and
the rotation in fp32 (relative error a few units of 2^-24) before the same
single rounding; the two differ only where the exact result lies within that
error of a rounding boundary.  So every element must agree to one unit in the
last place of its 16-bit format, and all but a small share (at most 1 in 200;
expected about 1 in 2000 for fp16 and 1 in 16000 for bf16) bit for bit.
Decode outputs use the tolerance of the other parity tests."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_decode_16_gb300 as pkv
from paged_kv_decode_16_gb300 import workloads as wl

from gpu_helpers import VARIANT_IDS, VARIANTS, assert_close, to_dev

pytestmark = pytest.mark.gpu


def assert_rounded_rows_equal(got_bits: np.ndarray, ref_bits: np.ndarray, what: str):
    g = got_bits.astype(np.int32)
    r = ref_bits.astype(np.int32)
    # adjacent patterns of the same sign are adjacent values: compare as integers
    same_sign = (g ^ r) & 0x8000 == 0
    diff = np.abs(g - r)
    assert np.all((diff <= 1) & (same_sign | (diff == 0)) |
                  ((g & 0x7FFF) == 0) & ((r & 0x7FFF) == 0)), f"{what}: beyond one ulp"
    mism = int(np.count_nonzero(diff))
    assert mism <= max(1, g.size // 200), f"{what}: {mism} of {g.size} differ in the last bit"


def _case(seed, dtype, D, B=6, Hq=8, Hkv=2, P=16):
    lens = np.random.default_rng(seed).integers(1, 300, size=B)
    w = wl.make_random(seed, batch=B, n_q_heads=Hq, n_kv_heads=Hkv, head_dim=D, page_size=P,
                       dtype=dtype, lens=lens, device="cuda")
    return w


@pytest.mark.parametrize("dtype,D,theta", [(torch.bfloat16, 128, 500000.0),
                                           (torch.float16, 128, 10000.0),
                                           (torch.float16, 64, 10000.0),
                                           (torch.bfloat16, 64, 1.0e6)])
def test_kv_append_rope_matches_oracle(dtype, D, theta):
    w = _case(31, dtype, D)
    table, lens, _ = to_dev(w)
    # positions: inside the sequence, zero, a padded slot, large angles
    pos_h = np.array([int(w.context_lens[0]) - 1, 0, -1, int(w.context_lens[3]) - 1, 5, 2],
                     dtype=np.int32)
    pos = torch.from_numpy(pos_h).cuda()
    pool = pkv.kv_pool_create(w.num_pages, w.page_size, w.n_kv_heads, w.head_dim, w.dtype,
                              w.k_pool, w.v_pool)
    before = (wl.to_bits(w.k_pool), wl.to_bits(w.v_pool))
    q_out = torch.empty_like(w.q)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.kv_append_rope(pool, w.q, w.k_new, w.v_new, table, pos, theta, q_out, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    dn = w.dtype_name
    q_ref = oracle.rope(wl.to_bits(w.q), pos_h, theta, dn)
    k_ref = oracle.rope(wl.to_bits(w.k_new), pos_h, theta, dn)
    kp_ref, vp_ref = oracle.kv_append(before[0], before[1], k_ref, wl.to_bits(w.v_new),
                                      w.page_table, pos_h)
    assert_rounded_rows_equal(wl.to_bits(q_out), q_ref, "rotated q")
    assert_rounded_rows_equal(wl.to_bits(w.k_pool), kp_ref, "k pool")
    assert np.array_equal(wl.to_bits(w.v_pool), vp_ref), "v pool (bit copy)"
    # position 0 leaves the row exactly as it was
    assert torch.equal(q_out[1].view(torch.int16), w.q[1].view(torch.int16))
    # in place (q_out is q) gives the same rows
    q2 = w.q.clone()
    pkv.kv_append_rope(pool, q2, w.k_new, w.v_new, table, pos, theta, q2)
    torch.cuda.synchronize()
    assert torch.equal(q2.view(torch.int16), q_out.view(torch.int16))
    pool.destroy()


@pytest.mark.parametrize("variant", VARIANTS, ids=VARIANT_IDS)
@pytest.mark.parametrize("name,theta", [("llama3_8b", 500000.0), ("mixed_append", 10000.0)])
def test_step_rope_matches_oracle(name, theta, variant):
    w = wl.make(name, seed=2, device="cuda", batch=12)
    table, lens, pos = to_dev(w)
    dn = w.dtype_name
    before = (wl.to_bits(w.k_pool), wl.to_bits(w.v_pool))
    ws = pkv.alloc_workspace(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, variant=variant)
    out = torch.full_like(w.q, float("nan"))
    q_keep = w.q.clone()
    pkv.paged_decode_step_rope(w.k_new, w.v_new, pos, w.q, w.k_pool, w.v_pool, table, lens,
                               w.scale, theta, out, ws, variant=variant)
    torch.cuda.synchronize()
    assert pkv.pkv_read_device_status(ws) == 0
    assert torch.equal(w.q.view(torch.int16), q_keep.view(torch.int16)), "q must stay as given"
    q_ref = oracle.rope(wl.to_bits(w.q), w.positions, theta, dn)
    k_ref = oracle.rope(wl.to_bits(w.k_new), w.positions, theta, dn)
    kp, vp = oracle.kv_append(before[0], before[1], k_ref, wl.to_bits(w.v_new), w.page_table,
                              w.positions)
    assert_rounded_rows_equal(wl.to_bits(w.k_pool), kp, "k pool")
    assert np.array_equal(wl.to_bits(w.v_pool), vp)
    ref = oracle.paged_decode(q_ref, kp, vp, w.page_table, w.context_lens, w.scale, dn)
    assert_close(out, ref, what=f"{name} rope step")


@pytest.mark.parametrize("variant", VARIANTS, ids=VARIANT_IDS)
def test_step_rope_equals_append_rope_then_attention(variant):
    """The fused step gives the bits of kv_append_rope followed by
    paged_decode_attention on the rotated queries (output and both pools)."""
    w1 = wl.make("llama3_8b", seed=5, device="cuda", batch=10)
    w2 = wl.make("llama3_8b", seed=5, device="cuda", batch=10)
    theta = 500000.0
    table, lens, pos = to_dev(w1)
    ws = pkv.alloc_workspace(w1.batch, w1.n_q_heads, w1.n_kv_heads, w1.head_dim, variant=variant)
    out1 = torch.empty_like(w1.q)
    pkv.paged_decode_step_rope(w1.k_new, w1.v_new, pos, w1.q, w1.k_pool, w1.v_pool, table, lens,
                               w1.scale, theta, out1, ws, variant=variant)
    pool = pkv.kv_pool_create(w2.num_pages, w2.page_size, w2.n_kv_heads, w2.head_dim, w2.dtype,
                              w2.k_pool, w2.v_pool)
    q_rot = torch.empty_like(w2.q)
    pkv.kv_append_rope(pool, w2.q, w2.k_new, w2.v_new, table, pos, theta, q_rot)
    out2 = torch.empty_like(w2.q)
    pkv.paged_decode_attention(q_rot, w2.k_pool, w2.v_pool, table, lens, w2.scale, out2, ws,
                               variant=variant)
    torch.cuda.synchronize()
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(w1.k_pool.view(torch.int16), w2.k_pool.view(torch.int16))
    assert torch.equal(w1.v_pool.view(torch.int16), w2.v_pool.view(torch.int16))
    pool.destroy()


def test_rope_rejects_bad_theta():
    w = _case(33, torch.bfloat16, 128)
    table, lens, pos = to_dev(w)
    pool = pkv.kv_pool_create(w.num_pages, w.page_size, w.n_kv_heads, w.head_dim, w.dtype,
                              w.k_pool, w.v_pool)
    for theta in (0.0, -5.0, float("nan"), float("inf")):
        with pytest.raises(pkv.PagedKVError) as e:
            pkv.kv_append_rope(pool, w.q, w.k_new, w.v_new, table, pos, theta,
                               torch.empty_like(w.q))
        assert e.value.name == "PKV_ERR_INVALID_ARG"
    pool.destroy()


def _norm_weights(dtype, D, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    wq = (1.0 + 0.3 * torch.randn(D, generator=g, device="cuda")).to(dtype)
    wk = (1.0 + 0.3 * torch.randn(D, generator=g, device="cuda")).to(dtype)
    return wq, wk


@pytest.mark.parametrize("sides", ["both", "q_only", "k_only"])
@pytest.mark.parametrize("dtype,D,theta", [(torch.bfloat16, 128, 1.0e6),
                                           (torch.float16, 128, 10000.0),
                                           (torch.float16, 64, 10000.0),
                                           (torch.bfloat16, 64, 500000.0)])
def test_kv_append_rope_norm_matches_oracle(dtype, D, theta, sides):
    """Per-head RMS norm (weights [D], eps 1e-6) before the rotation: rotated q
    and k rows within one ulp of the oracle's single rounding (bitwise for all
    but at most 1 in 200), v bit for bit."""
    w = _case(37, dtype, D)
    table, lens, _ = to_dev(w)
    pos_h = np.array([int(w.context_lens[0]) - 1, 0, -1, int(w.context_lens[3]) - 1, 5, 2],
                     dtype=np.int32)
    pos = torch.from_numpy(pos_h).cuda()
    wq, wk = _norm_weights(dtype, D, 38)
    qw = wq if sides != "k_only" else None
    kw = wk if sides != "q_only" else None
    eps = 1e-6
    pool = pkv.kv_pool_create(w.num_pages, w.page_size, w.n_kv_heads, w.head_dim, w.dtype,
                              w.k_pool, w.v_pool)
    before = (wl.to_bits(w.k_pool), wl.to_bits(w.v_pool))
    q_out = torch.empty_like(w.q)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.kv_append_rope(pool, w.q, w.k_new, w.v_new, table, pos, theta, q_out, dev_status=st,
                       q_norm_weight=qw, k_norm_weight=kw, norm_eps=eps)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    dn = w.dtype_name
    q_ref = (oracle.norm_rope(wl.to_bits(w.q), pos_h, wl.to_bits(qw), eps, theta, dn)
             if qw is not None else oracle.rope(wl.to_bits(w.q), pos_h, theta, dn))
    k_ref = (oracle.norm_rope(wl.to_bits(w.k_new), pos_h, wl.to_bits(kw), eps, theta, dn)
             if kw is not None else oracle.rope(wl.to_bits(w.k_new), pos_h, theta, dn))
    kp_ref, vp_ref = oracle.kv_append(before[0], before[1], k_ref, wl.to_bits(w.v_new),
                                      w.page_table, pos_h)
    assert_rounded_rows_equal(wl.to_bits(q_out), q_ref, "normalised rotated q")
    assert_rounded_rows_equal(wl.to_bits(w.k_pool), kp_ref, "k pool")
    assert np.array_equal(wl.to_bits(w.v_pool), vp_ref), "v pool (bit copy)"
    pool.destroy()


@pytest.mark.parametrize("variant", VARIANTS, ids=VARIANT_IDS)
def test_step_rope_norm_matches_oracle(variant):
    """paged_decode_step_rope with both norms: pools and attention output
    against the oracle's decode of the normalised, rotated q and k."""
    w = wl.make("llama3_8b", seed=3, device="cuda", batch=12)
    table, lens, pos = to_dev(w)
    dn = w.dtype_name
    theta, eps = 500000.0, 1e-6
    wq, wk = _norm_weights(w.dtype, w.head_dim, 39)
    before = (wl.to_bits(w.k_pool), wl.to_bits(w.v_pool))
    ws = pkv.alloc_workspace(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, variant=variant)
    out = torch.full_like(w.q, float("nan"))
    pkv.paged_decode_step_rope(w.k_new, w.v_new, pos, w.q, w.k_pool, w.v_pool, table, lens,
                               w.scale, theta, out, ws, variant=variant, q_norm_weight=wq,
                               k_norm_weight=wk, norm_eps=eps)
    torch.cuda.synchronize()
    assert pkv.pkv_read_device_status(ws) == 0
    q_ref = oracle.norm_rope(wl.to_bits(w.q), w.positions, wl.to_bits(wq), eps, theta, dn)
    k_ref = oracle.norm_rope(wl.to_bits(w.k_new), w.positions, wl.to_bits(wk), eps, theta, dn)
    kp, vp = oracle.kv_append(before[0], before[1], k_ref, wl.to_bits(w.v_new), w.page_table,
                              w.positions)
    assert_rounded_rows_equal(wl.to_bits(w.k_pool), kp, "k pool")
    assert np.array_equal(wl.to_bits(w.v_pool), vp)
    ref = oracle.paged_decode(q_ref, kp, vp, w.page_table, w.context_lens, w.scale, dn)
    assert_close(out, ref, what="rms-norm + rope step")
