"""Pins of the float64 oracle to facts outside the oracle itself.

Each ``check_*`` takes a loaded oracle (``oracle.Oracle``) and raises if the
oracle disagrees with something fixed by the pages' definition or by
mathematics: hand-derived worked examples (tests/golden/), closed forms,
invariants of the definition, library routines (numpy / torch dtype
conversion, torch scaled_dot_product_attention in float64) and brute force.
``tests/test_oracle.py`` runs them on the oracle; ``tests/test_oracle_mutations.py``
runs them on deliberately broken copies of the oracle to show that a plausible
mistake anywhere in it fails at least one of them.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

from paged_kv_decode_16_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "worked_examples.json")
NAN_BITS = {"f16": 0x7E00, "bf16": 0x7FC0}
TORCH_DT = {"f16": torch.float16, "bf16": torch.bfloat16}


def bits_of(values, dtype: str) -> np.ndarray:
    """Round float values to the dtype (library conversion) and return bit patterns."""
    t = torch.as_tensor(np.asarray(values, dtype=np.float64)).to(TORCH_DT[dtype])
    return t.view(torch.int16).numpy().view(np.uint16)


def values_of(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Library decode of bit patterns (numpy float16 / torch bfloat16) to float64."""
    if dtype == "f16":
        return bits.view(np.float16).astype(np.float64)
    return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()


def _rand_bits(rng, shape, dtype, scale=1.0):
    return bits_of(rng.standard_normal(shape) * scale, dtype)


def _sdpa(q, k, v, scale):
    """torch scaled_dot_product_attention in float64 (library routine)."""
    return torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v), scale=scale).numpy()


# ---------------------------------------------------------------------------
def check_decode_f16_all_patterns(orc):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = orc.decode_bits(bits, "f16")
    ref = values_of(bits, "f16")
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # signed zeros keep their sign
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def check_decode_bf16_all_patterns(orc):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = orc.decode_bits(bits, "bf16")
    ref = values_of(bits, "bf16")
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def _golden_case(case):
    dt = case["dtype"]
    B, Hq, Hkv, D, P = (case[k] for k in ("batch", "n_q_heads", "n_kv_heads", "head_dim",
                                            "page_size"))
    NP = case["num_pages"]
    table = np.array(case["page_table"], dtype=np.int32)
    lens = np.array(case["context_lens"], dtype=np.int32)
    kpool = np.full((NP, Hkv, P, D), NAN_BITS[dt], dtype=np.uint16)
    vpool = kpool.copy()
    dk = np.array(case["dense_k"], dtype=np.float64)
    dv = np.array(case["dense_v"], dtype=np.float64)
    for b in range(B):
        for t in range(int(lens[b])):
            pg, sl = table[b, t // P], t % P
            kpool[pg, :, sl, :] = bits_of(dk[b, :, t, :], dt)
            vpool[pg, :, sl, :] = bits_of(dv[b, :, t, :], dt)
    q = bits_of(np.array(case["q"], dtype=np.float64), dt)
    scale = float(eval(case["scale"], {"log": math.log}))
    return q, kpool, vpool, table, lens, scale, dt


def check_golden_worked_examples(orc):
    with open(GOLDEN) as f:
        cases = json.load(f)["cases"]
    assert cases
    for case in cases:
        q, kp, vp, table, lens, scale, dt = _golden_case(case)
        out = orc.paged_decode(q, kp, vp, table, lens, scale, dt)
        exp = np.array(case["expected"], dtype=np.float64)
        err = np.abs(out - exp).max()
        assert err <= case["atol"], (case["name"], out, exp)


def check_dense_vs_sdpa(orc):
    """Oracle on a permuted paged pool == torch SDPA (float64) on the dense cache,
    GQA expanded by repeating each KV head over its consecutive query heads."""
    rng = np.random.default_rng(11)
    for dt in ("f16", "bf16"):
        for (Hq, Hkv) in ((1, 1), (4, 2), (8, 2), (7, 1), (6, 3)):
            for D, P in ((8, 2), (64, 16), (16, 4)):
                B = 3
                lens = np.array([1, P + 1, 3 * P + rng.integers(0, P)], dtype=np.int64)
                Lmax = int(lens.max())
                dk = _rand_bits(rng, (B, Hkv, Lmax, D), dt)
                dv = _rand_bits(rng, (B, Hkv, Lmax, D), dt)
                kp, vp, table = wl.scatter_dense(dk, dv, lens, P, rng, extra_pages=2,
                                                 fill=NAN_BITS[dt])
                q = _rand_bits(rng, (B, Hq, D), dt)
                scale = 1.0 / math.sqrt(D)
                out = orc.paged_decode(q, kp, vp, table, lens, scale, dt)
                G = Hq // Hkv
                for b in range(B):
                    L = int(lens[b])
                    kk = np.repeat(values_of(dk[b, :, :L], dt), G, axis=0)  # [Hq, L, D]
                    vv = np.repeat(values_of(dv[b, :, :L], dt), G, axis=0)
                    qq = values_of(q[b], dt)[:, None, :]                     # [Hq, 1, D]
                    ref = _sdpa(qq, kk, vv, scale)[:, 0, :]
                    np.testing.assert_allclose(out[b], ref, rtol=1e-12, atol=1e-13)


def check_single_token_returns_v(orc):
    rng = np.random.default_rng(3)
    for dt in ("f16", "bf16"):
        B, Hq, Hkv, D, P = 4, 6, 2, 32, 16
        dk = _rand_bits(rng, (B, Hkv, 1, D), dt, 5.0)
        dv = _rand_bits(rng, (B, Hkv, 1, D), dt, 5.0)
        lens = np.ones(B, dtype=np.int64)
        kp, vp, table = wl.scatter_dense(dk, dv, lens, P, rng, extra_pages=3, fill=NAN_BITS[dt])
        q = _rand_bits(rng, (B, Hq, D), dt, 3.0)
        out = orc.paged_decode(q, kp, vp, table, lens, 0.37, dt)
        for b in range(B):
            for h in range(Hq):
                assert np.array_equal(out[b, h], values_of(dv[b, h // 3, 0], dt))


def check_constant_v_and_uniform_weights(orc):
    rng = np.random.default_rng(5)
    dt = "bf16"
    B, Hq, Hkv, D, P = 2, 4, 2, 16, 4
    lens = np.array([9, 13])
    Lmax = 13
    dk = _rand_bits(rng, (B, Hkv, Lmax, D), dt)
    row = _rand_bits(rng, (B, Hkv, 1, D), dt)
    dv = np.repeat(row, Lmax, axis=2)
    kp, vp, table = wl.scatter_dense(dk, dv, lens, P, rng, extra_pages=1, fill=NAN_BITS[dt])
    q = _rand_bits(rng, (B, Hq, D), dt)
    out = orc.paged_decode(q, kp, vp, table, lens, 0.25, dt)
    for b in range(B):
        for h in range(Hq):
            np.testing.assert_allclose(out[b, h], values_of(row[b, h // 2, 0], dt), rtol=1e-14,
                                       atol=0)
    # scale 0 (or q = 0): every weight equal -> arithmetic mean of the value rows
    dv2 = _rand_bits(rng, (B, Hkv, Lmax, D), dt)
    kp, vp, table = wl.scatter_dense(dk, dv2, lens, P, rng, extra_pages=1, fill=NAN_BITS[dt])
    out0 = orc.paged_decode(q, kp, vp, table, lens, 0.0, dt)
    qz = np.zeros_like(q)
    outq = orc.paged_decode(qz, kp, vp, table, lens, 0.7, dt)
    for b in range(B):
        for h in range(Hq):
            mean = values_of(dv2[b, h // 2, :lens[b]], dt).mean(axis=0)
            np.testing.assert_allclose(out0[b, h], mean, rtol=1e-13, atol=1e-15)
            np.testing.assert_allclose(outq[b, h], mean, rtol=1e-13, atol=1e-15)


def check_two_tokens_logistic(orc):
    """Two tokens: weight of token 1 = 1 / (1 + exp(-(s_1 - s_0)))."""
    rng = np.random.default_rng(9)
    dt = "f16"
    D, P = 8, 16
    for _ in range(5):
        dk = _rand_bits(rng, (1, 1, 2, D), dt)
        dv = _rand_bits(rng, (1, 1, 2, D), dt)
        kp, vp, table = wl.scatter_dense(dk, dv, [2], P, rng, extra_pages=1, fill=NAN_BITS[dt])
        q = _rand_bits(rng, (1, 1, D), dt)
        scale = 0.8
        out = orc.paged_decode(q, kp, vp, table, [2], scale, dt)
        k = values_of(dk[0, 0], dt)
        v = values_of(dv[0, 0], dt)
        qq = values_of(q[0, 0], dt)
        diff = scale * float(np.dot(qq, k[1] - k[0]))
        w1 = 1.0 / (1.0 + math.exp(-diff))
        np.testing.assert_allclose(out[0, 0], (1 - w1) * v[0] + w1 * v[1], rtol=1e-12, atol=1e-14)


def check_page_permutation_invariance(orc):
    rng = np.random.default_rng(17)
    dt = "bf16"
    B, Hq, Hkv, D, P = 3, 8, 2, 32, 4
    lens = np.array([5, 17, 12])
    dk = _rand_bits(rng, (B, Hkv, 17, D), dt)
    dv = _rand_bits(rng, (B, Hkv, 17, D), dt)
    q = _rand_bits(rng, (B, Hq, D), dt)
    outs = []
    for seed in (1, 2, 3):
        kp, vp, table = wl.scatter_dense(dk, dv, lens, P, np.random.default_rng(seed),
                                         extra_pages=4, fill=NAN_BITS[dt])
        outs.append(orc.paged_decode(q, kp, vp, table, lens, 0.3, dt))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def check_shared_prefix_equals_private_copies(orc):
    rng = np.random.default_rng(23)
    dt = "f16"
    B, Hq, Hkv, D, P = 4, 4, 1, 16, 4
    prefix = 8  # two full pages
    suffix = np.array([1, 4, 7, 3])
    lens = prefix + suffix
    NP = 2 + int(sum((suffix + P - 1) // P)) + B * 2
    kp = _rand_bits(rng, (NP, Hkv, P, D), dt)
    vp = _rand_bits(rng, (NP, Hkv, P, D), dt)
    MP = int(max((lens + P - 1) // P))
    shared = np.full((B, MP), -1, dtype=np.int32)
    private = np.full((B, MP), -1, dtype=np.int32)
    nxt = 2
    for b in range(B):
        shared[b, :2] = [0, 1]
        ns = (int(suffix[b]) + P - 1) // P
        shared[b, 2:2 + ns] = np.arange(nxt, nxt + ns)
        nxt += ns
    first_private = nxt
    for b in range(B):
        # private copies of the two prefix pages for every sequence
        c0, c1 = first_private + 2 * b, first_private + 2 * b + 1
        kp[c0], kp[c1], vp[c0], vp[c1] = kp[0], kp[1], vp[0], vp[1]
        private[b] = shared[b]
        private[b, :2] = [c0, c1]
    q = _rand_bits(rng, (B, Hq, D), dt)
    a = orc.paged_decode(q, kp, vp, shared, lens, 0.5, dt)
    c = orc.paged_decode(q, kp, vp, private, lens, 0.5, dt)
    assert np.array_equal(a, c)


def check_gqa_equals_repeated_kv_heads(orc):
    """Grouped heads == plain multi-head attention over a pool whose KV heads are
    each repeated for their consecutive query heads (repeat_kv)."""
    rng = np.random.default_rng(29)
    dt = "bf16"
    B, Hq, Hkv, D, P = 2, 6, 2, 16, 4
    G = Hq // Hkv
    lens = np.array([6, 11])
    dk = _rand_bits(rng, (B, Hkv, 11, D), dt)
    dv = _rand_bits(rng, (B, Hkv, 11, D), dt)
    kp, vp, table = wl.scatter_dense(dk, dv, lens, P, np.random.default_rng(1), extra_pages=1,
                                     fill=NAN_BITS[dt])
    kr, vr, table_r = wl.scatter_dense(np.repeat(dk, G, axis=1), np.repeat(dv, G, axis=1), lens,
                                       P, np.random.default_rng(2), extra_pages=1,
                                       fill=NAN_BITS[dt])
    q = _rand_bits(rng, (B, Hq, D), dt)
    a = orc.paged_decode(q, kp, vp, table, lens, 0.4, dt)
    c = orc.paged_decode(q, kr, vr, table_r, lens, 0.4, dt)
    assert np.array_equal(a, c)


def check_rows_match_full(orc):
    w = wl.make("tiny", seed=4)
    args = (wl.to_bits(w.q), wl.to_bits(w.k_pool), wl.to_bits(w.v_pool), w.page_table,
            w.context_lens, w.scale, w.dtype_name)
    full = orc.paged_decode(*args)
    rows = np.array([[0, 0], [1, 3], [0, 2], [1, 1]])
    part = orc.paged_decode_rows(*args, rows)
    for i, (b, h) in enumerate(rows):
        assert np.array_equal(part[i], full[b, h])


def check_append_then_gather_is_dense(orc):
    """Append of the new token followed by a gather through the table reproduces
    the dense cache with the new row at the end, bit for bit; padded slots
    (position < 0) write nothing; no other pool byte changes."""
    rng = np.random.default_rng(31)
    for dt in ("f16", "bf16"):
        B, Hkv, D, P = 5, 3, 16, 4
        before = np.array([0, 3, 4, 9, 6])
        lens_after = before + 1
        Lmax = int(lens_after.max())
        dk = _rand_bits(rng, (B, Hkv, Lmax, D), dt)
        dv = _rand_bits(rng, (B, Hkv, Lmax, D), dt)
        # pool built from the dense cache with the last row still missing (NaN)
        dk_old, dv_old = dk.copy(), dv.copy()
        for b in range(B):
            dk_old[b, :, before[b]:] = NAN_BITS[dt]
            dv_old[b, :, before[b]:] = NAN_BITS[dt]
        kp, vp, table = wl.scatter_dense(dk_old, dv_old, lens_after, P, rng, extra_pages=2,
                                         fill=NAN_BITS[dt])
        k_new = np.stack([dk[b, :, before[b]] for b in range(B)])
        v_new = np.stack([dv[b, :, before[b]] for b in range(B)])
        positions = before.astype(np.int32).copy()
        positions[2] = -1  # padded slot: must not write
        kp2, vp2 = orc.kv_append(kp, vp, k_new, v_new, table, positions)
        gk = orc.gather(kp2, table, lens_after, Lmax, fill=0)
        gv = orc.gather(vp2, table, lens_after, Lmax, fill=0)
        for b in range(B):
            L = int(lens_after[b]) if b != 2 else int(before[b])
            assert np.array_equal(gk[b, :, :L], dk[b, :, :L])
            assert np.array_equal(gv[b, :, :L], dv[b, :, :L])
        # sequence 2 was padded: its slot keeps the old (NaN) content
        pg, sl = table[2, before[2] // P], before[2] % P
        assert (kp2[pg, :, sl] == NAN_BITS[dt]).all() and (vp2[pg, :, sl] == NAN_BITS[dt]).all()
        # exactly the appended slots changed
        changed = np.argwhere((kp2 != kp).any(axis=(1, 3)))
        expect = sorted((int(table[b, before[b] // P]), int(before[b] % P))
                        for b in range(B) if b != 2)
        assert sorted(map(tuple, changed[:, [0, 1]].tolist())) == expect


def check_empty_context_and_errors(orc):
    from oracle import OracleError
    rng = np.random.default_rng(37)
    dt = "f16"
    B, Hq, Hkv, D, P = 2, 2, 1, 8, 4
    kp = _rand_bits(rng, (3, Hkv, P, D), dt)
    vp = _rand_bits(rng, (3, Hkv, P, D), dt)
    q = _rand_bits(rng, (B, Hq, D), dt)
    table = np.array([[0, 1], [2, -1]], dtype=np.int32)
    out = orc.paged_decode(q, kp, vp, table, [0, 3], 1.0, dt)
    assert np.array_equal(out[0], np.zeros((Hq, D)))
    assert np.isfinite(out[1]).all()
    for bad_table, lens, code in (([[0, 7], [2, -1]], [6, 3], 2),   # id beyond the pool
                                  ([[0, -1], [2, -1]], [6, 3], 2),  # unused id inside L
                                  ([[0, 1], [2, -1]], [9, 3], 3)):  # L beyond the row
        try:
            orc.paged_decode(q, kp, vp, np.array(bad_table, dtype=np.int32), lens, 1.0, dt)
        except OracleError as e:
            assert e.code == code
        else:
            raise AssertionError("bad input accepted")
    # an append beyond the table row is rejected and changes nothing
    try:
        orc.kv_append(kp, vp, q[:, :1], q[:, :1], table, [8, 0])
    except OracleError as e:
        assert e.code == 3
    else:
        raise AssertionError("append beyond the row accepted")




# ---- rotary embedding and rounding (the fused rotary + append path) ----

def check_encode_round_trips_and_matches_libraries(orc):
    """Rounding float64 to fp16 / bf16: every finite pattern survives a
    decode-encode round trip; random values round as numpy (fp16, from
    float64) and torch (bf16, from values exact in float32) round them; ties
    go to the even neighbour; overflow gives inf."""
    rng = np.random.default_rng(11)
    for dt in ("f16", "bf16"):
        allb = np.arange(65536, dtype=np.uint16)
        vals = orc.decode_bits(allb, dt)
        back = orc.encode(vals, dt)
        fin = np.isfinite(vals)
        assert np.array_equal(back[fin], allb[fin]), dt
        assert np.all(np.isnan(orc.decode_bits(back[np.isnan(vals)], dt)))
    x = rng.standard_normal(20000) * np.exp(rng.uniform(-20, 12, 20000))
    assert np.array_equal(orc.encode(x, "f16"), x.astype(np.float16).view(np.uint16))
    x32 = (rng.standard_normal(20000) * np.exp(rng.uniform(-40, 40, 20000))).astype(np.float32)
    ref = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(orc.encode(x32.astype(np.float64), "bf16"), ref)
    # halfway between 1 and the next fp16 (1 + 2^-10): ties to the even one, 1
    assert orc.encode([1 + 2.0 ** -11, 1 + 3 * 2.0 ** -11], "f16").tolist() == [0x3C00, 0x3C02]
    assert orc.encode([70000.0, -1e300], "f16").tolist() == [0x7C00, 0xFC00]


def check_rope_position_zero_is_identity(orc):
    rng = np.random.default_rng(12)
    for dt in ("f16", "bf16"):
        x = _rand_bits(rng, (3, 5, 64), dt)
        assert np.array_equal(orc.rope(x, [0, 0, 0], 10000.0, dt), x)


def check_rope_one_hot_closed_form(orc):
    """Unit vectors show the pairing (element i with i + D/2) and the angle
    pos * theta^(-2i/D): for D = 4, theta = 100, pair 0 turns by pos and pair 1
    by pos / 10."""
    one = {"f16": 0x3C00, "bf16": 0x3F80}
    for dt in ("f16", "bf16"):
        x = np.zeros((2, 2, 4), dtype=np.uint16)
        x[:, 0, 0] = one[dt]  # e_0
        x[:, 1, 1] = one[dt]  # e_1
        _, y = orc.rope(x, [1, 7], 100.0, dt, with_f64=True)
        for b, pos in enumerate((1, 7)):
            assert np.allclose(y[b, 0], [math.cos(pos), 0, math.sin(pos), 0], atol=1e-15)
            assert np.allclose(y[b, 1], [0, math.cos(pos / 10), 0, math.sin(pos / 10)],
                               atol=1e-15)


def check_rope_is_a_rotation(orc):
    """Each (i, i + D/2) pair keeps its length; turning by a then by b equals
    turning by a + b; and q.k after rotation depends only on the distance of
    the two positions (the defining property of rotary embeddings)."""
    rng = np.random.default_rng(13)
    dt, D, theta = "bf16", 64, 10000.0
    x = _rand_bits(rng, (4, 3, D), dt)
    xv = orc.decode_bits(x, dt)
    pos = np.array([5, 100, 2047, 32767], dtype=np.int32)
    _, y = orc.rope(x, pos, theta, dt, with_f64=True)
    h = D // 2
    assert np.allclose(y[..., :h] ** 2 + y[..., h:] ** 2, xv[..., :h] ** 2 + xv[..., h:] ** 2,
                       rtol=1e-12, atol=1e-12)
    # turn the float64 result for position a further by b and compare with a + b
    a, b = 37, 1000
    _, ya = orc.rope(x, np.full(4, a, np.int32), theta, dt, with_f64=True)
    _, yab = orc.rope(x, np.full(4, a + b, np.int32), theta, dt, with_f64=True)
    inv = theta ** (-2.0 * np.arange(h) / D)
    c, s_ = np.cos(b * inv), np.sin(b * inv)
    again = np.concatenate([ya[..., :h] * c - ya[..., h:] * s_, ya[..., h:] * c + ya[..., :h] * s_],
                           axis=-1)
    assert np.allclose(again, yab, atol=1e-9)
    q = _rand_bits(rng, (1, 1, D), dt)
    k = _rand_bits(rng, (1, 1, D), dt)
    dots = []
    for m, n in ((10, 3), (107, 100), (4007, 4000)):
        _, qm = orc.rope(q, [m], theta, dt, with_f64=True)
        _, kn = orc.rope(k, [n], theta, dt, with_f64=True)
        dots.append(float((qm * kn).sum()))
    assert np.allclose(dots, dots[0], atol=1e-9), dots


def check_rope_rounds_its_float64_result(orc):
    """The stored row is the float64 rotation rounded to the dtype."""
    rng = np.random.default_rng(14)
    for dt in ("f16", "bf16"):
        x = _rand_bits(rng, (2, 4, 128), dt)
        out, y = orc.rope(x, [9, 30000], 500000.0, dt, with_f64=True)
        assert np.array_equal(out, orc.encode(y, dt))
        if dt == "f16":  # numpy rounds float64 to float16 directly
            assert np.array_equal(out, y.astype(np.float16).view(np.uint16))




# ---- several query tokens per sequence (speculative / suffix decoding) ----

def _dense_kv(orc, w):
    """Dense float64 K/V [B][Hkv][Lmax][D] through the library-independent gather."""
    kb, vb = wl.to_bits(w.k_pool), wl.to_bits(w.v_pool)
    Lmax = int(max(w.context_lens))
    kd = orc.decode_bits(orc.gather(kb, w.page_table, w.context_lens, Lmax), w.dtype_name)
    vd = orc.decode_bits(orc.gather(vb, w.page_table, w.context_lens, Lmax), w.dtype_name)
    return kd, vd


def check_multi_query_vs_causal_sdpa(orc):
    """Each query token j attends to tokens 0 .. L - Qn + j: torch
    scaled_dot_product_attention in float64 with that causal mask on the dense
    cache, GQA by repeating KV heads.  Sequence 0 is shorter than Qn - 1, so
    its first queries see no token at all (zeros)."""
    rng = np.random.default_rng(21)
    for dt, Qn in (("bf16", 5), ("f16", 3)):
        w = wl.make_random(21, batch=3, n_q_heads=8, n_kv_heads=2, head_dim=64, page_size=16,
                           dtype=TORCH_DT[dt], lens=[2, 40, 70])
        q = _rand_bits(rng, (3, Qn, 8, 64), dt)
        got = orc.paged_decode_multi(q, wl.to_bits(w.k_pool), wl.to_bits(w.v_pool), w.page_table,
                                     w.context_lens, w.scale, dt)
        kd, vd = _dense_kv(orc, w)
        qv = orc.decode_bits(q, dt)
        for b in range(3):
            L = int(w.context_lens[b])
            k = torch.from_numpy(np.repeat(kd[b, :, :L], 4, axis=0))    # [Hq][L][D]
            v = torch.from_numpy(np.repeat(vd[b, :, :L], 4, axis=0))
            qq = torch.from_numpy(qv[b].transpose(1, 0, 2).copy())     # [Hq][Qn][D]
            pos = torch.arange(L)
            mask = pos[None, :] <= (L - Qn + torch.arange(Qn))[:, None]  # [Qn][L]
            ref = torch.nn.functional.scaled_dot_product_attention(
                qq, k, v, attn_mask=mask, scale=w.scale).numpy()        # [Hq][Qn][D]
            ref = np.nan_to_num(ref.transpose(1, 0, 2))                 # rows with no token: 0
            assert np.allclose(got[b], ref, rtol=1e-10, atol=1e-12), (dt, b)


def check_multi_query_single_token_and_causality(orc):
    """Qn = 1 is the plain decode; tokens after query j's position do not change
    row j but do change the last row."""
    rng = np.random.default_rng(22)
    dt = "bf16"
    w = wl.make_random(22, batch=2, n_q_heads=4, n_kv_heads=2, head_dim=64, page_size=16,
                       dtype=torch.bfloat16, lens=[33, 50])
    kb, vb = wl.to_bits(w.k_pool), wl.to_bits(w.v_pool)
    q1 = wl.to_bits(w.q)
    one = orc.paged_decode_multi(q1[:, None], kb, vb, w.page_table, w.context_lens, w.scale, dt)
    assert np.array_equal(one[:, 0], orc.paged_decode(q1, kb, vb, w.page_table, w.context_lens,
                                                      w.scale, dt))
    Qn = 5
    q = _rand_bits(rng, (2, Qn, 4, 64), dt)
    base = orc.paged_decode_multi(q, kb, vb, w.page_table, w.context_lens, w.scale, dt)
    L = int(w.context_lens[1])
    t = L - 2                                   # seen by queries 3 and 4 only
    page, slot = w.page_table[1, t // 16], t % 16
    kb2 = kb.copy()
    kb2[page, :, slot, :] = _rand_bits(rng, (2, 64), dt)
    moved = orc.paged_decode_multi(q, kb2, vb, w.page_table, w.context_lens, w.scale, dt)
    assert np.array_equal(moved[1, :3], base[1, :3])
    assert not np.allclose(moved[1, 3:], base[1, 3:])
    assert np.array_equal(moved[0], base[0])


def check_norm_rope_one_hot_closed_form(orc):
    """A row with one nonzero element a at d = i: the mean square is a^2 / D, so
    the normalised row is sign(a) sqrt(D) w_i at i (eps = 0), and the rotation
    at position p turns pair (i, i + D/2) by p * theta^(-2i/D).  With w_i !=
    w_{i+D/2} this also fixes the order: norm first, then the rotation."""
    D, theta = 8, 100.0
    w_vals = [1.5, 0.5, 1.0, 1.0, 0.25, 1.0, 1.0, 2.0]
    for dt in ("f16", "bf16"):
        w = bits_of(w_vals, dt)
        for i, a, p in ((0, 2.0, 3), (1, -0.75, 5), (3, 4.0, 1)):
            x = np.zeros((1, 1, D), dtype=np.uint16)
            x[0, 0, i] = bits_of([a], dt)[0]
            _, f = orc.norm_rope(x, np.array([p], np.int32), w, 0.0, theta, dt, with_f64=True)
            n = np.sign(a) * np.sqrt(D) * orc.decode_bits(w, dt)[i]
            ang = p * theta ** (-2.0 * i / D)
            want = np.zeros(D)
            want[i] = n * np.cos(ang)
            want[i + D // 2] = n * np.sin(ang)
            assert np.allclose(f[0, 0], want, rtol=1e-14, atol=1e-14), (dt, i)


def check_norm_rope_scale_invariance_and_weights(orc):
    """eps = 0: rows x and 2^k x give the same bits (exact power-of-two
    scaling); the weight multiplies element-wise (position 0: no rotation);
    with w = 1 the result is the plain rotation times 1 / rms(x); a zero row
    with eps > 0 stays zero."""
    rng = np.random.default_rng(41)
    for dt in ("f16", "bf16"):
        D = 64
        x = _rand_bits(rng, (3, 2, D), dt)
        xd = orc.decode_bits(x, dt)
        x4 = bits_of(xd * 4.0, dt)
        pos = np.array([0, 7, 1000], np.int32)
        w1 = bits_of(np.ones(D), dt)
        a = orc.norm_rope(x, pos, w1, 0.0, 10000.0, dt)
        b = orc.norm_rope(x4, pos, w1, 0.0, 10000.0, dt)
        assert np.array_equal(a, b)
        w = _rand_bits(rng, (D,), dt)
        _, fw = orc.norm_rope(x, np.zeros(3, np.int32), w, 1e-6, 10000.0, dt, with_f64=True)
        _, f1 = orc.norm_rope(x, np.zeros(3, np.int32), w1, 1e-6, 10000.0, dt, with_f64=True)
        assert np.allclose(fw, f1 * orc.decode_bits(w, dt), rtol=1e-14, atol=0)
        _, fr = orc.rope(x, pos, 10000.0, dt, with_f64=True)
        _, fn = orc.norm_rope(x, pos, w1, 0.0, 10000.0, dt, with_f64=True)
        rms = np.sqrt((xd ** 2).mean(axis=-1, keepdims=True))
        assert np.allclose(fn, fr / rms, rtol=1e-13, atol=1e-15)
        z = np.zeros((1, 1, D), np.uint16)
        zn = orc.norm_rope(z, np.array([3], np.int32), w1, 1e-6, 10000.0, dt)
        assert (orc.decode_bits(zn, dt) == 0).all()  # +0 or -0


ALL_CHECKS = [
    check_decode_f16_all_patterns,
    check_decode_bf16_all_patterns,
    check_golden_worked_examples,
    check_dense_vs_sdpa,
    check_single_token_returns_v,
    check_constant_v_and_uniform_weights,
    check_two_tokens_logistic,
    check_page_permutation_invariance,
    check_shared_prefix_equals_private_copies,
    check_gqa_equals_repeated_kv_heads,
    check_rows_match_full,
    check_append_then_gather_is_dense,
    check_empty_context_and_errors,
    check_encode_round_trips_and_matches_libraries,
    check_rope_position_zero_is_identity,
    check_rope_one_hot_closed_form,
    check_rope_is_a_rotation,
    check_rope_rounds_its_float64_result,
    check_multi_query_vs_causal_sdpa,
    check_multi_query_single_token_and_causality,
    check_norm_rope_one_hot_closed_form,
    check_norm_rope_scale_invariance_and_weights,
]
