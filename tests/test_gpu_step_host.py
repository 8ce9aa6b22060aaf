"""paged_decode_step_host: the step's inputs and its output in pinned host
memory, read and written by the kernels themselves.  Same kernels and schedule
as paged_decode_step, so the results must be the same bits; checked against
the float64 oracle as well."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import paged_kv_decode_16_gb300 as pkv
from paged_kv_decode_16_gb300 import workloads as wl
from gpu_helpers import VARIANT_IDS, VARIANTS, assert_close, oracle_full, to_dev

pytestmark = pytest.mark.gpu

INVALID, WORKSPACE = 1, 5


def _pin(x):
    t = torch.from_numpy(np.ascontiguousarray(x)) if isinstance(x, np.ndarray) else x.cpu()
    return t.contiguous().pin_memory()


def _host_args(w):
    """Pinned host copies of the step's inputs and a pinned output buffer."""
    return dict(k_new=_pin(w.k_new), v_new=_pin(w.v_new), positions=_pin(w.positions),
                q=_pin(w.q), table=_pin(w.page_table), lens=_pin(w.context_lens),
                out=torch.full(tuple(w.q.shape), float("nan"), dtype=w.q.dtype).pin_memory())


def _host_step(w, h, ws, **kw):
    pkv.paged_decode_step_host(h["k_new"], h["v_new"], h["positions"], h["q"], w.k_pool,
                               w.v_pool, h["table"], h["lens"], w.scale, h["out"], ws, **kw)
    torch.cuda.synchronize()
    return h["out"]


def _device_step(w, ws, **kw):
    table, lens, pos = to_dev(w)
    out = torch.empty_like(w.q)
    pkv.paged_decode_step(w.k_new, w.v_new, pos, w.q, w.k_pool, w.v_pool, table, lens, w.scale,
                          out, ws, **kw)
    torch.cuda.synchronize()
    return out


def _bits(t):
    return t.cpu().view(torch.int16)


@pytest.mark.parametrize("variant", VARIANTS, ids=VARIANT_IDS)
@pytest.mark.parametrize("name", ("tiny", "llama3_8b", "mixed_append"))
def test_host_step_equals_device_step(name, variant):
    """Bit for bit the device step's output and pools, on two copies of the
    same cache; and the oracle on the host step's output."""
    w1 = wl.make(name, seed=3, device="cuda")
    w2 = wl.make(name, seed=3, device="cuda")
    before = (wl.to_bits(w2.k_pool), wl.to_bits(w2.v_pool))
    ws1 = pkv.alloc_workspace(w1.batch, w1.n_q_heads, w1.n_kv_heads, w1.head_dim,
                              variant=variant)
    ref = _device_step(w1, ws1, variant=variant)
    assert pkv.pkv_read_device_status(ws1) == 0
    h = _host_args(w2)
    ws2 = pkv.alloc_step_host_workspace(w2.batch, w2.n_q_heads, w2.n_kv_heads, w2.head_dim,
                                        w2.page_table.shape[1], variant=variant)
    out = _host_step(w2, h, ws2, variant=variant)
    assert pkv.pkv_read_device_status(ws2) == 0
    assert torch.equal(_bits(out), _bits(ref))
    assert torch.equal(w1.k_pool.view(torch.int16), w2.k_pool.view(torch.int16))
    assert torch.equal(w1.v_pool.view(torch.int16), w2.v_pool.view(torch.int16))
    # every output element against the oracle, the step's append (at
    # positions[b]) applied on the host copy first; the append itself bit-exact
    assert_close(out.cuda(), oracle_full(w2, before, append=True), strict=True, what=name)
    kp, vp = oracle.kv_append(*before, wl.to_bits(w2.k_new), wl.to_bits(w2.v_new),
                              w2.page_table, w2.positions)
    assert np.array_equal(kp, wl.to_bits(w2.k_pool))
    assert np.array_equal(vp, wl.to_bits(w2.v_pool))


@pytest.mark.parametrize("workers", (1, 7, 1000))
def test_host_step_worker_counts(workers):
    """Forced worker counts (units split over many workers, and the combine):
    host step == device step, bit for bit."""
    w1 = wl.make("mixed_append", seed=11, device="cuda", batch=40)
    w2 = wl.make("mixed_append", seed=11, device="cuda", batch=40)
    ws1 = pkv.alloc_workspace(w1.batch, w1.n_q_heads, w1.n_kv_heads, w1.head_dim, workers)
    ref = _device_step(w1, ws1, num_workers=workers)
    h = _host_args(w2)
    ws2 = pkv.alloc_step_host_workspace(w2.batch, w2.n_q_heads, w2.n_kv_heads, w2.head_dim,
                                        w2.page_table.shape[1], workers)
    out = _host_step(w2, h, ws2, num_workers=workers)
    assert torch.equal(_bits(out), _bits(ref))
    assert pkv.pkv_read_device_status(ws2) == 0


def test_host_step_sees_new_host_inputs_each_call():
    """Inputs rewritten in the same pinned buffers between calls (after the
    previous call's stream work is done) are the ones the next call reads; a
    CUDA graph of the call, replayed, does the same."""
    w = wl.make("mixed_append", seed=5, device="cuda", batch=24)
    h = _host_args(w)
    ws = pkv.alloc_step_host_workspace(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim,
                                       w.page_table.shape[1])
    first = _host_step(w, h, ws).clone()
    h["q"].mul_(-1.0)
    second = _host_step(w, h, ws).clone()
    table, lens, _ = to_dev(w)
    ref = torch.empty_like(w.q)
    wsd = pkv.alloc_workspace(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim)
    pkv.paged_decode_attention(h["q"].cuda(), w.k_pool, w.v_pool, table, lens, w.scale, ref, wsd)
    torch.cuda.synchronize()
    assert torch.equal(_bits(second), _bits(ref))
    assert not torch.equal(_bits(first), _bits(second))
    # recorded once into a graph; the replays read the buffers' current contents
    h["out"].fill_(float("nan"))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            pkv.paged_decode_step_host(h["k_new"], h["v_new"], h["positions"], h["q"], w.k_pool,
                                       w.v_pool, h["table"], h["lens"], w.scale, h["out"], ws)
    torch.cuda.current_stream().wait_stream(s)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(_bits(h["out"]), _bits(ref))
    h["q"].mul_(-1.0)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(_bits(h["out"]), _bits(first))
    assert pkv.pkv_read_device_status(ws) == 0


@pytest.mark.parametrize("dtype,D,P", [(torch.float16, 64, 32), (torch.bfloat16, 128, 16)])
def test_host_step_empty_sequences_and_odd_shapes(dtype, D, P):
    """Empty sequences (their rows zeroed straight into host memory), lengths
    around page and chunk edges, group 6: host step == device step, bit for
    bit, and the oracle."""
    lens = [0, 1, 15, 16, 17, 0, 33, 64, 65, 200]
    w1 = wl.make_random(31, batch=len(lens), n_q_heads=12, n_kv_heads=2, head_dim=D,
                        page_size=P, dtype=dtype, lens=lens, device="cuda")
    w2 = wl.make_random(31, batch=len(lens), n_q_heads=12, n_kv_heads=2, head_dim=D,
                        page_size=P, dtype=dtype, lens=lens, device="cuda")
    before = (wl.to_bits(w2.k_pool), wl.to_bits(w2.v_pool))
    ws1 = pkv.alloc_workspace(w1.batch, w1.n_q_heads, w1.n_kv_heads, w1.head_dim)
    ref = _device_step(w1, ws1)
    h = _host_args(w2)
    ws2 = pkv.alloc_step_host_workspace(w2.batch, w2.n_q_heads, w2.n_kv_heads, w2.head_dim,
                                        w2.page_table.shape[1])
    out = _host_step(w2, h, ws2)
    assert pkv.pkv_read_device_status(ws2) == 0
    assert torch.equal(_bits(out), _bits(ref))
    assert not (out[0] != 0).any() and not (out[5] != 0).any()  # empty: zeros, not the NaN fill
    # per-element bound: a 1-token sequence returns its V row, where bf16 rounding
    # alone exceeds the absolute 2e-3 of the named workloads
    assert_close(out.cuda(), oracle_full(w2, before, append=True), what="odd")


def test_host_step_reports_bad_page_and_bad_position():
    """A page id outside the pool in a host table row and a position beyond
    the row: flagged in the device status like the device step, nothing
    written out of bounds (the append checked against the oracle)."""
    w = wl.make_random(21, batch=4, n_q_heads=8, n_kv_heads=2, head_dim=128, page_size=16,
                       dtype=torch.bfloat16, lens=[5, 17, 40, 3], device="cuda")
    before = (wl.to_bits(w.k_pool), wl.to_bits(w.v_pool))
    w.positions[1] = -1                               # padded slot: no write
    w.positions[2] = w.page_table.shape[1] * 16 + 3   # beyond the table row
    h = _host_args(w)
    ws = pkv.alloc_step_host_workspace(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim,
                                       w.page_table.shape[1])
    _host_step(w, h, ws)
    assert pkv.pkv_read_device_status(ws) & pkv.DEV_BAD_LEN
    pos_ok = w.positions.copy()
    pos_ok[2] = -1
    kp, vp = oracle.kv_append(*before, wl.to_bits(w.k_new), wl.to_bits(w.v_new), w.page_table,
                              pos_ok)
    assert np.array_equal(wl.to_bits(w.k_pool), kp) and np.array_equal(wl.to_bits(w.v_pool), vp)
    # a page id outside the pool in row 0 (read by the decode): flagged
    h["positions"].copy_(torch.from_numpy(pos_ok))
    h["table"][0, 0] = w.num_pages + 5
    _host_step(w, h, ws)
    assert pkv.pkv_read_device_status(ws) & pkv.DEV_BAD_PAGE
    # restored: a clean call clears the status
    h["table"][0, 0] = int(w.page_table[0, 0])
    _host_step(w, h, ws)
    assert pkv.pkv_read_device_status(ws) == 0


def test_host_step_rejects_unpinned_device_and_short_buffers():
    """Host-side checks before any launch: a pageable host buffer, a device
    buffer where host memory is expected, a too-small workspace."""
    w = wl.make("tiny", seed=1, device="cuda")
    h = _host_args(w)
    ws = pkv.alloc_step_host_workspace(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim,
                                       w.page_table.shape[1])
    lib = pkv.load_library()
    B, Hq, D = w.q.shape
    NP, Hkv, P, _ = w.k_pool.shape
    dt = 1 if w.q.dtype == torch.bfloat16 else 0

    def call(q=None, out=None, ws_bytes=None):
        q = h["q"].data_ptr() if q is None else q
        out = h["out"].data_ptr() if out is None else out
        return lib.paged_decode_step_host(
            h["k_new"].data_ptr(), h["v_new"].data_ptr(), h["positions"].data_ptr(), q,
            w.k_pool.data_ptr(), w.v_pool.data_ptr(), h["table"].data_ptr(),
            h["table"].shape[1], h["lens"].data_ptr(), B, Hq, Hkv, D, P, NP, dt,
            ctypes.c_float(w.scale), out, ws.data_ptr(),
            ws.numel() if ws_bytes is None else ws_bytes, 0, 0, None)

    pageable = np.zeros(B * Hq * D + 64, dtype=np.uint16)
    addr = (pageable.ctypes.data + 15) // 16 * 16
    assert call(q=addr) == INVALID
    assert call(out=addr) == INVALID
    q_dev = w.q.contiguous()
    assert call(q=q_dev.data_ptr()) == INVALID
    assert call(ws_bytes=ws.numel() - 256) == WORKSPACE
    with pytest.raises(ValueError):
        pkv.paged_decode_step_host(h["k_new"], h["v_new"], h["positions"], w.q, w.k_pool,
                                   w.v_pool, h["table"], h["lens"], w.scale, h["out"], ws)
    assert call() == 0
    torch.cuda.synchronize()
    assert pkv.pkv_read_device_status(ws) == 0
