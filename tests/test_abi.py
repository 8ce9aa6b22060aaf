"""The C ABI without a GPU: the library loads, exports every declared symbol,
and rejects bad arguments on the host before touching CUDA; the host page
allocator keeps correct reference counts."""
import ctypes
import os
import re
import threading

import pytest

import paged_kv_decode_16_gb300 as pkv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pagedkv.h")

OK, INVALID, UNSUPPORTED, ALIAS, OUT_OF_PAGES, WORKSPACE, CUDA, DEVCHECK, REFCOUNT = range(9)
F16, BF16 = 0, 1
A = 1 << 20  # fake, 256-byte aligned "device" addresses; validation never dereferences them


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s*([A-Za-z_][A-Za-z0-9_]*)\s*\(",
                       text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    return pkv.load_library()


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 20, names
    for name in names:
        assert hasattr(lib, name), f"{name} declared in pagedkv.h but not exported"


def test_status_strings(lib):
    for code in range(9):
        assert pkv.pkv_status_string(code)
    assert pkv.pkv_status_string(99) == "unknown status"
    assert pkv.pkv_version() >= 100


def _decode(lib, **kw):
    a = dict(q=A, k=A * 8, v=A * 16, table=A * 24, stride=4, lens=A * 25, batch=2, hq=8, hkv=2,
             d=128, p=16, np_=8, dt=BF16, scale=0.088, out=A * 26, ws=A * 27, ws_bytes=1 << 20,
             workers=0, variant=0)
    a.update(kw)
    V = ctypes.c_void_p
    return lib.paged_decode_attention(V(a["q"]), V(a["k"]), V(a["v"]), V(a["table"]), a["stride"],
                                      V(a["lens"]), a["batch"], a["hq"], a["hkv"], a["d"], a["p"],
                                      a["np_"], a["dt"], ctypes.c_float(a["scale"]), V(a["out"]),
                                      V(a["ws"]), a["ws_bytes"], a["workers"], a["variant"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(d=96), UNSUPPORTED),
    (dict(d=256), UNSUPPORTED),
    (dict(p=8), UNSUPPORTED),
    (dict(p=24), UNSUPPORTED),
    (dict(hq=6, hkv=4), INVALID),
    (dict(hkv=0), INVALID),
    (dict(batch=-1), INVALID),
    (dict(np_=0), INVALID),
    (dict(stride=0), INVALID),
    (dict(dt=5), INVALID),
    (dict(workers=-2), INVALID),
    (dict(variant=3), UNSUPPORTED),       # tcgen05: several query tokens only
    (dict(variant=4), INVALID),
    (dict(variant=-1), INVALID),
    (dict(scale=float("nan")), INVALID),
    (dict(scale=float("inf")), INVALID),
    (dict(q=0), INVALID),
    (dict(lens=0), INVALID),
    (dict(out=0), INVALID),
    (dict(ws=0), WORKSPACE),
    (dict(ws=A + 64), WORKSPACE),
    (dict(q=A + 8), INVALID),
    (dict(out=A * 26 + 4), INVALID),
    (dict(out=A), ALIAS),                 # out == q
    (dict(out=A * 8 + 4096), ALIAS),      # inside the K pool
    (dict(out=A * 24), ALIAS),            # on the page table
    (dict(out=A * 27 + 1024), ALIAS),     # inside the workspace
])
def test_decode_rejects_bad_arguments_on_host(lib, kw, code):
    assert _decode(lib, **kw) == code


def test_empty_batch_is_a_noop(lib):
    assert _decode(lib, batch=0, q=0, out=0, ws=0) == OK


def test_append_and_gather_host_checks(lib):
    V = ctypes.c_void_p
    h = V()
    assert lib.kv_pool_create(8, 16, 2, 128, BF16, V(A), V(A * 2), ctypes.byref(h)) == OK
    try:
        assert lib.kv_append(h, V(A * 3), V(A * 4), V(A * 5), 4, V(A * 6), 0, None, None) == OK
        assert lib.kv_append(h, None, V(A * 4), V(A * 5), 4, V(A * 6), 2, None, None) == INVALID
        assert lib.kv_append(h, V(A * 3 + 2), V(A * 4), V(A * 5), 4, V(A * 6), 2, None,
                             None) == INVALID
        # new rows inside the pool being written
        assert lib.kv_append(h, V(A + 256), V(A * 4), V(A * 5), 4, V(A * 6), 2, None,
                             None) == ALIAS
        assert lib.kv_append(None, V(A * 3), V(A * 4), V(A * 5), 4, V(A * 6), 2, None,
                             None) == INVALID
        assert lib.kv_gather(h, V(A * 5), 4, V(A * 6), 2, 64, V(A * 8), V(A * 8), None,
                             None) == ALIAS
        assert lib.kv_gather(h, V(A * 5), 0, V(A * 6), 2, 64, V(A * 8), V(A * 9), None,
                             None) == INVALID
    finally:
        assert lib.kv_pool_destroy(h) == OK


def test_pool_create_checks(lib):
    V = ctypes.c_void_p
    h = V()
    assert lib.kv_pool_create(8, 16, 2, 96, BF16, V(A), V(A), ctypes.byref(h)) == UNSUPPORTED
    assert lib.kv_pool_create(8, 12, 2, 128, BF16, V(A), V(A), ctypes.byref(h)) == UNSUPPORTED
    assert lib.kv_pool_create(0, 16, 2, 128, BF16, V(A), V(A), ctypes.byref(h)) == INVALID
    assert lib.kv_pool_create(8, 16, 2, 128, BF16, V(A), None, ctypes.byref(h)) == INVALID
    assert lib.kv_pool_create(8, 16, 2, 128, BF16, V(A + 4), V(A), ctypes.byref(h)) == INVALID
    assert lib.kv_pool_create(8, 16, 2, 128, 3, V(A), V(A), ctypes.byref(h)) == INVALID
    assert lib.kv_pool_destroy(None) == OK


def _borrowed_pool(lib, n):
    V = ctypes.c_void_p
    h = V()
    assert lib.kv_pool_create(n, 16, 2, 64, F16, V(A), V(A * 2), ctypes.byref(h)) == OK
    return h


def _ids(*v):
    return (ctypes.c_int32 * max(len(v), 1))(*v)


def test_allocator_refcounts(lib):
    h = _borrowed_pool(lib, 6)
    try:
        assert lib.kv_pool_free_count(h) == 6
        out = (ctypes.c_int32 * 4)()
        assert lib.kv_pool_alloc_pages(h, 4, out) == OK
        got = list(out)
        assert sorted(got) == [0, 1, 2, 3] and lib.kv_pool_free_count(h) == 2
        assert lib.kv_pool_alloc_pages(h, 3, out) == OUT_OF_PAGES
        assert lib.kv_pool_free_count(h) == 2  # all or nothing
        # share the first two pages (a prefix) with a second sequence
        assert lib.kv_pool_retain_pages(h, _ids(got[0], got[1]), 2) == OK
        assert lib.kv_pool_refcount(h, got[0]) == 2
        assert lib.kv_pool_release_pages(h, _ids(*got), 4) == OK
        assert lib.kv_pool_free_count(h) == 4
        assert lib.kv_pool_refcount(h, got[0]) == 1 and lib.kv_pool_refcount(h, got[2]) == 0
        # releasing a free page, or one page more often than held, changes nothing
        assert lib.kv_pool_release_pages(h, _ids(got[2]), 1) == REFCOUNT
        assert lib.kv_pool_release_pages(h, _ids(got[0], got[0]), 2) == REFCOUNT
        assert lib.kv_pool_refcount(h, got[0]) == 1
        assert lib.kv_pool_retain_pages(h, _ids(got[3]), 1) == REFCOUNT
        assert lib.kv_pool_retain_pages(h, _ids(99), 1) == INVALID
        assert lib.kv_pool_release_pages(h, _ids(-1), 1) == INVALID
        assert lib.kv_pool_release_pages(h, _ids(got[0], got[1]), 2) == OK
        assert lib.kv_pool_free_count(h) == 6
        assert lib.kv_pool_refcount(h, 99) == -1
    finally:
        lib.kv_pool_destroy(h)


def test_allocator_threads(lib):
    """Concurrent alloc/retain/release from several threads keeps the books."""
    h = _borrowed_pool(lib, 512)
    errors = []

    def worker(seed):
        import random
        rnd = random.Random(seed)
        held = []
        for _ in range(300):
            if held and rnd.random() < 0.5:
                ids = held.pop(rnd.randrange(len(held)))
                if lib.kv_pool_release_pages(h, _ids(*ids), len(ids)) != OK:
                    errors.append("release")
            else:
                n = rnd.randint(1, 4)
                out = (ctypes.c_int32 * n)()
                rc = lib.kv_pool_alloc_pages(h, n, out)
                if rc == OK:
                    ids = list(out)
                    if rnd.random() < 0.3:  # share them once more
                        if lib.kv_pool_retain_pages(h, _ids(*ids), n) != OK:
                            errors.append("retain")
                        held.append(ids)
                    held.append(ids)
                elif rc != OUT_OF_PAGES:
                    errors.append(f"alloc {rc}")
        for ids in held:
            if lib.kv_pool_release_pages(h, _ids(*ids), len(ids)) != OK:
                errors.append("final release")

    ts = [threading.Thread(target=worker, args=(s,)) for s in range(8)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    try:
        assert not errors, errors[:5]
        assert lib.kv_pool_free_count(h) == 512
        assert all(lib.kv_pool_refcount(h, i) == 0 for i in range(512))
    finally:
        lib.kv_pool_destroy(h)


def test_no_alloc_scratch_size_matches_header(lib):
    text = open(HEADER).read()
    m = re.search(r"#define\s+PKV_NO_ALLOC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", text)
    assert m, "PKV_NO_ALLOC_SCRATCH_BYTES not found"
    assert int(m.group(1)) << int(m.group(2)) == pkv.NO_ALLOC_SCRATCH_BYTES


def test_no_alloc_shape_checks_on_host(lib):
    V = ctypes.c_void_p

    def call(d=128, batch=2, hq=8, hkv=2):
        return lib.paged_decode_attention_no_alloc(V(A), V(A * 8), V(A * 16), V(A * 24), 4,
                                                   V(A * 25), batch, hq, hkv, d, 16, 8, BF16,
                                                   ctypes.c_float(0.088), V(A * 26), 0, 0, None)
    assert call(d=96) == UNSUPPORTED
    assert call(hq=6, hkv=4) == INVALID
    assert call(batch=-1) == INVALID
    assert call(batch=0) == OK


def test_rope_entry_points_check_theta_on_host(lib):
    V = ctypes.c_void_p
    for theta in (0.0, -1.0, float("nan"), float("inf")):
        rc = lib.paged_decode_step_rope(V(A * 30), V(A * 31), V(A * 32), V(A), V(A * 8),
                                        V(A * 16), V(A * 24), 4, V(A * 25), 2, 8, 2, 128, 16, 8,
                                        BF16, ctypes.c_float(0.088), ctypes.c_double(theta),
                                        None, None, ctypes.c_float(0.0),
                                        V(A * 26), V(A * 27), 1 << 20, 0, 0, None)
        assert rc == INVALID
    h = V()
    assert lib.kv_pool_create(8, 16, 2, 128, BF16, V(A), V(A * 2), ctypes.byref(h)) == OK
    F = ctypes.c_float

    def rope(batch=2, theta=1e4, q_out=A * 9, qw=None, kw=None, eps=0.0):
        return lib.kv_append_rope(h, V(A * 3), V(A * 4), V(A * 5), V(A * 6), 4, V(A * 7), batch,
                                  8, ctypes.c_double(theta), None if qw is None else V(qw),
                                  None if kw is None else V(kw), F(eps), V(q_out), None, None)
    try:
        assert rope(theta=0.0) == INVALID
        # q_out partly over q is refused; q_out == q (in place) passes the host checks
        assert rope(q_out=A * 3 + 256) == ALIAS
        assert rope(batch=0, q_out=A * 3) == OK
        # the norm before the rotation: 2-byte aligned weights, eps finite and >= 0
        assert rope(qw=A * 10 + 1) == INVALID
        assert rope(kw=A * 10 + 1) == INVALID
        assert rope(qw=A * 10, eps=-1e-6) == INVALID
        assert rope(kw=A * 10, eps=float("nan")) == INVALID
        assert rope(batch=0, qw=A * 10 + 1) == INVALID  # checked before the empty batch
        assert rope(batch=0, qw=A * 10, kw=A * 11, eps=1e-6) == OK
    finally:
        lib.kv_pool_destroy(h)


def test_host_step_checks_on_host(lib):
    """paged_decode_step_host: the decode checks, then k_new / v_new /
    positions, aliasing of out, and page-locked host memory for every host
    argument (the fake addresses here are not), all before any launch."""
    V = ctypes.c_void_p

    def step(batch=2, k_new=A * 30, out=A * 26, ws_bytes=1 << 20, stride=4):
        return lib.paged_decode_step_host(V(k_new), V(A * 31), V(A * 32), V(A), V(A * 8),
                                          V(A * 16), V(A * 24), stride, V(A * 25), batch, 8, 2,
                                          128, 16, 8, BF16, ctypes.c_float(0.088), V(out),
                                          V(A * 27), ws_bytes, 0, 0, None)
    assert step(batch=0) == OK
    assert step(batch=-1) == INVALID
    assert step(stride=0) == INVALID
    assert step(k_new=0) == INVALID
    assert step(k_new=A * 30 + 8) == INVALID      # not 16-byte aligned
    assert step(out=A * 30) == ALIAS              # out over k_new
    assert step(out=A * 27) == ALIAS              # out over the workspace
    assert step() == INVALID                      # not page-locked host memory
    n = ctypes.c_size_t(7)
    assert lib.paged_decode_step_host_workspace_size(2, 8, 2, 128, 0, 0, 0, ctypes.byref(n)) \
        == INVALID and n.value == 0
    assert lib.paged_decode_step_host_workspace_size(2, 8, 2, 96, 4, 0, 0, ctypes.byref(n)) \
        == UNSUPPORTED
    assert lib.paged_decode_step_host_workspace_size(2, 8, 2, 128, 4, 0, 0, None) == INVALID


def test_no_alloc_status_reader_rejects_null(lib):
    assert lib.pkv_read_no_alloc_status(None) == INVALID


class _FakeCudaTensor:
    """Stands in for a contiguous CUDA tensor (no GPU needed for the binding's checks)."""

    def __init__(self, index):
        import torch
        self.is_cuda = True
        self.dtype = torch.bfloat16
        self.device = torch.device("cuda", index)

    def is_contiguous(self):
        return True

    def dim(self):
        return 3


def test_binding_rejects_operands_on_another_device(monkeypatch):
    import torch
    t = _FakeCudaTensor(1)
    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    with pytest.raises(ValueError, match="current device is cuda:0"):
        pkv._dev(t, "q", torch.bfloat16, 3)
    monkeypatch.setattr(torch.cuda, "current_device", lambda: 1)
    assert pkv._dev(t, "q", torch.bfloat16, 3) is t


def test_host_step_binding_wants_pinned_host_tensors():
    """paged_decode_step_host's binding refuses CPU tensors that are not
    page-locked (and CUDA tensors where host memory is expected) before any
    call into the library."""
    import torch
    t = torch.zeros(2, 4, 64, dtype=torch.bfloat16)
    assert not t.is_pinned()
    with pytest.raises(ValueError, match="pinned host tensor"):
        pkv.paged_decode_step_host(t, t, t, t, t, t, t, t, 0.125, t, t)


def test_header_compiles_as_plain_c(tmp_path):
    """include/pagedkv.h is a C header: a C99 translation unit that includes it
    and names every declared function compiles with -pedantic, no warnings."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not found")
    names = declared_functions()
    src = tmp_path / "uses_header.c"
    src.write_text('#include "pagedkv.h"\n'
                   "typedef void (*any_fn)(void);\n"
                   "any_fn pkv_symbols[] = {\n" +
                   "".join(f"    (any_fn)&{n},\n" for n in names) +
                   "};\n")
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                        "-fsyntax-only", "-I", os.path.dirname(HEADER), str(src)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
