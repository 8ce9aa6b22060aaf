"""The host prefix cache (radix tree of whole pages of token ids over the pool)
against a brute-force model of the same policy, plus its reference counting,
LRU eviction and thread safety.  No GPU: the pool borrows fake addresses that
nothing dereferences."""
import ctypes
import random
import threading

import pytest

import paged_kv_decode_16_gb300 as pkv

A = 1 << 20
BF16 = 1


@pytest.fixture
def pool():
    lib = pkv.load_library()
    h = ctypes.c_void_p()
    assert lib.kv_pool_create(4096, 16, 2, 64, BF16, ctypes.c_void_p(A), ctypes.c_void_p(A * 4),
                              ctypes.byref(h)) == 0
    yield lib, h
    lib.kv_pool_destroy(h)


def alloc(lib, h, n):
    ids = (ctypes.c_int32 * max(n, 1))()
    assert lib.kv_pool_alloc_pages(h, n, ids) == 0
    return list(ids[:n])


def release(lib, h, ids):
    arr = (ctypes.c_int32 * max(len(ids), 1))(*ids)
    assert lib.kv_pool_release_pages(h, arr, len(ids)) == 0


def test_insert_then_match_whole_pages_only(pool):
    lib, h = pool
    c = pkv.PrefixCache(h)
    toks = list(range(1000, 1040))           # 2 full pages of 16 + 8 tokens
    pages = alloc(lib, h, 3)
    assert c.insert(toks, pages) == 2        # the partly filled page is not cached
    assert c.pages() == 2
    got = c.match(toks)
    assert got == pages[:2]
    # refcounts: the sequence's own, the cache's, the match's
    assert [lib.kv_pool_refcount(h, p) for p in pages] == [3, 3, 1]
    assert c.match(toks[:31]) == pages[:1]   # 31 tokens: one whole page
    assert c.match([7] * 40) == []           # no shared first page
    release(lib, h, pages[:1])               # the 31-token match
    release(lib, h, pages[:2])               # the 40-token match
    c.destroy()
    assert [lib.kv_pool_refcount(h, p) for p in pages] == [1, 1, 1]


def test_branches_and_first_insert_wins(pool):
    lib, h = pool
    c = pkv.PrefixCache(h)
    a = list(range(48))
    b = list(range(16)) + list(range(500, 532))     # shares page 0 with a
    pa, pb = alloc(lib, h, 3), alloc(lib, h, 3)
    assert c.insert(a, pa) == 3
    assert c.insert(b, pb) == 2                      # page 0 already cached (pa[0])
    assert c.match(b) == [pa[0], pb[1], pb[2]]
    assert c.match(a) == pa
    assert c.pages() == 5
    c.destroy()


def _model_match(model, toks, P):
    out = []
    for k in range(1, len(toks) // P + 1):
        key = tuple(toks[:k * P])
        if key not in model:
            break
        out.append(model[key])
    return out


def test_matches_a_brute_force_model(pool):
    lib, h = pool
    P = 16
    rnd = random.Random(5)
    c = pkv.PrefixCache(h)
    model = {}   # token prefix (whole pages) -> page of its first insertion
    held = []
    for _ in range(60):
        # few distinct page contents, so sequences share prefixes often
        n_pages = rnd.randint(1, 6)
        toks = []
        for _ in range(n_pages):
            toks += [rnd.randint(0, 2)] * P
        toks += [9] * rnd.randint(0, P - 1)
        pages = alloc(lib, h, (len(toks) + P - 1) // P)
        held.append(pages)
        new = c.insert(toks, pages)
        expect_new = 0
        for k in range(1, len(toks) // P + 1):
            key = tuple(toks[:k * P])
            if key not in model:
                model[key] = pages[k - 1]
                expect_new += 1
        assert new == expect_new
        q = []
        for _ in range(rnd.randint(0, 7)):
            q += [rnd.randint(0, 2)] * P
        got = c.match(q)
        assert got == _model_match(model, q, P)
        release(lib, h, got)
    assert c.pages() == len(model)
    for pages in held:
        release(lib, h, pages)
    # the cache alone keeps its pages
    assert all(lib.kv_pool_refcount(h, p) == 1 for p in model.values())
    c.destroy()
    assert lib.kv_pool_free_count(h) == 4096


def test_eviction_frees_lru_leaves_only_the_cache_holds(pool):
    lib, h = pool
    c = pkv.PrefixCache(h)
    s1, s2, s3 = ([1] * 16 + [2] * 16, [1] * 16 + [3] * 16, [4] * 16)
    p1, p2, p3 = alloc(lib, h, 2), alloc(lib, h, 2), alloc(lib, h, 1)
    c.insert(s1, p1)
    c.insert(s2, p2)
    c.insert(s3, p3)
    release(lib, h, p1)          # sequence 1 done: its pages stay cached
    release(lib, h, p3)          # sequence 3 done
    c.match(s3)                  # s3 recently used (and held again by this match)
    free0 = lib.kv_pool_free_count(h)
    # evictable now: s1's second page (leaf, cache-only); not s2 (held), not
    # s3 (held by the match), not page [1]*16 (has children)
    assert c.evict(10) == 1
    assert lib.kv_pool_free_count(h) == free0 + 1
    assert lib.kv_pool_refcount(h, p1[1]) == 0
    release(lib, h, p2)
    # now s2's second page, then the shared first page (a leaf in turn)
    assert c.evict(10) == 2
    assert c.match(s1) == [] and c.match(s2) == []
    release(lib, h, p3)          # the match's reference
    assert c.evict(10) == 1 and c.pages() == 0
    c.destroy()
    assert lib.kv_pool_free_count(h) == 4096


def test_eviction_order_matches_a_model(pool):
    """One page at a time, evict frees exactly the least recently used leaf
    whose page only the cache holds, as a model of the tree predicts: every
    match and insert stamps the nodes of its path with a fresh clock value;
    a parent whose last child goes becomes a leaf."""
    lib, h = pool
    c = pkv.PrefixCache(h)
    rnd = random.Random(11)
    P = 16
    systems = [[rnd.randrange(50) for _ in range(P * rnd.randint(1, 4))] for _ in range(6)]
    stamp, page = {}, {}     # path (tuple of page token tuples) -> last use, page id
    clock = 0
    held = []                # references the requests still hold

    def pages_of(toks):
        return [tuple(toks[i * P:(i + 1) * P]) for i in range(len(toks) // P)]

    for _ in range(60):
        toks = systems[rnd.randrange(6)] + [rnd.randrange(50) for _ in range(P * rnd.randint(0, 3))]
        got = c.match(toks)
        clock += 1
        keys = pages_of(toks)
        for k in range(len(got)):
            stamp[tuple(keys[:k + 1])] = clock
        fresh = alloc(lib, h, len(keys) - len(got)) if len(keys) > len(got) else []
        row = got + fresh
        c.insert(toks, row)
        clock += 1
        for k in range(len(keys)):
            path = tuple(keys[:k + 1])
            page.setdefault(path, row[k])
            stamp[path] = clock
        if rnd.random() < 0.7:
            release(lib, h, row)
        else:
            held.append(row)
    assert c.pages() == len(page)

    def expected():
        leaves = [q for q in page if not any(len(o) == len(q) + 1 and o[:-1] == q for o in page)]
        free = [q for q in leaves if lib.kv_pool_refcount(h, page[q]) == 1]
        return min(free, key=lambda q: stamp[q]) if free else None

    evicted = 0
    while True:
        q = expected()
        if q is None:
            assert c.evict(1) == 0
            break
        assert c.evict(1) == 1
        assert lib.kv_pool_refcount(h, page[q]) == 0, f"evicted the wrong page after {evicted}"
        del page[q]
        evicted += 1
    assert evicted > 10 and c.pages() == len(page)
    for row in held:
        release(lib, h, row)
    c.destroy()
    assert lib.kv_pool_free_count(h) == 4096


def test_insert_checks(pool):
    lib, h = pool
    c = pkv.PrefixCache(h)
    with pytest.raises(pkv.PagedKVError) as e:
        c.insert(list(range(16)), [5000])
    assert e.value.name == "PKV_ERR_INVALID_ARG"
    with pytest.raises(pkv.PagedKVError) as e:   # page 7 is not allocated
        c.insert(list(range(16)), [7])
    assert e.value.name == "PKV_ERR_REFCOUNT"
    # all or nothing: a prompt whose last new page is not allocated caches none
    # of its new pages and leaves their counts alone
    got = alloc(lib, h, 2)
    with pytest.raises(pkv.PagedKVError) as e:
        c.insert(list(range(48)), got + [7])
    assert e.value.name == "PKV_ERR_REFCOUNT"
    assert c.pages() == 0 and c.match(list(range(48))) == []
    assert [lib.kv_pool_refcount(h, p) for p in got] == [1, 1]
    release(lib, h, got)
    c.destroy()


def test_threads_keep_the_books(pool):
    lib, h = pool
    c = pkv.PrefixCache(h)
    errors = []

    def worker(seed):
        rnd = random.Random(seed)
        for _ in range(150):
            toks = []
            for _ in range(rnd.randint(1, 4)):
                toks += [rnd.randint(0, 3)] * 16
            try:
                got = c.match(toks)
                n_new = len(toks) // 16 - len(got)
                fresh = alloc(lib, h, n_new) if n_new else []
                row = got + fresh
                c.insert(toks, row)
                release(lib, h, row)
                if rnd.random() < 0.2:
                    c.evict(2)
            except Exception as ex:  # collected, asserted below
                errors.append(repr(ex))

    ts = [threading.Thread(target=worker, args=(s,)) for s in range(6)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    assert not errors, errors[:3]
    n = c.pages()
    assert 4096 - lib.kv_pool_free_count(h) == n   # only the cache holds pages
    c.destroy()
    assert lib.kv_pool_free_count(h) == 4096


def test_numpy_token_arrays_match_lists(pool):
    """int32 numpy arrays (passed without a copy) give what lists give."""
    import numpy as np
    lib, h = pool
    c = pkv.PrefixCache(h)
    toks = list(range(3000, 3048))
    pages = alloc(lib, h, 3)
    assert c.insert(np.array(toks, dtype=np.int32), pages) == 3
    assert c.match(np.array(toks, dtype=np.int32)) == pages
    assert c.match(toks) == pages
    release(lib, h, pages)
    release(lib, h, pages)
    release(lib, h, pages)
    c.destroy()


def test_counters_match_a_model(pool):
    """Hit/miss counters and page counts against the brute-force model."""
    lib, h = pool
    P = 16
    rnd = random.Random(17)
    c = pkv.PrefixCache(h)
    model = {}
    held = []
    exp = dict.fromkeys(pkv.PREFIX_STATS_FIELDS, 0)
    for _ in range(80):
        toks = []
        for _ in range(rnd.randint(0, 5)):
            toks += [rnd.randint(0, 3)] * P
        toks += [9] * rnd.randint(0, P - 1)
        pages = alloc(lib, h, (len(toks) + P - 1) // P)
        held.append(pages)
        exp["pages_inserted"] += c.insert(toks, pages)
        for k in range(1, len(toks) // P + 1):
            model.setdefault(tuple(toks[:k * P]), pages[k - 1])
        q = []
        for _ in range(rnd.randint(0, 6)):
            q += [rnd.randint(0, 3)] * P
        q += [9] * rnd.randint(0, P - 1)
        cap = rnd.choice([None, 0, 1, 3])
        got = c.match(q, cap)
        want = _model_match(model, q, P)[:cap]
        assert got == want
        asked = len(q) // P if cap is None else min(cap, len(q) // P)
        exp["lookups"] += 1
        exp["hits" if got else "misses"] += 1
        exp["pages_hit"] += len(got)
        exp["pages_missed"] += asked - len(got)
        release(lib, h, got)
    assert exp["pages_inserted"] == len(model)
    assert c.stats() == exp
    for pages in held:
        release(lib, h, pages)
    freed = c.evict(7)
    assert freed == 7
    exp["pages_evicted"] = 7
    assert c.stats(reset=True) == exp
    assert c.stats() == dict.fromkeys(pkv.PREFIX_STATS_FIELDS, 0)
    c.destroy()


def test_stats_rejects_null(pool):
    lib, _ = pool
    buf = (ctypes.c_uint64 * 7)()
    assert lib.pkv_prefix_cache_get_stats(None, 0, buf) == 1
