"""Host logic of the radix prefix cache (oscar_radix_*) on the page
allocator, checked against a plain Python model; no GPU."""
import numpy as np
import pytest

from bit_kv_cache_evict_gb300 import build as B
from bit_kv_cache_evict_gb300 import oscar as O

C = 64


@pytest.fixture(scope="module", autouse=True)
def _lib():
    B.build()
    O.lib()


def _ctx(chunks):
    """A context whose chunk i is filled with the value chunks[i]."""
    return np.repeat(np.asarray(chunks, np.int32), C)


def test_match_follows_the_whole_chain():
    P = O.Pages(16)
    R = O.Radix(P)
    pg = P.alloc(3)
    R.insert(_ctx([7, 1, 2, 3]), pg)                       # sink chunk 7, history pages for chunks 1..3
    assert R.cached_pages() == 3 and [P.refcount(int(p)) for p in pg] == [2, 2, 2]
    got = R.match(_ctx([7, 1, 2, 3, 4]), 8)
    assert list(got) == list(pg) and P.refcount(int(pg[0])) == 3
    assert list(R.match(_ctx([7, 1, 9, 3]), 8)) == [pg[0]]   # diverges at chunk 2
    assert len(R.match(_ctx([8, 1, 2, 3]), 8)) == 0          # another sink: nothing is reusable
    assert list(R.match(_ctx([7, 1, 2, 3]), 2)) == list(pg[:2])
    part = np.concatenate([_ctx([7, 1]), np.full(C - 1, 2, np.int32)])
    assert list(R.match(part, 8)) == [pg[0]]                 # only whole chunks


def test_insert_keeps_cached_pages_and_validates():
    P = O.Pages(16)
    R = O.Radix(P)
    a = P.alloc(2)
    R.insert(_ctx([1, 2, 3]), a)
    b = P.alloc(3)
    R.insert(_ctx([1, 2, 3, 4]), b)                         # chunks 1, 2 cached: only chunk 3's page is new
    assert R.cached_pages() == 3
    assert P.refcount(int(b[0])) == 1 and P.refcount(int(b[2])) == 2
    assert list(R.match(_ctx([1, 2, 3, 4]), 8)) == [a[0], a[1], b[2]]
    with pytest.raises(O.OscarError):
        R.insert(_ctx([1, 2]), P.alloc(2))                  # too few tokens for two pages
    with pytest.raises(O.OscarError):
        R.insert(_ctx([5, 6, 7]), [15, 14])                 # free pages
    assert R.cached_pages() == 3


def test_evict_frees_unreferenced_leaves_in_lru_order():
    P = O.Pages(16)
    R = O.Radix(P)
    x = P.alloc(2)
    y = P.alloc(2)
    R.insert(_ctx([1, 2, 3]), x)
    R.insert(_ctx([1, 5, 6]), y)
    P.release(x)
    P.release(y)                                            # only the cache holds them now
    held = R.match(_ctx([1, 2, 3]), 8)                      # a sequence holds x; x's path is the most recent
    free0 = P.free_count()
    assert R.evict(1) == 1 and P.refcount(int(y[1])) == 0   # y's leaf goes first (least recent, unheld)
    assert R.evict(10) == 1 and P.refcount(int(y[0])) == 0  # then y's first page; x's pages are held
    assert P.free_count() == free0 + 2 and R.cached_pages() == 2
    P.release(held)
    assert R.evict(10) == 2 and R.cached_pages() == 0 and P.free_count() == 16
    R.close()


def test_destroy_drops_the_cache_references():
    P = O.Pages(8)
    R = O.Radix(P)
    p = P.alloc(3)
    R.insert(_ctx([1, 1, 1, 1]), p)
    P.release(p)
    R.close()
    assert P.free_count() == 8


def test_random_operations_match_a_model():
    rng = np.random.default_rng(9)
    P = O.Pages(64)
    R = O.Radix(P)
    tree = {}          # chunk path (tuple) -> page (None for the sink level)
    stamp = {}         # chunk path -> last touch
    clock = 0
    held = []          # page lists handed to "sequences"
    for _ in range(400):
        op = int(rng.integers(0, 4))
        chunks = [int(v) for v in rng.integers(0, 3, int(rng.integers(1, 6)))]
        npg = len(chunks) - 1
        if op == 0 and npg > 0 and P.free_count() >= npg:      # a sequence caches its pages
            pg = P.alloc(npg)
            R.insert(_ctx(chunks), pg)
            clock += 1
            for c in range(len(chunks)):
                path = tuple(chunks[:c + 1])
                if path not in tree:
                    tree[path] = None if c == 0 else int(pg[c - 1])
                stamp[path] = clock
            P.release(pg)
        elif op == 1:                                           # a new request matches
            clock += 1
            got, path = [], ()
            for c in range(len(chunks)):
                path = path + (chunks[c],)
                if path not in tree:
                    break
                stamp[path] = clock
                if c > 0:
                    got.append(tree[path])
            assert list(R.match(_ctx(chunks), 16)) == got
            held.append(got)
        elif op == 2 and held:                                  # a sequence ends
            P.release(held.pop(int(rng.integers(0, len(held)))))
        elif op == 3:                                           # memory pressure
            want = int(rng.integers(1, 4))
            freed = 0
            while freed < want:
                leaves = [p for p in tree if not any(q[:len(p)] == p and len(q) > len(p) for q in tree)]
                refs = {pg: sum(pg in h for h in held) for pg in tree.values() if pg is not None}
                cand = [p for p in leaves if tree[p] is None or refs[tree[p]] == 0]
                if not cand:
                    break
                best = min(cand, key=lambda p: stamp[p])
                if tree[best] is not None:
                    freed += 1
                del tree[best]
            assert R.evict(want) == freed
        cached = sorted(pg for pg in tree.values() if pg is not None)
        assert R.cached_pages() == len(cached)
        for pg in range(64):
            want = (pg in cached) + sum(h.count(pg) for h in held)
            assert P.refcount(pg) == want, (pg, P.refcount(pg), want)
