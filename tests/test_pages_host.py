"""Host logic of the refcounted copy-on-write page allocator (oscar_pages_*),
checked against a plain Python model of reference counts; no GPU."""
import ctypes

import numpy as np
import pytest

from bit_kv_cache_evict_gb300 import build as B
from bit_kv_cache_evict_gb300 import oscar as O


@pytest.fixture(scope="module", autouse=True)
def _lib():
    B.build()
    O.lib()


def test_alloc_order_and_exhaustion():
    P = O.Pages(5)
    assert list(P.alloc(3)) == [0, 1, 2] and P.free_count() == 2
    with pytest.raises(O.OscarError) as e:
        P.alloc(3)
    assert e.value.status == O.OSCAR_ERR_OUT_OF_PAGES and P.free_count() == 2      # nothing taken
    P.release([1])
    assert P.refcount(1) == 0 and list(P.alloc(1)) == [1]                          # freed page reused first


def test_retain_release_validation_leaves_state():
    P = O.Pages(4)
    a = P.alloc(2)
    P.retain([a[0], a[0]])
    assert P.refcount(a[0]) == 3
    for bad in ([3], [a[1], a[1]], [-1], [9]):                                     # free, too many, out of range
        with pytest.raises(O.OscarError) as e:
            P.release(bad)
        assert e.value.status == O.OSCAR_ERR_INVALID_ARG
    with pytest.raises(O.OscarError):
        P.retain([a[1], 3])                                                        # 3 is free: nothing retained
    assert (P.refcount(a[0]), P.refcount(a[1]), P.free_count()) == (3, 1, 2)
    assert P.refcount(-1) == -1 and P.refcount(4) == -1


def test_unaligned_prefix_copy_on_write():
    # sequences 0 and 1 share 3 pages; the prefix ends inside page 2, so both
    # write into it: the first writer gets a copy, the second keeps the page
    P = O.Pages(8)
    pre = P.alloc(3)
    P.retain(pre)
    t = np.full((3, 5), -1, np.int32)
    t[0, :3] = pre
    t[1, :3] = pre
    src, dst = P.prepare_write([0, 1, 0, 1, 2], [2, 2, 3, 3, 0], t)
    assert list(src) == [pre[2]] and P.refcount(pre[2]) == 1
    assert t[0, 2] == dst[0] and t[1, 2] == pre[2]
    assert list(t[0, :2]) == list(pre[:2]) == list(t[1, :2])                      # read-only pages stay shared
    assert P.refcount(pre[0]) == 2
    assert t[0, 3] >= 0 and t[1, 3] >= 0 and t[2, 0] >= 0                         # empty entries filled
    assert P.free_count() == 8 - 3 - 4


def test_prepare_write_out_of_pages_changes_nothing():
    P = O.Pages(3)
    pre = P.alloc(2)
    P.retain(pre)
    t = np.full((2, 3), -1, np.int32)
    t[0, :2] = pre
    t[1, :2] = pre
    before = t.copy()
    with pytest.raises(O.OscarError) as e:
        P.prepare_write([0, 0, 1], [0, 1, 2], t)                                   # needs 3 fresh pages, 1 free
    assert e.value.status == O.OSCAR_ERR_OUT_OF_PAGES
    assert np.array_equal(t, before) and P.free_count() == 1 and P.refcount(pre[0]) == 2
    with pytest.raises(O.OscarError) as e:
        P.prepare_write([0, 5], [0, 0], t)                                         # sequence out of range
    assert e.value.status == O.OSCAR_ERR_INVALID_ARG and np.array_equal(t, before)


def test_random_operations_match_a_reference_model():
    rng = np.random.default_rng(5)
    npg, B_, M = 40, 6, 8
    P = O.Pages(npg)
    t = np.full((B_, M), -1, np.int32)
    for _ in range(300):
        op = rng.integers(0, 3)
        if op == 0:                                  # a sequence adopts another's first pages (prefix hit)
            a, b = rng.choice(B_, 2, replace=False)
            k = int(rng.integers(1, M))
            if np.all(t[a, :k] >= 0) and np.all(t[b, :k] < 0):
                P.retain(t[a, :k])
                t[b, :k] = t[a, :k]
        elif op == 1:                                # write targets
            n = int(rng.integers(1, 5))
            seq = rng.integers(0, B_, n)
            pg = rng.integers(0, M, n)
            before = t.copy()
            try:
                src, dst = P.prepare_write(seq, pg, t)
            except O.OscarError as e:
                assert e.status == O.OSCAR_ERR_OUT_OF_PAGES and np.array_equal(t, before)
                continue
            for s_, p_ in zip(seq, pg):
                assert t[s_, p_] >= 0
                assert np.sum(t == t[s_, p_]) == 1                               # private after the call
            for a_, b_ in zip(src, dst):
                assert np.sum(before == a_) > 1 and np.sum(before == b_) == 0
        else:                                        # a sequence finishes
            b = int(rng.integers(0, B_))
            row = t[b][t[b] >= 0]
            P.release(row)
            t[b] = -1
        # model: a page's references are the table entries that hold it
        ids, counts = np.unique(t[t >= 0], return_counts=True)
        model = np.zeros(npg, np.int64)
        model[ids] = counts
        assert [P.refcount(i) for i in range(npg)] == list(model)
        assert P.free_count() == int(np.sum(model == 0))


def test_copy_validates_before_any_device_work():
    lib = O.lib()
    sh = O.make_shape(8, 2)
    src = (ctypes.c_int32 * 2)(1, 2)
    dst = (ctypes.c_int32 * 2)(3, 2)
    fake = ctypes.c_void_p(4096)
    assert lib.oscar_pages_copy(ctypes.byref(sh), 0, None, None, None, None, 4, None) == O.OSCAR_OK
    assert lib.oscar_pages_copy(ctypes.byref(sh), 2, src, dst, fake, None, 4, None) == O.OSCAR_ERR_INVALID_ARG
    dst2 = (ctypes.c_int32 * 2)(3, 7)
    assert lib.oscar_pages_copy(ctypes.byref(sh), 2, src, dst2, fake, None, 4, None) == O.OSCAR_ERR_INVALID_ARG
