"""CPU tests of the C-ABI library: it loads, exports every declared entry
point, and its host-only logic (page-table layout, argument checks) matches
the oracle / the header's contract.  No compute call needs a GPU here."""
import ctypes

import numpy as np
import pytest

import oracle
from bit_kv_cache_evict_gb300 import build as B
from bit_kv_cache_evict_gb300 import oscar as O


@pytest.fixture(scope="module")
def lib():
    B.build()
    return O.lib()


def test_exports_every_declared_symbol(lib):
    names = O.declared_functions()
    assert {"oscar_pool_layout", "oscar_evict_quantize", "oscar_decode_attn"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def orc_block_bytes(g):
    import oracle as orcmod
    return orcmod.get().block_bytes(128, g, 64)


def test_block_bytes_and_status_strings(lib):
    assert O.block_bytes(O.make_shape(32, 8)) == 6144
    assert O.block_bytes(O.make_shape(32, 8, quant_group=64)) == 5120
    assert O.block_bytes(O.make_shape(32, 8, quant_group=128)) == 4608
    assert O.block_bytes(O.make_shape(32, 8, quant_group=16)) == 0       # unsupported
    for g in (32, 64, 128):   # the oracle's block size for the same shape
        assert O.block_bytes(O.make_shape(32, 8, quant_group=g)) == orc_block_bytes(g)
    for st in range(6):
        assert lib.oscar_status_string(st)


CASES = [
    (np.array([64, 1, 0, 130, 640]), None, 0, 0),
    (np.array([64, 1, 0, 130, 640]), None, 0, 77),
    (np.array([300, 200, 500, 256]), np.array([0, -1, 0, 0]), 128, 0),
    (np.array([300, 200, 500, 256, 700, 1000]), np.array([1, -1, 1, 1, 2, 2]), 256, 5),
    (np.random.default_rng(0).integers(0, 5000, 64), None, 0, 1003),
]


@pytest.mark.parametrize("g", [32, 128])
@pytest.mark.parametrize("cap,grp,shared,seed", CASES)
def test_pool_layout_matches_oracle(lib, orc, cap, grp, shared, seed, g):
    sh = O.make_shape(32, 8, quant_group=g)
    mp = int(max(1, (cap.max() + 63) // 64)) + 1
    t, n, nb = O.oscar_pool_layout(sh, cap, grp, shared, seed, mp)
    rc, t2, n2, nb2 = orc.pool_layout(oracle.Shape(128, g, 64, 256, 64, 32, 8), cap, grp, shared, seed, mp)
    assert rc == 0
    assert np.array_equal(t, t2) and n == n2 and nb == nb2


def test_pool_layout_errors(lib):
    sh = O.make_shape(32, 8)
    with pytest.raises(O.OscarError) as e:
        O.oscar_pool_layout(sh, np.array([65 * 64]), max_pages=64)
    assert e.value.status == O.OSCAR_ERR_OUT_OF_PAGES
    with pytest.raises(O.OscarError) as e:
        O.oscar_pool_layout(sh, np.array([300, 300]), np.array([0, 0]), 100, 0, 8)
    assert e.value.status == O.OSCAR_ERR_INVALID_ARG
    with pytest.raises(O.OscarError) as e:
        O.oscar_pool_layout(O.make_shape(24, 8), np.array([10]), max_pages=4)     # G = 3
    assert e.value.status == O.OSCAR_ERR_UNSUPPORTED


def test_argument_checks_before_launch(lib):
    """Host-side validation returns before touching the GPU (NULL / bad sizes)."""
    sh = O.make_shape(32, 8)
    ws = ctypes.c_size_t(0)
    # workspace query needs no device
    assert lib.oscar_decode_attn(ctypes.byref(sh), 4, None, None, None, None, None, 10, 0, None, None,
                                 ctypes.c_float(1.0), None, None, ctypes.byref(ws), None, None) == O.OSCAR_OK
    assert ws.value > 0
    small = ctypes.c_size_t(ws.value - 1)
    fake = ctypes.c_void_p(256)
    assert lib.oscar_decode_attn(ctypes.byref(sh), 4, fake, fake, fake, fake, fake, 10, 1, fake, fake,
                                 ctypes.c_float(1.0), fake, fake, ctypes.byref(small), None,
                                 None) == O.OSCAR_ERR_WORKSPACE
    assert lib.oscar_decode_attn(ctypes.byref(sh), 4, None, None, None, None, None, 0, 0, None, None,
                                 ctypes.c_float(1.0), None, fake, ctypes.byref(ws), None,
                                 None) == O.OSCAR_ERR_INVALID_ARG       # max_pages = 0
    assert lib.oscar_decode_attn(ctypes.byref(sh), 4, None, None, None, None, None, 10, 0, None, None,
                                 ctypes.c_float(1.0), None, fake, ctypes.byref(ws), None,
                                 None) == O.OSCAR_ERR_INVALID_ARG       # NULL q
    mis = ctypes.c_void_p(258)
    assert lib.oscar_decode_attn(ctypes.byref(sh), 4, mis, fake, fake, fake, fake, 10, 1, fake, fake,
                                 ctypes.c_float(1.0), fake, fake, ctypes.byref(ws), None,
                                 None) == O.OSCAR_ERR_INVALID_ARG       # misaligned q
    # eviction: n_tok = 0 is a no-op; NULL pointers are rejected
    assert lib.oscar_evict_quantize(ctypes.byref(sh), 0, None, 0, None, None, None, None, None, None, None, None,
                                    1, 1, 1, None, None) == O.OSCAR_OK
    assert lib.oscar_evict_quantize(ctypes.byref(sh), 3, None, 3, None, None, None, None, None, None, None, None,
                                    1, 1, 1, None, None) == O.OSCAR_ERR_INVALID_ARG
    bad = O.make_shape(32, 8, head_dim=96)
    assert lib.oscar_evict_quantize(ctypes.byref(bad), 3, fake, 3, None, fake, fake, None, fake, fake, fake, fake,
                                    1, 1, 1, None, None) == O.OSCAR_ERR_UNSUPPORTED


def test_variant_calls_validate_before_launch(lib):
    """The Lloyd-Max and channel-boost calls reject a missing or misaligned
    codebook or boost array before touching the GPU."""
    fake = ctypes.c_void_p(4096)
    ws = ctypes.c_size_t(1 << 30)
    for fn, extra in (("oscar_decode_attn_codebook", "codebook"), ("oscar_decode_attn_boost", "boost")):
        f = getattr(lib, fn)
        if extra == "codebook":
            args = lambda sh, cb: (ctypes.byref(sh), 4, fake, fake, fake, fake, fake, 10, 1, fake, fake, cb,  # noqa: E731
                                   ctypes.c_float(1.0), fake, fake, ctypes.byref(ws), None, None)
        else:
            args = lambda sh, cb: (ctypes.byref(sh), 4, fake, fake, fake, fake, cb, fake, 10, 1, fake, fake,  # noqa: E731
                                   ctypes.c_float(1.0), fake, fake, ctypes.byref(ws), None, None)
        assert f(*args(O.make_shape(32, 8), None)) == O.OSCAR_ERR_INVALID_ARG
        assert f(*args(O.make_shape(32, 8), ctypes.c_void_p(4098))) == O.OSCAR_ERR_INVALID_ARG   # misaligned
    sh = O.make_shape(32, 8)
    assert lib.oscar_evict_quantize_codebook(ctypes.byref(sh), 3, fake, 3, None, fake, fake, None, fake, fake, None,
                                             fake, fake, 1, 1, 1, None, None) == O.OSCAR_ERR_INVALID_ARG
    assert lib.oscar_evict_quantize_boost(ctypes.byref(sh), 3, fake, 3, None, fake, fake, None, fake, fake, fake,
                                          None, fake, 1, 1, 1, None, None) == O.OSCAR_ERR_INVALID_ARG
    assert lib.oscar_evict_quantize_boost(ctypes.byref(sh), 0, None, 0, None, None, None, None, None, None, None,
                                          None, None, 1, 1, 1, None, None) == O.OSCAR_OK          # nothing to do


def test_workspace_query_rejects_int32_overflow(lib):
    """Split-K item counts and partial offsets are int32 on the device: a
    batch x pages shape whose item count (or partial-buffer word count) does
    not fit is rejected by the workspace query itself, on the host, instead
    of wrapping.  Items per (sequence, KV head) = ceil(max_pages / pps) + 2
    short tail items, pps = 256 pages for these sizes."""
    sh = O.make_shape(32, 8)                       # G = 4: a partial is 4 x 130 floats
    ws = ctypes.c_size_t(0)

    def query(batch, max_pages):
        return lib.oscar_decode_attn(ctypes.byref(sh), batch, None, None, None, None, None, max_pages, 0, None,
                                     None, ctypes.c_float(1.0), None, None, ctypes.byref(ws), None, None)

    assert query(1024, 2048) == O.OSCAR_OK         # 8192 x (8 + 2) items
    assert 81920 * 520 * 4 < ws.value < 2 * 81920 * 520 * 4 + (1 << 28)
    assert query(1 << 20, 1 << 16) == O.OSCAR_ERR_INVALID_ARG    # 2^23 x 258 items > 2^31 - 1
    assert query(1 << 16, 1 << 12) == O.OSCAR_ERR_INVALID_ARG    # 9.4e6 items x 520 words > 4e9 words
    assert query(1 << 14, 1 << 12) == O.OSCAR_OK                 # 2.4e6 items x 520 words = 1.2e9 words
