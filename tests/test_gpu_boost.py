"""GPU parity of the K channel precision boost (oscar_evict_quantize_boost,
oscar_decode_attn_boost) against the float64 oracle (oracle/kitty.py on top
of the C oracle's eviction).

Eviction: the pool is checked like the uniform eviction's; the boost records
are bit-exact except where the oracle leaves the choice open within the
eviction's error window: a position chosen on one side only has an oracle
error within 1e-5 of the oracle's eighth largest (a near-tie of the
ranking), and a 4-bit code may differ only where 5u lies within 5e-5 of a
rounding midpoint (u within 1e-5 of (k + 1/2) / 5).  Decode: the oracle
attends over the GPU-written pool and records; max-abs 2e-3, rel-L2 1e-3.
"""
import numpy as np
import pytest

import oracle
from bit_kv_cache_evict_gb300 import synth as S
from oracle import kitty as K

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import gpu_harness as H  # noqa: E402
from bit_kv_cache_evict_gb300 import build as B  # noqa: E402
from bit_kv_cache_evict_gb300 import oscar as O  # noqa: E402

BOUND = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    B.build()
    O.lib()


def _setup(hist, hq, hk, g, seed, perm_seed=0):
    w = S.Workload(seed, "boost", batch=len(hist), hq=hq, hk=hk)
    orc = oracle.get()
    shape = oracle.Shape(S.D, g, S.SINK, S.RECENT, S.PAGE, hq, hk)
    hist = np.asarray(hist, np.int32)
    rc, table, npages, nbytes = orc.pool_layout(shape, hist + 64, None, 0, perm_seed, None)
    assert rc == 0
    rng = S.rng_for(w, 3)
    prof = S.channel_profile(w)
    src = np.concatenate([S.kv_tokens(w, int(h), rng, prof) for h in hist])
    seq = np.concatenate([np.full(h, b, np.int32) for b, h in enumerate(hist)])
    pos = np.concatenate([np.arange(h, dtype=np.int32) for h in hist])
    U = S.rotation_U(w).astype(np.float32)
    clip = S.clip_ratios(w)
    bf16_kv = S.kv_tokens(w, len(hist) * S.NSLOT, rng, prof).reshape(len(hist), S.NSLOT, hk, 2, S.D)
    q = S.queries(w, rng, len(hist))
    return orc, shape, hist, table, npages, nbytes, src, seq, pos, U, clip, bf16_kv, q


def _evict_gpu(shape, src, seq, pos, U, clip, table, npages, nbytes, B_):
    sh = O.oscar_shape(*[getattr(shape, f) for f in ("head_dim", "quant_group", "sink", "recent", "page_size",
                                                      "num_q_heads", "num_kv_heads")])
    hk = shape.num_kv_heads
    pool = torch.zeros(max(nbytes, 16), dtype=torch.uint8, device="cuda")
    boost = torch.full((max(npages * hk * K.BLOCK, 16),), 0xEE, dtype=torch.uint8, device="cuda")
    O.oscar_evict_quantize_boost(sh, H.bf16_t(src), H.i32_t(seq), H.i32_t(pos), H.f32_t(U), H.f32_t(clip), pool,
                                 boost, H.i32_t(table), B_, table.shape[1], npages)
    torch.cuda.synchronize()
    return sh, pool, boost


def _check_records(pool_g, pool_o, boost_g, table, seq, pos, u, hk, g):
    """Returns the number of exempt records; asserts the rest bit-exact.

    A record is a function of the clipped values and the STORED s and z; where
    the GPU stored another s or z than the oracle (the fp16-midpoint window
    of the eviction's parity rule), the expected record is taken from the
    oracle's clipped values y_c = z + s u with the GPU's s and z."""
    exempt = 0
    for i in range(seq.size):
        b, p = int(seq[i]), int(pos[i])
        page = int(table[b, p // 64])
        for kv in range(hk):
            off = (page * hk + kv) * K.BLOCK + (p % 64) * K.RECORD
            rg = boost_g[off:off + K.RECORD]
            codes, s, z = K.read_k(pool_g, table, b, p, kv, hk, g)
            _, so, zo = K.read_k(pool_o, table, b, p, kv, hk, g)
            grp = np.arange(128) // g
            uu = u[i, kv, 0]
            if not (np.array_equal(s, so) and np.array_equal(z, zo)):
                yc = zo[grp] + so[grp] * uu
                uu = np.where(s[grp] != 0, (yc - z[grp]) / np.where(s[grp] != 0, s[grp], 1.0), 0.0)
            nz = np.repeat(s != 0, g)
            ro = K.record(uu, codes, nz)
            if np.array_equal(rg, ro):
                continue
            pg, qg = K.parse(rg)
            po, qo = K.parse(ro)
            err = np.where(nz, np.abs(uu - codes), 0.0)
            eighth = np.sort(err)[::-1][K.NB - 1]
            for p_ in np.setxor1d(pg, po):
                assert abs(err[p_] - eighth) < BOUND, (b, p, kv, int(p_), err[p_], eighth, list(pg), list(po))
            for p_ in np.intersect1d(pg, po):
                a, c = qg[list(pg).index(p_)], qo[list(po).index(p_)]
                if a != c:
                    f = 5 * uu[p_]
                    assert abs(f - np.floor(f) - 0.5) < 5 * BOUND, (b, p, kv, int(p_), a, c, f)
            exempt += 1
    return exempt


@pytest.mark.parametrize("g,hq,hk,perm", [(32, 8, 2, 0), (128, 8, 2, 7), (64, 4, 2, 0), (32, 16, 2, 3)])
def test_boost_eviction_and_decode_match_oracle(g, hq, hk, perm):
    hist = [700, 1300, 2050]
    orc, shape, hist, table, npages, nbytes, src, seq, pos, U, clip, bf16_kv, q = _setup(hist, hq, hk, g, 51, perm)
    sh, pool_t, boost_t = _evict_gpu(shape, src, seq, pos, U, clip, table, npages, nbytes, len(hist))
    pool_g, boost_g = pool_t.cpu().numpy(), boost_t.cpu().numpy()
    pool_o = np.zeros(max(nbytes, 16), np.uint8)
    boost_o = np.zeros(max(npages * hk * K.BLOCK, 16), np.uint8)
    aux = K.evict(orc, shape, src, seq, pos, U.astype(np.float64), clip, pool_o, table, table.shape[1], boost_o)
    u = aux[0]
    items = [(int(seq[i]), int(pos[i]), i) for i in range(seq.size)]
    allowed = np.zeros_like(pool_o)
    H.compare_evicted(pool_g, pool_o, table, items, aux, hk, g, allowed=allowed)
    H.assert_pools_equal_except(pool_g, pool_o, allowed)
    n_ex = _check_records(pool_g, pool_o, boost_g, table, seq, pos, u, hk, g)
    assert n_ex <= max(2, 2e-3 * seq.size * hk), n_ex

    B_ = len(hist)
    bf16_len = np.full(B_, S.NSLOT, np.int32)
    out = torch.zeros((B_, hq, S.D), dtype=torch.float32, device="cuda")
    ws = torch.zeros(O.oscar_decode_workspace_bytes(sh, B_, table.shape[1]), dtype=torch.uint8, device="cuda")
    O.oscar_decode_attn_boost(sh, H.bf16_t(q), H.bf16_t(bf16_kv), H.i32_t(bf16_len), pool_t, boost_t,
                              H.i32_t(table), table.shape[1], npages, H.i32_t(hist), H.f32_t(U), 1 / np.sqrt(S.D),
                              out, ws)
    torch.cuda.synchronize()
    ref = K.decode(orc, shape, q, bf16_kv, bf16_len, pool_g, table, hist, U.astype(np.float64), boost_g,
                   1 / np.sqrt(S.D))
    err, rel = H.assert_close(out.cpu().numpy(), ref)
    print(f"boost g={g} G={hq // hk}: max-abs {err:.3e} rel-L2 {rel:.3e} exempt records {n_ex}")


@pytest.mark.parametrize("hist,hq,hk", [([0, 17, 64, 130], 2, 2), ([1, 63, 65], 4, 1)])
def test_boost_edge_histories(hist, hq, hk):
    """Empty, one-token, page-sized and ragged histories, G = 1 and G = 4."""
    orc, shape, hist, table, npages, nbytes, src, seq, pos, U, clip, bf16_kv, q = _setup(hist, hq, hk, 32, 57)
    sh, pool_t, boost_t = _evict_gpu(shape, src, seq, pos, U, clip, table, npages, nbytes, len(hist))
    pool_g, boost_g = pool_t.cpu().numpy(), boost_t.cpu().numpy()
    pool_o = np.zeros(max(nbytes, 16), np.uint8)
    boost_o = np.zeros(max(npages * hk * K.BLOCK, 16), np.uint8)
    aux = K.evict(orc, shape, src, seq, pos, U.astype(np.float64), clip, pool_o, table, table.shape[1], boost_o)
    items = [(int(seq[i]), int(pos[i]), i) for i in range(seq.size)]
    allowed = np.zeros_like(pool_o)
    H.compare_evicted(pool_g, pool_o, table, items, aux, hk, 32, allowed=allowed)
    H.assert_pools_equal_except(pool_g, pool_o, allowed)
    _check_records(pool_g, pool_o, boost_g, table, seq, pos, aux[0], hk, 32)
    B_ = len(hist)
    bf16_len = np.array([S.NSLOT, 5, S.NSLOT, 200][:B_], np.int32)
    out = torch.zeros((B_, hq, S.D), dtype=torch.float32, device="cuda")
    ws = torch.zeros(O.oscar_decode_workspace_bytes(sh, B_, table.shape[1]), dtype=torch.uint8, device="cuda")
    O.oscar_decode_attn_boost(sh, H.bf16_t(q), H.bf16_t(bf16_kv), H.i32_t(bf16_len), pool_t, boost_t,
                              H.i32_t(table), table.shape[1], npages, H.i32_t(hist), H.f32_t(U), 1 / np.sqrt(S.D),
                              out, ws)
    torch.cuda.synchronize()
    ref = K.decode(orc, shape, q, bf16_kv, bf16_len, pool_g, table, hist, U.astype(np.float64), boost_g,
                   1 / np.sqrt(S.D))
    H.assert_close(out.cpu().numpy(), ref)


def test_records_without_correction_give_the_uniform_decode():
    """Records whose 4-bit codes equal 5c (written on the host from the
    GPU pool) make oscar_decode_attn_boost equal oscar_decode_attn."""
    hist = [900, 333]
    hq, hk = 4, 1
    orc, shape, hist, table, npages, nbytes, src, seq, pos, U, clip, bf16_kv, q = _setup(hist, hq, hk, 32, 53)
    sh, pool_t, boost_t = _evict_gpu(shape, src, seq, pos, U, clip, table, npages, nbytes, len(hist))
    pool_g, boost_g = pool_t.cpu().numpy(), boost_t.cpu().numpy()
    for i in range(seq.size):
        b, p = int(seq[i]), int(pos[i])
        off = int(table[b, p // 64]) * K.BLOCK + (p % 64) * K.RECORD
        ps, _ = K.parse(boost_g[off:off + K.RECORD])
        codes, _, _ = K.read_k(pool_g, table, b, p, 0, 1, 32)
        c = codes[ps].astype(np.int64)
        boost_g[off:off + K.RECORD] = (ps | (5 * c << 8) | (c << 12)).astype("<u2").view(np.uint8)
    B_ = len(hist)
    bf16_len = np.full(B_, S.NSLOT, np.int32)
    a = (sh, H.bf16_t(q), H.bf16_t(bf16_kv), H.i32_t(bf16_len), pool_t)
    rest = (H.i32_t(table), table.shape[1], npages, H.i32_t(hist), H.f32_t(U), 1 / np.sqrt(S.D))
    outs = []
    for boosted in (False, True):
        out = torch.zeros((B_, hq, S.D), dtype=torch.float32, device="cuda")
        ws = torch.zeros(O.oscar_decode_workspace_bytes(sh, B_, table.shape[1]), dtype=torch.uint8, device="cuda")
        if boosted:
            O.oscar_decode_attn_boost(*a, H.u8_t(boost_g), *rest, out, ws)
        else:
            O.oscar_decode_attn(*a, *rest, out, ws)
        torch.cuda.synchronize()
        outs.append(out.cpu().numpy().astype(np.float64))
    assert np.abs(outs[0] - outs[1]).max() <= 1e-5 * max(1.0, np.abs(outs[0]).max())
