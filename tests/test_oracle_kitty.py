"""Pins of the channel precision boost oracle (oracle/kitty.py)."""
import numpy as np

import oracle
from bit_kv_cache_evict_gb300 import synth as S
from oracle import kitty as K

D = 128


def _quant(y, g=32, clip=1.0):
    codes, s16, z16, u = oracle.get().quantize_vec(y, g, clip)[:4]
    s = np.asarray(s16, np.uint16).view(np.float16).astype(np.float64)
    z = np.asarray(z16, np.uint16).view(np.float16).astype(np.float64)
    return codes, s16, z16, u, s, z


def test_record_bytes_of_a_hand_built_case():
    # u = 0 everywhere except four positions; with c = rint(u) (half to even)
    # the errors are 0.5 (pos 5: c 0, q4 rint(2.5) = 2), 0.45 (pos 100:
    # u 1.45, c 1, q4 rint(7.25) = 7), 0.4 (pos 31: u 2.6, c 3, q4 13),
    # 0.3 (pos 64: u 0.3, c 0, q4 rint(1.5) = 2); the other four entries are
    # the lowest error-0 positions 0, 1, 2, 3 (q4 0); the code copy sits in
    # bits 12-13 (c = 1 at pos 100, 3 at pos 31)
    u = np.zeros(D)
    u[5], u[100], u[31], u[64] = 0.5, 1.45, 2.6, 0.3
    codes = np.clip(np.rint(u), 0, 3).astype(np.uint8)
    rec = K.record(u, codes, np.ones(D, bool))
    want = bytes([0, 0, 1, 0, 2, 0, 3, 0, 5, 2, 31, 0x3D, 64, 2, 100, 0x17])
    assert rec.tobytes() == want


def test_selected_errors_dominate_and_entries_are_sorted():
    rng = np.random.default_rng(7)
    for g in (32, 64, 128):
        for _ in range(20):
            y = rng.standard_normal(D) * rng.uniform(0.1, 5)
            codes, s16, z16, u, s, z = _quant(y, g, 0.9)
            nz = np.repeat(s != 0, g)
            rec = K.record(u, codes, nz)
            pos, q4 = K.parse(rec)
            assert pos.size == K.NB and np.all(np.diff(pos) > 0)
            assert np.array_equal(K.parse_codes(rec), codes[pos])
            err = np.abs(u - codes)
            others = np.setdiff1d(np.arange(D), pos)
            assert err[pos].min() >= err[others].max()


def test_boosted_codes_are_the_nearest_of_sixteen_levels():
    rng = np.random.default_rng(8)
    for _ in range(30):
        y = rng.standard_normal(D) * 2
        codes, s16, z16, u, s, z = _quant(y, 32, 0.95)
        pos, q4 = K.parse(K.record(u, codes, np.repeat(s != 0, 32)))
        yc = z[pos // 32] + s[pos // 32] * u[pos]          # the clipped value, from its definition of u
        for j, p in enumerate(pos):
            lv = z[p // 32] + s[p // 32] * np.arange(16) / 5.0
            assert int(np.argmin(np.abs(lv - yc[j]))) == q4[j]


def test_on_grid_vector_dequantises_like_the_uniform_path():
    # values on the 2-bit grid of every group: all errors 0, the boosted
    # positions are 0..7 with q4 = 5 c, and the K values equal the C
    # oracle's uniform dequantisation
    rng = np.random.default_rng(9)
    y = np.concatenate([rng.integers(0, 4, 32) * 0.25 - 0.5 for _ in range(4)])
    y[0::32] = -0.5
    y[1::32] = 0.25
    codes, s16, z16, u, s, z = _quant(y, 32, 1.0)
    rec = K.record(u, codes, np.repeat(s != 0, 32))
    pos, q4 = K.parse(rec)
    assert np.array_equal(pos, np.arange(8)) and np.array_equal(q4, 5 * codes[:8])
    ref = oracle.get().dequantize_vec(codes, s16, z16, 32)
    assert np.array_equal(K.dequantize_k(codes, s, z, rec, 32), ref)


def test_constant_groups_keep_their_value():
    y = np.full(D, 1.25)
    codes, s16, z16, u, s, z = _quant(y, 32, 1.0)
    rec = K.record(u, codes, np.repeat(s != 0, 32))
    assert np.all(K.dequantize_k(codes, s, z, rec, 32) == 1.25)


def _scene(seed):
    w = S.Workload(seed, "kitty_pin", batch=1, hq=1, hk=1)
    orc = oracle.get()
    shape = oracle.Shape(D, 32, 64, 256, 64, 1, 1)
    rc, table, npages, nbytes = orc.pool_layout(shape, np.array([64], np.int32))
    assert rc == 0
    rng = S.rng_for(w, 1)
    toks = S.kv_tokens(w, 2, rng, S.channel_profile(w))      # [2][1][2][d]
    toks[1, 0, 0] = toks[0, 0, 0]                            # identical K, different V
    U = S.rotation_U(w)[:1].astype(np.float64)
    clip = np.full((1, 2), 0.95)
    pool = np.zeros(nbytes, np.uint8)
    boost = np.zeros(npages * K.BLOCK, np.uint8)
    K.evict(orc, shape, toks, np.zeros(2, np.int32), np.arange(2, dtype=np.int32), U, clip, pool, table,
            table.shape[1], boost)
    q = S.queries(w, rng, 1)                                 # [1][1][d] bf16 bits
    return orc, shape, table, pool, boost, U, q


def test_decode_closed_form_of_one_changed_boost_code():
    """Two history tokens with the same stored K: moving token 1's first
    boosted code by dq shifts its logit by sm (q R_K)[pos] s dq / 5, so the
    output is (v0 + e^D v1) / (1 + e^D); v0 and v1 come from the C oracle's
    plain decode of the same pool."""
    orc, shape, table, pool, boost, U, q = _scene(21)
    sm = 0.3
    empty = np.zeros((1, 320, 1, 2, D), np.uint16)
    blen = np.zeros(1, np.int32)
    v0 = orc.decode(shape, q, empty, blen, pool, table, table.shape[1], np.array([1], np.int32), U, sm)[0, 0]
    mean = orc.decode(shape, q, empty, blen, pool, table, table.shape[1], np.array([2], np.int32), U, sm)[0, 0]
    v1 = 2 * mean - v0
    rec1 = boost[K.RECORD:2 * K.RECORD].copy()
    assert np.array_equal(rec1, boost[:K.RECORD])            # same K, same record
    pos, q4 = K.parse(rec1)
    p, dq = int(pos[0]), (1 if q4[0] < 15 else -1)
    ent = rec1.view("<u2").copy()
    ent[0] = (int(ent[0]) & ~0x0F00) | ((int(q4[0]) + dq) << 8)
    boost2 = boost.copy()
    boost2[K.RECORD:2 * K.RECORD] = ent.view(np.uint8)
    _, s, _ = K.read_k(pool, table, 0, 1, 0, 1, 32)
    qf = S.bf16_to_f32(q[0, 0]).astype(np.float64)
    qr = qf @ orc.build_R(U[0, 0])
    delta = sm * qr[p] * s[p // 32] * dq / 5.0
    want = (v0 + np.exp(delta) * v1) / (1 + np.exp(delta))
    got = K.decode(orc, shape, q, empty, blen, pool, table, np.array([2], np.int32), U, boost2, sm)[0, 0]
    assert np.abs(got - want).max() < 1e-12


def test_decode_without_correction_is_the_plain_oracle():
    """Records whose 4-bit codes equal 5 c change nothing: the decode equals
    the C oracle's."""
    orc, shape, table, pool, boost, U, q = _scene(22)
    for t in range(2):
        rec = boost[t * K.RECORD:(t + 1) * K.RECORD]
        pos, _ = K.parse(rec)
        codes, _, _ = K.read_k(pool, table, 0, t, 0, 1, 32)
        c = codes[pos].astype(np.int64)
        ent = (pos | (5 * c << 8) | (c << 12)).astype("<u2")
        boost[t * K.RECORD:(t + 1) * K.RECORD] = ent.view(np.uint8)
    rng = np.random.default_rng(3)
    bkv = S.bf16_bits(rng.standard_normal((1, 320, 1, 2, D)).astype(np.float32))
    blen = np.array([5], np.int32)
    hist = np.array([2], np.int32)
    ref = orc.decode(shape, q, bkv, blen, pool, table, table.shape[1], hist, U, 0.1)
    got = K.decode(orc, shape, q, bkv, blen, pool, table, hist, U, boost, 0.1)
    assert np.abs(got - ref).max() < 1e-12
