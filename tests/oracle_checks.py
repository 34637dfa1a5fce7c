"""Pins for the float64 oracle: each check ties an oracle function to
something other than itself (a library routine, a closed form, a published
test vector, a hand-derived golden value, brute force on small inputs, an
algebraic identity).  Checks are plain functions of an ``oracle.Oracle`` so
that tests/test_oracle_mutants.py can run them against oracle builds with a
planted mistake and confirm that each mistake is caught."""
from __future__ import annotations

import os

import numpy as np
import scipy.linalg

import oracle
from bit_kv_cache_evict_gb300 import synth as S

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def strrev_bits(j: int, nbits: int) -> int:
    return int(format(j, f"0{nbits}b")[::-1], 2)


def qr_U(seed: int, d: int = 128) -> np.ndarray:
    rng = np.random.default_rng(seed)
    q, r = np.linalg.qr(rng.standard_normal((d, d)))
    return q * np.sign(np.diag(r))[None, :]


# --------------------------------------------------------------------------
# rotation
# --------------------------------------------------------------------------

def check_hadamard(o: oracle.Oracle):
    """Sylvester Hadamard against scipy.linalg.hadamard (library)."""
    for k in range(1, 8):
        d = 1 << k
        H = o.hadamard(d)
        assert np.array_equal(H * np.sqrt(d), scipy.linalg.hadamard(d).astype(np.float64)) or \
            np.max(np.abs(H * np.sqrt(d) - scipy.linalg.hadamard(d))) < 1e-13
        assert np.max(np.abs(H @ H.T - np.eye(d))) < 1e-13


def check_bitrev(o: oracle.Oracle):
    """Bit reversal against string reversal of the binary digits; it is an
    involution."""
    for nb in range(1, 9):
        for j in range(1 << nb):
            r = o.bitrev(j, nb)
            assert r == strrev_bits(j, nb)
            assert o.bitrev(r, nb) == j


def check_R(o: oracle.Oracle):
    """R = U.H.P: orthogonal to 1e-12 and equal to the composition built
    from scipy's Hadamard and a string-reversal permutation."""
    d = 128
    U = qr_U(5, d)
    R = o.build_R(U)
    assert np.max(np.abs(R @ R.T - np.eye(d))) < 1e-12
    Hs = scipy.linalg.hadamard(d) / np.sqrt(d)
    perm = np.array([strrev_bits(j, 7) for j in range(d)])
    ref = (U @ Hs)[:, perm]
    assert np.max(np.abs(R - ref)) < 1e-13
    x = np.random.default_rng(1).standard_normal(d)
    assert np.max(np.abs(x @ R - ((x @ U) @ Hs)[perm])) < 1e-12
    # a non-orthogonal U is rejected by nothing: R must still equal U.H.P
    A = np.random.default_rng(2).standard_normal((d, d))
    assert np.max(np.abs(o.build_R(A) - (A @ Hs)[:, perm])) < 1e-11


def check_group_structure(o: oracle.Oracle):
    """With d=128, g=32, stored group k holds the Hadamard outputs j with
    j mod 4 == bitrev2(k): each group samples the whole spectrum, which is
    what the bit-reversal is there for."""
    for k in range(4):
        outs = {o.bitrev(p, 7) for p in range(32 * k, 32 * k + 32)}
        assert {j % 4 for j in outs} == {strrev_bits(k, 2)}
        assert len(outs) == 32


# --------------------------------------------------------------------------
# number formats
# --------------------------------------------------------------------------

def f16_edge_values() -> np.ndarray:
    tiny = 2.0 ** -24
    vals = [0.0, tiny, tiny * 0.5, tiny * 1.5, tiny * 2.5, tiny * 0.49999, tiny * 1023, tiny * 1023.5,
            tiny * 1024, 2.0 ** -14, 2.0 ** -14 * (1 - 2 ** -12), 65504.0, 65519.99, 65520.0, 65536.0, 1e9,
            1.0, 1.0 + 2 ** -11, 1.0 + 3 * 2 ** -11, 1.0 + 2 ** -11 + 1e-12, 2048.0 + 1.0, 2048.0 + 3.0,
            0.1, 1 / 3, 2 / 3, 1e-5, 6.1e-5, 3.14159265]
    vals = np.array(vals)
    return np.concatenate([vals, -vals])


def check_f16(o: oracle.Oracle):
    """float64 -> binary16 round-to-nearest-even against numpy.float16
    (library), on edge cases (subnormal, ties, overflow) and random values
    spanning the exponent range."""
    rng = np.random.default_rng(3)
    rand = rng.standard_normal(3000) * np.exp2(rng.uniform(-27, 17, 3000))
    x = np.concatenate([f16_edge_values(), rand])
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    got = o.f16_from_f64(x)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(x[i], hex(got[i]), hex(ref[i])) for i in bad[:5]]


def check_f16_decode(o: oracle.Oracle):
    """binary16 -> float64 for every non-NaN bit pattern, against numpy."""
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = pats.view(np.float16).astype(np.float64)
    keep = ~np.isnan(ref)
    got = o.f64_from_f16(pats[keep])
    assert np.array_equal(got, ref[keep])


def check_bf16(o: oracle.Oracle):
    rng = np.random.default_rng(4)
    pats = rng.integers(0, 65536, 4000).astype(np.uint16)
    pats = pats[(pats & 0x7F80) != 0x7F80]          # drop Inf/NaN patterns
    ref = (pats.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    keep = ~np.isnan(ref)
    assert np.array_equal(o.f64_from_bf16(pats[keep]), ref[keep])


def check_pack(o: oracle.Oracle):
    """Four codes per byte: exhaustive round trip, and the fixed bit order
    (code i in bits 2i..2i+1)."""
    for byte in range(256):
        c = o.unpack4(byte)
        assert o.pack4(c) == byte
        assert all(int(c[i]) == (byte >> (2 * i)) & 3 for i in range(4))
    assert o.pack4([1, 2, 3, 0]) == 0b00111001
    assert o.pack4([0, 0, 0, 3]) == 0xC0


# --------------------------------------------------------------------------
# quantiser
# --------------------------------------------------------------------------

def check_on_grid(o: oracle.Oracle):
    """Values already on the 4-level grid (dyadic s, z, each group using
    levels 0 and 3) requantise to the same codes, s and z exactly; exact
    midpoints round half to even."""
    rng = np.random.default_rng(6)
    for trial in range(200):
        g = [32, 64, 128][trial % 3]
        d = 128
        ng = d // g
        s = (rng.integers(1, 1024, ng) * 2.0 ** rng.integers(-12, 2, ng))
        z = (rng.integers(-1024, 1024, ng) * 2.0 ** rng.integers(-10, 2, ng))
        codes = rng.integers(0, 4, d)
        for k in range(ng):
            codes[k * g] = 0
            codes[k * g + 1] = 3
        y = np.repeat(s, g) * codes + np.repeat(z, g)
        c, s16, z16, u, sp, zp = o.quantize_vec(y, g, 1.0)
        assert np.array_equal(c, codes)
        assert np.array_equal(s16, s.astype(np.float16).view(np.uint16))
        assert np.array_equal(z16, z.astype(np.float16).view(np.uint16))
    # exact midpoints: u = 0.5 -> 0, 1.5 -> 2, 2.5 -> 2
    y = np.zeros(32)
    y[0], y[1] = 0.0, 3.0
    y[2], y[3], y[4] = 0.5, 1.5, 2.5
    c = o.quantize_vec(y, 32, 1.0)[0]
    assert list(c[:5]) == [0, 3, 0, 2, 2]


def check_nearest_level(o: oracle.Oracle):
    """Every code names the nearest level of the *stored* grid
    {s*c + z : c = 0..3}, clamped, ties aside; this fixes that codes come
    from the fp16 scale and zero, not the pre-rounding ones."""
    rng = np.random.default_rng(7)
    for trial in range(300):
        y = rng.standard_normal(128) * np.exp2(rng.uniform(-6, 6))
        clip = [1.0, 0.95, 0.8][trial % 3]
        c, s16, z16, u, sp, zp = o.quantize_vec(y, 32, clip)
        s = s16.view(np.float16).astype(np.float64)
        z = z16.view(np.float16).astype(np.float64)
        for k in range(4):
            yg = y[32 * k:32 * k + 32]
            t = clip * np.max(np.abs(yg))
            yc = np.minimum(np.maximum(yg, -t), t)
            levels = s[k] * np.arange(4) + z[k]
            dist = np.abs(yc[:, None] - levels[None, :])
            best = np.argmin(dist, axis=1)
            srt = np.sort(dist, axis=1)
            clear = (srt[:, 1] - srt[:, 0]) > 1e-9 * s[k]
            assert np.array_equal(c[32 * k:32 * k + 32][clear], best[clear])


def check_error_bound(o: oracle.Oracle):
    """|yhat - clamp(y)| <= s/2 plus the fp16 rounding of s and z."""
    rng = np.random.default_rng(8)
    for trial in range(300):
        y = rng.standard_normal(128) * np.where(rng.random(128) < 0.05, 20.0, 1.0)
        clip = 1.0 if trial % 2 else 0.95
        c, s16, z16, u, sp, zp = o.quantize_vec(y, 32, clip)
        yhat = o.dequantize_vec(c, s16, z16, 32)
        s = s16.view(np.float16).astype(np.float64)
        z = z16.view(np.float16).astype(np.float64)
        for k in range(4):
            yg = y[32 * k:32 * k + 32]
            t = clip * np.max(np.abs(yg))
            yc = np.minimum(np.maximum(yg, -t), t)
            err = np.abs(yhat[32 * k:32 * k + 32] - yc)
            bound = s[k] / 2 + 3 * 2.0 ** -11 * s[k] + 2.0 ** -11 * abs(z[k]) + 1e-12
            assert np.all(err <= bound)


def check_minmax_textbook(o: oracle.Oracle):
    """Clip ratio 1 reduces to textbook asymmetric min-max INT2 with an
    fp16 scale/zero (numpy float16 rounding, numpy half-to-even rint)."""
    rng = np.random.default_rng(9)
    for g in (32, 64, 128):
        for trial in range(100):
            y = rng.standard_normal(128) * 3
            c, s16, z16, *_ = o.quantize_vec(y, g, 1.0)
            assert len(s16) == 128 // g
            for k in range(128 // g):
                yg = y[g * k:g * k + g]
                s = np.float16((yg.max() - yg.min()) / 3)
                z = np.float16(yg.min())
                ref = np.clip(np.rint((yg - np.float64(z)) / np.float64(s)), 0, 3)
                assert s16[k] == s.view(np.uint16) and z16[k] == z.view(np.uint16)
                assert np.array_equal(c[g * k:g * k + g], ref)


def check_clip(o: oracle.Oracle):
    """With ratio c < 1 the group range shrinks to +-c*max|y| and the
    clipped extremes map to codes 0 / 3."""
    rng = np.random.default_rng(10)
    for trial in range(100):
        y = rng.standard_normal(128)
        y[5] = 40.0
        y[70] = -35.0
        for g in (32, 128):
            c, s16, z16, u, sp, zp = o.quantize_vec(y, g, 0.5)
            for k in range(128 // g):
                yg = y[g * k:g * k + g]
                t = 0.5 * np.max(np.abs(yg))
                yc = np.clip(yg, -t, t)
                assert abs(sp[k] - (yc.max() - yc.min()) / 3) <= 1e-15 * abs(sp[k]) + 1e-300
                assert zp[k] == yc.min()
            assert c[5] == 3 and c[70] == 0
            assert sp[0] < (40.0 + 1.0) / 3


def check_degenerate(o: oracle.Oracle):
    """A constant group has s = 0: codes 0 and yhat = z = fp16(clipped
    value); the clip applies to a constant group too."""
    y = np.full(128, 0.3)
    c, s16, z16, *_ = o.quantize_vec(y, 32, 1.0)
    assert not c.any() and not s16.any()
    assert np.all(z16 == np.float16(0.3).view(np.uint16))
    c, s16, z16, *_ = o.quantize_vec(y, 32, 0.95)
    assert not c.any() and not s16.any()
    assert np.all(z16 == np.float16(0.95 * 0.3).view(np.uint16))
    y = np.zeros(128)
    c, s16, z16, *_ = o.quantize_vec(y, 32, 0.95)
    assert not c.any() and not s16.any() and not z16.any()


def load_golden(name: str) -> dict:
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                key, *rest = line.split()
                vals[key] = rest
    return vals


def check_evict_golden(o: oracle.Oracle):
    """Hand-derived eviction of x = e_4 with U = I (tests/golden/evict_e4.txt),
    checked at the pool-format addresses for K and V."""
    gold = load_golden("evict_e4.txt")
    s_bits = int(gold["scale_bits"][0], 16)
    z_bits = int(gold["zero_bits"][0], 16)
    code_bytes = np.array([int(v, 16) for v in gold["code_bytes"]], np.uint8)
    sh = oracle.Shape(128, 32, 64, 256, 64, 1, 1)
    x = np.zeros((1, 1, 2, 128), np.float64)
    x[0, 0, :, 4] = 1.0
    src = S.bf16_bits(x)
    U = np.stack([np.eye(128), np.eye(128)])[None]
    bb = o.block_bytes(128, 32, 64)
    assert bb == 6144
    pool = np.zeros(2 * bb, np.uint8)
    table = np.array([[1]], np.int32)
    slot = 5
    o.evict(sh, src, [0], [slot], U, np.ones((1, 2)), pool, table, 1)
    blk = pool[bb:]
    assert np.array_equal(blk[slot * 32:slot * 32 + 32], code_bytes)              # K, token-major
    assert np.array_equal(blk[2048 + np.arange(32) * 64 + slot], code_bytes)      # V, byte-plane-major
    for which in range(2):
        sz = blk[4096 + which * 1024 + slot * 16: 4096 + which * 1024 + slot * 16 + 16].view(np.uint16)
        assert np.all(sz[0::2] == s_bits) and np.all(sz[1::2] == z_bits)
    assert not pool[:bb].any()
    touched = np.zeros(bb, bool)
    touched[slot * 32:slot * 32 + 32] = True
    touched[2048 + np.arange(32) * 64 + slot] = True
    for which in range(2):
        touched[4096 + which * 1024 + slot * 16: 4096 + which * 1024 + slot * 16 + 16] = True
    assert not blk[~touched].any()


# --------------------------------------------------------------------------
# decode attention
# --------------------------------------------------------------------------

def numpy_read_pool(pool, table, b, n, kv, Hk, d=128, g=32, P=64):
    """Independent numpy reading of the pool format: dequantised
    stored-order K and V of the first n history tokens of (b, kv)."""
    ng = d // g
    bb = 2 * P * d // 4 + 2 * P * ng * 4
    K = np.zeros((n, d))
    V = np.zeros((n, d))
    shifts = np.array([0, 2, 4, 6], np.uint8)
    for pos in range(n):
        page = table[b, pos // P]
        t = pos % P
        blk = pool[(page * Hk + kv) * bb:(page * Hk + kv + 1) * bb]
        kb = blk[t * (d // 4):(t + 1) * (d // 4)]
        vb = blk[P * d // 4 + np.arange(d // 4) * P + t]
        # byte j holds positions j + i*d/4 in bits 2i..2i+1
        kc = ((kb[None, :] >> shifts[:, None]) & 3).reshape(-1).astype(np.float64)
        vc = ((vb[None, :] >> shifts[:, None]) & 3).reshape(-1).astype(np.float64)
        ksz = blk[2 * P * d // 4 + t * ng * 4: 2 * P * d // 4 + (t + 1) * ng * 4].view(np.float16).astype(np.float64)
        vo = 2 * P * d // 4 + P * ng * 4
        vsz = blk[vo + t * ng * 4: vo + (t + 1) * ng * 4].view(np.float16).astype(np.float64)
        K[pos] = kc * np.repeat(ksz[0::2], g) + np.repeat(ksz[1::2], g)
        V[pos] = vc * np.repeat(vsz[0::2], g) + np.repeat(vsz[1::2], g)
    return K, V


def numpy_R(U):
    d = U.shape[0]
    Hs = scipy.linalg.hadamard(d) / np.sqrt(d)
    perm = np.array([strrev_bits(j, int(np.log2(d))) for j in range(d)])
    return (U @ Hs)[:, perm]


def brute_force_decode(sc) -> np.ndarray:
    """softmax(q K^T * scale) V over [BF16 tokens ; history mapped back by
    R^T], float64, numpy."""
    sh = sc.shape
    B, Hq, d = sc.q.shape
    Hk = sh.num_kv_heads
    G = Hq // Hk
    out = np.zeros((B, Hq, d))
    f = lambda a: S.bf16_to_f32(a).astype(np.float64)
    for b in range(B):
        for kv in range(Hk):
            nb = int(sc.bf16_len[b])
            Kb = f(sc.bf16_kv[b, :nb, kv, 0])
            Vb = f(sc.bf16_kv[b, :nb, kv, 1])
            Kh, Vh = numpy_read_pool(sc.pool, sc.page_table, b, int(sc.hist_len[b]), kv, Hk, d, sh.quant_group,
                                     sh.page_size)
            K = np.concatenate([Kb, Kh @ numpy_R(sc.U[kv, 0]).T])
            V = np.concatenate([Vb, Vh @ numpy_R(sc.U[kv, 1]).T])
            for hh in range(G):
                h = kv * G + hh
                if K.shape[0] == 0:
                    continue
                lg = (K @ f(sc.q[b, h])) * sc.sm_scale
                p = np.exp(lg - lg.max())
                out[b, h] = (p @ V) / p.sum()
    return out


def small_scenes(o: oracle.Oracle):
    from scene import make_scene
    w = S.WORKLOADS["tiny"]
    yield make_scene(w, orc=o)
    w2 = S.Workload(90, "small", batch=3, hq=4, hk=2, n_outlier=2)
    yield make_scene(w2, ctx=np.array([700, 385, 100], np.int32), perm_seed=11, orc=o)


def check_decode_bruteforce(o: oracle.Oracle):
    for sc in small_scenes(o):
        out = o.decode(sc.shape, sc.q, sc.bf16_kv, sc.bf16_len, sc.pool, sc.page_table, sc.max_pages,
                       sc.hist_len, sc.U, sc.sm_scale)
        ref = brute_force_decode(sc)
        assert np.max(np.abs(out - ref)) < 1e-11, np.max(np.abs(out - ref))


def check_segmented_equals_plain(o: oracle.Oracle):
    """Two-segment online-softmax merge (rotated INT2 segment + BF16
    segment) equals the single-pass softmax over the concatenation."""
    from scene import make_scene
    w = S.Workload(91, "edges", batch=8, hq=4, hk=1, n_outlier=2)
    ctx = np.array([1, 100, 320, 321, 383, 384, 385, 1000], np.int32)
    scenes = list(small_scenes(o)) + [make_scene(w, ctx=ctx, orc=o)]
    for sc in scenes:
        a = o.decode(sc.shape, sc.q, sc.bf16_kv, sc.bf16_len, sc.pool, sc.page_table, sc.max_pages,
                     sc.hist_len, sc.U, sc.sm_scale)
        b = o.decode(sc.shape, sc.q, sc.bf16_kv, sc.bf16_len, sc.pool, sc.page_table, sc.max_pages,
                     sc.hist_len, sc.U, sc.sm_scale, segmented=True)
        assert np.max(np.abs(a - b)) < 1e-12


def check_rotation_invariance(o: oracle.Oracle):
    """Attending in the rotated domain (q.R_K against the stored rotated
    keys, output mapped back by R_V^T) equals attention on the un-rotated
    dequantised cache (history-only context)."""
    from scene import make_scene
    w = S.Workload(92, "histonly", batch=1, hq=4, hk=1, n_outlier=2)
    sc = make_scene(w, ctx=np.array([900], np.int32), orc=o)
    sc.bf16_len[:] = 0
    out = o.decode(sc.shape, sc.q, sc.bf16_kv, sc.bf16_len, sc.pool, sc.page_table, sc.max_pages,
                   sc.hist_len, sc.U, sc.sm_scale)
    Kh, Vh = numpy_read_pool(sc.pool, sc.page_table, 0, int(sc.hist_len[0]), 0, 1)
    RK, RV = numpy_R(sc.U[0, 0]), numpy_R(sc.U[0, 1])
    for h in range(4):
        q = S.bf16_to_f32(sc.q[0, h]).astype(np.float64)
        lg = (Kh @ (q @ RK)) * sc.sm_scale
        p = np.exp(lg - lg.max())
        o_rot = (p @ Vh) / p.sum()
        assert np.max(np.abs(o_rot @ RV.T - out[0, h])) < 1e-12


def check_decode_special(o: oracle.Oracle):
    """One-token context returns that token's V; equal logits average V;
    an empty context returns zeros."""
    sh = oracle.Shape(128, 32, 64, 256, 64, 2, 1)
    rng = np.random.default_rng(12)
    kv = np.zeros((1, 320, 1, 2, 128), np.uint16)
    kv[0, :3] = S.bf16_bits(rng.standard_normal((3, 1, 2, 128)))
    q = S.bf16_bits(rng.standard_normal((1, 2, 128)))
    U = np.stack([np.eye(128)] * 2)[None]
    one = o.decode(sh, q, kv, np.array([1]), None, None, 0, np.array([0]), U, 0.1)
    v0 = S.bf16_to_f32(kv[0, 0, 0, 1]).astype(np.float64)
    assert np.array_equal(one[0, 0], v0) and np.array_equal(one[0, 1], v0)
    qz = np.zeros_like(q)
    avg = o.decode(sh, qz, kv, np.array([3]), None, None, 0, np.array([0]), U, 0.1)
    vm = S.bf16_to_f32(kv[0, :3, 0, 1]).astype(np.float64).mean(0)
    assert np.max(np.abs(avg[0, 0] - vm)) < 1e-14
    empty = o.decode(sh, q, kv, np.array([0]), None, None, 0, np.array([0]), U, 0.1)
    assert not empty.any()


# --------------------------------------------------------------------------
# page-table layout
# --------------------------------------------------------------------------

SPLITMIX64_SEED0 = [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]  # published test vector


def check_splitmix(o: oracle.Oracle):
    assert [int(v) for v in o.splitmix64(0, 3)] == SPLITMIX64_SEED0


def check_pool_layout(o: oracle.Oracle):
    sh = oracle.Shape(128, 32, 64, 256, 64, 32, 8)
    cap = np.array([64, 1, 0, 130, 640], np.int32)
    rc, table, n, nbytes = o.pool_layout(sh, cap, max_pages=10)
    assert rc == 0 and n == 1 + 1 + 0 + 3 + 10
    assert nbytes == n * 8 * 6144
    used = [table[b, :(c + 63) // 64] for b, c in enumerate(cap)]
    assert np.array_equal(np.concatenate(used), np.arange(n))       # contiguous order
    assert (table[0, 1:] == -1).all() and (table[2] == -1).all()
    # shuffled: a bijection onto the same ids, following Fisher-Yates on
    # SplitMix64 draws
    rc, t2, n2, _ = o.pool_layout(sh, cap, perm_seed=77, max_pages=10)
    assert rc == 0 and n2 == n
    ids = np.concatenate([t2[b, :(c + 63) // 64] for b, c in enumerate(cap)])
    assert sorted(ids.tolist()) == list(range(n))
    draws = [int(v) for v in o.splitmix64(77, n)]
    pi = list(range(n))
    for k, i in enumerate(range(n - 1, 0, -1)):
        j = draws[k] % (i + 1)
        pi[i], pi[j] = pi[j], pi[i]
    assert ids.tolist() == [pi[L] for L in range(n)]
    # shared prefix: sequences of one group alias their first pages
    cap = np.array([300, 200, 500, 256], np.int32)
    grp = np.array([0, -1, 0, 0], np.int32)
    rc, t3, n3, _ = o.pool_layout(sh, cap, grp, 128, 0, 8)
    assert rc == 0
    assert (t3[0, :2] == t3[2, :2]).all() and (t3[0, :2] == t3[3, :2]).all()
    assert n3 == 2 + (5 - 2) + 4 + (8 - 2) + (4 - 2)
    priv = np.concatenate([t3[0, 2:5], t3[1, :4], t3[2, 2:8], t3[3, 2:4]])
    assert len(set(priv.tolist()) | set(t3[0, :2].tolist())) == n3
    # errors
    assert o.pool_layout(sh, np.array([65 * 64], np.int32), max_pages=64)[0] == oracle.ERR_OUT_OF_PAGES
    assert o.pool_layout(sh, cap, grp, 100, 0, 8)[0] == oracle.ERR_INVALID_ARG        # not page aligned
    assert o.pool_layout(sh, cap, grp, 320, 0, 8)[0] == oracle.ERR_INVALID_ARG        # prefix > capacity


ALL_CHECKS = [check_hadamard, check_bitrev, check_R, check_group_structure, check_f16, check_f16_decode,
              check_bf16, check_pack, check_on_grid, check_nearest_level, check_error_bound,
              check_minmax_textbook, check_clip, check_degenerate, check_evict_golden, check_decode_bruteforce,
              check_segmented_equals_plain, check_rotation_invariance, check_decode_special, check_splitmix,
              check_pool_layout]
