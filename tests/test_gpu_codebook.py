"""GPU parity of the Lloyd-Max codebook variant (oscar_evict_quantize_codebook,
oscar_decode_attn_codebook) against the float64 oracle (oracle/lloyd.py on
top of the C oracle's eviction).

Eviction: s and z are those of the uniform path (bit-exact except within the
fp16-midpoint window), codes are the nearest codebook levels of the oracle's
pre-rounding u (bit-exact except within 1e-5 of a threshold a/2, 3/2,
3 - a/2).  Decode: the oracle attends over the same stored codes, s and z,
dequantised with the levels and mapped back by R^T; max-abs 2e-3, rel-L2 1e-3.
"""
import numpy as np
import pytest

import oracle
from bit_kv_cache_evict_gb300 import synth as S
from oracle import lloyd as L

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


def _setup(hist, hq, hk, g, seed):
    w = S.Workload(seed, "codebook", batch=len(hist), hq=hq, hk=hk)
    orc = oracle.get()
    shape = oracle.Shape(S.D, g, S.SINK, S.RECENT, S.PAGE, hq, hk)
    hist = np.asarray(hist, np.int32)
    rc, table, npages, nbytes = orc.pool_layout(shape, hist + 64, None, 0, 5, None)
    assert rc == 0
    max_pages = table.shape[1]
    rng = S.rng_for(w, 3)
    prof = S.channel_profile(w)
    toks = [S.kv_tokens(w, int(h), rng, prof) for h in hist]
    src = np.concatenate(toks)                                   # bf16 bits [sum h][hk][2][d]
    seq = np.concatenate([np.full(h, b, np.int32) for b, h in enumerate(hist)])
    pos = np.concatenate([np.arange(h, dtype=np.int32) for h in hist])
    U = S.rotation_U(w).astype(np.float32)
    clip = S.clip_ratios(w)
    bf16_kv = S.kv_tokens(w, len(hist) * S.NSLOT, rng, prof).reshape(len(hist), S.NSLOT, hk, 2, S.D)
    q = S.queries(w, rng, len(hist))
    return orc, shape, hist, table, max_pages, npages, nbytes, src, seq, pos, U, clip, bf16_kv, q


def _evict_gpu(shape, src, seq, pos, U, clip, cb, table, max_pages, npages, nbytes, B_):
    sh = O.oscar_shape(*[getattr(shape, f) for f in ("head_dim", "quant_group", "sink", "recent", "page_size",
                                                      "num_q_heads", "num_kv_heads")])
    pool = torch.zeros(max(nbytes, 16), dtype=torch.uint8, device="cuda")
    args = (sh, H.bf16_t(src), H.i32_t(seq), H.i32_t(pos), H.f32_t(U), H.f32_t(clip))
    if cb is None:
        O.oscar_evict_quantize(*args, pool, H.i32_t(table), B_, max_pages, npages)
    else:
        O.oscar_evict_quantize_codebook(*args, H.f32_t(cb), pool, H.i32_t(table), B_, max_pages, npages)
    torch.cuda.synchronize()
    return sh, pool


@pytest.mark.parametrize("g,hq", [(32, 8), (64, 8), (32, 16)])
def test_codebook_eviction_and_decode_match_oracle(g, hq):
    hist = [700, 1300, 2050]
    hk = 2
    orc, shape, hist, table, max_pages, npages, nbytes, src, seq, pos, U, clip, bf16_kv, q = _setup(hist, hq, hk, g, 41)
    cb = np.array([[1.2, 0.8], [1.1, 1.3]], np.float32)[:hk]
    sh, pool_t = _evict_gpu(shape, src, seq, pos, U, clip, cb, table, max_pages, npages, nbytes, len(hist))
    pool_g = pool_t.cpu().numpy()
    # oracle: s, z and pre-rounding u of the same vectors (uniform eviction)
    pool_o = np.zeros(max(nbytes, 16), np.uint8)
    u, sp, zp = orc.evict(shape, src, seq, pos, U.astype(np.float64), clip, pool_o, table, max_pages, want_aux=True)
    exempt = 0
    total = 0
    ng = 128 // g
    for i in range(seq.size):
        for kv in range(hk):
            for wv in range(2):
                cg, sg, zg = H.read_vec(pool_g, table, int(seq[i]), int(pos[i]), kv, wv, hk, g)
                _, so, zo = H.read_vec(pool_o, table, int(seq[i]), int(pos[i]), kv, wv, hk, g)
                grp_ex = np.zeros(ng, bool)
                for k in range(ng):
                    if sg[k] != so[k] or zg[k] != zo[k]:
                        assert H.near_f16_midpoint(sp[i, kv, wv, k]) or H.near_f16_midpoint(zp[i, kv, wv, k])
                        grp_ex[k] = True
                uu = u[i, kv, wv]
                a = float(cb[kv, wv])
                want = L.codes_from_u(uu, a)
                total += 128
                for j in np.nonzero(cg != want)[0]:
                    near = min(abs(uu[j] - t) for t in (a / 2, 1.5, 3 - a / 2)) < BOUND
                    assert near or grp_ex[j // g], (i, kv, wv, j, int(cg[j]), int(want[j]), uu[j])
                    exempt += 1
    assert exempt <= max(1, 1e-4 * total), (exempt, total)

    # decode over the GPU-written history
    B_ = len(hist)
    bf16_len = np.full(B_, S.NSLOT, np.int32)
    out = torch.zeros((B_, hq, S.D), dtype=torch.float32, device="cuda")
    ws = torch.zeros(O.oscar_decode_workspace_bytes(sh, B_, max_pages), dtype=torch.uint8, device="cuda")
    O.oscar_decode_attn_codebook(sh, H.bf16_t(q), H.bf16_t(bf16_kv), H.i32_t(bf16_len), pool_t, H.i32_t(table),
                                 max_pages, npages, H.i32_t(hist), H.f32_t(U), H.f32_t(cb), 1 / np.sqrt(S.D), out, ws)
    torch.cuda.synchronize()
    ref = L.decode(q, bf16_kv, bf16_len, pool_g, table, hist, U.astype(np.float64), orc.build_R, cb.astype(np.float64),
                   1 / np.sqrt(S.D), g)
    err, rel = H.assert_close(out.cpu().numpy(), ref)
    print(f"codebook g={g} G={hq // hk}: max-abs {err:.3e} rel-L2 {rel:.3e} exempt codes {exempt}")


@pytest.mark.parametrize("hist,hq,hk", [([0, 17, 64, 130], 2, 2), ([1, 63, 65], 4, 1)])
def test_codebook_edge_histories(hist, hq, hk):
    """Empty, one-token, page-sized and ragged histories, G = 1 and G = 4."""
    orc, shape, hist, table, max_pages, npages, nbytes, src, seq, pos, U, clip, bf16_kv, q = _setup(hist, hq, hk, 32, 59)
    cb = np.array([[0.7, 1.3], [1.2, 0.9]], np.float32)[:hk]
    sh, pool_t = _evict_gpu(shape, src, seq, pos, U, clip, cb, table, max_pages, npages, nbytes, len(hist))
    pool_g = pool_t.cpu().numpy()
    B_ = len(hist)
    bf16_len = np.array([S.NSLOT, 5, S.NSLOT, 200][:B_], np.int32)
    out = torch.zeros((B_, hq, S.D), dtype=torch.float32, device="cuda")
    ws = torch.zeros(O.oscar_decode_workspace_bytes(sh, B_, max_pages), dtype=torch.uint8, device="cuda")
    O.oscar_decode_attn_codebook(sh, H.bf16_t(q), H.bf16_t(bf16_kv), H.i32_t(bf16_len), pool_t, H.i32_t(table),
                                 max_pages, npages, H.i32_t(hist), H.f32_t(U), H.f32_t(cb), 1 / np.sqrt(S.D), out, ws)
    torch.cuda.synchronize()
    ref = L.decode(q, bf16_kv, bf16_len, pool_g, table, hist, U.astype(np.float64), orc.build_R, cb.astype(np.float64),
                   1 / np.sqrt(S.D), 32)
    H.assert_close(out.cpu().numpy(), ref)


def test_codebook_one_is_the_uniform_path():
    hist = [900, 400]
    hq, hk = 4, 1
    orc, shape, hist, table, max_pages, npages, nbytes, src, seq, pos, U, clip, bf16_kv, q = _setup(hist, hq, hk, 32, 43)
    ones = np.ones((hk, 2), np.float32)
    sh, pool_u = _evict_gpu(shape, src, seq, pos, U, clip, None, table, max_pages, npages, nbytes, len(hist))
    _, pool_c = _evict_gpu(shape, src, seq, pos, U, clip, ones, table, max_pages, npages, nbytes, len(hist))
    diff = (pool_u != pool_c).sum().item()
    assert diff <= 2, diff                                       # exact ties of u at k + 1/2 may round either way
    B_ = len(hist)
    bf16_len = np.full(B_, S.NSLOT, np.int32)
    outs = []
    for cb in (None, ones):
        out = torch.zeros((B_, hq, S.D), dtype=torch.float32, device="cuda")
        ws = torch.zeros(O.oscar_decode_workspace_bytes(sh, B_, max_pages), dtype=torch.uint8, device="cuda")
        a = (sh, H.bf16_t(q), H.bf16_t(bf16_kv), H.i32_t(bf16_len), pool_u, H.i32_t(table), max_pages, npages,
             H.i32_t(hist), H.f32_t(U))
        if cb is None:
            O.oscar_decode_attn(*a, 1 / np.sqrt(S.D), out, ws)
        else:
            O.oscar_decode_attn_codebook(*a, H.f32_t(cb), 1 / np.sqrt(S.D), out, ws)
        torch.cuda.synchronize()
        outs.append(out.cpu().numpy().astype(np.float64))
    assert np.abs(outs[0] - outs[1]).max() <= 1e-5 * max(1.0, np.abs(outs[0]).max())


@pytest.mark.parametrize("g", [32, 128])
def test_codebook_fit_matches_oracle(g):
    """The Lloyd-Max fit of a on calibration tokens (fp32 rotation on the
    GPU, float64 in the oracle) agrees within 1e-4."""
    hk, n_t = 2, 400
    w = S.Workload(47, "fit", batch=1, hq=4 * hk, hk=hk)
    rng = S.rng_for(w, 5)
    kvb = S.kv_tokens(w, n_t, rng, S.channel_profile(w))
    U = S.rotation_U(w).astype(np.float32)
    clip = S.clip_ratios(w)
    sh = O.oscar_shape(128, g, 64, 256, 64, 4 * hk, hk)
    a_t = torch.zeros((hk, 2), dtype=torch.float32, device="cuda")
    O.oscar_calibrate_codebook(sh, H.bf16_t(kvb), H.f32_t(U), H.f32_t(clip), a_t)
    torch.cuda.synchronize()
    a_ref = L.fit_from_tokens(S.bf16_to_f32(kvb).astype(np.float64), U.astype(np.float64), clip, g)
    a_g = a_t.cpu().numpy().astype(np.float64)
    print(f"codebook fit g={g}: gpu {a_g.ravel()} oracle {a_ref.ravel()}")
    assert np.abs(a_g - a_ref).max() <= 1e-4, (a_g, a_ref)
    assert np.all(a_ref > 0.3) and np.all(a_ref < 1.5)
