"""Prefix sharing with copy-on-write on the GPU: two sequences share a
1000-token history prefix that ends inside a page; both then evict their own
tokens, the shared last page is copied for the first writer
(oscar_pages_prepare_write + oscar_pages_copy), and the decode of every
sequence matches the oracle run on a private (unshared) layout of the same
tokens.  Also with the K channel boost (records copied with the pages)."""
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


@pytest.fixture(scope="module", autouse=True)
def _lib():
    B.build()
    O.lib()


@pytest.mark.parametrize("boost", [False, True])
def test_unaligned_shared_prefix_with_copy_on_write(boost):
    hq, hk, g = 8, 2, 32
    npre, suffix = 1000, [700, 333]
    hist = np.array([npre + suffix[0], npre + suffix[1], 900], np.int32)
    Bn = len(hist)
    w = S.Workload(61, "cow", batch=Bn, hq=hq, hk=hk)
    rng = S.rng_for(w, 3)
    prof = S.channel_profile(w)
    pre = S.kv_tokens(w, npre, rng, prof)
    own = [S.kv_tokens(w, int(n), rng, prof) for n in (suffix[0], suffix[1], hist[2])]
    U = S.rotation_U(w).astype(np.float32)
    clip = S.clip_ratios(w)
    bf16_kv = S.kv_tokens(w, Bn * S.NSLOT, rng, prof).reshape(Bn, S.NSLOT, hk, 2, S.D)
    q = S.queries(w, rng, Bn)

    sh = O.make_shape(hq, hk, quant_group=g)
    max_pages = int((hist.max() + 63) // 64)
    num_pages = 3 * max_pages + 4
    P = O.Pages(num_pages)
    table = np.full((Bn, max_pages), -1, np.int32)
    pool = torch.zeros(num_pages * hk * O.block_bytes(sh), dtype=torch.uint8, device="cuda")
    brec = torch.zeros(num_pages * hk * O.BOOST_BLOCK_BYTES, dtype=torch.uint8, device="cuda") if boost else None

    def evict(tokens, seq, pos):
        src, dst = P.prepare_write(seq, pos // 64, table)
        O.oscar_pages_copy(sh, src, dst, pool, brec, num_pages)
        args = (sh, H.bf16_t(tokens), H.i32_t(seq), H.i32_t(pos), H.f32_t(U), H.f32_t(clip), pool)
        tail = (H.i32_t(table), Bn, max_pages, num_pages)
        if boost:
            O.oscar_evict_quantize_boost(*args, brec, *tail)
        else:
            O.oscar_evict_quantize(*args, *tail)
        return src

    # sequence 0 writes the prefix; sequence 1 adopts its pages (a prefix hit)
    evict(pre, np.zeros(npre, np.int32), np.arange(npre, dtype=np.int32))
    npg_pre = (npre + 63) // 64
    P.retain(table[0, :npg_pre])
    table[1, :npg_pre] = table[0, :npg_pre]
    shared_last = int(table[0, npg_pre - 1])
    # every sequence evicts its own tokens: the shared last page is copied once
    seq = np.concatenate([np.full(suffix[0], 0), np.full(suffix[1], 1), np.full(hist[2], 2)]).astype(np.int32)
    pos = np.concatenate([np.arange(npre, hist[0]), np.arange(npre, hist[1]), np.arange(hist[2])]).astype(np.int32)
    copied = evict(np.concatenate(own), seq, pos)
    assert list(copied) == [shared_last]
    assert table[1, npg_pre - 1] == shared_last and table[0, npg_pre - 1] != shared_last
    assert np.array_equal(table[0, :npg_pre - 1], table[1, :npg_pre - 1])
    assert all(P.refcount(int(p)) == 2 for p in table[0, :npg_pre - 1]) and P.refcount(shared_last) == 1

    bf16_len = np.full(Bn, S.NSLOT, np.int32)
    out = torch.zeros((Bn, hq, S.D), dtype=torch.float32, device="cuda")
    ws = torch.zeros(O.oscar_decode_workspace_bytes(sh, Bn, max_pages), dtype=torch.uint8, device="cuda")
    common = (sh, H.bf16_t(q), H.bf16_t(bf16_kv), H.i32_t(bf16_len), pool)
    rest = (H.i32_t(table), max_pages, num_pages, H.i32_t(hist), H.f32_t(U), 1 / np.sqrt(S.D), out, ws)
    if boost:
        O.oscar_decode_attn_boost(*common, brec, *rest)
    else:
        O.oscar_decode_attn(*common, *rest)
    torch.cuda.synchronize()

    # the shared pages hold the prefix once; the copy and the original agree
    # on the prefix's 40 tokens of the last page (K codes of those slots)
    pool_g = pool.cpu().numpy()
    bb = O.block_bytes(sh)
    ntail = npre - 64 * (npg_pre - 1)
    for kv in range(hk):
        a = pool_g[(int(table[0, npg_pre - 1]) * hk + kv) * bb:][:ntail * 32]
        b = pool_g[(shared_last * hk + kv) * bb:][:ntail * 32]
        assert np.array_equal(a, b)

    # oracle on a private layout of the same tokens
    orc = oracle.get()
    shape = oracle.Shape(S.D, g, S.SINK, S.RECENT, S.PAGE, hq, hk)
    rc, t_o, np_o, nb_o = orc.pool_layout(shape, hist, None, 0, 0, max_pages)
    assert rc == 0
    toks = [np.concatenate([pre, own[0]]), np.concatenate([pre, own[1]]), own[2]]
    src_o = np.concatenate(toks)
    seq_o = np.concatenate([np.full(h, b, np.int32) for b, h in enumerate(hist)])
    pos_o = np.concatenate([np.arange(h, dtype=np.int32) for h in hist])
    pool_o = np.zeros(max(nb_o, 16), np.uint8)
    if boost:
        boost_o = np.zeros(max(np_o * hk * K.BLOCK, 16), np.uint8)
        K.evict(orc, shape, src_o, seq_o, pos_o, U.astype(np.float64), clip, pool_o, t_o, max_pages, boost_o)
        ref = K.decode(orc, shape, q, bf16_kv, bf16_len, pool_o, t_o, hist, U.astype(np.float64), boost_o,
                       1 / np.sqrt(S.D))
    else:
        orc.evict(shape, src_o, seq_o, pos_o, U.astype(np.float64), clip, pool_o, t_o, max_pages)
        ref = orc.decode(shape, q, bf16_kv, bf16_len, pool_o, t_o, max_pages, hist, U.astype(np.float64),
                         1 / np.sqrt(S.D))
    err, rel = H.assert_close(out.cpu().numpy(), ref)
    print(f"copy-on-write prefix (boost={boost}): max-abs {err:.3e} rel-L2 {rel:.3e}")


def test_radix_prefix_hit_reuses_cached_pages():
    """Sequence 0's history pages go into the radix cache; sequence 1 (the
    same first 64 + 640 context tokens, then its own) matches 10 pages,
    evicts only its own tokens after them, and its decode equals the oracle
    on a private layout of its tokens."""
    hq, hk, g = 8, 2, 32
    nshare = 10 * 64                                       # shared history tokens (whole pages)
    hist = np.array([1300, nshare + 437], np.int32)
    Bn = 2
    w = S.Workload(63, "radix", batch=Bn, hq=hq, hk=hk)
    rng = S.rng_for(w, 3)
    prof = S.channel_profile(w)
    toks0 = S.kv_tokens(w, int(hist[0]), rng, prof)
    own1 = S.kv_tokens(w, int(hist[1]) - nshare, rng, prof)
    toks1 = np.concatenate([toks0[:nshare], own1])
    ids0 = np.arange(64 + hist[0], dtype=np.int32)        # token ids of the contexts' first chunks
    ids1 = np.concatenate([ids0[:64 + nshare], 100000 + np.arange(hist[1] - nshare, dtype=np.int32)])
    U = S.rotation_U(w).astype(np.float32)
    clip = S.clip_ratios(w)
    bf16_kv = S.kv_tokens(w, Bn * S.NSLOT, rng, prof).reshape(Bn, S.NSLOT, hk, 2, S.D)
    q = S.queries(w, rng, Bn)

    sh = O.make_shape(hq, hk, quant_group=g)
    max_pages = int((hist.max() + 63) // 64)
    num_pages = 2 * max_pages + 4
    P = O.Pages(num_pages)
    R = O.Radix(P)
    table = np.full((Bn, max_pages), -1, np.int32)
    pool = torch.zeros(num_pages * hk * O.block_bytes(sh), dtype=torch.uint8, device="cuda")

    def evict(tokens, seq, pos):
        src, dst = P.prepare_write(seq, pos // 64, table)
        O.oscar_pages_copy(sh, src, dst, pool, None, num_pages)
        O.oscar_evict_quantize(sh, H.bf16_t(tokens), H.i32_t(seq), H.i32_t(pos), H.f32_t(U), H.f32_t(clip), pool,
                               H.i32_t(table), Bn, max_pages, num_pages)

    evict(toks0, np.zeros(hist[0], np.int32), np.arange(hist[0], dtype=np.int32))
    full0 = int(hist[0]) // 64
    R.insert(ids0, table[0, :full0])                       # cache sequence 0's whole pages
    got = R.match(ids1, max_pages)
    assert list(got) == list(table[0, :nshare // 64])       # a hit on the 10 shared pages
    table[1, :len(got)] = got
    evict(own1, np.ones(hist[1] - nshare, np.int32), np.arange(nshare, hist[1], dtype=np.int32))
    assert np.array_equal(table[1, :10], table[0, :10]) and P.refcount(int(table[0, 0])) == 3

    bf16_len = np.full(Bn, S.NSLOT, np.int32)
    out = torch.zeros((Bn, hq, S.D), dtype=torch.float32, device="cuda")
    ws = torch.zeros(O.oscar_decode_workspace_bytes(sh, Bn, max_pages), dtype=torch.uint8, device="cuda")
    O.oscar_decode_attn(sh, H.bf16_t(q), H.bf16_t(bf16_kv), H.i32_t(bf16_len), pool, H.i32_t(table), max_pages,
                        num_pages, H.i32_t(hist), H.f32_t(U), 1 / np.sqrt(S.D), out, ws)
    torch.cuda.synchronize()

    orc = oracle.get()
    shape = oracle.Shape(S.D, g, S.SINK, S.RECENT, S.PAGE, hq, hk)
    rc, t_o, np_o, nb_o = orc.pool_layout(shape, hist, None, 0, 0, max_pages)
    assert rc == 0
    src_o = np.concatenate([toks0, toks1])
    seq_o = np.concatenate([np.full(h, b, np.int32) for b, h in enumerate(hist)])
    pos_o = np.concatenate([np.arange(h, dtype=np.int32) for h in hist])
    pool_o = np.zeros(max(nb_o, 16), np.uint8)
    orc.evict(shape, src_o, seq_o, pos_o, U.astype(np.float64), clip, pool_o, t_o, max_pages)
    ref = orc.decode(shape, q, bf16_kv, bf16_len, pool_o, t_o, max_pages, hist, U.astype(np.float64),
                     1 / np.sqrt(S.D))
    err, rel = H.assert_close(out.cpu().numpy(), ref)
    print(f"radix prefix hit: max-abs {err:.3e} rel-L2 {rel:.3e}")
    R.close()
