"""GPU parity of the C-ABI path against the float64 oracle on the same seeded
inputs (small and edge-case sizes spanning several tiles and ragged
tails).  Eviction: codes and packed bytes bit-exact except listed boundary
codes; attention: max-abs 2e-3 and relative-L2 1e-3."""
import dataclasses

import numpy as np
import pytest

import oracle
from bit_kv_cache_evict_gb300 import synth as S
from scene import make_scene, oracle_step

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


def run_and_compare(orc, sc, label=""):
    out_o, pool_o, kv_o, hist_o, bl_o, seqs, aux = oracle_step(orc, sc)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out_g, pool_g, kv_g, hist_g, bl_g = H.gpu_step(sc, status=status)
    assert int(status.item()) == 0
    assert np.array_equal(hist_g, hist_o) and np.array_equal(bl_g, bl_o)
    assert np.array_equal(kv_g, kv_o)                        # ring append fused into the eviction
    exempt = []
    allowed = np.zeros_like(pool_o)
    if seqs.size:
        items = [(int(b), int(sc.hist_len[b]), i) for i, b in enumerate(seqs)]
        exempt = H.compare_evicted(pool_g, pool_o, sc.page_table, items, aux, sc.shape.num_kv_heads,
                                   sc.shape.quant_group, allowed=allowed)
    # every other bit of the pool is equal: no stray writes anywhere
    H.assert_pools_equal_except(pool_g, pool_o, allowed)
    # attention: the oracle on the pool the GPU wrote would differ only by
    # exempt codes; compare with the oracle's own step
    mx, rel = H.assert_close(out_g, out_o)
    print(f"{label}: max-abs {mx:.3e} rel-L2 {rel:.3e} exempt codes {len(exempt)}")
    return out_g, out_o


def test_tiny_step(orc):
    """Tiny: 1 sequence, 1 KV head, 4 query heads, 64 + 704 + 256 tokens;
    one eviction and one decode step (attends over 1025 tokens)."""
    run_and_compare(orc, make_scene(S.WORKLOADS["tiny"], orc=orc), "tiny")


@pytest.mark.parametrize("hq,hk", [(4, 1), (2, 2), (8, 1), (16, 2)])
def test_edge_contexts(orc, hq, hk):
    """Contexts with empty history, 1 token of history, page boundaries
    (63/64/65), several pages with a ragged tail, and more than one split."""
    w = S.Workload(40 + hq + hk, "edges", batch=10, hq=hq, hk=hk, n_outlier=2)
    ctx = np.array([1, 100, 320, 321, 383, 384, 385, 1000, 320 + 64 * 9 + 5, 320 + 64 * 17 + 63], np.int32)
    run_and_compare(orc, make_scene(w, ctx=ctx, perm_seed=9, orc=orc), f"edges G={hq // hk}")


def test_heavy_tails_shuffled(orc):
    """Student-t(3) values with lognormal channel scales (Qwen3-32B-shaped
    heads, G = 8), shuffled page table."""
    w = dataclasses.replace(S.WORKLOADS["qwen3_32b"], batch=3)
    ctx = np.array([1500, 2900, 700], np.int32)
    run_and_compare(orc, make_scene(w, ctx=ctx, hq=16, hk=2, perm_seed=21, orc=orc), "student-t")


def test_prefix_sharing(orc):
    """Sequences sharing prefix pages read the same physical pages."""
    w = S.Workload(55, "prefix", batch=4, hq=4, hk=1, n_outlier=2)
    ctx = np.array([1200, 900, 1500, 2000], np.int32)
    grp = np.array([0, -1, 0, 0], np.int32)
    sc = make_scene(w, ctx=ctx, prefix_group=grp, shared_hist_tokens=256, perm_seed=3, orc=orc)
    run_and_compare(orc, sc, "prefix")


@pytest.mark.parametrize("g", [32, 64, 128])
def test_bulk_evict_matches_oracle(orc, g):
    """Bulk eviction (no src_row, no append) of a whole history at once,
    across page boundaries of a shuffled table, for each group size."""
    w = S.Workload(56, "bulk", batch=2, hq=8, hk=2, n_outlier=4)
    sh = oracle.Shape(128, g, 64, 256, 64, 8, 2)
    rng = S.rng_for(w, 3)
    n = 700
    toks = S.kv_tokens(w, n, rng, S.channel_profile(w))
    U = S.rotation_U(w).astype(np.float32)
    clip = S.clip_ratios(w)
    seq = np.repeat(np.arange(2, dtype=np.int32), n // 2)
    pos = np.tile(np.arange(n // 2, dtype=np.int32), 2)
    rc, table, npages, nbytes = orc.pool_layout(sh, np.array([n // 2, n // 2]), perm_seed=5, max_pages=8)
    pool_o = np.zeros(nbytes, np.uint8)
    aux = orc.evict(sh, toks, seq, pos, U.astype(np.float64), clip, pool_o, table, 8, want_aux=True)
    pool = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    O.oscar_evict_quantize(O.make_shape(8, 2, quant_group=g), H.bf16_t(toks), H.i32_t(seq), H.i32_t(pos), H.f32_t(U),
                           H.f32_t(clip), pool, H.i32_t(table), 2, 8, npages, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    items = [(int(seq[i]), int(pos[i]), i) for i in range(n)]
    pool_g = pool.cpu().numpy()
    allowed = np.zeros_like(pool_o)
    exempt = H.compare_evicted(pool_g, pool_o, table, items, aux, 2, g, allowed=allowed)
    H.assert_pools_equal_except(pool_g, pool_o, allowed)
    print("bulk exempt", exempt)


@pytest.mark.parametrize("g", [64, 128])
def test_quant_groups_64_128(orc, g):
    """One decode step with scale/zero groups of 64 and 128 stored positions
    (one (s, z) pair per two / four 32-position MMA blocks), G = 4 and 8."""
    for hq, hk in ((8, 2), (8, 1)):
        w = S.Workload(95 + g, f"g{g}", batch=6, hq=hq, hk=hk, n_outlier=2)
        sc = make_scene(w, ctx=np.array([3000, 1025, 700, 321, 5000, 64], np.int32), perm_seed=3, orc=orc,
                        quant_group=g)
        run_and_compare(orc, sc, f"g={g} G={hq // hk}")


def test_degenerate_and_extreme_groups(orc):
    """Constant vectors (scale 0), all-zero vectors, and magnitudes near the
    fp16 limit; clip ratio 1.0 and 0.5."""
    sh = oracle.Shape(128, 32, 64, 256, 64, 4, 1)
    n = 6
    x = np.zeros((n, 1, 2, 128))
    x[0] = 0.0
    x[1, :, :, 0] = 3.0                        # e_0: constant after the Hadamard (U = I)
    x[2] = 7e3 * np.random.default_rng(1).standard_normal((1, 2, 128))
    x[3, :, :, 5] = -1e4
    x[4] = np.random.default_rng(2).standard_normal((1, 2, 128)) * 1e-6
    x[5] = np.random.default_rng(3).standard_normal((1, 2, 128))
    toks = S.bf16_bits(x)
    for U in (np.stack([np.eye(128)] * 2)[None], S.rotation_U(S.WORKLOADS["tiny"])):
        U = U.astype(np.float32)
        for c in (1.0, 0.5):
            clip = np.full((1, 2), c)
            table = np.array([[0]], np.int32)
            pool_o = np.zeros(6144, np.uint8)
            seq = np.zeros(n, np.int32)
            pos = np.arange(n, dtype=np.int32) * 7
            aux = orc.evict(sh, toks, seq, pos, U.astype(np.float64), clip, pool_o, table, 1, want_aux=True)
            pool = torch.zeros(6144, dtype=torch.uint8, device="cuda")
            O.oscar_evict_quantize(O.make_shape(4, 1), H.bf16_t(toks), H.i32_t(seq), H.i32_t(pos), H.f32_t(U),
                                   H.f32_t(clip), pool, H.i32_t(table), 1, 1, 1)
            torch.cuda.synchronize()
            pool_g = pool.cpu().numpy()
            allowed = np.zeros_like(pool_o)
            H.compare_evicted(pool_g, pool_o, table, [(0, int(pos[i]), i) for i in range(n)], aux, 1,
                              allowed=allowed)
            H.assert_pools_equal_except(pool_g, pool_o, allowed)


def test_bad_indices_are_skipped_and_reported(orc):
    """Out-of-range rows, sequences, positions and page ids are skipped on
    the device and reported in dev_status; nothing is written."""
    sh = O.make_shape(4, 1)
    toks = H.bf16_t(S.bf16_bits(np.random.default_rng(0).standard_normal((4, 1, 2, 128))))
    U = H.f32_t(np.stack([np.eye(128)] * 2)[None])
    clip = H.f32_t(np.ones((1, 2)))
    table = H.i32_t(np.array([[0, 5]], np.int32))            # page 5 does not exist (num_pages = 1)
    pool = torch.zeros(6144, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    # tokens: ok | bad sequence | bad position | page id 5 >= num_pages | bad source row
    O.oscar_evict_quantize(sh, toks, H.i32_t([0, 1, 0, 0, 0]), H.i32_t([3, 3, 200, 70, 4]), U, clip, pool, table,
                           batch=1, max_pages=2, num_pages=1, src_row=H.i32_t([0, 1, 2, 3, 9]), dev_status=status)
    torch.cuda.synchronize()
    st = int(status.item())
    assert st & O.OSCAR_STATUS_BAD_POS and st & O.OSCAR_STATUS_BAD_PAGE
    # only token 0 (row 0, seq 0, pos 3) was written
    pool_np = pool.cpu().numpy()
    assert pool_np[3 * 32:4 * 32].any()
    written = np.zeros(6144, bool)
    written[3 * 32:4 * 32] = True
    written[2048 + np.arange(32) * 64 + 3] = True
    written[4096 + 3 * 16:4096 + 4 * 16] = True
    written[5120 + 3 * 16:5120 + 4 * 16] = True
    assert not pool_np[~written].any()
    # decode with a bad page id: that page contributes nothing, status set
    status.zero_()
    q = H.bf16_t(S.bf16_bits(np.random.default_rng(1).standard_normal((1, 4, 128))))
    kv = torch.zeros((1, 320, 1, 2, 128), dtype=torch.bfloat16, device="cuda")
    kv[0, :5] = toks[:4].repeat(2, 1, 1, 1)[:5]
    out = torch.zeros((1, 4, 128), dtype=torch.float32, device="cuda")
    ws = torch.zeros(O.oscar_decode_workspace_bytes(sh, 1, 2), dtype=torch.uint8, device="cuda")
    O.oscar_decode_attn(sh, q, kv, H.i32_t([5]), pool, table, 2, 1, H.i32_t([100]), U, 0.088, out, ws,
                        dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & O.OSCAR_STATUS_BAD_PAGE
    assert np.isfinite(out.cpu().numpy()).all()


def test_two_streams_and_repeat(orc):
    """Same call on a side stream and twice in a row gives identical results
    (the workspace plan is rebuilt each call)."""
    sc = make_scene(S.WORKLOADS["tiny"], orc=orc)
    s = torch.cuda.Stream()
    a = H.gpu_step(sc, stream=s)[0]
    b = H.gpu_step(sc)[0]
    assert np.array_equal(a, b)
