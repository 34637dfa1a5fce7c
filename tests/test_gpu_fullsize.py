"""Parity at full workload sizes, in the launch configuration bench.py times.

For each workload the whole batch is built on the GPU exactly as the
benchmark builds it (bench.GpuState: every sequence's history evicted by
the GPU), so the decode launch covers the full batch, page table and split
plan.  A few (sequence, KV head) units are then overwritten with data whose
history the float64 oracle quantised itself (pages copied into the pool at
the sequence's real page ids, plus that unit's BF16 segment, queries and
appended token).  One decode step runs for the whole batch; the sampled
units' evicted token and attention outputs are compared with the oracle's
own step on the same inputs."""
import dataclasses
import os
import sys

import numpy as np
import pytest

import oracle
from bit_kv_cache_evict_gb300 import synth as S
from scene import make_scene, oracle_step

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402
import gpu_harness as H  # noqa: E402
from bit_kv_cache_evict_gb300 import build as B  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _lib():
    B.build()


# sampled (sequence, KV head) units per workload: eight for the workloads
# with the widest value ranges (Student-t values) and length mixes (1K-128K
# with a shared prefix), three or four elsewhere
N_UNITS = {"qwen3_32b": 8, "stress": 8}


def pick_units(w: S.Workload, ctx: np.ndarray):
    """Sampled (sequence, KV head) units: the shortest and the longest
    sequence, one in the middle (and two prefix sharers for the stress mix),
    then sequences at evenly spaced length ranks up to N_UNITS."""
    order = np.argsort(ctx, kind="stable")
    seqs = [int(order[0]), int(order[-1]), int(order[len(order) // 2])]
    if w.prefix_seqs:
        seqs += [1, w.prefix_seqs - 1]
    n = N_UNITS.get(w.name, len(seqs))
    for r in np.linspace(0, len(order) - 1, n + 2)[1:-1]:
        if len(dict.fromkeys(seqs)) >= n:
            break
        seqs.append(int(order[int(round(r))]))
    seqs = list(dict.fromkeys(seqs))[:max(n, 3)]
    if len(seqs) == 1:  # one sequence: two of its KV heads
        return [(seqs[0], 1), (seqs[0], w.hk - 2)]
    return [(b, (3 * i + 1) % w.hk) for i, b in enumerate(seqs)]


def inject(st, w, b, kv, orc):
    """Oracle-built state for unit (b, kv), written into the GPU state."""
    ctx = np.array([st.ctx0[b]], np.int32)
    wl = dataclasses.replace(w, batch=1)
    sc = make_scene(wl, ctx=ctx, orc=orc, extra_capacity=64, only_kv=kv)  # one-KV-head scene
    lay = st.layers[0]
    hist = int(sc.hist_len[0])
    table = st.table.cpu().numpy()
    # pages holding history positions 0..hist (hist = the position the step
    # evicts into) of this KV head: mini page i -> real page table[b][i]
    npg = hist // S.PAGE + 1
    pool = lay["pool"]
    for i in range(npg):
        mp = int(sc.page_table[0, i])
        src = sc.pool[mp * 6144:(mp + 1) * 6144]
        dst = (int(table[b, i]) * w.hk + kv) * 6144
        pool[dst:dst + 6144] = torch.from_numpy(src.copy()).to(pool.device)
    lay["kv"][b, :, kv] = H.bf16_t(np.ascontiguousarray(sc.bf16_kv[0, :, 0]))
    G = w.hq // w.hk
    lay["q"][b, kv * G:(kv + 1) * G] = H.bf16_t(sc.q[0])
    lay["new_kv"][b, kv] = H.bf16_t(sc.new_kv[0, 0])
    return sc


@pytest.mark.parametrize("name", ["qwen3_4b", "gate", "qwen3_8b_36l", "qwen3_32b", "stress", "longctx_b1"])
def test_full_size_sampled(orc, name):
    w = S.WORKLOADS[name]
    st = bench.GpuState(w, 1, 1, 0)
    units = pick_units(w, st.ctx0)
    scenes = [inject(st, w, b, kv, orc) for b, kv in units]
    torch.cuda.synchronize()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    # one step: fused eviction + append for every sequence, then decode
    lay = st.layers[0]
    from bit_kv_cache_evict_gb300 import oscar as O
    O.oscar_evict_quantize(st.shape, lay["kv"].view(st.B * S.NSLOT, st.Hk, 2, S.D), st.seqs, st.hist_before[0],
                           lay["U"], lay["clip"], lay["pool"], st.table, st.B, st.max_pages, st.num_pages,
                           src_row=st.src_row[0], new_kv=lay["new_kv"], dev_status=status)
    O.oscar_decode_attn(st.shape, lay["q"], lay["kv"], st.bf16_len, lay["pool"], st.table, st.max_pages,
                        st.num_pages, st.hist_after[0], lay["U"], st.sm_scale, lay["out"], st.ws, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    out = lay["out"].cpu().numpy()
    table = st.table.cpu().numpy()
    G = w.hq // w.hk
    for (b, kv), sc in zip(units, scenes):
        out_o, pool_o, kv_o, hist_o, bl_o, seqs, aux = oracle_step(orc, sc)
        # evicted token of this unit: bit-exact codes (boundary exemptions listed)
        pos = int(sc.hist_len[0])
        page = int(table[b, pos // S.PAGE])
        blk_g = lay["pool"][(page * w.hk + kv) * 6144:(page * w.hk + kv + 1) * 6144].cpu().numpy()
        mini_page = int(sc.page_table[0, pos // S.PAGE])
        blk_o = pool_o[mini_page * 6144:(mini_page + 1) * 6144]
        slot = pos % S.PAGE
        H.compare_evicted(blk_g, blk_o, np.zeros((1, 1), np.int32), [(0, slot, 0)], aux, 1)
        got = out[b, kv * G:(kv + 1) * G]
        ref = out_o[0]
        mx, rel = H.assert_close(got, ref)
        print(f"{name} b={b} kv={kv} ctx={int(st.ctx0[b])}: max-abs {mx:.2e} rel-L2 {rel:.2e}")
