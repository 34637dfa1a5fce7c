"""The decode step inside a CUDA graph.

One layer's step (fused eviction + append, then decode attention) is
captured once with torch's graph capture on the C ABI's stream argument and
replayed; its results match the same step run eagerly.  The split-K work
queue makes the floating-point summation order depend on scheduling, so
the attention outputs are compared with a tight relative bound rather than
bit for bit; the pool and the BF16 segment must match exactly."""
import numpy as np
import pytest

from bit_kv_cache_evict_gb300 import synth as S
from scene import make_scene

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


def test_step_captured_in_a_cuda_graph(orc):
    w = S.Workload(61, "graph", batch=6, hq=8, hk=2, n_outlier=2)
    sc = make_scene(w, ctx=np.array([4000, 900, 321, 2500, 1400, 700], np.int32), perm_seed=9, orc=orc)
    sh = H.shape_of(sc)
    Bsz, Hq, d = sc.q.shape
    Hk = sc.shape.num_kv_heads
    full = sc.bf16_len == S.NSLOT
    assert full.all()
    seqs = H.i32_t(np.arange(Bsz))
    rows = H.i32_t(np.arange(Bsz) * S.NSLOT + S.SINK + sc.ring_head)
    hist_before = H.i32_t(sc.hist_len)
    hist_after = H.i32_t(sc.hist_len + 1)
    bf16_len = H.i32_t(sc.bf16_len)
    q, U, clip, table = H.bf16_t(sc.q), H.f32_t(sc.U32), H.f32_t(sc.clip), H.i32_t(sc.page_table)
    new_kv = H.bf16_t(sc.new_kv)
    nump = H.num_pages_of(sc)
    ws = torch.zeros(O.oscar_decode_workspace_bytes(sh, Bsz, sc.max_pages), dtype=torch.uint8, device="cuda")

    def fresh():
        return H.u8_t(sc.pool), H.bf16_t(sc.bf16_kv), torch.zeros((Bsz, Hq, d), dtype=torch.float32, device="cuda")

    def step(pool, kv, out, stream):
        O.oscar_evict_quantize(sh, kv.view(Bsz * S.NSLOT, Hk, 2, d), seqs, hist_before, U, clip, pool, table, Bsz,
                               sc.max_pages, nump, src_row=rows, new_kv=new_kv, stream=stream)
        O.oscar_decode_attn(sh, q, kv, bf16_len, pool, table, sc.max_pages, nump, hist_after, U, sc.sm_scale, out,
                            ws, stream=stream)

    # eager reference (also sets the kernels' attributes before any capture)
    pool_e, kv_e, out_e = fresh()
    step(pool_e, kv_e, out_e, torch.cuda.current_stream())
    torch.cuda.synchronize()

    pool_g, kv_g, out_g = fresh()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            step(pool_g, kv_g, out_g, side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    assert float(out_g.abs().max()) == 0.0   # capturing ran nothing
    graph.replay()
    torch.cuda.synchronize()

    assert torch.equal(pool_g, pool_e)
    assert torch.equal(kv_g.view(torch.int16), kv_e.view(torch.int16))
    a, b = out_g.cpu().numpy().astype(np.float64), out_e.cpu().numpy().astype(np.float64)
    assert np.isfinite(a).all()
    assert np.abs(a - b).max() <= 1e-5 * max(1.0, np.abs(b).max())
