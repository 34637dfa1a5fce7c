"""Full-size parity of the Lloyd-Max and K channel-boost decodes, in the
launch configuration bench.py times (bench.GpuState with --codebook /
--boost: the whole batch's history evicted by the GPU, one bench step of
eviction + decode).  For sampled (sequence, KV head) units the float64
oracle of the variant (oracle/lloyd.py, oracle/kitty.py) attends over the
same stored values (codes, s, z, boost records, BF16 segment after the
step's append, queries); max-abs 2e-3, rel-L2 1e-3."""
import os
import sys

import numpy as np
import pytest

import oracle
from bit_kv_cache_evict_gb300 import synth as S
from oracle import kitty as K
from oracle import lloyd as L

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402
import gpu_harness as H  # noqa: E402
from bit_kv_cache_evict_gb300 import build as B  # noqa: E402

CB_A = 1.1


@pytest.fixture(scope="module", autouse=True)
def _lib():
    B.build()


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("name,mode", [("gate", "codebook"), ("gate", "boost"), ("qwen3_8b_36l", "codebook"),
                                       ("qwen3_8b_36l", "boost"), ("qwen3_32b", "codebook"), ("qwen3_32b", "boost")])
def test_variant_full_size_sampled(name, mode):
    w = S.WORKLOADS[name]
    st = bench.GpuState(w, 1, 1, 0, 32, CB_A if mode == "codebook" else None, mode == "boost")
    st.layer_step(0, 0)
    torch.cuda.synchronize()
    lay = st.layers[0]
    out = lay["out"].cpu().numpy()
    table = st.table.cpu().numpy()
    hist_all = st.hist_after[0].cpu().numpy()
    G = w.hq // w.hk
    bb = 4096 + 512 * 4
    orc = oracle.get()
    order = np.argsort(st.ctx0)
    units = [(int(order[0]), 1), (int(order[-1]), w.hk - 2), (int(order[len(order) // 2]), 4)]
    for b, kv in units:
        hist = int(hist_all[b])
        npg = (hist + S.PAGE - 1) // S.PAGE
        pages = table[b, :npg]
        pool_u = np.concatenate([lay["pool"][(int(pg) * w.hk + kv) * bb:][:bb].cpu().numpy() for pg in pages])
        mini_table = np.arange(npg, dtype=np.int32)[None, :]
        q = _bits(lay["q"][b, kv * G:(kv + 1) * G])[None]
        kvb = _bits(lay["kv"][b, :, kv:kv + 1])[None]
        U = lay["U"][kv:kv + 1].cpu().numpy().astype(np.float64)
        blen = np.array([S.NSLOT], np.int32)
        hl = np.array([hist], np.int32)
        if mode == "codebook":
            a = np.full((1, 2), float(np.float32(CB_A)))    # the fp32 value the GPU reads
            ref = L.decode(q, kvb, blen, pool_u, mini_table, hl, U, orc.build_R, a, st.sm_scale, 32)
        else:
            rec = np.concatenate([lay["boost"][(int(pg) * w.hk + kv) * K.BLOCK:][:K.BLOCK].cpu().numpy()
                                  for pg in pages])
            shape = oracle.Shape(S.D, 32, S.SINK, S.RECENT, S.PAGE, G, 1)
            ref = K.decode(orc, shape, q, kvb, blen, pool_u, mini_table, hl, U, rec, st.sm_scale)
        mx, rel = H.assert_close(out[b, kv * G:(kv + 1) * G], ref[0])
        print(f"{name} {mode} b={b} kv={kv} hist={hist}: max-abs {mx:.2e} rel-L2 {rel:.2e}")
