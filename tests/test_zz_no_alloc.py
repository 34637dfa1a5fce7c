"""oscar_decode_attn_noalloc: the decode entry point for callers that cannot
allocate device memory (for instance code inside a runtime that owns all
device memory, or a plugin limited to the buffers it is handed).  Its
scratch is the library's fixed device array instead of a caller workspace.

Checked through the C ABI against oscar_decode_attn with a workspace and
against the float64 oracle on the same inputs, on two calls in a row with
different inputs (the second call must not see anything the first one left
in the shared array), within the attention tolerance the other GPU tests
use; requests larger than the array are rejected before any launch.  This
file is collected last on purpose."""
import ctypes

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


def device_inputs(sc):
    return dict(q=H.bf16_t(sc.q), kv=H.bf16_t(sc.bf16_kv), bl=H.i32_t(sc.bf16_len), pool=H.u8_t(sc.pool),
                table=H.i32_t(sc.page_table), hist=H.i32_t(sc.hist_len), U=H.f32_t(sc.U32))


def with_workspace(sc, d):
    sh = H.shape_of(sc)
    out = torch.zeros(sc.q.shape, dtype=torch.float32, device="cuda")
    ws = torch.empty(O.oscar_decode_workspace_bytes(sh, sc.q.shape[0], sc.max_pages), dtype=torch.uint8,
                     device="cuda")
    O.oscar_decode_attn(sh, d["q"], d["kv"], d["bl"], d["pool"], d["table"], sc.max_pages, H.num_pages_of(sc),
                        d["hist"], d["U"], sc.sm_scale, out, ws)
    return out


def without_workspace(sc, d, status):
    out = torch.full(sc.q.shape, float("nan"), dtype=torch.float32, device="cuda")
    O.oscar_decode_attn_noalloc(H.shape_of(sc), d["q"], d["kv"], d["bl"], d["pool"], d["table"], sc.max_pages,
                                H.num_pages_of(sc), d["hist"], d["U"], sc.sm_scale, out, dev_status=status)
    return out


def test_noalloc_matches_workspace_entry_twice(orc):
    # call 1: several sequences, some with several split-K items; call 2: a
    # different batch and head layout, so stale scratch would show up
    w1 = S.Workload(70, "noalloc1", batch=5, hq=8, hk=2, n_outlier=2)
    sc1 = make_scene(w1, ctx=np.array([2000, 321, 5000, 100, 1300], np.int32), perm_seed=4, orc=orc)
    w2 = S.Workload(71, "noalloc2", batch=3, hq=4, hk=1, n_outlier=2)
    sc2 = make_scene(w2, ctx=np.array([900, 3100, 640], np.int32), orc=orc)
    d1, d2 = device_inputs(sc1), device_inputs(sc2)
    ref1, ref2 = with_workspace(sc1, d1), with_workspace(sc2, d2)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got1 = without_workspace(sc1, d1, status)
    got2 = without_workspace(sc2, d2, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for sc, got, ref in ((sc1, got1, ref1), (sc2, got2, ref2)):
        g, r = got.cpu().numpy(), ref.cpu().numpy().astype(np.float64)
        assert np.isfinite(g).all()
        H.assert_close(g, r)
        # and against the oracle's decode of the same pool and BF16 segment
        o = orc.decode(sc.shape, sc.q, sc.bf16_kv, sc.bf16_len, sc.pool, sc.page_table, sc.max_pages, sc.hist_len,
                       sc.U, sc.sm_scale)
        H.assert_close(g, o)


def test_noalloc_rejects_requests_beyond_the_array():
    """A request whose scratch would exceed the fixed array returns
    OSCAR_ERR_WORKSPACE before launching anything (all pointers are fake)."""
    sh = O.make_shape(32, 8)
    need = O.oscar_decode_workspace_bytes(sh, 256, 4096)
    assert need > O.NOALLOC_SCRATCH_BYTES
    fake = ctypes.c_void_p(256)
    st = O.lib().oscar_decode_attn_noalloc(ctypes.byref(sh), 256, fake, fake, fake, fake, fake, 4096, 1, fake,
                                           fake, ctypes.c_float(0.1), fake, None, None)
    assert st == O.OSCAR_ERR_WORKSPACE
