"""GPU parity of oscar_calibrate_rotation against the float64 oracle
(oracle/calibrate.py), on seeded anisotropic calibration activations.

The GPU computes in fp32 (attention, covariance sums, Jacobi), the oracle in
float64 on the same bf16 inputs.  Checked per (KV head, K/V) matrix:
eigenvalues within 2e-5 of the largest; the eigen-equation C u = lam u of the
oracle's covariance; orthogonality of U; and, for every eigenvector whose
eigenvalue is separated from its neighbours by a relative gap g, the angle to
the oracle's eigenvector within 2e-5 / g (first-order perturbation bound
with the fp32 error of C), with the same sign once that angle is small.
"""
import numpy as np
import pytest

from bit_kv_cache_evict_gb300 import synth as S
from oracle import calibrate as OC

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from bit_kv_cache_evict_gb300 import build as B  # noqa: E402
from bit_kv_cache_evict_gb300 import oscar as O  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _lib():
    B.build()
    O.lib()


def _shape(hq, hk):
    return O.oscar_shape(128, 32, 64, 256, 64, hq, hk)


@pytest.mark.parametrize("n_q,n_t,hq,hk", [(256, 512, 8, 2), (97, 333, 4, 4), (64, 1000, 8, 1)])
def test_calibration_matches_oracle(n_q, n_t, hq, hk):
    qb, kvb = S.calibration_inputs(17 + n_q, n_q, n_t, hq, hk)
    scale = 1 / np.sqrt(128)
    sh = _shape(hq, hk)
    q_t = torch.from_numpy(qb.view(np.int16)).cuda().view(torch.bfloat16)
    kv_t = torch.from_numpy(kvb.view(np.int16)).cuda().view(torch.bfloat16)
    U_t = torch.zeros((hk, 2, 128, 128), dtype=torch.float32, device="cuda")
    lam_t = torch.zeros((hk, 2, 128), dtype=torch.float32, device="cuda")
    ws = torch.zeros(O.oscar_calibrate_workspace_bytes(sh, n_q), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    O.oscar_calibrate_rotation(sh, q_t, kv_t, scale, U_t, ws, eigvals=lam_t, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    U_g, lam_g = U_t.cpu().numpy().astype(np.float64), lam_t.cpu().numpy().astype(np.float64)

    q = S.bf16_to_f32(qb).astype(np.float64)
    kv = S.bf16_to_f32(kvb).astype(np.float64)
    ck = OC.query_covariance(q, hk)
    cv = OC.value_covariance(OC.attention_outputs(q, kv[:, :, 0], kv[:, :, 1], scale), hk)
    for h in range(hk):
        for w, cm in enumerate((ck[h], cv[h])):
            U_r, lam_r = OC.rotation_from_covariance(cm)
            top = lam_r[0]
            u, lam = U_g[h, w], lam_g[h, w]
            assert np.abs(lam - lam_r).max() <= 2e-5 * top, (h, w)
            assert np.abs(u.T @ u - np.eye(128)).max() <= 2e-5, (h, w)
            assert np.abs(cm @ u - u * lam).max() <= 5e-5 * top, (h, w)
            gaps = np.full(128, np.inf)
            gaps[:-1] = np.minimum(gaps[:-1], lam_r[:-1] - lam_r[1:])
            gaps[1:] = np.minimum(gaps[1:], lam_r[:-1] - lam_r[1:])
            rel = gaps / top
            for j in np.nonzero(rel > 1e-3)[0]:
                dot = float(u[:, j] @ U_r[:, j]) / float(np.linalg.norm(u[:, j]))  # cosine: U is orthonormal to ~1e-6
                bound = 2e-5 / rel[j]
                assert 1.0 - abs(dot) <= 0.5 * bound * bound + 1e-9, (h, w, j, dot, bound)
                mags = np.sort(np.abs(U_r[:, j]))
                if mags[-1] - mags[-2] > 10 * bound:  # the sign convention's pivot entry is unambiguous
                    assert dot > 0, (h, w, j, dot)


@pytest.mark.parametrize("n_t,hk,qg", [(300, 2, 32), (130, 1, 128)])
def test_clip_search_matches_oracle(n_t, hk, qg):
    """Per-candidate mean squared errors within 2e-4 (relative) of the
    oracle's, and the chosen ratio equal to the oracle's unless the oracle's
    two best candidates are that close."""
    _, kvb = S.calibration_inputs(90 + n_t, 8, n_t, 4 * hk, hk)
    w = S.Workload(77, "clip", batch=1, hq=4 * hk, hk=hk)
    U = S.rotation_U(w).astype(np.float32)
    grid = np.round(np.arange(0.80, 1.0001, 0.02), 4).astype(np.float32)
    sh = O.oscar_shape(128, qg, 64, 256, 64, 4 * hk, hk)
    kv_t = torch.from_numpy(kvb.view(np.int16)).cuda().view(torch.bfloat16)
    U_t = torch.from_numpy(U).cuda()
    grid_t = torch.from_numpy(grid).cuda()
    clip_t = torch.zeros((hk, 2), dtype=torch.float32, device="cuda")
    mse_t = torch.zeros((hk, 2, grid.size), dtype=torch.float32, device="cuda")
    O.oscar_calibrate_clip(sh, kv_t, U_t, grid_t, clip_t, mse=mse_t)
    torch.cuda.synchronize()
    clip_r, mse_r = OC.clip_search(S.bf16_to_f32(kvb).astype(np.float64), U.astype(np.float64), grid, qg)
    mse_g, clip_g = mse_t.cpu().numpy(), clip_t.cpu().numpy()
    assert np.abs(mse_g - mse_r).max() <= 2e-4 * mse_r.max()
    for h in range(hk):
        for wv in range(2):
            srt = np.sort(mse_r[h, wv])
            if srt[1] - srt[0] > 2e-4 * srt[0]:
                assert clip_g[h, wv] == clip_r[h, wv], (h, wv, clip_g[h, wv], clip_r[h, wv], mse_r[h, wv])
