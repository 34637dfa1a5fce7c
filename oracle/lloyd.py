"""Float64 oracle of the Lloyd-Max codebook variant.

TEST INFRASTRUCTURE ONLY: imported by tests/ and by the CPU leg of
``bench.py``; the product library never imports it.

Source: "卓绝TurboQuant：Together AI把2-bit KV Cache推向实在行状", section
"为什么这对长陡立文 Agent 很遑急": OSCAR's code repository pairs the
attention-aware rotation with a stronger Lloyd-Max codebook.  The pages give
no format; the plainest reading that keeps everything else of the method,
taken here:

  - the stored format is unchanged (four 2-bit codes per byte, fp16 scale s
    and zero z per group: z = the clipped group minimum, s = range / 3);
  - the four levels, in units of s above z, are {0, a, 3 - a, 3} instead of
    {0, 1, 2, 3}: the end levels stay at the group's extremes and the inner
    pair is placed symmetrically, a in (0, 1.5) per (layer, KV head, K/V),
    fixed offline like U and the clip ratio; a = 1 is the uniform grid;
  - a code is the nearest level to u = (y_c - z) / s, i.e. the number of the
    thresholds a/2, 3/2, 3 - a/2 that u reaches (u >= t);
  - a value is dequantised as z + s * level[code];
  - a is fitted by Lloyd's iteration on the calibration tokens' u values: by
    the symmetry, on u' = min(u, 3 - u) in [0, 3/2], whose two levels are 0
    (fixed: every group has its minimum and maximum at u' = 0) and a; the
    cell of a is u' >= a/2 and a moves to the mean of that cell until it
    stops moving.
"""
from __future__ import annotations

import numpy as np


def levels(a: float) -> np.ndarray:
    return np.array([0.0, a, 3.0 - a, 3.0])


def codes_from_u(u: np.ndarray, a: float) -> np.ndarray:
    """Nearest-level codes (u >= threshold moves up)."""
    u = np.asarray(u, np.float64)
    return ((u >= a / 2).astype(np.uint8) + (u >= 1.5).astype(np.uint8) + (u >= 3.0 - a / 2).astype(np.uint8))


def fit_a(u: np.ndarray, a0: float = 1.0, iters: int = 200, tol: float = 1e-12) -> float:
    """Lloyd's iteration for the inner level a on u' = min(u, 3 - u)."""
    v = np.minimum(np.asarray(u, np.float64).ravel(), 3.0 - np.asarray(u, np.float64).ravel())
    a = float(a0)
    for _ in range(iters):
        cell = v[v >= a / 2]
        if cell.size == 0:
            break
        a_new = float(cell.mean())
        if abs(a_new - a) <= tol:
            a = a_new
            break
        a = a_new
    return a


# ---------------------------------------------------------------------------
# decode on the stored values
# ---------------------------------------------------------------------------

def _f16(h: np.ndarray) -> np.ndarray:
    return np.asarray(h, np.uint16).view(np.float16).astype(np.float64)


def read_stored(pool: np.ndarray, table: np.ndarray, b: int, pos: int, kv: int, which: int, hk: int, g: int):
    """Codes [128] (stored order), s and z (float64, per group) of one stored
    token-vector, from the pool layout of the C ABI (include/oscar.h)."""
    ng = 128 // g
    bb = 4096 + 512 * ng
    page = int(table[b, pos // 64])
    t = pos % 64
    blk = pool[(page * hk + kv) * bb:(page * hk + kv + 1) * bb]
    byts = blk[t * 32:(t + 1) * 32] if which == 0 else blk[2048 + np.arange(32) * 64 + t]
    codes = np.empty(128, np.uint8)
    for i in range(4):                        # byte j holds stored position 32 i + j in bits 2 i
        codes[32 * i:32 * i + 32] = (byts >> (2 * i)) & 3
    off = 4096 + which * 256 * ng + t * 4 * ng
    sz = blk[off:off + 4 * ng].view(np.uint16)
    return codes, _f16(sz[0::2]), _f16(sz[1::2])


def dequantize(codes: np.ndarray, s: np.ndarray, z: np.ndarray, a: float, g: int) -> np.ndarray:
    lv = levels(a)[codes]
    grp = np.arange(128) // g
    return z[grp] + s[grp] * lv


def decode(q_bits, bf16_kv_bits, bf16_len, pool, table, hist_len, U, R_of, a, sm_scale: float, g: int = 32):
    """out [B][Hq][d] (float64): softmax attention over the valid BF16 slots
    and the stored history dequantised with the codebook levels (a [Hk][2])
    and mapped back by R^T (R_of(U[kv, which]) builds R)."""
    bf = lambda x: (np.asarray(x, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)  # noqa: E731
    q = bf(q_bits)
    kvb = bf(bf16_kv_bits)
    B, hq, d = q.shape
    hk = kvb.shape[2]
    G = hq // hk
    R = [[R_of(U[h, w]) for w in range(2)] for h in range(hk)]
    out = np.zeros((B, hq, d))
    for b in range(B):
        nb = int(bf16_len[b])
        for kv in range(hk):
            keys = [kvb[b, :nb, kv, 0, :]]
            vals = [kvb[b, :nb, kv, 1, :]]
            h = int(hist_len[b])
            if h:
                K = np.empty((h, d))
                V = np.empty((h, d))
                for pos in range(h):
                    for w, dst in ((0, K), (1, V)):
                        c, s, z = read_stored(pool, table, b, pos, kv, w, hk, g)
                        dst[pos] = dequantize(c, s, z, float(a[kv, w]), g) @ R[kv][w].T
                keys.append(K)
                vals.append(V)
            Kc, Vc = np.concatenate(keys), np.concatenate(vals)
            for j in range(G):
                hh = kv * G + j
                if Kc.shape[0] == 0:
                    continue
                lg = Kc @ q[b, hh] * sm_scale
                p = np.exp(lg - lg.max())
                out[b, hh] = p @ Vc / p.sum()
    return out


def fit_from_tokens(kv: np.ndarray, U: np.ndarray, clip: np.ndarray, group: int = 32) -> np.ndarray:
    """a [Hk][2] fitted on calibration tokens kv (float64 [n_t][Hk][2][d]):
    the u of every element of the groups whose stored s is non-zero, from
    the C oracle's quantiser (rotation y = x . R in float64), folded and
    passed to fit_a."""
    from oracle import get
    orc = get()
    n_t, hk, _, d = kv.shape
    out = np.zeros((hk, 2))
    for h in range(hk):
        for w in range(2):
            R = orc.build_R(U[h, w])
            samples = []
            for x in kv[:, h, w, :]:
                codes, s16, z16, u = orc.quantize_vec(x @ R, group, float(clip[h, w]))[:4]
                keep = np.repeat(s16 != 0, group)
                samples.append(u[keep])
            out[h, w] = fit_a(np.concatenate(samples))
    return out
