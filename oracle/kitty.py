"""Float64 oracle of the channel precision boost variant (K history).

TEST INFRASTRUCTURE ONLY: imported by tests/ and by the CPU leg of
``bench.py``; the product library never imports it.

Source: the "Zhongzhu (Charlie) Zhou" home page, Featured Projects, entry
"KITTY: Accurate and Efficient 2-bit KV Cache Quantization with Dynamic
Channel-wise Precision Boost": a sibling method of OSCAR keeps a small
fraction of the K cache's channels at 4 bits and the rest at 2 bits,
choosing them dynamically.  The pages say nothing more; the reading taken
here keeps OSCAR's stored format and adds to it:

  - K only.  Every stored K token-vector keeps its 2-bit codes, s and z
    exactly as the uniform eviction writes them;
  - of its 128 stored positions (the rotated channels), the NB = 8 whose
    2-bit rounding error |u - c| is largest are boosted (ties to the lower
    stored position; u = (y_c - z) / s from the stored s and z, u = 0 and
    error 0 where s = 0): "dynamic" = chosen per token from its own values;
  - a boosted position holds a 4-bit code q4 = clamp(rint(5 u), 0, 15) on
    the same group range, i.e. levels z + s * q4 / 5 (sixteen levels from z
    to z + 3 s, step s / 5; rint = round half to even);
  - the boost record of a token is NB little-endian 16-bit entries
    (stored position in bits 0-6, q4 in bits 8-11, and a copy of the
    position's 2-bit code c in bits 12-13, so that a reader finds the
    correction q4 / 5 - c without the code bytes), in increasing stored
    position, 16 bytes; the records of a (page, KV head) form a 1024-byte
    block (token t at byte 16 t) of a separate array indexed like the pool;
  - a K value is z + s * q4 / 5 at a boosted position, z + s * c elsewhere;
    V is unchanged.
"""
from __future__ import annotations

import numpy as np

NB = 8                      # boosted positions per K token-vector
RECORD = 2 * NB             # bytes per token
BLOCK = 64 * RECORD         # bytes per (page, KV head)


def select(u: np.ndarray, codes: np.ndarray, s_nonzero: np.ndarray) -> np.ndarray:
    """Boosted stored positions of one vector (sorted): the NB largest
    rounding errors |u - c|, ties to the lower position.  s_nonzero [d]
    marks positions whose group has s != 0 (error 0 elsewhere)."""
    err = np.where(s_nonzero, np.abs(np.asarray(u, np.float64) - codes), 0.0)
    order = sorted(range(err.size), key=lambda j: (-err[j], j))
    return np.array(sorted(order[:NB]), np.int64)


def q4_of(u: np.ndarray) -> np.ndarray:
    return np.clip(np.rint(5.0 * np.asarray(u, np.float64)), 0, 15).astype(np.int64)


def record(u: np.ndarray, codes: np.ndarray, s_nonzero: np.ndarray) -> np.ndarray:
    """The 16-byte boost record of one vector."""
    pos = select(u, codes, s_nonzero)
    q4 = np.where(s_nonzero[pos], q4_of(u[pos]), 0)
    ent = (pos | (q4 << 8) | (np.asarray(codes, np.int64)[pos] << 12)).astype("<u2")
    return ent.view(np.uint8)


def parse(rec: np.ndarray):
    """(positions, 4-bit codes) of a record."""
    ent = np.asarray(rec, np.uint8).view("<u2").astype(np.int64)
    return ent & 0x7F, (ent >> 8) & 0xF


def parse_codes(rec: np.ndarray):
    """The 2-bit code copies of a record's entries."""
    return (np.asarray(rec, np.uint8).view("<u2").astype(np.int64) >> 12) & 3


def evict(orc, shape, src, seq, pos, U, clip, pool, table, max_pages, boost):
    """The uniform eviction (the C oracle) plus the boost records of the K
    vectors written into ``boost`` (uint8, num_pages * Hk * 1024).  Returns
    the C oracle's (u, s_pre, z_pre)."""
    u, sp, zp = orc.evict(shape, src, seq, pos, U, clip, pool, table, max_pages, want_aux=True)
    hk, g = shape.num_kv_heads, shape.quant_group
    for i in range(len(seq)):
        b, p = int(seq[i]), int(pos[i])
        page = int(table[b, p // 64])
        for kv in range(hk):
            codes, s, _ = read_k(pool, table, b, p, kv, hk, g)
            nz = np.repeat(s != 0, g)
            off = (page * hk + kv) * BLOCK + (p % 64) * RECORD
            boost[off:off + RECORD] = record(u[i, kv, 0], codes, nz)
    return u, sp, zp


def _f16(h) -> np.ndarray:
    return np.asarray(h, np.uint16).view(np.float16).astype(np.float64)


def read_k(pool, table, b, pos, kv, hk, g):
    """Stored codes [128], s and z (float64 per group) of one K vector."""
    ng = 128 // g
    bb = 4096 + 512 * ng
    page = int(table[b, pos // 64])
    t = pos % 64
    blk = pool[(page * hk + kv) * bb:(page * hk + kv + 1) * bb]
    byts = blk[t * 32:(t + 1) * 32]
    codes = np.empty(128, np.uint8)
    for i in range(4):                        # byte j holds stored position 32 i + j in bits 2 i
        codes[32 * i:32 * i + 32] = (byts >> (2 * i)) & 3
    sz = blk[4096 + t * 4 * ng:4096 + (t + 1) * 4 * ng].view(np.uint16)
    return codes, _f16(sz[0::2]), _f16(sz[1::2])


def dequantize_k(codes, s, z, rec, g):
    """K value in the rotated domain: 2-bit levels, boosted positions on the
    4-bit grid."""
    grp = np.arange(128) // g
    v = z[grp] + s[grp] * codes
    pos, q4 = parse(rec)
    v[pos] = z[grp[pos]] + s[grp[pos]] * (q4 / 5.0)
    return v


def decode(orc, shape, q_bits, bf16_kv_bits, bf16_len, pool, table, hist_len, U, boost, sm_scale):
    """out [B][Hq][d] (float64): softmax attention over the valid BF16 slots
    and the stored history (K with the boost, V uniform) mapped back by R^T."""
    bf = lambda x: (np.asarray(x, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)  # noqa: E731
    q = bf(q_bits)
    kvb = bf(bf16_kv_bits)
    B, hq, d = q.shape
    hk = kvb.shape[2]
    G = hq // hk
    g = shape.quant_group
    ng = 128 // g
    bb = 4096 + 512 * ng
    out = np.zeros((B, hq, d))
    for b in range(B):
        nb = int(bf16_len[b])
        for kv in range(hk):
            RK, RV = orc.build_R(U[kv, 0]), orc.build_R(U[kv, 1])
            keys = [kvb[b, :nb, kv, 0, :]]
            vals = [kvb[b, :nb, kv, 1, :]]
            h = int(hist_len[b])
            if h:
                K = np.empty((h, d))
                V = np.empty((h, d))
                for p in range(h):
                    page = int(table[b, p // 64])
                    t = p % 64
                    codes, s, z = read_k(pool, table, b, p, kv, hk, g)
                    off = (page * hk + kv) * BLOCK + t * RECORD
                    K[p] = dequantize_k(codes, s, z, boost[off:off + RECORD], g) @ RK.T
                    blk = pool[(page * hk + kv) * bb:(page * hk + kv + 1) * bb]
                    byts = blk[2048 + np.arange(32) * 64 + t]
                    vc = np.concatenate([(byts >> (2 * i)) & 3 for i in range(4)]).astype(np.float64)
                    vo = 4096 + 256 * ng + t * 4 * ng
                    sz = blk[vo:vo + 4 * ng].view(np.uint16)
                    grp = np.arange(128) // g
                    V[p] = (_f16(sz[1::2])[grp] + _f16(sz[0::2])[grp] * vc) @ RV.T
                keys.append(K)
                vals.append(V)
            Kc, Vc = np.concatenate(keys), np.concatenate(vals)
            for j in range(G):
                hh = kv * G + j
                if Kc.shape[0] == 0:
                    continue
                lg = Kc @ q[b, hh] * sm_scale
                p_ = np.exp(lg - lg.max())
                out[b, hh] = p_ @ Vc / p_.sum()
    return out
