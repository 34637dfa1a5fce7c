"""Helpers for the GPU parity tests: move scenes to the device, run one
decode step through the C ABI, and compare pools with the eviction
tolerance (bit-exact codes except values within 1e-5 of a rounding
boundary; fp16 scale/zero except pre-rounding values within 2^-20 of an
fp16 midpoint)."""
from __future__ import annotations

import numpy as np

import torch

from bit_kv_cache_evict_gb300 import oscar as O
from bit_kv_cache_evict_gb300 import synth as S

BOUNDARY = 1e-5          # code units: exempt codes this close to k + 0.5
MAX_EXEMPT_FRAC = 1e-4   # of all codes
MIDPOINT_REL = 2.0 ** -20
ATOL, RTOL_L2 = 2e-3, 1e-3


def dev():
    return torch.device("cuda")


def bf16_t(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev()).view(torch.bfloat16)


def i32_t(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(dev())


def f32_t(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(dev())


def u8_t(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.uint8)).to(dev())


def shape_of(sc) -> O.oscar_shape:
    return O.make_shape(sc.shape.num_q_heads, sc.shape.num_kv_heads, quant_group=sc.shape.quant_group)


def block_bytes_g(g: int) -> int:
    return 4096 + 512 * (128 // g)


def num_pages_of(sc) -> int:
    return sc.pool.size // (sc.shape.num_kv_heads * block_bytes_g(sc.shape.quant_group))


def gpu_step(sc, stream=None, status=None):
    """One decode step through the C ABI: fused evict + ring append for the
    sequences whose BF16 window is full, plain append for the others (a test
    convenience: a torch copy), then decode.  Returns (out, pool, bf16_kv,
    hist_after, bf16_len_after) as numpy."""
    sh = shape_of(sc)
    B, Hq, d = sc.q.shape
    Hk = sc.shape.num_kv_heads
    q = bf16_t(sc.q)
    kv = bf16_t(sc.bf16_kv)
    pool = u8_t(sc.pool)
    table = i32_t(sc.page_table)
    U = f32_t(sc.U32)
    clip = f32_t(sc.clip)
    new_kv = bf16_t(sc.new_kv)
    nump = num_pages_of(sc)
    full = sc.bf16_len == S.NSLOT
    seqs = np.nonzero(full)[0].astype(np.int32)
    hist = sc.hist_len.copy()
    if seqs.size:
        rows = seqs * S.NSLOT + S.SINK + sc.ring_head[seqs]
        O.oscar_evict_quantize(sh, kv.view(B * S.NSLOT, Hk, 2, d), i32_t(seqs), i32_t(hist[seqs]), U, clip, pool,
                               table, B, sc.max_pages, nump, src_row=i32_t(rows), new_kv=new_kv[i32_t(seqs).long()],
                               dev_status=status, stream=stream)
        hist[seqs] += 1
    bf16_len = sc.bf16_len.copy()
    for b in np.nonzero(~full)[0]:
        kv[b, bf16_len[b]] = new_kv[b]
        bf16_len[b] += 1
    out = torch.zeros((B, Hq, d), dtype=torch.float32, device=dev())
    ws = torch.zeros(O.oscar_decode_workspace_bytes(sh, B, sc.max_pages), dtype=torch.uint8, device=dev())
    O.oscar_decode_attn(sh, q, kv, i32_t(bf16_len), pool, table, sc.max_pages, nump, i32_t(hist), U, sc.sm_scale,
                        out, ws, dev_status=status, stream=stream)
    torch.cuda.synchronize()
    return (out.cpu().numpy(), pool.cpu().numpy(), kv.view(torch.int16).cpu().numpy().view(np.uint16), hist,
            bf16_len)


def vec_offsets(table, b, pos, kv, which, Hk, g=32):
    """Pool byte offsets of one stored token-vector: its 32 code bytes (byte j
    holds stored positions j + 32 i in bits 2i, 2i + 1) and the 4 bytes of
    each of its 128/g (fp16 s, fp16 z) pairs, as ([32], [128/g][4])."""
    bb, ng = block_bytes_g(g), 128 // g
    page = int(table[b, pos // 64])
    t = pos % 64
    base = (page * Hk + kv) * bb
    if which == 0:
        code = base + t * 32 + np.arange(32)
    else:
        code = base + 2048 + np.arange(32) * 64 + t
    sz = base + 4096 + which * 256 * ng + t * 4 * ng + 4 * np.arange(ng)[:, None] + np.arange(4)[None, :]
    return code, sz


def read_vec(pool, table, b, pos, kv, which, Hk, g=32):
    """Raw codes[128], s16[128/g], z16[128/g] of one stored token-vector (numpy)."""
    code_off, sz_off = vec_offsets(table, b, pos, kv, which, Hk, g)
    byts = pool[code_off]
    codes = ((byts[None, :] >> np.array([0, 2, 4, 6], np.uint8)[:, None]) & 3).reshape(-1)  # byte j: j + 32 i
    sz = np.ascontiguousarray(pool[sz_off.reshape(-1)]).view(np.uint16)
    return codes, sz[0::2].copy(), sz[1::2].copy()


def _allow_code(allowed, code_off, p):
    """Mark the two bits of stored position p of a vector as allowed to differ."""
    allowed[code_off[p % 32]] |= np.uint8(3 << (2 * (p // 32)))


def near_f16_midpoint(v: float) -> bool:
    """True if v lies within 2^-20 (relative) of a binary16 rounding
    midpoint, where a correctly rounded float64 and an fp64-from-another-
    summation-order value may round differently."""
    if v == 0.0 or not np.isfinite(v):
        return False
    h = np.float16(v)
    lo, hi = np.nextafter(h, np.float16(-np.inf)), np.nextafter(h, np.float16(np.inf))
    mids = [(float(h) + float(lo)) / 2, (float(h) + float(hi)) / 2]
    return any(abs(v - m) <= MIDPOINT_REL * abs(v) for m in mids)


def compare_evicted(pool_g, pool_o, table, items, aux, Hk, g=32, allowed=None):
    """items: list of (b, pos, aux_index); aux = (u, s_pre, z_pre) from the
    oracle [n][Hk][2][...].  Returns the list of exempt codes; asserts the
    rest are bit-exact.  With ``allowed`` (a uint8 array shaped like the
    pools), the bits each exemption lets differ are set there: the two bits
    of an exempt code, and the (s, z) bytes and every code of a group whose
    s or z was exempt."""
    u, sp, zp = aux
    exempt = []
    total = 0
    for (b, pos, ai) in items:
        for kv in range(Hk):
            for which in range(2):
                cg, sg, zg = read_vec(pool_g, table, b, pos, kv, which, Hk, g)
                co, so, zo = read_vec(pool_o, table, b, pos, kv, which, Hk, g)
                code_off, sz_off = vec_offsets(table, b, pos, kv, which, Hk, g)
                total += cg.size
                group_exempt = np.zeros(128 // g, bool)
                for k in range(128 // g):
                    if sg[k] != so[k] or zg[k] != zo[k]:
                        assert near_f16_midpoint(sp[ai, kv, which, k]) or near_f16_midpoint(zp[ai, kv, which, k]), \
                            (b, pos, kv, which, k, hex(sg[k]), hex(so[k]), hex(zg[k]), hex(zo[k]))
                        group_exempt[k] = True
                        if allowed is not None:
                            allowed[sz_off[k]] = 0xFF
                            for p in range(g * k, g * (k + 1)):
                                _allow_code(allowed, code_off, p)
                bad = np.nonzero(cg != co)[0]
                for j in bad:
                    uu = u[ai, kv, which, j]
                    near = abs((uu - np.floor(uu)) - 0.5) < BOUNDARY
                    assert near or group_exempt[j // g], (b, pos, kv, which, j, int(cg[j]), int(co[j]), uu)
                    exempt.append((b, pos, kv, which, int(j), float(uu)))
                    if allowed is not None:
                        _allow_code(allowed, code_off, int(j))
    assert len(exempt) <= max(1, MAX_EXEMPT_FRAC * total), (len(exempt), total)
    return exempt


def assert_pools_equal_except(pool_g, pool_o, allowed):
    """Every pool bit outside the exempted ones is equal (no stray writes)."""
    diff = np.bitwise_and(np.bitwise_xor(pool_g, pool_o), np.bitwise_not(allowed))
    bad = np.nonzero(diff)[0]
    assert bad.size == 0, (bad[:8].tolist(), int(bad.size))


def assert_close(out_g, out_o, atol=ATOL, rtol_l2=RTOL_L2):
    err = np.abs(out_g.astype(np.float64) - out_o)
    rel = np.linalg.norm(out_g.astype(np.float64) - out_o) / max(np.linalg.norm(out_o), 1e-30)
    assert err.max() <= atol and rel <= rtol_l2, (float(err.max()), float(rel))
    return float(err.max()), float(rel)
