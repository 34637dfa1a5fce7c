"""Decode scenes for tests: seeded inputs plus an INT2 history written by
the oracle's eviction (so no stored value or oracle input comes from the
CUDA path).  Test infrastructure only."""
from __future__ import annotations

import dataclasses

import numpy as np

import oracle
from bit_kv_cache_evict_gb300 import synth as S


@dataclasses.dataclass
class Scene:
    shape: oracle.Shape
    hist_len: np.ndarray      # [B] history tokens already in the pool
    bf16_len: np.ndarray      # [B] valid BF16 slots
    ring_head: np.ndarray     # [B] ring index of the oldest recent token
    q: np.ndarray             # bf16 bits [B][Hq][d]
    bf16_kv: np.ndarray       # bf16 bits [B][320][Hk][2][d]
    pool: np.ndarray          # uint8 [num_pages * Hk * block_bytes]
    page_table: np.ndarray    # int32 [B][max_pages]
    max_pages: int
    U: np.ndarray             # float64 [Hk][2][d][d] (fp32-exact values)
    U32: np.ndarray           # float32 copy of U
    clip: np.ndarray          # float64 [Hk][2]
    new_kv: np.ndarray        # bf16 bits [B][Hk][2][d]: the token appended by a step
    sm_scale: float


def make_scene(w: S.Workload, ctx: np.ndarray | None = None, hq: int | None = None, hk: int | None = None,
               extra_capacity: int = 64, perm_seed: int = 0, prefix_group=None, shared_hist_tokens: int = 0,
               orc: oracle.Oracle | None = None, quant_group: int = S.GROUP, only_kv: int | None = None) -> Scene:
    """Build a decode state: sink = first 64 tokens, recent ring = last 256,
    history = the rest (quantised by the oracle).  With only_kv, the draws
    are those of the full head layout, but only KV head only_kv (and its G
    query heads) is kept: a one-KV-head scene of that unit."""
    orc = orc or oracle.get()
    hq = hq or w.hq
    hk = hk or w.hk
    ctx = S.context_lengths(w) if ctx is None else np.asarray(ctx, np.int32)
    B = ctx.shape[0]
    wl = dataclasses.replace(w, hq=hq, hk=hk, batch=B)
    rng = S.rng_for(wl, 7)
    prof = S.channel_profile(wl)
    G = hq // hk
    keep = slice(None) if only_kv is None else slice(only_kv, only_kv + 1)
    keep_q = slice(None) if only_kv is None else slice(only_kv * G, (only_kv + 1) * G)
    if only_kv is not None:
        hq, hk = G, 1
    shape = oracle.Shape(S.D, quant_group, S.SINK, S.RECENT, S.PAGE, hq, hk)
    hist = np.maximum(ctx - S.NSLOT, 0).astype(np.int32)
    bf16_len = np.minimum(ctx, S.NSLOT).astype(np.int32)
    cap = hist + extra_capacity
    max_pages = int(max(1, (cap.max() + S.PAGE - 1) // S.PAGE))
    rc, table, npages, nbytes = orc.pool_layout(shape, cap, prefix_group, shared_hist_tokens, perm_seed,
                                                max_pages)
    assert rc == 0, rc
    pool = np.zeros(max(nbytes, 16), np.uint8)
    U = S.rotation_U(wl).astype(np.float32)[keep]
    clip = S.clip_ratios(wl)
    bf16_kv = np.zeros((B, S.NSLOT, hk, 2, S.D), np.uint16)
    clip_keep = clip[keep]
    ring_head = np.zeros(B, np.int32)
    prefix_toks = {}
    for b in range(B):
        toks = S.kv_tokens(wl, int(ctx[b]), rng, prof)[:, keep]
        if prefix_group is not None and prefix_group[b] >= 0:
            # sharers see identical sink + shared-history tokens
            n_pre = S.SINK + shared_hist_tokens
            if prefix_group[b] in prefix_toks:
                toks[:n_pre] = prefix_toks[prefix_group[b]]
            else:
                prefix_toks[prefix_group[b]] = toks[:n_pre].copy()
        nb = int(bf16_len[b])
        if ctx[b] <= S.NSLOT:
            bf16_kv[b, :nb] = toks[:nb]
        else:
            bf16_kv[b, :S.SINK] = toks[:S.SINK]
            bf16_kv[b, S.SINK:] = toks[ctx[b] - S.RECENT:]
            h = int(hist[b])
            if h:
                pos = np.arange(h, dtype=np.int32)
                # shared prefix pages are written once, by the first sharer
                if prefix_group is not None and prefix_group[b] >= 0:
                    first = int(np.argmax(np.asarray(prefix_group) == prefix_group[b]))
                    if first != b:
                        pos = pos[pos >= shared_hist_tokens]
                if pos.size:
                    orc.evict(shape, toks[S.SINK:S.SINK + h], np.full(pos.size, b, np.int32), pos,
                              U.astype(np.float64), clip_keep, pool, table, max_pages,
                              src_row=pos)
    q = S.queries(wl, rng, B)[:, keep_q]
    new_kv = S.kv_tokens(wl, B, rng, prof)[:, keep]
    return Scene(shape, hist, bf16_len, ring_head, np.ascontiguousarray(q), bf16_kv, pool, table, max_pages,
                 U.astype(np.float64), np.ascontiguousarray(U), clip[keep], np.ascontiguousarray(new_kv),
                 1.0 / np.sqrt(S.D))


def oracle_step(orc: oracle.Oracle, sc: Scene):
    """One decode step on the oracle side (append -> evict oldest recent ->
    attend).  Returns (out, pool_after, bf16_kv_after, hist_after, aux)."""
    B = sc.q.shape[0]
    pool = sc.pool.copy()
    kv = sc.bf16_kv.copy()
    hist = sc.hist_len.copy()
    full = sc.bf16_len == S.NSLOT
    seqs = np.nonzero(full)[0].astype(np.int32)
    rows = (seqs * S.NSLOT + S.SINK + sc.ring_head[seqs]).astype(np.int32)
    aux = None
    if seqs.size:
        flat = kv.reshape(B * S.NSLOT, sc.shape.num_kv_heads, 2, S.D)
        aux = orc.evict(sc.shape, flat, seqs, hist[seqs], sc.U, sc.clip, pool, sc.page_table, sc.max_pages,
                        src_row=rows, want_aux=True)
        flat[rows] = sc.new_kv[seqs]
        hist[seqs] += 1
    bf16_len = sc.bf16_len.copy()
    for b in np.nonzero(~full)[0]:
        kv[b, bf16_len[b]] = sc.new_kv[b]
        bf16_len[b] += 1
    out = orc.decode(sc.shape, sc.q, kv, bf16_len, pool, sc.page_table, sc.max_pages, hist, sc.U, sc.sm_scale)
    return out, pool, kv, hist, bf16_len, seqs, aux
