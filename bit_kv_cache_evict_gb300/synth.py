"""Seeded synthetic inputs for the OSCAR hot path.

This module only draws random inputs and encodes them (float -> bf16 bits);
it holds none of the method's arithmetic.  Both the CUDA path's tests and
the float64 oracle are fed from here, so neither side generates inputs for
the other.

The workloads stand in for the pages' Qwen3-4B / 8B / 32B serving runs
("卓绝TurboQuant：Together AI把2-bit KV Cache推向实在行状", accuracy and
systems sections): only head layouts, context lengths and the
outlier-channel structure of K/V activations (a few channels of large
magnitude, section "不是更会'压缩向量'，而是运转保护 attention") are taken
from them.  No model weights, calibration data or benchmark items are used.

Seeds: numpy ``Generator(PCG64(seed))`` with ``seed = 1000 + workload id``.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

D = 128          # head_dim
GROUP = 32       # quantisation group along head_dim
SINK = 64        # BF16 sink tokens
RECENT = 256     # BF16 recent window
PAGE = 64        # tokens per history page
NSLOT = SINK + RECENT


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic decode workload.  ``ctx`` is the context length per
    sequence *before* the step (sink + history + recent); a step evicts one
    token per sequence and layer, appends one, and attends over ctx + 1."""
    wid: int
    name: str
    batch: int
    hq: int
    hk: int
    layers: int = 1
    ctx_kind: str = "fixed"        # fixed | uniform | loguniform
    ctx_lo: int = 32768
    ctx_hi: int = 32768
    shuffled: bool = False         # seeded permutation of the page pool
    dist: str = "gauss_outlier"    # gauss_outlier | student_t
    n_outlier: int = 4
    outlier_scale: float = 20.0
    clip: float = 0.95
    prefix_seqs: int = 0           # sequences sharing one prefix
    prefix_tokens: int = 0         # shared prefix length (tokens)
    evict_per_step: int = 1        # evictions per sequence per layer and step

    @property
    def seed(self) -> int:
        return 1000 + self.wid

    @property
    def group(self) -> int:
        return self.hq // self.hk

    @property
    def shared_hist_tokens(self) -> int:
        """History tokens of the shared prefix (sink excluded), rounded down
        to whole pages so shared pages are full and never written."""
        if self.prefix_seqs == 0:
            return 0
        return ((self.prefix_tokens - SINK) // PAGE) * PAGE


WORKLOADS: dict[str, Workload] = {
    # 1 sequence, 1 KV head, 4 query heads, context 1024 = 64 + 704 + 256.
    "tiny": Workload(1, "tiny", batch=1, hq=4, hk=1, ctx_lo=1024, ctx_hi=1024, n_outlier=2),
    # Qwen3-4B-shaped single layer: batch 8, 32/8 heads, 32K, contiguous pages.
    "qwen3_4b": Workload(2, "qwen3_4b", batch=8, hq=32, hk=8),
    # Qwen3-8B-shaped full decode step over 36 layers: batch 64, context
    # uniform in [4096, 32768], shuffled page table.
    "qwen3_8b_36l": Workload(3, "qwen3_8b_36l", batch=64, hq=32, hk=8, layers=36, ctx_kind="uniform",
                             ctx_lo=4096, ctx_hi=32768, shuffled=True),
    # Qwen3-32B-shaped single layer: batch 128, 64/8 heads, 32K,
    # Student-t(3) K/V with lognormal(sigma=1) per-channel scales.
    "qwen3_32b": Workload(4, "qwen3_32b", batch=128, hq=64, hk=8, dist="student_t"),
    # Large-batch mixed-length stress: batch 256, Qwen3-8B heads, context
    # log-uniform in [1K, 128K], sequences 0..31 share a 2K-token prefix.
    "stress": Workload(5, "stress", batch=256, hq=32, hk=8, ctx_kind="loguniform", ctx_lo=1024,
                       ctx_hi=131072, prefix_seqs=32, prefix_tokens=2048),
    # Qwen3-8B layout, batch 64, context exactly 32768, one layer.
    "gate": Workload(6, "gate", batch=64, hq=32, hk=8),
    # One sequence of 100K tokens (the long-context, batch-1 decode of a full
    # prefix-cache hit: all of the history is already in the pool), Qwen3-8B
    # heads, 36 layers; the split-K plan has to fill the GPU from one sequence.
    "longctx_b1": Workload(7, "longctx_b1", batch=1, hq=32, hk=8, layers=36, ctx_lo=100000, ctx_hi=100000),
}


def rng_for(w: Workload, stream: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([w.seed, stream]))


# ---------------------------------------------------------------------------
# encodings
# ---------------------------------------------------------------------------

def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float64/float32 -> bf16 bit patterns (uint16), round to nearest even
    from the float32 value.  NaN is not expected in synthetic inputs."""
    f = np.ascontiguousarray(np.asarray(x, np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------------------
# draws
# ---------------------------------------------------------------------------

def context_lengths(w: Workload) -> np.ndarray:
    rng = rng_for(w, 1)
    if w.ctx_kind == "fixed":
        ctx = np.full(w.batch, w.ctx_lo, np.int64)
    elif w.ctx_kind == "uniform":
        ctx = rng.integers(w.ctx_lo, w.ctx_hi + 1, size=w.batch)
    elif w.ctx_kind == "loguniform":
        ctx = np.exp(rng.uniform(math.log(w.ctx_lo), math.log(w.ctx_hi), size=w.batch)).astype(np.int64)
        if w.prefix_seqs:
            # prefix sharers: long enough that the prefix lies wholly in
            # sink + history (prefix + a full recent window)
            lo = w.prefix_tokens + RECENT
            ctx[: w.prefix_seqs] = np.exp(rng.uniform(math.log(lo), math.log(w.ctx_hi),
                                                      size=w.prefix_seqs)).astype(np.int64)
    else:
        raise ValueError(w.ctx_kind)
    return ctx.astype(np.int32)


def rotation_U(w: Workload, layer: int = 0) -> np.ndarray:
    """Per (KV head, K/V) random orthogonal U: QR of a seeded Gaussian with
    sign-fixed diag(R) > 0.  float64 [Hk][2][d][d]."""
    rng = rng_for(w, 100 + layer)
    U = np.empty((w.hk, 2, D, D), np.float64)
    for h in range(w.hk):
        for kv in range(2):
            a = rng.standard_normal((D, D))
            q, r = np.linalg.qr(a)
            U[h, kv] = q * np.sign(np.diag(r))[None, :]
    return U


def clip_ratios(w: Workload) -> np.ndarray:
    return np.full((w.hk, 2), w.clip, np.float64)


def channel_profile(w: Workload, layer: int = 0):
    """Per (KV head, K/V, channel) multiplier of the unrotated K/V values."""
    rng = rng_for(w, 200 + layer)
    if w.dist == "gauss_outlier":
        scale = np.ones((w.hk, 2, D))
        for h in range(w.hk):
            ch = rng.choice(D, size=w.n_outlier, replace=False)
            scale[h, :, ch] = w.outlier_scale
        return scale
    if w.dist == "student_t":
        return rng.lognormal(0.0, 1.0, size=(w.hk, 2, D))
    raise ValueError(w.dist)


def kv_tokens(w: Workload, n: int, rng: np.random.Generator, profile: np.ndarray) -> np.ndarray:
    """n token rows of K/V, bf16 bits [n][Hk][2][d]."""
    if w.dist == "gauss_outlier":
        x = rng.standard_normal((n, w.hk, 2, D))
    else:
        x = rng.standard_t(3.0, size=(n, w.hk, 2, D))
    return bf16_bits(x * profile[None])


def queries(w: Workload, rng: np.random.Generator, batch: int | None = None) -> np.ndarray:
    return bf16_bits(rng.standard_normal((batch or w.batch, w.hq, D)))


# ---------------------------------------------------------------------------
# torch (device) draws for large benchmark pools; same distributions, not
# the same values as the numpy draws
# ---------------------------------------------------------------------------

def kv_tokens_torch(w: Workload, n: int, gen, profile_t, device):
    import torch
    if w.dist == "gauss_outlier":
        x = torch.randn((n, w.hk, 2, D), generator=gen, device=device, dtype=torch.float32)
    else:
        # Student-t(3) = N / sqrt(chi2_3 / 3)
        z = torch.randn((n, w.hk, 2, D), generator=gen, device=device, dtype=torch.float32)
        c = torch.randn((n, w.hk, 2, D, 3), generator=gen, device=device, dtype=torch.float32)
        x = z / torch.sqrt((c * c).sum(-1) / 3.0)
    return (x * profile_t).to(torch.bfloat16)


# ---------------------------------------------------------------------------
# offline rotation calibration
# ---------------------------------------------------------------------------

CALIB_SPECTRUM_SCALE = 24.0   # eigenvalue i of each drawn covariance: exp(-i / 24)


def calibration_inputs(seed: int, n_q: int, n_t: int, hq: int, hk: int):
    """Seeded calibration activations for the offline rotation calibration:
    query tokens q [n_q][hq][D] and K/V tokens [n_t][hk][2][D], as bf16 bit
    patterns.  Each KV head draws three orthogonal bases (queries of its
    group, keys, values) and the values are Gaussian along them with the
    spectrum exp(-i / 24) (every eigenvalue distinct), scaled so that the
    attention of a query over the tokens is selective (logits of a few
    units), as the pages' calibration on real activations would be.  They
    stand in for model activations, which this build has none of."""
    rng = np.random.Generator(np.random.PCG64([seed, 7]))
    g = hq // hk
    sd = np.sqrt(np.exp(-np.arange(D) / CALIB_SPECTRUM_SCALE))
    q = np.empty((n_q, hq, D))
    kv = np.empty((n_t, hk, 2, D))
    for h in range(hk):
        bases = []
        for _ in range(3):
            a, r = np.linalg.qr(rng.standard_normal((D, D)))
            bases.append(a * np.sign(np.diag(r))[None, :])
        for j in range(g):
            q[:, h * g + j, :] = 3.0 * (rng.standard_normal((n_q, D)) * sd) @ bases[0].T
        kv[:, h, 0, :] = 3.0 * (rng.standard_normal((n_t, D)) * sd) @ bases[1].T
        kv[:, h, 1, :] = 2.0 * (rng.standard_normal((n_t, D)) * sd) @ bases[2].T
    return bf16_bits(q), bf16_bits(kv)
