"""The numeric property the INT2 decode's tensor-core products rest on.

The decode feeds 2-bit codes to mma.sync (fp16, both products) without
unpacking them into values: a code c left at bits P, P + 1 of an otherwise
clear 16-bit half is the bit pattern c << P, whose value read as fp16 is
c * 2^(P - 24), because the fp16 subnormals and the first normal binade join
without a gap (patterns below 0x0400; read as bf16 it is c * 2^(P - 133) for
P <= 6).  The power of two is folded into the scales.  The tensor core keeps
the products of such operands to a fixed number of bits below their nominal
exponent, so the precision of a product depends on P: the kernel takes the
codes of byte slot 0 at bits 8-9 (from the code word with the bytes of each
half swapped) and slots 1, 2, 3 at bits 2, 4, 6.

One warp and one MMA per case, A built by the library's operand helpers
from random code words, B a sweep of magnitudes over the range the scale
folding uses (fp16: 2^-6 .. 2^15: q' * 2^e with the largest |q'| of a KV
group at 2^13 .. 2^14 and W = p * s up to 65504, low parts and small
elements below, down into the fp16 subnormals; bf16, slots 1-3 only, for
comparison: 2^8 .. 2^125); checked here against exact float64 products:

- every A register is the expected bit pattern, and the pattern's value is
  c * 2^(P - 24) (fp16) or c * 2^(P - 133) (bf16);
- products of short-mantissa B values (exactly representable sums) come out
  exact for every slot;
- for full-mantissa B with mixed magnitudes (hi and lo parts, tiny values),
  |D - exact| <= 2^-r * sum |terms| with r = 22, 22, 20, 18 retained bits
  for P = 8, 6, 4, 2 (a bit of margin over the bits each slot keeps: P = 8
  and 6 lose nothing, P = 4 two bits, P = 2 four bits).
"""
import ctypes
import os
import subprocess
import tempfile

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from bit_kv_cache_evict_gb300 import build as B  # noqa: E402

HERE = os.path.dirname(os.path.abspath(__file__))
SLOT_BIT = {0: 8, 1: 2, 2: 4, 3: 6}          # bit of the code inside its operand half, per byte slot
RETAINED = {8: 22, 6: 22, 4: 20, 2: 18}      # bits kept relative to sum |terms|, with margin


@pytest.fixture(scope="module")
def probe():
    out = os.path.join(tempfile.mkdtemp(), "tc_code_operands.so")
    subprocess.run([B.nvcc_path(), *B.ARCH, "-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-shared", "-cudart",
                    "shared", os.path.join(HERE, "cuda", "tc_code_operands.cu"), "-o", out], check=True)
    lib = ctypes.CDLL(out)
    lib.run_tc_code_operands.argtypes = [ctypes.c_int, ctypes.c_int] + [ctypes.c_void_p] * 5
    return lib


def bf16_value(bits: np.ndarray) -> np.ndarray:
    """float64 value of bf16 bit patterns from the format's definition."""
    bits = np.asarray(bits, np.int64)
    sign = np.where(bits >> 15, -1.0, 1.0)
    e = (bits >> 7) & 0xFF
    m = (bits & 0x7F).astype(np.float64)
    val = np.where(e == 0, np.ldexp(m, -133), np.ldexp(128.0 + m, e - 134))
    return sign * val


def f16_value(bits: np.ndarray) -> np.ndarray:
    """float64 value of IEEE binary16 bit patterns from the format's definition."""
    bits = np.asarray(bits, np.int64)
    sign = np.where(bits >> 15, -1.0, 1.0)
    e = (bits >> 10) & 0x1F
    m = (bits & 0x3FF).astype(np.float64)
    val = np.where(e == 0, np.ldexp(m, -24), np.ldexp(1024.0 + m, e - 25))
    return sign * val


def a_matrix(slot: int, words: np.ndarray, f16: bool = False):
    """Expected A register bits [32][4] and the exact A values [16][16] of one
    case from its code words [32][2] (row gID of lane 4 gID + tq from word
    0, row gID + 8 from word 1; bytes 0, 2 -> k 2tq, 2tq + 1; bytes 1, 3 ->
    k 2tq + 8, 2tq + 9)."""
    P = SLOT_BIT[slot]
    regs = np.zeros((32, 4), np.uint32)
    A = np.zeros((16, 16))
    for lane in range(32):
        gid, tq = lane >> 2, lane & 3
        for wi, row in ((0, gid), (1, gid + 8)):
            w = int(words[lane, wi])
            byts = [(w >> (8 * i)) & 0xFF for i in range(4)]
            codes = [(bb >> (2 * slot)) & 3 for bb in byts]
            pat = [c << P for c in codes]
            regs[lane, wi] = pat[0] | (pat[2] << 16)          # a0 (row gID) / a1 (row gID + 8)
            regs[lane, 2 + wi] = pat[1] | (pat[3] << 16)      # a2 / a3
            for (k, bi) in ((2 * tq, 0), (2 * tq + 1, 2), (2 * tq + 8, 1), (2 * tq + 9, 3)):
                v = (f16_value if f16 else bf16_value)(np.array([pat[bi]]))[0]
                assert v == codes[bi] * 2.0 ** (P - (24 if f16 else 133))  # subnormal / first-binade reading
                A[row, k] = v
    return regs, A


def b_matrix(rng, expo: int, short: bool, f16: bool = False) -> np.ndarray:
    """bf16 or fp16 bits [16][8] around 2^expo: short mantissas (4
    significant bits, one exponent) or full mantissas with mixed magnitudes
    (fp16: the smallest reach the subnormals, as the low parts of small q'
    elements do)."""
    if short:
        m = rng.integers(8, 16, size=(16, 8)).astype(np.float64)      # 4-bit significands
        vals = m * 2.0 ** (expo - 3) * rng.choice([-1.0, 1.0], size=(16, 8))
    else:
        offs = [0, -1, -2, -11, -20] if f16 else [0, -1, -2, -9, -20]
        off = rng.choice(offs, p=[0.4, 0.2, 0.2, 0.15, 0.05], size=(16, 8))
        vals = rng.uniform(1.0, 2.0, size=(16, 8)) * 2.0 ** (expo + off) * rng.choice([-1.0, 1.0], size=(16, 8))
    if f16:
        return vals.astype(np.float16).view(np.uint16)                   # round to nearest fp16
    f = vals.astype(np.float32)
    return (f.view(np.uint32) >> 16).astype(np.uint16)                   # truncate to bf16


def run_cases(probe, slots, words, bmats, f16=False):
    n = len(slots)
    sl = np.ascontiguousarray(slots, np.int32)
    wd = np.ascontiguousarray(words, np.uint32)
    bm = np.ascontiguousarray(bmats, np.uint16)
    regs = np.zeros((n, 32, 4), np.uint32)
    d = np.zeros((n, 16, 8), np.float32)
    rc = probe.run_tc_code_operands(n, int(f16), sl.ctypes.data, wd.ctypes.data, bm.ctypes.data, regs.ctypes.data,
                                    d.ctypes.data)
    assert rc == 0, rc
    return regs, d


@pytest.mark.parametrize("kind", ["bf16", "f16"])
@pytest.mark.parametrize("short", [True, False])
def test_code_operands_on_tensor_cores(probe, short, kind):
    f16 = kind == "f16"
    rng = np.random.default_rng(20260 + int(short) + 2 * int(f16))
    # bf16 B magnitudes 2^8 .. 2^125 (the smallest mixed-in parts sit 2^-20
    # below 2^expo, so every product stays a normal fp32 number, as in the
    # kernel); fp16 B magnitudes 2^-6 .. 2^15
    expos = list(range(-6, 16, 2)) if f16 else list(range(28, 125, 6))
    slots, words, bmats = [], [], []
    for slot in (range(4) if f16 else range(1, 4)):   # slot 0's bit 8 is an exponent bit in bf16
        for e in expos:
            for _ in range(3):
                slots.append(slot)
                words.append(rng.integers(0, 2 ** 32, size=(32, 2), dtype=np.uint64).astype(np.uint32))
                bmats.append(b_matrix(rng, e, short, f16))
    regs, d = run_cases(probe, slots, words, bmats, f16)
    worst = {}
    for c, slot in enumerate(slots):
        exp_regs, A = a_matrix(slot, words[c], f16)
        assert np.array_equal(regs[c], exp_regs), (c, slot)
        Bv = (f16_value if f16 else bf16_value)(bmats[c]).reshape(16, 8)
        terms = A[:, :, None] * Bv[None, :, :]                          # [16 rows][16 k][8 cols]
        exact = terms.sum(axis=1)
        mag = np.abs(terms).sum(axis=1)
        err = np.abs(d[c].astype(np.float64) - exact)
        P = SLOT_BIT[slot]
        if short:
            assert np.all(err == 0), (c, slot, float(err.max()))
        else:
            rel = np.where(mag > 0, err / np.where(mag > 0, mag, 1), 0.0)
            worst[P] = max(worst.get(P, 0.0), float(rel.max()))
            assert rel.max() <= 2.0 ** -RETAINED[P], (c, slot, expos[(c // 3) % len(expos)], float(rel.max()))
    print(kind, "worst error / sum|terms| per code bit position:", {p: f"{v:.2e}" for p, v in sorted(worst.items())})
