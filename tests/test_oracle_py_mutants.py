"""Plant plausible mistakes in copies of the numpy oracles of the variants
(oracle/lloyd.py, oracle/kitty.py) and check that their pins catch each one
(CPU only: the mutated copy is loaded as a module and the pin functions run
against it)."""
import os
import types

import pytest

import oracle
import test_oracle_calibrate as PC
import test_oracle_kitty as PK
import test_oracle_lloyd as PL

ORACLE_DIR = os.path.dirname(oracle.__file__)

LLOYD = [
    ("inner levels not symmetric", "return np.array([0.0, a, 3.0 - a, 3.0])", "return np.array([0.0, a, 2.0 * a, 3.0])"),
    ("middle threshold at 1", "(u >= 1.5).astype(np.uint8)", "(u >= 1.0).astype(np.uint8)"),
    ("Lloyd cell starts at a", "cell = v[v >= a / 2]", "cell = v[v >= a]"),
    ("no folding", "v = np.minimum(np.asarray(u, np.float64).ravel(), 3.0 - np.asarray(u, np.float64).ravel())",
     "v = np.asarray(u, np.float64).ravel()"),
    ("dequantised with the codes", "    lv = levels(a)[codes]\n", "    lv = codes.astype(np.float64)\n"),
    ("history mapped back by R", "@ R[kv][w].T", "@ R[kv][w]"),
    ("scale and zero swapped", "return codes, _f16(sz[0::2]), _f16(sz[1::2])", "return codes, _f16(sz[1::2]), _f16(sz[0::2])"),
]

KITTY = [
    ("step s/4", "(q4 / 5.0)", "(q4 / 4.0)"),
    ("smallest errors chosen", "key=lambda j: (-err[j], j)", "key=lambda j: (err[j], j)"),
    ("q4 field shifted", "return ent & 0x7F, (ent >> 8) & 0xF", "return ent & 0x7F, (ent >> 7) & 0xF"),
    ("K mapped back by R", "@ RK.T", "@ RK"),
    ("4-bit code truncated", "np.rint(5.0 *", "np.floor(5.0 *"),
    ("group 0's scale everywhere", "z[grp[pos]] + s[grp[pos]]", "z[grp[pos]] + s[0]"),
    ("code copy missing", "(np.asarray(codes, np.int64)[pos] << 12)", "0"),
]


CALIBRATE = [
    ("eigenvalues ascending", "order = np.argsort(-w, kind=\"stable\")", "order = np.argsort(w, kind=\"stable\")"),
    ("no sign convention", "        if u[i, j] < 0:\n            u[:, j] = -u[:, j]", "        if u[i, j] < -1e300:\n            u[:, j] = -u[:, j]"),
    ("sum instead of mean", "out[kv] = s.T @ s / (n * g)", "out[kv] = s.T @ s"),
    ("query heads interleaved over KV heads", "x = np.asarray(q, np.float64).reshape(n, num_kv_heads, g, d)",
     "x = np.asarray(q, np.float64).reshape(n, g, num_kv_heads, d).transpose(0, 2, 1, 3)"),
    ("softmax scale dropped", "logits = (q64[:, h, :] @ k64[:, kv, :].T) * sm_scale", "logits = (q64[:, h, :] @ k64[:, kv, :].T)"),
    ("weights not normalised", "        p /= p.sum(axis=1, keepdims=True)\n", ""),
    ("V covariance from the queries", "cv = value_covariance(attention_outputs(q, kv[:, :, 0, :], kv[:, :, 1, :], sm_scale), hk)",
     "cv = value_covariance(q, hk)"),
    ("clip error against the clipped value", "err += float(((y - orc.dequantize_vec(codes, s16, z16, group)) ** 2).sum())",
     "err += float(((np.clip(y, -0.0, 0.0) - orc.dequantize_vec(codes, s16, z16, group)) ** 2).sum())"),
]


def _load(name: str, text: str) -> types.ModuleType:
    mod = types.ModuleType(f"oracle.{name}_mutant")
    mod.__file__ = os.path.join(ORACLE_DIR, f"{name}.py")
    exec(compile(text, mod.__file__, "exec"), mod.__dict__)
    return mod


def _pins_fail(pins, attr: str, mutant) -> bool:
    original = getattr(pins, attr)
    setattr(pins, attr, mutant)
    try:
        for fn in [getattr(pins, n) for n in dir(pins) if n.startswith("test_")]:
            try:
                fn()
            except Exception:
                return True
        return False
    finally:
        setattr(pins, attr, original)


@pytest.mark.parametrize("module,pins,attr,mutants", [("lloyd", PL, "L", LLOYD), ("kitty", PK, "K", KITTY),
                                                       ("calibrate", PC, "C", CALIBRATE)],
                         ids=["lloyd", "kitty", "calibrate"])
def test_planted_mistakes_fail_a_pin(module, pins, attr, mutants):
    with open(os.path.join(ORACLE_DIR, f"{module}.py")) as f:
        src = f.read()
    assert not _pins_fail(pins, attr, _load(module, src)), "the unmodified oracle must pass its pins"
    missed = []
    for name, old, new in mutants:
        assert src.count(old) == 1, name
        if not _pins_fail(pins, attr, _load(module, src.replace(old, new))):
            missed.append(name)
    assert not missed, missed
