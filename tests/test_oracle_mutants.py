"""Plant plausible mistakes in copies of the oracle source (CPU only) and
check that the pins in oracle_checks.py catch every one of them."""
import os
import subprocess
import sys
import tempfile

import pytest

import oracle
import oracle_checks as C

SRC = os.path.join(os.path.dirname(oracle.__file__), "oscar_oracle.c")
TESTS = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(TESTS)

# (name, text to replace, replacement)
MUTANTS = [
    ("U transposed in R", "acc += U[(size_t)i * d + k] * H[(size_t)k * d + l];",
     "acc += U[(size_t)k * d + i] * H[(size_t)k * d + l];"),
    ("Hadamard sign uses OR", "(popcount_u((unsigned)(i & j)) & 1) ? -c : c",
     "(popcount_u((unsigned)(i | j)) & 1) ? -c : c"),
    ("Hadamard not normalised", "double c = 1.0 / sqrt((double)d);", "double c = 1.0;"),
    ("no bit reversal", "UH[(size_t)i * d + oracle_bitrev(j, nb)]", "UH[(size_t)i * d + j]"),
    ("scale divides by 4", "double sp = (hi - lo) / 3.0, zp = lo;", "double sp = (hi - lo) / 4.0, zp = lo;"),
    ("zero is the maximum", "double sp = (hi - lo) / 3.0, zp = lo;", "double sp = (hi - lo) / 3.0, zp = hi;"),
    ("codes from pre-rounding scale/zero", "uj = (yc - z) / s;", "uj = (yc - zp) / sp;"),
    ("round half away from zero", "double r = nearbyint(uj);", "double r = round(uj);"),
    ("clip ignored", "double t = clip * amax;", "double t = amax;"),
    ("pack order reversed", "return (uint8_t)((c[0] & 3u) | ((c[1] & 3u) << 2) | ((c[2] & 3u) << 4) | ((c[3] & 3u) << 6));",
     "return (uint8_t)((c[3] & 3u) | ((c[2] & 3u) << 2) | ((c[1] & 3u) << 4) | ((c[0] & 3u) << 6));"),
    ("consecutive positions share a byte", "for (int i = 0; i < 4; ++i) four[i] = codes[j + i * nbytes];",
     "for (int i = 0; i < 4; ++i) four[i] = codes[4 * j + i];"),
    ("V stored token-major", "else block[codes_bytes + (size_t)j * P + slot] = byte;",
     "else block[codes_bytes + (size_t)slot * nbytes + j] = byte;"),
    ("V scale/zero written over K's", "    uint8_t* sz = block + 2 * codes_bytes + (size_t)which * sz_bytes;",
     "    uint8_t* sz = block + 2 * codes_bytes;"),
    ("f16 subnormal scale off by one", "double m = nearbyint(ldexp(a, 24));", "double m = nearbyint(ldexp(a, 23));"),
    ("f16 mantissa truncated", "double m = nearbyint((ldexp(a, -E) - 1.0) * 1024.0);",
     "double m = floor((ldexp(a, -E) - 1.0) * 1024.0);"),
    ("history mapped back by R instead of R^T",
     "for (int j = 0; j < d; ++j) acc += yh[j] * RK[(size_t)a * d + j];",
     "for (int j = 0; j < d; ++j) acc += yh[j] * RK[(size_t)j * d + a];"),
    ("GQA mapping interleaved", "int h = kv * G + hh;", "int h = hh * Hk + kv;"),
    ("softmax scale dropped", "logit[t] = sm_scale * acc;", "logit[t] = acc;"),
    ("page index from slot", "int page = page_table[(size_t)b * max_pages + pos / P];\n            const uint8_t* block = pool + ((size_t)page * Hk + kv) * bb;\n            double* kr",
     "int page = page_table[(size_t)b * max_pages + pos % P];\n            const uint8_t* block = pool + ((size_t)page * Hk + kv) * bb;\n            double* kr"),
    ("segment merge ignores BF16 weight", "double w_bf = (l_bf > 0.0) ? exp(m_bf - M) : 0.0;",
     "double w_bf = (l_bf > 0.0) ? 1.0 : 0.0;"),
    ("Fisher-Yates off by one", "long j = (long)(r % (uint64_t)(i + 1));", "long j = (long)(r % (uint64_t)(i));"),
    ("SplitMix64 shift", "z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;", "z = (z ^ (z >> 31)) * 0xBF58476D1CE4E5B9ull;"),
    ("shared pages not aliased", "page_table[(size_t)b * max_pages + p] = page_table[(size_t)first * max_pages + p];",
     "page_table[(size_t)b * max_pages + p] = (int32_t)(next++);"),
]


@pytest.fixture(scope="module")
def src_text():
    with open(SRC) as f:
        return f.read()


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(src_text, name, old, new):
    assert src_text.count(old) == 1, f"mutation site not unique: {name}"
    with tempfile.TemporaryDirectory() as tmp:
        path = os.path.join(tmp, "mutant.c")
        with open(path, "w") as f:
            f.write(src_text.replace(old, new))
        so = os.path.join(tmp, "libmutant.so")
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", path,
                        "-o", so, "-lm"], check=True)
        # run the pins in a child process: a mutant may also crash, which
        # counts as caught
        code = ("import sys; sys.path[:0] = %r; import oracle, oracle_checks as C\n"
                "o = oracle.Oracle(%r)\n"
                "for ch in C.ALL_CHECKS:\n"
                "    try:\n"
                "        ch(o)\n"
                "    except Exception:\n"
                "        print('CAUGHT', ch.__name__); sys.exit(3)\n"
                "print('MISSED')\n") % ([TESTS, ROOT], so)
        r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
        assert "MISSED" not in r.stdout and r.returncode != 0, f"no pin catches the mutant '{name}'"
