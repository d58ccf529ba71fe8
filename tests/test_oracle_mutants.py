"""The oracle's pins are sensitive: each plausible mistake planted in a copy of the oracle makes
the pin suite fail (CPU only).

Each mutant is the oracle source with one edit (a dropped term, a wrong sign, index or
comparison, a transposed operand), compiled to a temporary library; the pin tests run against it
in a subprocess (GQ_ORACLE_LIB) and must fail.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "gq_oracle.c")

# (name, text in the oracle, replacement)
MUTANTS = [
    ("round-up compare <=", "k = lo + (r < T ? 1 : 0);", "k = lo + (r <= T ? 1 : 0);"),
    ("round-up compare inverted", "k = lo + (r < T ? 1 : 0);", "k = lo + (r >= T ? 1 : 0);"),
    ("worker dropped from counter", "ctr[1] = (uint32_t)i;", "ctr[1] = 0u;"),
    ("step dropped from counter", "ctr[2] = (uint32_t)step;", "ctr[2] = 0u;"),
    ("wrong half of the call", "int h = (int)(j & 7);", "int h = (int)((j + 1) & 7);"),
    ("halves of r swapped", "return (half16(a, h) << 16) | half16(b, h);",
     "return (half16(b, h) << 16) | half16(a, h);"),
    ("second counter space dropped", "ctr[0] |= 0x80000000u;", "ctr[0] |= 0u;"),
    ("philox key bump dropped", "k1 += weyl1;", "k1 += 0u;"),
    ("philox halves swapped", "uint32_t n1 = lo1;", "uint32_t n1 = hi1;"),
    ("E level off by one", "*lo = s + e; /* 2^e = 2^-(s - lo) */", "*lo = s + e + 1;"),
    ("E first interval scale", "f = (double)v / smallest;", "f = (double)v / (2.0 * smallest);"),
    ("L fraction dropped", "f = t - m; /* exact */", "f = 0.0;"),
    ("sign dropped", "codes[i * w + j] = (int8_t)(xv < 0.0f ? -k : k);",
     "codes[i * w + j] = (int8_t)k;"),
    ("window keyed by its local column", "r = gqo_philox_word(seed, step, i, j0 + j);",
     "r = gqo_philox_word(seed, step, i, j);"),
    ("E decode 2^k", "int64_t units = (int64_t)1 << (k - 1);", "int64_t units = (int64_t)1 << k;"),
    ("mean not divided by n", "out[j] = ldexp(num, -(s - 1)) / (double)n;",
     "out[j] = ldexp(num, -(s - 1));"),
    ("L scale drops s", "out[j] = num / ((double)n * (double)s);", "out[j] = num / (double)n;"),
    ("norm transposed", "double v = (double)load_x(x, dtype, i * d + j);",
     "double v = (double)load_x(x, dtype, (i * d + j) % n * d + (i * d + j) / n);"),
    ("q=2 inner sqrt dropped", "        if (q == 2)\n            inner = sqrt(inner);", ""),
    ("bf16 widened wrong", "<< 16;", "<< 8;"),
    ("re-round probability over the wrong gap", "*T = (uint32_t)(frac << (32 - e));",
     "*T = (uint32_t)(frac << (31 - e));"),
    ("re-round level off by one", "    *lo = e + 1;\n", "    *lo = e;\n"),
    ("re-round drops the sign", "    return t < 0 ? -k : k;\n}", "    return k;\n}"),
    ("tree stream ignores the level", "return (int64_t)0x80000000LL + ((int64_t)l << 24) + m;",
     "return (int64_t)0x80000000LL + m;"),
    ("p=2 outer sum of norms, not squares", "outer += inner * inner;", "outer += inner;"),
    ("q=inf signed maximum", "else if (fabs(v) > inner)\n                inner = fabs(v);",
     "else if (v > inner)\n                inner = v;"),
    ("NaN not propagated", "if (has_nan)\n        return NAN;", "if (0)\n        return NAN;"),
    ("final square root dropped", "return p == 2 ? sqrt(outer) : outer;", "return outer;"),
    ("ring starts at worker c", "int code = codes[((c + 1) % n) * w + j];",
     "int code = codes[(c % n) * w + j];"),
    ("16-bit mode: a tie rounds up", "lvl = lo + (int32_t)((word >> 16) < F);",
     "lvl = lo + (int32_t)((word >> 16) <= F);"),
    ("16-bit mode: low half of the word", "lvl = lo + (int32_t)((word >> 16) < F);",
     "lvl = lo + (int32_t)((word & 0xFFFFu) < F);"),
    ("16-bit mode: L truncates", "double p16 = round_half_odd((double)ax * (double)c1 * 65536.0);",
     "double p16 = floor((double)ax * (double)c1 * 65536.0);"),
    ("16-bit mode: E fraction from the low bits", "*F = (bits & 0x7FFFFFu) >> 7;",
     "*F = bits & 0xFFFFu;"),
    ("16-bit mode: no clamp at the top level",
     "        if (p16 > (double)s * 65536.0)\n            p16 = (double)s * 65536.0;\n", ""),
    ("16-bit mode: E level off by one", "*lo = s + (ex - 1);", "*lo = s + ex;"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, name
    mutant_c = tmp_path / "mutant.c"
    mutant_c.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-o",
                    str(so), str(mutant_c), "-lm"], check=True)
    env = dict(os.environ, GQ_ORACLE_LIB=str(so))
    pins = [os.path.join(ROOT, "tests", f) for f in
            ("test_oracle_philox.py", "test_oracle_norm.py", "test_oracle_quantize.py",
             "test_oracle_exp_allreduce.py", "test_oracle_u16.py")]
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        *pins], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, "pins did not catch mutant %r" % name
