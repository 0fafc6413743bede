"""The oracle's pins must reject plausible mistakes.

Each case plants one mistake in a temporary copy of the oracle's C source (on
the CPU; the oracle in the repository is untouched), compiles it, and runs the
pin suite against it: at least one pin must fail.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "ragged_oracle.c")

MUTANTS = [
    ("rotation sign", "y[i1] = t2 + t3;", "y[i1] = t2 - t3;"),
    ("fp64 rotation sign", "y[i1] = x1 * c + x0 * s;", "y[i1] = x1 * c - x0 * s;"),
    ("GQA head map", "int32_t c = h / g;", "int32_t c = h % J->Hkv;"),
    ("slot offset", "int32_t off = (int32_t)(p % bs);", "int32_t off = (int32_t)((p + 1) % bs);"),
    ("bf16 rounding", "u += 0x7fffu + lsb;", "u += 0x8000u;"),
    ("token position", "tok_pos[cu_seqlens[i] + j] = seen[i] + j;", "tok_pos[cu_seqlens[i] + j] = j;"),
    ("drops the diagonal", "double w = exp(z[u] - zmax);", "double w = exp(z[u] - zmax) * (u < p ? 1.0 : 0.0);"),
    ("frequency exponent", "float fk = (float)pow((double)theta, -2.0 * (double)k / (double)d);",
     "float fk = (float)pow((double)theta, -1.0 * (double)k / (double)d);"),
    ("fp64 frequency index", "double fk = pow(theta, -2.0 * (double)k / (double)d);",
     "double fk = pow(theta, -2.0 * (double)(k + 1) / (double)d);"),
    ("pairing", "        *i1 = k + d / 2;", "        *i1 = d - 1 - k;"),
    ("value from key", "pool[pool_index(blk, 1, h, off, e, Hkv, bs, d)] = v[e];",
     "pool[pool_index(blk, 1, h, off, e, Hkv, bs, d)] = k[e];"),
    ("value column", "const uint16_t* v = row + (int64_t)(Hq + Hkv + h) * d;",
     "const uint16_t* v = row + (int64_t)(Hq + h) * d;"),
    ("fp16 decode exponent", "v = ldexp((double)(1024 + m), e - 25);", "v = ldexp((double)(1024 + m), e - 24);"),
    ("softmax scale", "scale > 0.0f ? (double)scale : 1.0 / sqrt((double)d)", "scale > 0.0f ? (double)scale : 1.0 / (double)d"),
    ("block offsets", "blk_off[i + 1] = blk_off[i] + (int32_t)nb;", "blk_off[i + 1] = blk_off[i] + (int32_t)nb + 1;"),
]


@pytest.mark.parametrize("label,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_reject_mutant(tmp_path, label, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, label
    mut = tmp_path / "mutant.c"
    mut.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
                           str(mut), "-o", str(lib), "-lm"])
    env = dict(os.environ, RAGGED_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, "pins accepted the mutant '%s'" % label
