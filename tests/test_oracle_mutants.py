"""The oracle's pins catch plausible mistakes (no GPU).

Each case plants one mistake in a copy of oracle.c (a dropped term, a wrong
sign, index or constant, a transposed operand, a wrong rounding rule), builds
it into a separate library, and runs the pin tests against that library in a
subprocess: they must fail. The real oracle is never modified.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTANTS = [
    ("m uses 1-b2", "(1.0 - b1) * gi", "(1.0 - b2) * gi", "test_oracle_adamw.py"),
    ("no m bias correction", "double mhat = mi / bc1", "double mhat = mi", "test_oracle_adamw.py"),
    ("bc2 index t-1", "pow(b2, (double)hp->step)", "pow(b2, (double)(hp->step - 1))", "test_oracle_adamw.py"),
    ("eps inside sqrt", "(sqrt(vhat) + eps)", "sqrt(vhat + eps)", "test_oracle_adamw.py"),
    ("decay sign", "(1.0 - lr * wd)", "(1.0 + lr * wd)", "test_oracle_adamw.py"),
    ("v uses g not g^2", "(1.0 - b2) * gi * gi", "(1.0 - b2) * gi", "test_oracle_adamw.py"),
    ("reduce drops rank 1", "for (int32_t r = 1; r < n_ranks; ++r)", "for (int32_t r = 2; r < n_ranks; ++r)",
     "test_oracle_reduce.py"),
    ("reduce reversed order", "float acc = ora_widen16(ranks[0][i], dtype);\n    for (int32_t r = 1; r < n_ranks; ++r) acc = acc + ora_widen16(ranks[r][i], dtype);",
     "float acc = ora_widen16(ranks[n_ranks - 1][i], dtype);\n    for (int32_t r = n_ranks - 2; r >= 0; --r) acc = acc + ora_widen16(ranks[r][i], dtype);",
     "test_oracle_reduce.py"),
    ("reduce seeded with +0", "float acc = ora_widen16(ranks[0][i], dtype);\n    for (int32_t r = 1;",
     "float acc = 0.0f;\n    for (int32_t r = 0;", "test_oracle_reduce.py"),
    ("bf16 ties away from zero", "drop > 0x8000u || (drop == 0x8000u && (keep & 1u))", "drop >= 0x8000u",
     "test_oracle_cast.py"),
    ("fp16 subnormal spacing", "q = ldexp(1.0, -24);", "q = ldexp(1.0, -23);", "test_oracle_cast.py"),
    ("fp16 widen exponent bias", "e - 25);", "e - 24);", "test_oracle_cast.py"),
    ("ceil shard rule", "bounds[k] = (int64_t)(((__int128)k * (__int128)P) / (__int128)n_ranks);",
     "bounds[k] = (int64_t)(((__int128)k * (__int128)P + n_ranks - 1) / (__int128)n_ranks);",
     "test_oracle_layout.py"),
    ("segment offset", "out[c].shard_offset = a - lo;", "out[c].shard_offset = a - offsets[t];",
     "test_oracle_layout.py"),
    ("adam bytes 4P", "out->fp32_adam = 8 * p;", "out->fp32_adam = 4 * p;", "test_oracle_accounting.py"),
    ("unshard at next bound", "(char*)flat + bounds[k] * elem_size", "(char*)flat + (bounds[k + 1] - len) * elem_size + (k ? 1 : 0) * elem_size",
     "test_oracle_unshard_clip.py"),
    ("clip coefficient uncapped", "return (float)(c < 1.0 ? c : 1.0);", "return (float)c;", "test_oracle_unshard_clip.py"),
]


@pytest.mark.slow
@pytest.mark.parametrize("name,old,new,testfile", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new, testfile):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site not unique for {name!r}"
    mutant = tmp_path / "oracle.c"
    mutant.write_text(src.replace(old, new))
    (tmp_path / "oracle.h").write_text(open(os.path.join(ROOT, "oracle", "oracle.h")).read())
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-fopenmp", "-std=c11", str(mutant),
                    "-o", str(so), "-lm"], check=True, capture_output=True)
    env = dict(os.environ, ORACLE_SO=str(so))
    args = [sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
            os.path.join(ROOT, "tests", testfile), "-k", "not exhaustive"]
    p = subprocess.run(args, env=env, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert p.returncode != 0, f"pins did not catch mutant {name!r}:\n{p.stdout[-2000:]}"
