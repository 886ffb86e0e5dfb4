"""The oracle's pins have power: each test below compiles a copy of the oracle
with one plausible mistake written into it (a dropped rounding, a wrong tie
rule, an operation order the readings do not take) and checks that the CPU
pin suite FAILS against that copy.  The copies live in a temporary folder;
the oracle itself is not changed.  The unmutated oracle passes the same
suite (the rest of tests/).

Each mistake is a textual replacement in qta_oracle.c that must match
exactly once, so a change to the oracle that moves the line makes the test
fail loudly instead of testing nothing.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ORACLE = os.path.join(ROOT, "oracle")

# the fast CPU pins (the exhaustive 2^32-pattern E4M3 sweeps are left out)
PIN_FILES = ["tests/test_oracle_exact.py", "tests/test_oracle_codec.py", "tests/test_oracle_transform.py",
             "tests/test_oracle_formats.py", "tests/test_oracle_ring.py", "tests/test_golden.py"]
PIN_FILTER = "not exhaustive_band and not every_pattern_outside"

_ASYM_FUSED_HELPER = """static float mut_fused_term(int scheme, const void* codes, const void* scales,
                            const void* zeros, int64_t e, float acc)
{
    float s = orc_f16_to_f32(((const uint16_t*)scales)[e / 128]);
    float z = orc_f16_to_f32(((const uint16_t*)zeros)[e / 128]);
    int q = scheme == ORC_INT8_ASYM ? ((const uint8_t*)codes)[e]
                                    : (((const uint8_t*)codes)[e >> 1] >> ((e & 1) * 4)) & 15;
    return fmaf((float)q, s, acc + z);
}

static void reduce_sums("""

MUTANTS = {
    # EQuARX INT8: the stored scale a/127 rounded twice
    "int8_scale_two_roundings": [("float s = a / 127.0f;", "float s = a * (1.0f / 127.0f);")],
    # EQuARX INT8 codes: ties away from zero instead of to even
    "int8_codes_ties_away": [("float q = rintf(load_elem(x, dtype, off + b * 64 + i) * inv);",
                              "float q = roundf(load_elem(x, dtype, off + b * 64 + i) * inv);")],
    # Flash asymmetric codes: ties away from zero instead of to even
    "asym_codes_ties_away": [("float q = rintf((load_elem(x, dtype, off + g * G + i) - z) * inv);",
                              "float q = roundf((load_elem(x, dtype, off + g * G + i) - z) * inv);")],
    # Flash asymmetric reduce: the zero-point added to the partial sum first,
    # then one fused multiply-add
    "asym_reduce_fused": [("acc = acc + dequant(scheme, B, codes[r], scales[r], z, st, e);",
                           "acc = mut_fused_term(scheme, codes[r], scales[r], z, e, acc);"),
                          ("static void reduce_sums(", _ASYM_FUSED_HELPER)],
    # TACO / INT8 reduce: the product rounded before the add (two roundings)
    "sym_reduce_two_roundings": [("acc = fmaf(code, sc, acc);", "acc = acc + code * sc;")],
    # round-to-nearest with ties away from zero in the E4M3 / fp16 encoders
    "rne_ties_away": [("if (rem > half || (rem == half && (q & 1u))) q += 1u;", "if (rem >= half) q += 1u;")],
    # the butterfly with descending strides (same matrix, other roundings)
    "fwht_descending": [("for (int h = 1; h < B; h <<= 1)", "for (int h = B / 2; h >= 1; h >>= 1)")],
    # the per-tensor factor 1/(448 S) formed as (1/448)/S
    "taco_tinv_two_roundings": [("float tinv = 1.0f / (448.0f * S);", "float tinv = (1.0f / 448.0f) / S;")],
    # no 2^-9 floor for a non-zero block whose scale byte rounds to zero
    "taco_no_scale_floor": [("if (r == 0 && a > 0.0f) r = 0x01;", "(void)0;")],
}


def _build_mutant(tmp_path, edits):
    with open(os.path.join(ORACLE, "qta_oracle.c")) as f:
        src = f.read()
    for old, new in edits:
        assert src.count(old) == 1, f"mutation site not found exactly once: {old!r}"
        src = src.replace(old, new)
    d = tmp_path / "mut"
    d.mkdir()
    (d / "qta_oracle.c").write_text(src)
    with open(os.path.join(ORACLE, "qta_oracle.h")) as f:
        (d / "qta_oracle.h").write_text(f.read())
    so = d / "liboracle_mut.so"
    subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fexcess-precision=standard",
                    "-fPIC", "-shared", "-o", str(so), str(d / "qta_oracle.c"), "-lm"], check=True)
    return str(so)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(tmp_path, name):
    so = _build_mutant(tmp_path, MUTANTS[name])
    env = dict(os.environ, QTA_ORACLE_LIB=so)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", "-m", "not gpu",
                        "-k", PIN_FILTER, *PIN_FILES], cwd=ROOT, env=env, capture_output=True, text=True)
    tail = "\n".join((r.stdout + r.stderr).splitlines()[-6:])
    assert r.returncode == 1, f"the pins did not catch mutant {name} (rc {r.returncode}):\n{tail}"
