"""The quantizers' division scheme equals IEEE x / S on every BF16 input pair.

Compiles tests/division_domain_check.c (plain C, -ffp-contract=off) and runs
it over all ~1.07e9 (x, amax) pairs; see that file for the scheme.
"""
import os
import subprocess
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))


def test_division_scheme_matches_ieee_over_all_bf16_pairs():
    src = os.path.join(HERE, "division_domain_check.c")
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "check")
        subprocess.run(["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-pthread", src, "-o", exe, "-lm"],
                       check=True)
        r = subprocess.run([exe], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "mismatches=0" in r.stdout
