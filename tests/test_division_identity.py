"""The key encoder's division-free quotient gives the same codes as IEEE division.

The kernel replaces x/scale by Markstein's correction step (see
tests/helpers/markstein_check.c); this CPU test checks the claim on generated
bf16 groups of every magnitude class, and the same for the per-group scale and
zero point computed without a division.  CPU only.
"""
import os
import subprocess

from conftest import ROOT


def test_markstein_quotient_matches_ieee_codes(tmp_path):
    exe = tmp_path / "markstein_check"
    src = os.path.join(ROOT, "tests", "helpers", "markstein_check.c")
    subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-o", str(exe), src, "-lm"], check=True)
    out = subprocess.run([str(exe), "300000"], check=True, capture_output=True, text=True).stdout.split()
    elems, bad, groups, pbad = (int(v) for v in out)
    assert elems > 10_000_000 and bad == 0
    assert groups > 400_000 and pbad == 0
