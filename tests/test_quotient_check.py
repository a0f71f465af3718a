"""The tile quantiser's division-free arithmetic against the oracle's IEEE
quotient (CPU only).

The TMA-staged quantisation kernel forms s = amax/448 from a correction step
on a/7 and x/s from an approximate reciprocal plus one correction step (see
quotient_check.c).  These tests compile that arithmetic in C, with explicit
fused multiply-adds and no contraction, and compare every e4m3 code and every
scale with the oracle (RNE_e4m3(clamp(fl32(x/s), +-448)), s = fl32(amax/448)):
a strided subset of the bf16 amax values by default, all of them (about 1.07e9
(amax, x, sign) cases, each with four reciprocal candidates) in the slow test.
"""
import os
import subprocess

import pytest

import oracle as O

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


@pytest.fixture(scope="module")
def checker(tmp_path_factory):
    exe = str(tmp_path_factory.mktemp("qc") / "quotient_check")
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           os.path.join(HERE, "quotient_check.c"), os.path.join(ROOT, "oracle", "bfp8_oracle.c"),
           "-lm", "-o", exe]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return exe


def _run(exe, stride):
    out = subprocess.run([exe, str(stride)], check=True, capture_output=True, text=True).stdout
    fields = dict(kv.split("=") for kv in out.split())
    return int(fields["tot"]), int(fields["bad"]), int(fields["scale_bad"])


def test_quotient_and_scale_strided(checker):
    tot, bad, scale_bad = _run(checker, 97)
    assert tot > 5_000_000
    assert bad == 0 and scale_bad == 0


@pytest.mark.slow
def test_quotient_and_scale_exhaustive(checker):
    tot, bad, scale_bad = _run(checker, 1)
    assert tot == 1_065_402_240
    assert bad == 0 and scale_bad == 0
