"""The quantizers' replacements for IEEE division give the same E4M3 codes.

The blockwise quantizers encode the fp32 quotient x / s (s = amax / 448, the
"AIS: Adaptive Importance Sampling for Quantized RL" explainer, equation
Q(X)).  The CUDA kernels form s from amax * RN(1/448), and x / s from
x * RN(1/s), each with one FMA correction (Markstein's method; the latter
when s >= 2^-100, run on the negated quotient so that a zero keeps its
sign).  This test compiles a host restatement
of that formula and checks it against the IEEE quotient over every bf16 input
and every bf16 group maximum: the E4M3 codes must agree everywhere.
"""
import os
import shutil
import subprocess
import tempfile

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_fma_corrected_quotients_match_ieee_exhaustively():
    with tempfile.TemporaryDirectory() as tmp:
        exe = os.path.join(tmp, "division_check")
        subprocess.run(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-o", exe,
                        os.path.join(HERE, "division_check.c"), "-lm"], check=True)
        out = subprocess.run([exe], capture_output=True, text=True, timeout=900)
    fields = dict(zip(out.stdout.split()[0::2], map(int, out.stdout.split()[1::2])))
    assert out.returncode == 0, out.stdout
    assert fields["scale_diffs"] == 0
    assert fields["code_diffs"] == 0
    assert fields["pairs"] > 10**9  # every (x, group maximum) pair with s >= 2^-100


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_exact_quotient_of_full_significand_values():
    """The saved-FP8 re-quantization divides values with full fp32
    significands, where one correction is not always enough: two Markstein
    corrections on the negated quotient must give the IEEE quotient bit for
    bit (and its E4M3 code, signed zeros included) over 6.7e8 sampled pairs,
    among them the rare inputs that a single correction gets wrong."""
    with tempfile.TemporaryDirectory() as tmp:
        exe = os.path.join(tmp, "division_exact_check")
        subprocess.run(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-o", exe,
                        os.path.join(HERE, "division_exact_check.c"), "-lm"], check=True)
        out = subprocess.run([exe], capture_output=True, text=True, timeout=900)
    fields = dict(zip(out.stdout.split()[0::2], map(int, out.stdout.split()[1::2])))
    assert out.returncode == 0, out.stdout
    assert fields["quotient_diffs"] == 0
    assert fields["code_diffs"] == 0
    assert fields["checked"] > 6 * 10**8
    assert fields["single_correction_misses"] >= 1
