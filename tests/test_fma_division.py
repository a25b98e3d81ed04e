"""The CUDA block quantizer replaces its 16 correctly rounded divisions by the
block scale with one reciprocal and an FMA correction per element. This CPU
test compiles a small C program (fma_division_check.c, beside this file) that
checks the identity bit for bit against IEEE division for every non-zero E4M3
scale and every f32 mantissa (about 10^9 quotients, a few seconds)."""
import os
import shutil
import subprocess
import tempfile

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def test_fma_corrected_quotient_is_correctly_rounded():
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "fma_division_check")
        subprocess.run([cc, "-O2", "-ffp-contract=off", os.path.join(HERE, "fma_division_check.c"), "-o", exe,
                        "-lm"], check=True)
        r = subprocess.run([exe], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert " 0 mismatches" in r.stdout
