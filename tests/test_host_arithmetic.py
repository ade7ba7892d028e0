"""Host checks of arithmetic identities the kernels rely on (no GPU)."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_nvfp4_reciprocal_encode_equals_ieee_quotient(tmp_path):
    """The NVFP4 quantizer encodes RN(x * r), r any fp32 within 1 ulp of
    1/D (the hardware reciprocal), unless the bracket RN(y (1 -+ 2^-20))
    straddles an E2M1 rounding boundary, where it uses RN(x / D); the
    codes must equal those of RN(x / D) for every bf16 x, and the block
    scale's E4M3 code the same way (and the check must be able to fail:
    without the fallback it finds mismatches)."""
    exe = tmp_path / "e2m1_check"
    subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-o", str(exe),
                    os.path.join(HERE, "host", "e2m1_reciprocal_check.c"), "-lm"], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
