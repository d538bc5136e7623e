"""GPU checks of the arithmetic identities the codec kernels use in place of
IEEE divisions: the block scale absmax/qmax by reciprocal + one FMA correction
equals the IEEE quotient for every non-negative float (both bit widths,
exhaustive), and the quantizer's FMA-division codes equal rint of the IEEE
quotient on 2^33 seeded draws of 8 values per bit width, most of them within
3 ulps of a rounding boundary; the Adam bias-correction reciprocal and FMA
division equal the IEEE ones (exhaustive over the divisors, 2^32 seeded
dividend pairs); and the one-FMA int4 dequantize-and-add, a subnormal code
times the scale scaled by 2^133, equals the product and sum rounded one after
the other for every code and every scale below 2^-5 (exhaustive), for int4
and for int8."""
import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
pytestmark = pytest.mark.gpu


def test_exhaustive_device_identities(tmp_path):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    exe = tmp_path / "device_checks"
    subprocess.check_call([
        "nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-fmad=false",
        "-I", os.path.join(ROOT, "gradient_comm_codecs_gb300", "csrc"),
        os.path.join(ROOT, "tests", "device_checks.cu"), "-o", str(exe)])
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stdout + out.stderr
    res = {line.split()[0]: int(line.split()[1]) for line in out.stdout.splitlines()}
    assert res == {"div_qmax7": 0, "div_qmax127": 0, "quantize_q7": 0, "quantize_q127": 0,
                   "bias_rcp": 0, "bias_div": 0, "i4_fma": 0, "i8_fma": 0}, out.stdout
