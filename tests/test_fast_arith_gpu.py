"""Bit-exactness of the fast paths' arithmetic against CUDA's own IEEE
operations: the reciprocal-plus-one-remainder-correction quotient equals
__fdiv_rn for every bf16 operand pair (and for float32 scales RN(a/qmax) of
every bf16 abs-max, and 2^30 random float32 pairs) inside its domain when
|x| and |x/s| are at least 2^-100, the rounded integer codes agree for every
pair, the 1.5*2^23 rounding trick equals rintf for every float of magnitude
< 2^21, and a group range divided by any integer 1..255 this way equals
__fdiv_rn for every float in [2^-100, 2^127]."""
import os
import subprocess

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_fast_quotient_and_rounding_are_exact(tmp_path):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kv_cache_quantization_kvq_gb300 import builder
    exe = str(tmp_path / "quot_check")
    subprocess.run([builder._nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-fmad=false",
                    "-I", builder.INCLUDE, "-I", builder.CSRC, os.path.join(ROOT, "tests", "cuda", "quot_check.cu"),
                    "-o", exe], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=600)
    print(r.stdout)
    assert r.returncode == 0, r.stdout + r.stderr
