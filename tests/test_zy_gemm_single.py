"""The single-CTA GEMM kernel on the shapes the CTA-pair kernel takes by
default (output width a multiple of 256), against the oracle: NVQ_GEMM_PAIR=0
routes every GEMM to the single-CTA kernel, so the GEMM tests run again here in
a child process with the variable set ("Add an NVFP4 quantization converter":
NVFP4 GEMM; "Hybrid quantization": MXFP8 GEMM)."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_single_cta_kernel_parity():
    env = dict(os.environ, NVQ_GEMM_PAIR="0")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", os.path.join(ROOT, "tests", "test_gpu_gemm.py"),
                        os.path.join(ROOT, "tests", "test_gpu_grouped.py")],
                       env=env, capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
