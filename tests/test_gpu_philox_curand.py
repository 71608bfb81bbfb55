"""The oracle's Philox4x32-10 against cuRAND's device implementation of the
same generator (a library routine written by others), evaluated on the GPU by
a test-only probe kernel on random counters and keys: every output word must
agree.  Stochastic rounding draws its bits from this generator ("Add an NVFP4
quantization converter", "What changed": a Philox key per rank)."""
import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


def test_oracle_philox_equals_curand(tmp_path):
    so = str(tmp_path / "libphilox_probe.so")
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-shared", "-Xcompiler", "-fPIC",
                    os.path.join(HERE, "probes", "curand_philox_probe.cu"), "-o", so], check=True,
                   capture_output=True, text=True, timeout=600)
    lib = ctypes.CDLL(so)
    lib.philox_probe.restype = ctypes.c_int
    lib.philox_probe.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
    rng = np.random.default_rng(11)
    n = 4096
    ctr = rng.integers(0, 1 << 32, (n, 4), dtype=np.uint64).astype(np.uint32)
    key = rng.integers(0, 1 << 32, (n, 2), dtype=np.uint64).astype(np.uint32)
    ctr[0], key[0] = 0, 0
    ctr[1], key[1] = 0xFFFFFFFF, 0xFFFFFFFF
    # the stochastic-rounding counter layout: (block lo, block hi, direction, offset), key = seed words
    ctr[2] = (123456, 0, 1, 0)
    key[2] = (1234, 0)
    dc = torch.from_numpy(ctr.view(np.int32)).cuda()
    dk = torch.from_numpy(key.view(np.int32)).cuda()
    do = torch.zeros(n * 4, dtype=torch.int32, device="cuda")
    assert lib.philox_probe(dc.data_ptr(), dk.data_ptr(), do.data_ptr(), n) == 0
    got = do.cpu().numpy().view(np.uint32).reshape(n, 4)
    want = np.stack([oracle.philox4x32_10(ctr[i], key[i]) for i in range(n)])
    assert np.array_equal(got, want)
