"""Pin of the oracle's Philox4x32-10 against the CUDA toolkit's own Philox4x32-10 (cuRAND device API).

cuRAND's Philox4x32-10 state for (seed, subsequence s, offset 0) starts at
counter (0, 0, s_lo, s_hi) with key (seed_lo, seed_hi); its first curand4()
call returns that counter's four output words.  The oracle computes the same
words from the round definition alone, so agreement pins the multipliers,
Weyl constants, round structure and word order to an outside implementation.
"""
import ctypes
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def helper():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    d = tempfile.mkdtemp(prefix="kvq_curand_")
    so = os.path.join(d, "curand_philox.so")
    subprocess.check_call([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-shared", "-Xcompiler", "-fPIC",
                           "-o", so, os.path.join(HERE, "cuda", "curand_philox.cu")])
    lib = ctypes.CDLL(so)
    lib.curand_philox_first4.restype = ctypes.c_int
    lib.curand_philox_first4.argtypes = [ctypes.c_uint64, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
    yield lib
    shutil.rmtree(d, ignore_errors=True)


@pytest.mark.parametrize("seed", [0, 1, 0x0123456789ABCDEF, 0xFFFFFFFFFFFFFFFF])
def test_oracle_philox_matches_curand(helper, seed):
    from oracle.philox import philox4x32_10

    subseq = np.array([0, 1, 2, 7, 1 << 31, (1 << 32) + 5, 0xDEADBEEFCAFEF00D], dtype=np.uint64)
    out = np.zeros(4 * subseq.size, dtype=np.uint32)
    assert helper.curand_philox_first4(seed, subseq.ctypes.data, subseq.size, out.ctypes.data) == 0
    ref = philox4x32_10((np.zeros_like(subseq), np.zeros_like(subseq), subseq & np.uint64(0xFFFFFFFF),
                         subseq >> np.uint64(32)), (seed & 0xFFFFFFFF, seed >> 32))
    ref = np.stack([r.astype(np.uint32) for r in ref], axis=1).reshape(-1)
    assert np.array_equal(out, ref)
