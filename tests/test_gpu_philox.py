"""Philox4x32-10 on the GPU: the library's device generator against cuRAND's
device block function curand_Philox4x32_10 (every counter word, including
word 3, which carries the draw's purpose), and the CPU oracle's Philox against
the same cuRAND outputs.  The uniform map is checked bit for bit against the
oracle's fp64 values."""
import ctypes
import os
import subprocess
import tempfile

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "speculative_decoding_verification_80_gb300", "csrc")


@pytest.fixture(scope="module")
def pin_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.init()
    out = os.path.join(tempfile.mkdtemp(prefix="philox_pin_"), "philox_pin.so")
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-shared", "-Xcompiler",
                    "-fPIC", f"-I{CSRC}", os.path.join(HERE, "cuda", "philox_pin.cu"), "-o", out], check=True)
    lib = ctypes.CDLL(out)
    lib.philox_pin.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int]
    lib.uniform_pin.argtypes = [ctypes.c_void_p] * 2 + [ctypes.c_int]
    return lib


def test_device_philox_matches_curand_and_oracle(pin_lib):
    rng = np.random.default_rng(0)
    n = 4096
    ctr = rng.integers(0, 2**32, size=(n, 4), dtype=np.uint64).astype(np.uint32)
    key = rng.integers(0, 2**32, size=(n, 2), dtype=np.uint64).astype(np.uint32)
    ctr[:16] = 0
    ctr[16:32, 3] = np.arange(16)  # counter word 3 alone
    c = torch.from_numpy(ctr.view(np.int32)).cuda()
    k = torch.from_numpy(key.view(np.int32)).cuda()
    a = torch.empty(n, 4, dtype=torch.int32, device="cuda")
    b = torch.empty(n, 4, dtype=torch.int32, device="cuda")
    assert pin_lib.philox_pin(c.data_ptr(), k.data_ptr(), a.data_ptr(), b.data_ptr(), n) == 0
    by_curand = a.cpu().numpy().view(np.uint32)
    by_lib = b.cpu().numpy().view(np.uint32)
    assert (by_curand == by_lib).all()
    for i in range(0, n, 37):
        assert list(oracle.philox4x32_10(ctr[i], key[i])) == list(by_curand[i]), i


def test_device_uniform_map_is_exact(pin_lib):
    rng = np.random.default_rng(1)
    w = rng.integers(0, 2**32, size=20000, dtype=np.uint64).astype(np.uint32)
    w[:4] = [0, 511, 512, 0xFFFFFFFF]
    wt = torch.from_numpy(w.view(np.int32)).cuda()
    u = torch.empty(w.size, dtype=torch.float32, device="cuda")
    assert pin_lib.uniform_pin(wt.data_ptr(), u.data_ptr(), w.size) == 0
    got = u.cpu().numpy().astype(np.float64)
    exp = np.array([oracle.uniform(int(x)) for x in w])
    assert (got == exp).all()
