"""spec_verify_no_alloc: the verify step for callers that cannot allocate
device memory when they verify (code inside an allocator or memory-pool
callback, runtimes that forbid cudaMalloc after start-up because it
synchronises the device, C hosts that only own the tensors they pass).

The entry point is called through the C ABI (ctypes) and must give exactly
what spec_verify gives with a caller-allocated workspace, on two calls in a
row (the second call reuses the library's array).  This file is collected
last so that a run stopping at its first failure has run everything else."""
import ctypes

import pytest
import torch

from tests.parity import wait_gpu
from workloads import make_config, make_random

pytestmark = pytest.mark.gpu

sd = pytest.importorskip("speculative_decoding_verification_80_gb300")


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return sd.load_library()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _no_alloc(lib, w, seed):
    dev = w.target.device
    acc = torch.full((w.B,), -7, dtype=torch.int32, device=dev)
    out = torch.full((w.B, w.n_max + 1), -7, dtype=torch.int32, device=dev)
    lse = torch.full((w.B, w.n_max + 1, 2), float("nan"), device=dev)
    dtype = sd.F32 if w.target.dtype == torch.float32 else sd.BF16
    st = lib.spec_verify_no_alloc(_ptr(w.target), _ptr(w.draft), dtype, w.B, w.n_max, w.V,
                                  _ptr(w.draft_tokens), _ptr(w.draft_len), _ptr(w.temperature),
                                  seed, _ptr(acc), _ptr(out), _ptr(lse),
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, st
    wait_gpu()
    return acc, out, lse


def _reference(w, seed):
    lse = torch.full((w.B, w.n_max + 1, 2), float("nan"), device=w.target.device)
    acc, out = sd.spec_verify(w.target, w.draft, w.draft_tokens, w.draft_len, w.temperature,
                              seed=seed, row_lse=lse)
    wait_gpu()
    return acc, out, lse


@pytest.mark.parametrize("case", ["tiny_fp32", "bf16_128k_ragged_mixed_T"])
def test_no_alloc_matches_spec_verify_twice(lib, case):
    if case == "tiny_fp32":
        w = make_config(1, device="cuda")
    else:
        w = make_random(48, 4, 128256, dtype="bf16", device="cuda", seed=21,
                        temperatures=(0.7, 0.0, 1.2), ragged=True, philox_seed=99)
    acc_r, out_r, lse_r = _reference(w, w.seed)
    for _ in range(2):  # the second call runs on what the first left in the array
        acc, out, lse = _no_alloc(lib, w, w.seed)
        assert torch.equal(acc, acc_r)
        assert torch.equal(out, out_r)
        scored = ~torch.isnan(lse_r)
        assert torch.equal(scored, ~torch.isnan(lse))
        err = (lse[scored] - lse_r[scored]).abs() / lse_r[scored].abs().clamp_min(1.0)
        assert err.numel() == 0 or err.max().item() <= 1e-5


def test_no_alloc_rejects_batches_beyond_its_array(lib):
    B, n, V = 60000, 7, 152064
    need = lib.specdec_verify_workspace_bytes(B, n, V)
    assert need > (8 << 20)
    fake = ctypes.c_void_p(0x1000)
    st = lib.spec_verify_no_alloc(fake, fake, sd.BF16, B, n, V, fake, fake, fake, 0, fake, fake,
                                  None, None)
    assert st == 3  # SPECDEC_ERR_WORKSPACE, nothing enqueued
