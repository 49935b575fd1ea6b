"""The failure path on the GPU, without a fault: a build of the library in
which one warp waits for a word that nothing writes (SPECDEC_TEST_WAIT_RUNS_OUT,
with a 0.05 s wait budget).  Every wait of that call runs out in turn; the call
reports SPECDEC_ERR_TIMEOUT through specdec_get_error, the context stays
usable, and the production library's next call on the same workspace gives
the oracle's outputs with no error: the timed-out call re-armed the
workspace."""
import ctypes
import os
import subprocess
import tempfile

import numpy as np
import pytest
import torch

from tests.parity import compare, oracle_on, wait_gpu
from workloads import make_config

pytestmark = pytest.mark.gpu

sd = pytest.importorskip("speculative_decoding_verification_80_gb300")
PKG = os.path.dirname(sd.__file__)
ROOT = os.path.dirname(PKG)


@pytest.fixture(scope="module")
def stall_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sd.load_library()
    out = os.path.join(tempfile.mkdtemp(prefix="specdec_stall_"), "libspecdec_stall.so")
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-shared",
                    "-Xcompiler", "-fPIC", f"-I{os.path.join(ROOT, 'include')}", f"-I{os.path.join(PKG, 'csrc')}",
                    "-DSPECDEC_TEST_WAIT_RUNS_OUT", "-DSPECDEC_WAIT_BUDGET_CYCLES=100000000LL",
                    os.path.join(PKG, "csrc", "api.cu"), "-o", out], check=True)
    return sd.load_library(path=out)


@pytest.mark.parametrize("config", [1, 2])
def test_a_wait_that_runs_out_reports_timeout_and_rearms(stall_lib, config):
    w = make_config(config, device="cuda")
    ws = sd.new_workspace(w.B, w.n_max, w.V)
    acc = torch.empty(w.B, dtype=torch.int32, device="cuda")
    out = torch.empty(w.B, w.n_max + 1, dtype=torch.int32, device="cuda")
    P = ctypes.c_void_p
    st = stall_lib.spec_verify(P(w.target.data_ptr()), P(w.draft.data_ptr()), sd.F32 if w.dtype == "f32" else sd.BF16,
                               w.B, w.n_max, w.V, P(w.draft_tokens.data_ptr()), P(w.draft_len.data_ptr()),
                               P(w.temperature.data_ptr()), w.seed, P(acc.data_ptr()), P(out.data_ptr()), None,
                               P(ws.data_ptr()), ws.numel(), P(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    wait_gpu(timeout_s=60.0)  # bounded: a few 0.05 s budgets
    bits = ctypes.c_uint32(0)
    assert stall_lib.specdec_get_error(P(ws.data_ptr()), ctypes.byref(bits)) == 6  # SPECDEC_ERR_TIMEOUT
    assert bits.value & sd.DEV_ERR_TIMEOUT
    # the production library, same workspace: the oracle's outputs, no error
    acc2, out2 = sd.spec_verify(w.target, w.draft, w.draft_tokens, w.draft_len, w.temperature, seed=w.seed,
                                workspace=ws)
    wait_gpu()
    ref = oracle_on(w, want_lse=False)
    compare(w, acc2, out2, ref, None, f"config{config} after a timed-out call")
    assert sd.get_error(ws) == 0
