"""spec_verify does not need all of its CTAs resident at once: with half the
SMs held by another kernel (bounded, 200 KB of shared memory per block, so no
verify CTA fits beside it), the CTAs that do run take every segment and race
job from the counters and finish the whole batch; the CTAs that start later
find nothing left and leave.  The outputs are read on a third stream while
the other kernel still holds its SMs."""
import ctypes
import os
import subprocess
import tempfile
import time

import numpy as np
import pytest
import torch

from tests.parity import compare, oracle_on, wait_gpu
from workloads import make_random

pytestmark = pytest.mark.gpu

sd = pytest.importorskip("speculative_decoding_verification_80_gb300")
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def hold_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sd.load_library()
    out = os.path.join(tempfile.mkdtemp(prefix="hold_sm_"), "hold_sm.so")
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-shared", "-Xcompiler", "-fPIC",
                    os.path.join(HERE, "cuda", "hold_sm.cu"), "-o", out], check=True)
    lib = ctypes.CDLL(out)
    lib.launch_hold.argtypes = [ctypes.c_int, ctypes.c_longlong, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    lib.launch_hold.restype = ctypes.c_int
    return lib


def test_verify_finishes_on_the_sms_it_gets(hold_lib):
    dev = torch.device("cuda")
    w = make_random(48, 4, 65536, dtype="bf16", device="cuda", seed=21, temperatures=(0.7, 0.0, 1.2),
                    ragged=True, philox_seed=77)
    ws = sd.new_workspace(w.B, w.n_max, w.V, device=dev)
    acc = torch.full((w.B,), -7, dtype=torch.int32, device=dev)
    out = torch.full((w.B, w.n_max + 1), -7, dtype=torch.int32, device=dev)
    acc_h = torch.empty(w.B, dtype=torch.int32).pin_memory()
    out_h = torch.empty(w.B, w.n_max + 1, dtype=torch.int32).pin_memory()
    finished = torch.zeros(1, dtype=torch.int32, device=dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    s_hold, s_verify, s_read = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    # Load the kernels first: a module's first launch may wait for running work.
    sd.spec_verify(w.target, w.draft, w.draft_tokens, w.draft_len, w.temperature, seed=w.seed,
                   accepted_len=acc, out_tokens=out, workspace=ws, stream=s_verify)
    wait_gpu()
    acc.fill_(-7)
    out.fill_(-7)
    wait_gpu()
    clock_hz = 2.0e9
    hold_s = 0.4
    assert hold_lib.launch_hold(sms // 2, int(hold_s * clock_hz), 200 * 1024, ctypes.c_void_p(finished.data_ptr()),
                                ctypes.c_void_p(s_hold.cuda_stream)) == 0
    t0 = time.perf_counter()
    sd.spec_verify(w.target, w.draft, w.draft_tokens, w.draft_len, w.temperature, seed=w.seed,
                   accepted_len=acc, out_tokens=out, workspace=ws, stream=s_verify)
    time.sleep(0.1)  # the held SMs stay held for hold_s; the verify work needs well under a millisecond
    with torch.cuda.stream(s_read):
        acc_h.copy_(acc, non_blocking=True)
        out_h.copy_(out, non_blocking=True)
        fin_h = finished.to("cpu", non_blocking=True)
    s_read.synchronize()
    read_at = time.perf_counter() - t0
    still_held = int(fin_h.item()) == 0
    wait_gpu()
    wall = time.perf_counter() - t0
    assert still_held, "the holding kernel ended before the outputs were read"
    assert read_at < hold_s
    ref = oracle_on(w, want_lse=False)
    compare(w, acc_h, out_h, ref, None, "half the SMs held")  # complete before the late CTAs could run
    assert sd.get_error(ws) == 0
    assert wall < 1.5, wall  # far below the ~2 s budget of a device wait
    # the late CTAs left the workspace re-armed: the next call is correct too
    acc2, out2 = sd.spec_verify(w.target, w.draft, w.draft_tokens, w.draft_len, w.temperature, seed=w.seed,
                                workspace=ws)
    wait_gpu()
    assert torch.equal(acc2.cpu(), acc_h) and torch.equal(out2.cpu(), out_h)
