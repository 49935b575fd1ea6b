"""GPU parity of spec_verify against the CPU oracle (calls go through the C ABI
via the ctypes binding).  Requires a GB300 and the built library."""
import numpy as np
import pytest
import torch

import oracle
from tests.parity import compare, oracle_on, wait_gpu
from workloads import make_config, make_random

pytestmark = pytest.mark.gpu

sd = pytest.importorskip("speculative_decoding_verification_80_gb300")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sd.load_library()


def _run(w, seed=None, stream=None):
    dev = w.target.device
    lse = torch.full((w.B, w.n_max + 1, 2), float("nan"), device=dev)
    ws = sd.new_workspace(w.B, w.n_max, w.V, device=dev)
    acc, out = sd.spec_verify(w.target, w.draft, w.draft_tokens, w.draft_len, w.temperature,
                              seed=w.seed if seed is None else seed, row_lse=lse, workspace=ws,
                              stream=stream)
    wait_gpu()
    return acc, out, lse, ws


def test_config1_tiny_fp32_all_rows():
    w = make_config(1, device="cuda")
    acc, out, lse, ws = _run(w)
    ref = oracle_on(w)
    st = compare(w, acc, out, ref, lse, "config1")
    assert st["mismatch"] == 0
    assert sd.get_error(ws) == 0


@pytest.mark.parametrize("V", [7, 8, 1000, 1024, 4097])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_random_small_shapes(V, dtype):
    w = make_random(24, 4, V, dtype=dtype, device="cuda", seed=V, temperatures=(0.0, 0.3, 1.0, 1.3),
                    ragged=True, philox_seed=V * 7919)
    acc, out, lse, ws = _run(w)
    ref = oracle_on(w)
    compare(w, acc, out, ref, lse, f"V={V} {dtype}")
    assert sd.get_error(ws) == 0


@pytest.mark.parametrize("V,dtype", [(40000, "bf16"), (50001, "bf16"), (70000, "f32"),
                                     (128256, "bf16"), (262144, "bf16"), (150001, "f32")])
def test_multi_cta_rows(V, dtype):
    # Rows cut into many chunks streamed by different groups and CTAs (their
    # partials merged by the request combine), aligned (bulk copy) and ragged
    # (plain-load) rows, and the largest vocabulary.
    w = make_random(6, 3, V, dtype=dtype, device="cuda", seed=V % 1000,
                    temperatures=(0.7, 0.0, 1.3), ragged=True, philox_seed=12345)
    acc, out, lse, ws = _run(w)
    ref = oracle_on(w)
    compare(w, acc, out, ref, lse, f"V={V} {dtype}")
    assert sd.get_error(ws) == 0


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_stream_sum_reference_edges(dtype):
    # A sampled row's sum takes each thread's largest element of its first
    # vector in the segment as its reference.  Two rows leave that path:
    # request 0's rows start with 4096 -inf logits (no finite value in the
    # first vector of any thread: the reference comes from the whole chunk),
    # and requests 1 and 2 carry one logit far above the rest in a later
    # chunk of the segment (its term overflows: the chunk is summed again
    # against its own maximum).  Outputs and LSEs must match the oracle.
    w = make_random(8, 3, 40000, dtype=dtype, device="cuda", seed=5, temperatures=(1.0, 1.0, 0.3, 0.7),
                    philox_seed=123)
    w.target[0, :, :4096] = float("-inf")
    w.draft[0, :, :4096] = float("-inf")
    w.draft_tokens[0] = torch.tensor([5000, 6000, 7000], dtype=torch.int32, device="cuda")
    w.target[1, 1, 20000] = 200.0
    w.draft[1, 1, 20000] = 150.0
    w.target[2, 0, 30000] = 120.0
    acc, out, lse, ws = _run(w)
    ref = oracle_on(w)
    st = compare(w, acc, out, ref, lse, f"reference edges {dtype}")
    assert st["mismatch"] == 0
    assert sd.get_error(ws) == 0
    # the spiked rows' log-sum-exp is the spike's scaled logit
    assert abs(float(lse[1, 1, 0]) - 200.0 / float(w.temperature[1])) < 1e-3
    assert abs(float(lse[2, 0, 0]) - 120.0 / float(w.temperature[2])) < 1e-3


def test_plan_records_written_per_warp_mixed_batch():
    # Above 256 requests the plan kernel's warps write their lanes' unit
    # records together (each lane finds its request by a shuffle search):
    # requests with 1 to 9 units (greedy ones, n_b = 0, ragged lengths) must
    # still be verified exactly as the oracle does.
    w = make_random(300, 4, 3000, dtype="bf16", device="cuda", seed=17, temperatures=(0.0, 0.7, 1.0, 1.3),
                    ragged=True, philox_seed=2024)
    acc, out, lse, ws = _run(w)
    ref = oracle_on(w)
    st = compare(w, acc, out, ref, lse, "plan per warp")
    assert st["requests"] == 300
    assert sd.get_error(ws) == 0


def test_identical_distributions_accept_all_on_gpu():
    w = make_random(32, 5, 5000, dtype="bf16", device="cuda", seed=3, temperatures=(0.5, 1.0, 2.0))
    w.draft = w.target[:, : w.n_max].contiguous()
    acc, out, _, _ = _run(w)
    assert (acc.cpu() == w.n_max).all()


def test_near_identical_distributions_rerun_races_without_threshold():
    # Draft and target logits 0.02 apart: rows are rarely rejected, and a
    # rejected row's residual mass R is small, so its thresholded race finds
    # no key at or above 1/64 with probability exp(-64 R) and runs again
    # without the threshold (the job tag travels through the rerun).
    w = make_random(512, 8, 4096, dtype="f32", device="cuda", seed=31, temperatures=(0.8, 1.0, 1.2),
                    draft_noise=0.02, philox_seed=13)
    acc, out, lse, _ = _run(w)
    ref = oracle_on(w)
    compare(w, acc, out, ref, lse, "near-identical drafts")
    a = ref["accepted_len"]
    t = w.target.double().cpu().numpy()
    d = w.draft.double().cpu().numpy()
    T = w.temperature.cpu().numpy()
    small = 0
    for b in range(w.B):
        if a[b] >= w.n_max:
            continue  # every draft accepted: a race on p, R = 1
        k = int(a[b])
        p = np.exp(t[b, k] / T[b] - np.logaddexp.reduce(t[b, k] / T[b]))
        q = np.exp(d[b, k] / T[b] - np.logaddexp.reduce(d[b, k] / T[b]))
        if np.maximum(p - q, 0.0).sum() < 1.0 / 128:
            small += 1  # reruns with probability > exp(-1/2)
    assert small >= 4, small


def test_zero_drafts_is_plain_sampling():
    # No draft tensor at all: T > 0 requests sample from the target row, T = 0
    # ones take its argmax, and nothing is flagged.
    w = make_random(64, 0, 3000, dtype="bf16", device="cuda", seed=4, temperatures=(0.8, 0.0))
    w.draft = None
    acc, out, lse, ws = _run(w)
    ref = oracle_on(w)
    compare(w, acc, out, ref, lse, "n=0")
    assert (acc.cpu() == 0).all()
    assert sd.get_error(ws) == 0
    sampled = (w.temperature.cpu() > 0).numpy()
    top = w.target[:, 0].float().argmax(dim=1).cpu().numpy()
    assert (out.cpu().numpy()[sampled, 0] != top[sampled]).any()


def test_missing_draft_logits_only_bind_requests_with_drafts():
    # draft_len 0 requests sample without draft logits; requests with drafts
    # and T > 0 fall back to greedy and flag the temperature bit.
    w = make_random(32, 3, 5000, dtype="bf16", device="cuda", seed=9, temperatures=(1.0,), ragged=True,
                    philox_seed=4)
    w.draft_len[: w.B // 2] = 0
    w.draft = None
    acc, out, lse, ws = _run(w)
    ref = oracle_on(w)
    compare(w, acc, out, ref, lse, "no draft logits")
    has = (w.draft_len.cpu() > 0).any().item()
    assert sd.get_error(ws) == (sd.DEV_ERR_TEMPERATURE if has else 0)


def test_same_seed_is_deterministic_and_seed_matters():
    w = make_random(64, 4, 2048, dtype="bf16", device="cuda", seed=5, temperatures=(1.0,))
    a1, o1, _, _ = _run(w, seed=11)
    a2, o2, _, _ = _run(w, seed=11)
    a3, o3, _, _ = _run(w, seed=12)
    assert torch.equal(a1, a2) and torch.equal(o1, o2)
    assert not torch.equal(o1, o3)


def test_workspace_is_reusable_call_after_call():
    w = make_random(20, 3, 3000, dtype="bf16", device="cuda", seed=6, temperatures=(0.9, 0.0),
                    ragged=True)
    w.seed = 1
    ws = sd.new_workspace(w.B, w.n_max, w.V)
    outs = []
    for _ in range(3):
        acc, out = sd.spec_verify(w.target, w.draft, w.draft_tokens, w.draft_len, w.temperature,
                                  seed=w.seed, workspace=ws)
        outs.append((acc.clone(), out.clone()))
    wait_gpu()
    for acc, out in outs[1:]:
        assert torch.equal(acc, outs[0][0]) and torch.equal(out, outs[0][1])
    ref = oracle_on(w, want_lse=False)
    compare(w, outs[-1][0], outs[-1][1], ref, None, "third call")


def test_device_data_errors_match_oracle():
    w = make_random(6, 3, 500, dtype="f32", device="cuda", seed=7, temperatures=(1.0,))
    x = w.draft_tokens.clone()
    x[0, 0] = w.V + 3  # out-of-range token at a scored row
    L = w.draft_len.clone()
    L[1] = w.n_max + 2  # clamped
    T = w.temperature.clone()
    T[2], T[3], T[4] = -1.0, float("nan"), 1e-9
    w.draft_tokens, w.draft_len, w.temperature = x, L, T
    acc, out, lse, ws = _run(w)
    ref = oracle_on(w, want_lse=False)
    compare(w, acc, out, ref, None, "bad data")
    bits = sd.get_error(ws)
    assert bits == ref["err"] == (sd.DEV_ERR_TOKEN | sd.DEV_ERR_DRAFT_LEN | sd.DEV_ERR_TEMPERATURE)
    assert sd.get_error(ws) == 0  # read-and-clear


def test_graph_capture_has_no_host_sync():
    # Capturing spec_verify + mtp_shift_insert into a CUDA graph fails if
    # either call synchronises or copies to the host.
    w = make_config(1, device="cuda")
    R = w.B * (w.n_max + 1)
    ws = sd.new_workspace(w.B, w.n_max, w.V)
    acc = torch.empty(w.B, dtype=torch.int32, device="cuda")
    out = torch.empty(w.B, w.n_max + 1, dtype=torch.int32, device="cuda")
    tok_in = torch.arange(R, dtype=torch.int32, device="cuda")
    tok_out = torch.empty_like(tok_in)
    s = torch.cuda.Stream()
    wait_gpu()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        sd.spec_verify(w.target, w.draft, w.draft_tokens, w.draft_len, w.temperature, seed=w.seed,
                       accepted_len=acc, out_tokens=out, workspace=ws)
        sd.mtp_shift_insert(tok_in, tok_out, w.draft_len, acc, out.view(-1), w.n_max + 1)
    for _ in range(3):
        g.replay()
    wait_gpu()
    ref = oracle_on(w, want_lse=False)
    compare(w, acc, out, ref, None, "graph")
    expect = tok_in.cpu().numpy().copy()
    oracle.mtp_shift_insert(tok_in.cpu().numpy(), expect, w.draft_len.cpu().numpy(),
                            acc.cpu().numpy(), out.cpu().numpy().ravel(), w.n_max + 1)
    assert (tok_out.cpu().numpy() == expect).all()


# ---------------------------------------------------------- full-size workloads
def test_config2_linear_full():
    w = make_config(2, device="cuda")
    acc, out, lse, ws = _run(w)
    ref = oracle_on(w)
    st = compare(w, acc, out, ref, lse, "config2")
    print("config2", st)
    assert sd.get_error(ws) == 0


def test_config3_mtp_full():
    w = make_config(3, device="cuda")
    acc, out, lse, ws = _run(w)
    ref = oracle_on(w)
    st = compare(w, acc, out, ref, lse, "config3")
    print("config3", st)
    # MTP step on the verify outputs, hidden carried to a second buffer
    R = w.mtp_tokens.numel()
    tok_out = torch.empty_like(w.mtp_tokens)
    hid_out = torch.empty_like(w.hidden)
    sd.mtp_shift_insert(w.mtp_tokens, tok_out, w.draft_len, acc, out.view(-1), w.n_max + 1,
                        hidden_in=w.hidden, hidden_out=hid_out)
    wait_gpu()
    expect = w.mtp_tokens.cpu().numpy().copy()
    oracle.mtp_shift_insert(w.mtp_tokens.cpu().numpy(), expect, w.draft_len.cpu().numpy(),
                            acc.cpu().numpy(), out.cpu().numpy().ravel(), w.n_max + 1)
    assert (tok_out.cpu().numpy() == expect).all()
    assert torch.equal(hid_out.view(torch.int16), w.hidden.view(torch.int16))
    assert R == 512


def test_config4_greedy_full():
    w = make_config(4, device="cuda")
    acc, out, lse, ws = _run(w)
    ref = oracle_on(w, want_lse=False)
    st = compare(w, acc, out, ref, None, "config4")
    assert st["mismatch"] == 0
    mean_emitted = float((acc.float() + 1).mean())
    assert 2.5 < mean_emitted < 3.6, mean_emitted  # about 3.05 by construction


def test_config5_ragged_every_request():
    # The largest workload (B=1024, n_b ~ U{1..7}, V=152 064, per-request T):
    # every request against the oracle (the oracle runs on several threads).
    w = make_config(5, device="cuda")
    acc, out, lse, ws = _run(w)
    ref = oracle_on(w)
    st = compare(w, acc, out, ref, lse, "config5")
    print("config5", st)
    assert st["requests"] == w.B
    assert st["near_tie_rows"] <= max(1, int(1e-4 * st["rows"]))
    assert sd.get_error(ws) == 0


def test_side_stream_without_a_workspace():
    # stream= given and no workspace: the default workspace and outputs are
    # allocated and zeroed on that stream, so the call is ordered after them.
    w = make_random(40, 4, 20000, dtype="bf16", device="cuda", seed=31, temperatures=(0.9, 0.0), ragged=True,
                    philox_seed=8)
    s = torch.cuda.Stream()
    wait_gpu()
    results = []
    for _ in range(4):
        acc, out = sd.spec_verify(w.target, w.draft, w.draft_tokens, w.draft_len, w.temperature, seed=w.seed,
                                  stream=s)
        results.append((acc, out))
    s.synchronize()
    ref = oracle_on(w, want_lse=False)
    for acc, out in results:
        compare(w, acc, out, ref, None, "side stream")
    # a raw stream handle works the same way
    acc, out = sd.spec_verify(w.target, w.draft, w.draft_tokens, w.draft_len, w.temperature, seed=w.seed,
                              stream=s.cuda_stream)
    s.synchronize()
    compare(w, acc, out, ref, None, "raw handle")
