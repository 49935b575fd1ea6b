"""GPU parity of spec_verify_packed (packed ragged rows, optional position
offsets) against the CPU oracle, through the C ABI.

The oracle runs on the dense form of the same batch; the packed outputs are
unpacked and compared row by row with the tolerances of tests/parity.py."""
import numpy as np
import pytest
import torch

from tests.parity import compare, oracle_on, wait_gpu
from workloads import make_config, make_random, pack, unpack_rows

pytestmark = pytest.mark.gpu

sd = pytest.importorskip("speculative_decoding_verification_80_gb300")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sd.load_library()


def _run_packed(w, pos=None, want_lse=True):
    t, d, x, cu = pack(w)
    R = t.shape[0]
    lse = torch.full((R, 2), float("nan"), device=t.device) if want_lse else None
    ws = sd.new_workspace(w.B, w.n_max, w.V, device=t.device)
    acc, out = sd.spec_verify_packed(t, d, cu, x, w.temperature, w.n_max, seed=w.seed, pos_offset=pos,
                                     row_lse=lse, workspace=ws)
    wait_gpu()
    out_d = unpack_rows(out, cu, w.n_max, -1)
    lse_d = None if lse is None else unpack_rows(lse, cu, w.n_max, float("nan"))
    return acc, out, out_d, lse_d, cu, ws


@pytest.mark.parametrize("V,dtype", [(1000, "f32"), (4097, "bf16"), (50001, "bf16"), (128256, "bf16")])
def test_packed_matches_oracle_with_offsets(V, dtype):
    w = make_random(24, 5, V, dtype=dtype, device="cuda", seed=V % 97, temperatures=(0.0, 0.6, 1.0, 1.4),
                    ragged=True, philox_seed=V * 31)
    pos = torch.randint(0, 1 << 30, (w.B,), generator=torch.Generator().manual_seed(V), dtype=torch.int64)
    pos = pos.to(torch.int32).to("cuda")
    acc, out, out_d, lse_d, cu, ws = _run_packed(w, pos)
    ref = oracle_on(w, pos_off=pos.cpu().numpy())
    compare(w, acc, out_d, ref, lse_d, f"packed V={V} {dtype}")
    assert sd.get_error(ws) == 0


def test_packed_without_offsets_equals_dense():
    w = make_random(40, 4, 20000, dtype="bf16", device="cuda", seed=11, temperatures=(0.8, 0.0, 1.2),
                    ragged=True, philox_seed=5)
    lse = torch.full((w.B, w.n_max + 1, 2), float("nan"), device="cuda")
    acc_d, out_dense = sd.spec_verify(w.target, w.draft, w.draft_tokens, w.draft_len, w.temperature,
                                      seed=w.seed, row_lse=lse)
    acc_p, _, out_p, lse_p, _, _ = _run_packed(w)
    wait_gpu()
    assert torch.equal(acc_d, acc_p)
    assert torch.equal(out_dense, out_p)
    both = ~torch.isnan(lse)
    assert torch.equal(both, ~torch.isnan(lse_p))
    assert torch.equal(lse[both], lse_p[both])


def test_packed_config5_every_request():
    # The ragged workload (B=1024, n_b ~ U{1..7}, V=152 064) in its natural
    # packed form, with position offsets: every request against the oracle.
    w = make_config(5, device="cuda")
    pos = (torch.arange(w.B, dtype=torch.int32, device="cuda") * 37) % 4096
    acc, out, out_d, lse_d, cu, ws = _run_packed(w, pos)
    ref = oracle_on(w, pos_off=pos.cpu().numpy())
    st = compare(w, acc, out_d, ref, lse_d, "packed config5")
    print("packed config5", st)
    assert st["requests"] == w.B
    a = acc.cpu().numpy()
    L = w.draft_len.cpu().numpy()
    o = out_d.cpu().numpy()
    for b in range(w.B):
        assert 0 <= o[b, a[b]] < w.V and (o[b, a[b] + 1: L[b] + 1] == -1).all()
    assert sd.get_error(ws) == 0


def test_packed_bad_segments_are_skipped_and_flagged():
    # Request 1 has an empty segment, request 3 more rows than n_max + 1 (its
    # draft length is clamped), request 4's segment reaches past total_rows.
    # Nothing outside the tensors is read and the other requests are verified
    # as usual.
    w = make_random(6, 2, 3000, dtype="bf16", device="cuda", seed=3, temperatures=(0.9, 0.0))
    V = w.V
    g = torch.Generator(device="cuda").manual_seed(9)
    R = 2 + 0 + 3 + 5 + 3 + 3  # rows as laid out below; request 4 is cut short
    t = (torch.randn(R, V, generator=g, device="cuda") * 3).to(torch.bfloat16)
    d = (torch.randn(R - w.B, V, generator=g, device="cuda") * 3).to(torch.bfloat16)
    x = torch.randint(0, V, (R - w.B,), generator=g, device="cuda").to(torch.int32)
    cu = torch.tensor([0, 2, 2, 5, 10, 13, 16], dtype=torch.int32, device="cuda")
    cu_bad = cu.clone()
    cu_bad[5] = 40  # request 4 reaches past the tensor; request 5 then starts past it too
    T = torch.tensor([0.9, 0.9, 0.0, 0.9, 0.9, 0.9], dtype=torch.float32, device="cuda")
    ws = sd.new_workspace(w.B, 2, V)
    out = torch.full((R,), -7, dtype=torch.int32, device="cuda")
    acc, _ = sd.spec_verify_packed(t, d, cu_bad, x, T, 2, seed=1, out_tokens=out, workspace=ws)
    wait_gpu()
    a = acc.cpu().tolist()
    o = out.cpu().tolist()
    assert a[1] == -1 and a[4] == -1 and a[5] == -1  # not verified
    assert o[13:16] == [-7, -7, -7]                   # request 5's rows were not written
    assert 0 <= a[0] <= 1 and 0 <= a[2] <= 2 and 0 <= a[3] <= 2
    assert sd.get_error(ws) & sd.DEV_ERR_DRAFT_LEN


def test_packed_and_early_exit_capture_into_one_graph():
    # Neither call synchronises or copies to the host: both capture into a
    # CUDA graph, and replays give the oracle's outputs.
    from workloads import make_config

    w = make_config(1, device="cuda")
    t, d, x, cu = pack(w)
    ws1 = sd.new_workspace(w.B, w.n_max, w.V)
    ws2 = sd.new_workspace(w.B, w.n_max, w.V)
    acc_p = torch.empty(w.B, dtype=torch.int32, device="cuda")
    out_p = torch.empty(t.shape[0], dtype=torch.int32, device="cuda")
    acc_e = torch.empty(w.B, dtype=torch.int32, device="cuda")
    out_e = torch.empty(w.B, w.n_max + 1, dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()
    wait_gpu()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        sd.spec_verify_packed(t, d, cu, x, w.temperature, w.n_max, seed=w.seed, accepted_len=acc_p,
                              out_tokens=out_p, workspace=ws1)
        sd.spec_verify_early_exit(w.target, w.draft, w.draft_tokens, w.draft_len, w.temperature, seed=w.seed,
                                  accepted_len=acc_e, out_tokens=out_e, workspace=ws2)
    for _ in range(3):
        g.replay()
    wait_gpu()
    ref = oracle_on(w, want_lse=False)
    compare(w, acc_p, unpack_rows(out_p, cu, w.n_max, -1), ref, None, "graph packed")
    compare(w, acc_e, out_e, ref, None, "graph early exit")


def test_two_streams_two_workspaces():
    # Two calls in flight on two streams, each with its own workspace.  Each
    # kernel takes one CTA per SM, so the second may start only as the first
    # one's CTAs leave.  Every segment and race job is claimed from a counter,
    # so a CTA that starts late finds the work taken: neither call waits on
    # the other's CTAs, and both finish with the oracle's outputs.
    w1 = make_random(48, 4, 30000, dtype="bf16", device="cuda", seed=1, temperatures=(0.8, 0.0), ragged=True,
                     philox_seed=11)
    w2 = make_random(40, 3, 50000, dtype="bf16", device="cuda", seed=2, temperatures=(1.1,), ragged=True,
                     philox_seed=22)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    ws1 = sd.new_workspace(w1.B, w1.n_max, w1.V)
    ws2 = sd.new_workspace(w2.B, w2.n_max, w2.V)
    wait_gpu()
    outs = []
    for _ in range(3):
        a1, o1 = sd.spec_verify(w1.target, w1.draft, w1.draft_tokens, w1.draft_len, w1.temperature, seed=w1.seed,
                                workspace=ws1, stream=s1)
        a2, o2 = sd.spec_verify(w2.target, w2.draft, w2.draft_tokens, w2.draft_len, w2.temperature, seed=w2.seed,
                                workspace=ws2, stream=s2)
        outs.append((a1, o1, a2, o2))
    torch.cuda.synchronize()
    r1 = oracle_on(w1, want_lse=False)
    r2 = oracle_on(w2, want_lse=False)
    for a1, o1, a2, o2 in outs:
        compare(w1, a1, o1, r1, None, "stream 1")
        compare(w2, a2, o2, r2, None, "stream 2")
    assert sd.get_error(ws1) == 0 and sd.get_error(ws2) == 0
