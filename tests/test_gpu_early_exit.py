"""GPU tests of spec_verify_early_exit (rows after a request's first rejection
are not read).  Its outputs must equal spec_verify's bit for bit and match
the oracle; only the bytes read may differ, and they are bounded below by the
rows the outcome needs and above by every row plus the race's re-reads."""
import numpy as np
import pytest
import torch

from tests.parity import compare, oracle_on, wait_gpu
from workloads import make_config, make_random

pytestmark = pytest.mark.gpu

sd = pytest.importorskip("speculative_decoding_verification_80_gb300")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sd.load_library()


def _byte_bounds(w, acc):
    """(needed, full): logits bytes the outcome needs (target rows 0..a, draft
    rows 0..min(a, n_b - 1) of sampled requests) and every valid row plus
    one race re-read of row a per sampled request."""
    elt = w.target.element_size()
    row = w.V * elt
    a = acc.cpu().numpy().astype(np.int64)
    L = w.draft_len.cpu().numpy().clip(0, w.n_max).astype(np.int64)
    T = w.temperature.cpu().numpy()
    sampled = (T > 0) & (w.draft is not None)
    need = ((a + 1) + np.where(sampled, np.minimum(a + 1, L), 0)).sum() * row
    full = ((L + 1) + np.where(sampled, L, 0)).sum() * row
    race = np.where(sampled, 1 + (a < L), 0).sum() * row
    return int(need), int(full + race)


def _both(w):
    ws = sd.new_workspace(w.B, w.n_max, w.V)
    acc_f, out_f = sd.spec_verify(w.target, w.draft, w.draft_tokens, w.draft_len, w.temperature, seed=w.seed)
    sd.bytes_read(ws)  # starts at zero; clears anything left
    acc_e, out_e = sd.spec_verify_early_exit(w.target, w.draft, w.draft_tokens, w.draft_len, w.temperature,
                                             seed=w.seed, workspace=ws)
    wait_gpu()
    return acc_f, out_f, acc_e, out_e, ws


@pytest.mark.parametrize("V,dtype", [(1000, "f32"), (4097, "bf16"), (50001, "bf16")])
def test_early_exit_equals_full_and_oracle(V, dtype):
    w = make_random(40, 6, V, dtype=dtype, device="cuda", seed=V % 89, temperatures=(0.0, 0.5, 1.0, 1.5),
                    ragged=True, philox_seed=V * 13)
    acc_f, out_f, acc_e, out_e, ws = _both(w)
    assert torch.equal(acc_f, acc_e) and torch.equal(out_f, out_e)
    ref = oracle_on(w, want_lse=False)
    compare(w, acc_e, out_e, ref, None, f"early exit V={V} {dtype}")
    need, full = _byte_bounds(w, acc_e)
    got = sd.bytes_read(ws)
    assert need <= got <= full, (need, got, full)
    assert sd.get_error(ws) == 0


@pytest.mark.parametrize("k", [2, 4])
def test_early_exit_full_configs(k):
    w = make_config(k, device="cuda")
    acc_f, out_f, acc_e, out_e, ws = _both(w)
    assert torch.equal(acc_f, acc_e) and torch.equal(out_f, out_e)
    need, full = _byte_bounds(w, acc_e)
    got = sd.bytes_read(ws)
    assert need <= got <= full, (need, got, full)
    print(f"config {k}: bytes read {got / 1e6:.1f} MB, needed {need / 1e6:.1f} MB, full {full / 1e6:.1f} MB")
    assert sd.get_error(ws) == 0


def test_early_exit_workspace_reuse_and_mixing():
    # Early-exit state is cleared at the end of each call, so a workspace
    # serves repeated early-exit calls and full calls in any order.
    w = make_random(64, 5, 20000, dtype="bf16", device="cuda", seed=21, temperatures=(0.9, 0.0, 1.3),
                    ragged=True, philox_seed=77)
    ws = sd.new_workspace(w.B, w.n_max, w.V)
    results = []
    for call in ("ee", "ee", "full", "ee", "full", "ee"):
        fn = sd.spec_verify_early_exit if call == "ee" else sd.spec_verify
        acc, out = fn(w.target, w.draft, w.draft_tokens, w.draft_len, w.temperature, seed=w.seed, workspace=ws)
        results.append((acc.clone(), out.clone()))
    wait_gpu()
    for acc, out in results[1:]:
        assert torch.equal(acc, results[0][0]) and torch.equal(out, results[0][1])
    assert sd.get_error(ws) == 0
