"""GPU parity of mtp_shift_insert on multi-token segments (n_b drafts, n_b + 1
tokens per request) against the oracle, through the C ABI.

After a verify step with several drafts per request, the draft model is run
again over each request's whole window with the target's hidden states: the
token buffer is shifted left by one within each segment and the token the
target sampled at the first rejection a_b is inserted at position a_b, while
the hidden states stay in place (copied bitwise when an output buffer is
given).  Segments here are ragged and packed (explicit starts), as the packed
verify lays them out."""
import numpy as np
import pytest
import torch

import oracle
from tests.parity import wait_gpu
from workloads import make_random, pack

pytestmark = pytest.mark.gpu

sd = pytest.importorskip("speculative_decoding_verification_80_gb300")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sd.load_library()


def _oracle(tok_in, L, acc, nxt, stride, seg=None, hid_in=None):
    expect = tok_in.copy()
    hid_out = None if hid_in is None else np.zeros_like(hid_in)
    oracle.mtp_shift_insert(tok_in, expect, L, acc, nxt, stride, seg_start=seg, hidden_in=hid_in,
                            hidden_out=hid_out)
    return expect, hid_out


@pytest.mark.parametrize("H,in_place", [(7168, False), (33, False), (0, True)])
def test_mtp_after_packed_verify(H, in_place):
    # Verify a ragged batch in packed form, then shift/insert its token window.
    w = make_random(48, 7, 5000, dtype="bf16", device="cuda", seed=H + 1, temperatures=(0.8, 0.0, 1.2),
                    ragged=True, philox_seed=3)
    t, d, x, cu = pack(w)
    R = t.shape[0]
    acc, out = sd.spec_verify_packed(t, d, cu, x, w.temperature, w.n_max, seed=w.seed)
    seg = cu[:-1].contiguous()
    nxt = out[(seg + acc).long()].contiguous()  # the token sampled at a_b
    g = torch.Generator(device="cuda").manual_seed(H)
    tok_in = torch.randint(0, w.V, (R,), generator=g, device="cuda").to(torch.int32)
    tok_ref_in = tok_in.cpu().numpy().copy()
    hid_in = hid_out = None
    if H:
        hid_in = torch.randn(R, H, generator=g, device="cuda").to(torch.bfloat16)
        hid_out = torch.empty_like(hid_in)
    tok_out = tok_in if in_place else torch.empty_like(tok_in)
    sd.mtp_shift_insert(tok_in, tok_out, w.draft_len, acc, nxt, 0, seg_start=seg, hidden_in=hid_in,
                        hidden_out=hid_out)
    wait_gpu()
    expect, hid_ref = _oracle(tok_ref_in, w.draft_len.cpu().numpy(), acc.cpu().numpy(), nxt.cpu().numpy(), 0,
                              seg=seg.cpu().numpy(),
                              hid_in=None if hid_in is None else hid_in.view(torch.int16).cpu().numpy())
    assert (tok_out.cpu().numpy() == expect).all()
    if H:
        assert (hid_out.view(torch.int16).cpu().numpy() == hid_ref).all()


def test_mtp_dense_stride_and_edge_segments():
    # Uniform windows of n_max + 1 tokens with next_token read through the
    # out_tokens stride; requests with a_b = 0 and a_b = n_b, and one segment
    # whose accepted length is out of range (left untouched, as the oracle).
    B, n = 16, 4
    rows = n + 1
    g = torch.Generator().manual_seed(5)
    tok_in = torch.randint(0, 1000, (B * rows,), generator=g, dtype=torch.int32)
    L = torch.full((B,), n, dtype=torch.int32)
    acc = torch.randint(0, n + 1, (B,), generator=g, dtype=torch.int32)
    acc[0], acc[1], acc[2] = 0, n, n + 3  # request 2: invalid
    out = torch.randint(0, 1000, (B, rows), generator=g, dtype=torch.int32)
    expect, _ = _oracle(tok_in.numpy().copy(), L.numpy(), acc.numpy(), out.numpy().ravel(), rows)
    dev = [v.cuda() for v in (tok_in, L, acc, out)]
    tok_out = torch.full_like(dev[0], -5)
    err = sd.new_workspace(B, n, 1000)  # a verify workspace: its first word is the error word
    sd.mtp_shift_insert(dev[0], tok_out, dev[1], dev[2], dev[3].view(-1), rows, error_word=err)
    wait_gpu()
    got = tok_out.cpu().numpy()
    valid = np.ones(B * rows, dtype=bool)
    valid[2 * rows: 3 * rows] = False  # the invalid segment is left unchanged
    assert (got[valid] == expect[valid]).all()
    assert (got[~valid] == -5).all()
    assert sd.get_error(err) == sd.DEV_ERR_SEGMENT
    # without an error word the bad segment is skipped the same way, silently
    sd.mtp_shift_insert(dev[0], tok_out, dev[1], dev[2], dev[3].view(-1), rows)
    wait_gpu()
    assert (tok_out.cpu().numpy()[valid] == expect[valid]).all()
