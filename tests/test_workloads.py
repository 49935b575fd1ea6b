"""The synthetic inputs (CPU only): each workload follows its stated recipe,
rows past a request's draft length are poisoned (NaN logits, -1 tokens) so a
kernel that read them would fail parity, and the packed layout round-trips.
The recipes are cut to a few requests here (same generator, same shapes per
request)."""
import math

import numpy as np
import pytest
import torch

from workloads import make_config, make_random, pack, unpack_rows
from workloads.gen import CONFIGS, algorithmic_bytes


def _valid_rows(w):
    L = w.draft_len.long()
    j = torch.arange(w.n_max + 1).view(1, -1)
    return j <= L.view(-1, 1), j[:, : w.n_max] < L.view(-1, 1)


@pytest.mark.parametrize("k", [1, 2, 3, 4, 5])
def test_config_shapes_and_poisoned_padding(k):
    c = CONFIGS[k]
    B = min(c["B"], 6)
    w = make_config(k, B=B)
    V, n = c["V"], c["n"]
    dt = torch.float32 if c["dtype"] == "f32" else torch.bfloat16
    assert (w.B, w.n_max, w.V) == (B, n, V)
    assert w.target.shape == (B, n + 1, V) and w.target.dtype == dt
    assert w.draft.shape == (B, n, V) and w.draft.dtype == dt
    assert w.draft_tokens.dtype == torch.int32 and w.draft_len.dtype == torch.int32
    assert w.temperature.dtype == torch.float32
    vt, vd = _valid_rows(w)
    assert torch.isfinite(w.target[vt].float()).all() and torch.isfinite(w.draft[vd].float()).all()
    assert torch.isnan(w.target[~vt].float()).all() and torch.isnan(w.draft[~vd].float()).all()
    x = w.draft_tokens
    assert ((x[vd] >= 0) & (x[vd] < V)).all() and (x[~vd] == -1).all()
    L = w.draft_len
    if k == 5:
        assert ((L >= 1) & (L <= 7)).all()
        assert ((w.temperature >= 0.3) & (w.temperature <= 1.3)).all()
    else:
        assert (L == n).all()
        assert torch.allclose(w.temperature, torch.full((B,), {1: 1.0, 2: 0.7, 3: 1.0, 4: 0.0}[k]))
    if k == 3:
        assert w.mtp_tokens.shape == (B * (n + 1),) and w.hidden.shape == (B * (n + 1), 7168)


def test_config4_drafts_are_the_draft_argmax_and_mostly_the_target_argmax():
    w = make_config(4, B=8)
    d_arg = w.draft.float().argmax(dim=-1)
    assert torch.equal(d_arg.to(torch.int32), w.draft_tokens)
    t_arg = w.target[:, : w.n_max].float().argmax(dim=-1).to(torch.int32)
    frac = (t_arg == w.draft_tokens).float().mean().item()
    assert 0.5 < frac < 0.95  # the recipe: top-1 with probability 0.75, else the second best


def test_config_is_seeded_and_repeatable():
    a = make_config(2, B=3)
    b = make_config(2, B=3)
    assert torch.equal(a.target, b.target) and torch.equal(a.draft_tokens, b.draft_tokens)


def test_algorithmic_bytes_counts_valid_rows_once():
    w = make_config(5, B=5)
    vt, vd = _valid_rows(w)
    sampled = (w.temperature > 0).view(-1, 1)
    rows = int(vt.sum()) + int((vd & sampled).sum())
    assert algorithmic_bytes(w) == rows * w.V * 2
    g = make_config(4, B=5)  # greedy: target rows only
    assert algorithmic_bytes(g) == 5 * (g.n_max + 1) * g.V * 2


def test_pack_round_trips_the_valid_rows():
    w = make_random(7, 4, 300, dtype="f32", seed=2, temperatures=(0.5, 0.0), ragged=True)
    t, d, x, cu = pack(w)
    L = w.draft_len.tolist()
    assert cu.tolist() == list(np.cumsum([0] + [n + 1 for n in L]))
    assert t.shape == (sum(L) + w.B, w.V) and d.shape == (sum(L), w.V) and x.shape == (sum(L),)
    dense = unpack_rows(t, cu, w.n_max, float("nan"))
    vt, vd = _valid_rows(w)
    assert torch.equal(dense[vt], w.target[vt])
    for b in range(w.B):
        s = int(cu[b]) - b  # draft rows and tokens of request b start here
        assert torch.equal(d[s: s + L[b]], w.draft[b, : L[b]])
        assert torch.equal(x[s: s + L[b]], w.draft_tokens[b, : L[b]])
