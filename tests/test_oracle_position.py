"""Pins of the oracle's position offset (CPU only).

With a position offset o, row j of a request draws its random numbers at row
coordinate o + j.  The pin is an invariant that holds only if every draw of
the request (the acceptance tests, the residual race and the bonus race)
moves with the offset: a request whose row 0 is always accepted (its draft
distribution equals the target's, so p(x)/q(x) = 1 > u for any u < 1) behaves
from row 1 on exactly like the same request with row 0 removed and offset 1.
The accepted length then grows by one and the emitted tokens gain x_0 in
front.  Dropping the offset, applying it with the wrong sign, or applying it
to only some of the draws breaks the equality on most seeds.
"""
import numpy as np
import pytest

import oracle


def _request(rng, n, V, sigma, noise):
    t = rng.normal(0.0, sigma, size=(n + 1, V)).astype(np.float32)
    d = (t[:n] + rng.normal(0.0, noise, size=(n, V))).astype(np.float32)
    d[0] = t[0]  # row 0: identical distributions, always accepted
    x = np.empty(n, dtype=np.int32)
    for j in range(n):
        q = np.exp(d[j].astype(np.float64) - d[j].max())
        x[j] = rng.choice(V, p=q / q.sum())
    return t, d, x


@pytest.mark.parametrize("T", [0.7, 1.0, 1.6])
def test_offset_moves_every_draw(T):
    rng = np.random.default_rng(int(T * 1000))
    n, V, trials = 4, 64, 60
    outcomes = set()
    for k in range(trials):
        t, d, x = _request(rng, n, V, sigma=2.0, noise=1.5)
        seed = 1000 + k
        b = 7  # same request coordinate on both sides
        full = oracle.spec_verify(t[None], d[None], x[None], np.array([n]), np.array([T], np.float32),
                                  seed, req_ids=np.array([b]), pos_off=np.array([0]), want_stats=False)
        tail = oracle.spec_verify(t[None, 1:], d[None, 1:], x[None, 1:], np.array([n - 1]),
                                  np.array([T], np.float32), seed, req_ids=np.array([b]),
                                  pos_off=np.array([1]), want_stats=False)
        a_full, a_tail = int(full["accepted_len"][0]), int(tail["accepted_len"][0])
        assert a_full >= 1  # row 0 always passes
        assert a_full == a_tail + 1
        assert full["out_tokens"][0, 0] == x[0]
        assert list(full["out_tokens"][0, 1:]) == list(tail["out_tokens"][0])
        outcomes.add(a_tail)
    # both a residual race (a_tail < n-1) and the bonus race (a_tail = n-1) ran
    assert min(outcomes) < n - 1 and max(outcomes) == n - 1


def test_offset_zero_is_the_default_and_offsets_change_draws():
    rng = np.random.default_rng(5)
    n, V, B = 3, 48, 64
    t = rng.normal(0.0, 2.0, size=(B, n + 1, V)).astype(np.float32)
    d = (t[:, :n] + rng.normal(0.0, 1.5, size=(B, n, V))).astype(np.float32)
    x = rng.integers(0, V, size=(B, n)).astype(np.int32)
    L = np.full(B, n, np.int32)
    T = np.full(B, 1.0, np.float32)
    plain = oracle.spec_verify(t, d, x, L, T, 3, want_stats=False)
    zero = oracle.spec_verify(t, d, x, L, T, 3, pos_off=np.zeros(B, np.int32), want_stats=False)
    moved = oracle.spec_verify(t, d, x, L, T, 3, pos_off=np.full(B, 1000, np.int32), want_stats=False)
    assert np.array_equal(plain["accepted_len"], zero["accepted_len"])
    assert np.array_equal(plain["out_tokens"], zero["out_tokens"])
    assert not np.array_equal(plain["out_tokens"], moved["out_tokens"])
