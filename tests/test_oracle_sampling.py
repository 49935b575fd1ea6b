"""Pins of the oracle's verify/accept step (CPU only).

Each test ties the oracle to something other than itself:
  * the greedy branch to a numpy argmax restatement (T = 0 accepts while the
    draft token is the target's top token and then emits that top token);
  * identical draft and target distributions to "always accept every draft";
  * output lengths to 1 <= a+1 <= n+1 with the accepted prefix equal to the
    drafts;
  * the whole stochastic rule to the target's exact autoregressive
    distribution, by brute-force enumeration over every sequence at V <= 8,
    n <= 3, with a chi-square test over 10^6 trials;
  * the law of (accepted length, emitted token) for fixed drafts to its closed
    form prod_j min(1, p/q) times the residual or bonus distribution;
  * the exponential race to "winner frequency = r_i / sum r";
  * row log-sum-exp to scipy.special.logsumexp and to the closed form for a
    constant row.
Sources: "Accelerating Sonar through speculation", §Speculative decoding
(stages Acceptance and Target generation) and §Target-draft; the acceptance
rule of "Fast Inference from Transformers via Speculative Decoding".
"""
import itertools

import numpy as np
import pytest
from scipy import special, stats

import oracle


def _softmax(z):
    z = np.asarray(z, dtype=np.float64)
    m = z.max(axis=-1, keepdims=True)
    e = np.exp(z - m)
    return e / e.sum(axis=-1, keepdims=True)


def _chi2_pvalue(obs, exp, min_expected=5.0):
    obs = np.asarray(obs, dtype=np.float64)
    exp = np.asarray(exp, dtype=np.float64)
    zero = exp == 0.0
    assert (obs[zero] == 0).all(), "an outcome of probability zero occurred"
    obs, exp = obs[~zero], exp[~zero]
    small = exp < min_expected
    if small.any():
        obs = np.concatenate([obs[~small], [obs[small].sum()]])
        exp = np.concatenate([exp[~small], [exp[small].sum()]])
    assert abs(obs.sum() - exp.sum()) < 1e-6 * exp.sum()
    return stats.chisquare(obs, exp).pvalue


def _random_batch(rng, B, n, V, T, dtype=np.float32, ragged=False):
    t = (rng.normal(0, 2.0, size=(B, n + 1, V))).astype(np.float32)
    d = (t[:, :n] + rng.normal(0, 1.0, size=(B, n, V))).astype(np.float32)
    L = rng.integers(0, n + 1, size=B).astype(np.int32) if ragged else np.full(B, n, np.int32)
    x = np.zeros((B, n), np.int32)
    for b in range(B):
        for j in range(n):
            if T[b] > 0:
                x[b, j] = rng.choice(V, p=_softmax(d[b, j] / T[b]))
            else:
                x[b, j] = int(np.argmax(d[b, j]))
    if dtype == np.uint16:  # round to bf16 (RNE) and pass the raw bits
        def to_bf16(a):
            u = a.view(np.uint32).astype(np.uint64)
            r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
            return r
        return to_bf16(t), to_bf16(d), x, L
    return t, d, x, L


def _as_f64(a):
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


# ---------------------------------------------------------------- (a) greedy
@pytest.mark.parametrize("dtype", [np.float32, np.uint16])
def test_greedy_matches_numpy_restatement(dtype):
    rng = np.random.default_rng(1)
    B, n, V = 200, 4, 37
    T = np.zeros(B, np.float32)
    t, d, x, L = _random_batch(rng, B, n, V, T, dtype=dtype, ragged=True)
    tf = _as_f64(t)
    # make half of the drafts the target's argmax so that long prefixes occur
    for b in range(B):
        for j in range(n):
            if rng.random() < 0.7:
                x[b, j] = int(np.argmax(tf[b, j]))
    # exact ties: the lowest index must win
    tf_tie = t.copy()
    tf_tie[0, 0, 5] = tf_tie[0, 0].max()
    tf_tie[0, 0, 9] = tf_tie[0, 0, 5]
    t = tf_tie
    tf = _as_f64(t)
    res = oracle.spec_verify(t, d, x, L, T, seed=3)
    for b in range(B):
        a_ref, y_ref = L[b], int(np.argmax(tf[b, L[b]]))
        for j in range(L[b]):
            g = int(np.argmax(tf[b, j]))  # numpy: first index of the maximum
            if x[b, j] != g:
                a_ref, y_ref = j, g
                break
        assert res["accepted_len"][b] == a_ref
        assert res["out_tokens"][b, a_ref] == y_ref
    assert res["err"] == 0


def test_greedy_needs_no_draft_logits():
    rng = np.random.default_rng(2)
    t, d, x, L = _random_batch(rng, 8, 3, 11, np.zeros(8, np.float32))
    a = oracle.spec_verify(t, d, x, L, np.zeros(8, np.float32), seed=0)
    b = oracle.spec_verify(t, None, x, L, np.zeros(8, np.float32), seed=0)
    assert (a["accepted_len"] == b["accepted_len"]).all()
    assert (a["out_tokens"] == b["out_tokens"]).all()


# ------------------------------------------------------ (b) identical rows
@pytest.mark.parametrize("T", [0.3, 1.0, 2.5])
@pytest.mark.parametrize("dtype", [np.float32, np.uint16])
def test_identical_distributions_accept_everything(T, dtype):
    rng = np.random.default_rng(4)
    B, n, V = 300, 5, 50
    t, _, x, L = _random_batch(rng, B, n, V, np.full(B, T, np.float32), dtype=dtype)
    d = np.ascontiguousarray(t[:, :n])
    for seed in (0, 1, 2**40 + 3):
        res = oracle.spec_verify(t, d, x, L, np.full(B, T, np.float32), seed=seed)
        assert (res["accepted_len"] == n).all()
        assert (res["out_tokens"][:, :n] == x).all()
        assert (res["out_tokens"][:, n] >= 0).all()


# ----------------------------------------------------------- (c) lengths
def test_output_length_bounds_and_prefix():
    rng = np.random.default_rng(5)
    B, n, V = 400, 6, 23
    T = rng.choice([0.0, 0.4, 1.0, 1.7], size=B).astype(np.float32)
    t, d, x, L = _random_batch(rng, B, n, V, T, ragged=True)
    res = oracle.spec_verify(t, d, x, L, T, seed=9)
    a, out = res["accepted_len"], res["out_tokens"]
    assert ((0 <= a) & (a <= L)).all()
    for b in range(B):
        assert (out[b, : a[b]] == x[b, : a[b]]).all()
        assert 0 <= out[b, a[b]] < V
        assert (out[b, a[b] + 1:] == -1).all()
    assert res["err"] == 0


def test_replacement_token_lies_in_residual_support():
    # On a rejection the emitted token y must satisfy p(y) > q(y).
    rng = np.random.default_rng(6)
    B, n, V = 300, 3, 13
    T = np.full(B, 0.8, np.float32)
    t, d, x, L = _random_batch(rng, B, n, V, T)
    res = oracle.spec_verify(t, d, x, L, T, seed=1)
    rej = 0
    for b in range(B):
        a = res["accepted_len"][b]
        if a < L[b]:
            rej += 1
            p = _softmax(t[b, a].astype(np.float64) / T[b])
            q = _softmax(d[b, a].astype(np.float64) / T[b])
            y = res["out_tokens"][b, a]
            assert p[y] > q[y]
    assert rej > 50


# ---------------------------------------------------------------- LSE
def test_row_lse_matches_scipy_and_closed_form():
    rng = np.random.default_rng(7)
    B, n, V = 20, 2, 300
    T = np.array([0.5, 1.0, 1.3, 2.0] * 5, np.float32)
    t, d, x, L = _random_batch(rng, B, n, V, T)
    lse = oracle.row_lse_all(t, d, L, T)
    for b in range(B):
        s = 1.0 / np.float64(T[b])
        for j in range(n + 1):
            ref = special.logsumexp(s * t[b, j].astype(np.float64))
            assert abs(lse[b, j, 0] - ref) <= 1e-12 * max(1.0, abs(ref))
            if j < n:
                ref = special.logsumexp(s * d[b, j].astype(np.float64))
                assert abs(lse[b, j, 1] - ref) <= 1e-12 * max(1.0, abs(ref))
    # constant row c: LSE(s c) = s c + ln V exactly (up to rounding)
    c = np.full((1, 1, 1000), 3.25, np.float32)
    lse = oracle.row_lse_all(c, np.zeros((1, 0, 1000), np.float32), np.zeros(1, np.int32),
                             np.array([0.5], np.float32))
    assert abs(lse[0, 0, 0] - (6.5 + np.log(1000.0))) < 1e-12


# --------------------------------------------- (d) autoregressive chi-square
def _ar_tables(rng, V, n):
    tgt = [rng.normal(0, 1.5, size=(V ** k, V)).astype(np.float32) for k in range(n + 1)]
    drf = [(tgt[k] + rng.normal(0, 1.0, size=tgt[k].shape)).astype(np.float32) for k in range(n)]
    return tgt, drf


def _sample_categorical(rng, probs):
    u = rng.random(probs.shape[0])
    c = np.cumsum(probs, axis=1)
    return np.minimum((c < u[:, None]).sum(axis=1), probs.shape[1] - 1)


@pytest.mark.parametrize("V,n,T", [(6, 3, 1.0), (8, 2, 0.6), (4, 3, 1.4)])
def test_emitted_sequence_law_equals_target_autoregressive_law(V, n, T):
    """North-star pin (d): drafts drawn from q, verify, then complete the
    sequence to n+1 tokens from the exact p tables; the law of the n+1 tokens
    must be the target's autoregressive product, whatever q is."""
    rng = np.random.default_rng(1000 + V * 10 + n)
    tgt, drf = _ar_tables(rng, V, n)
    N, chunk = 1_000_000, 250_000
    counts = np.zeros(V ** (n + 1), np.int64)
    for c0 in range(0, N, chunk):
        m = min(chunk, N - c0)
        pid = np.zeros(m, np.int64)
        pids = [pid]
        x = np.zeros((m, n), np.int32)
        for k in range(n):
            q = _softmax(drf[k][pid].astype(np.float64) / T)
            x[:, k] = _sample_categorical(rng, q)
            pid = pid * V + x[:, k]
            pids.append(pid)
        t_rows = np.stack([tgt[k][pids[k]] for k in range(n + 1)], axis=1)
        d_rows = np.stack([drf[k][pids[k]] for k in range(n)], axis=1)
        res = oracle.spec_verify(t_rows, d_rows, x, np.full(m, n, np.int32),
                                 np.full(m, T, np.float32), seed=77,
                                 req_ids=np.arange(c0, c0 + m, dtype=np.int32), want_stats=False)
        a, out = res["accepted_len"], res["out_tokens"]
        seq = out.astype(np.int64).copy()
        # complete positions a+1..n from the exact target conditionals
        for k in range(1, n + 1):
            need = a + 1 <= k
            if need.any():
                pid_k = np.zeros(m, np.int64)
                for i in range(k):
                    pid_k = pid_k * V + seq[:, i]
                p = _softmax(tgt[k][pid_k[need]].astype(np.float64) / T)
                seq[need, k] = _sample_categorical(rng, p)
        code = np.zeros(m, np.int64)
        for k in range(n + 1):
            code = code * V + seq[:, k]
        counts += np.bincount(code, minlength=V ** (n + 1))
    # exact law by enumeration
    expected = np.zeros(V ** (n + 1))
    for cell, s in enumerate(itertools.product(range(V), repeat=n + 1)):
        pr, pid = 1.0, 0
        for k in range(n + 1):
            pr *= _softmax(tgt[k][pid].astype(np.float64) / T)[s[k]]
            pid = pid * V + s[k]
        expected[cell] = pr
    assert abs(expected.sum() - 1) < 1e-9
    pval = _chi2_pvalue(counts, expected * N)
    assert pval > 1e-3, pval


def test_autoregressive_pin_detects_a_wrong_rule():
    """The chi-square above has power: sampling the emitted token from q
    (a plausible mistake) is rejected on the same tables."""
    rng = np.random.default_rng(3)
    V, n, T, N = 6, 1, 1.0, 200_000
    tgt, drf = _ar_tables(rng, V, n)
    # simulate "always accept the draft and emit a bonus from p": law q(x0) p(x1|x0)
    q0 = _softmax(drf[0][0] / T)
    x0 = _sample_categorical(rng, np.broadcast_to(q0, (N, V)))
    p1 = _softmax(tgt[1][x0].astype(np.float64) / T)
    x1 = _sample_categorical(rng, p1)
    counts = np.bincount(x0 * V + x1, minlength=V * V)
    p0 = _softmax(tgt[0][0] / T)
    expected = np.array([p0[s0] * _softmax(tgt[1][s0] / T)[s1] for s0 in range(V) for s1 in range(V)])
    assert _chi2_pvalue(counts, expected * N) < 1e-6


# ------------------------------------------ closed-form law of (a, y)
@pytest.mark.parametrize("dtype", [np.float32, np.uint16])
def test_outcome_law_for_fixed_drafts(dtype):
    rng = np.random.default_rng(11)
    V, n, T, N, chunk = 7, 3, 0.9, 1_000_000, 250_000
    t1, d1, _, _ = _random_batch(rng, 1, n, V, np.full(1, T, np.float32), dtype=dtype)
    x1 = np.array([[2, 5, 0]], np.int32)
    tf, df = _as_f64(t1)[0], _as_f64(d1)[0]
    s = 1.0 / np.float64(np.float32(T))
    p = _softmax(tf * s)
    q = _softmax(df * s)
    law = np.zeros((n + 1, V))
    alive = 1.0
    for j in range(n):
        acc = min(1.0, p[j, x1[0, j]] / q[j, x1[0, j]])
        res = np.maximum(p[j] - q[j], 0.0)
        law[j] = alive * (1 - acc) * res / res.sum()
        alive *= acc
    law[n] = alive * p[n]
    assert abs(law.sum() - 1) < 1e-12
    counts = np.zeros((n + 1) * V, np.int64)
    for c0 in range(0, N, chunk):
        m = min(chunk, N - c0)
        t = np.ascontiguousarray(np.broadcast_to(t1, (m,) + t1.shape[1:]))
        d = np.ascontiguousarray(np.broadcast_to(d1, (m,) + d1.shape[1:]))
        x = np.ascontiguousarray(np.broadcast_to(x1, (m, n)))
        r = oracle.spec_verify(t, d, x, np.full(m, n, np.int32), np.full(m, T, np.float32),
                               seed=2024, req_ids=np.arange(c0, c0 + m, dtype=np.int32),
                               want_stats=False)
        a = r["accepted_len"].astype(np.int64)
        y = r["out_tokens"][np.arange(m), a].astype(np.int64)
        counts += np.bincount(a * V + y, minlength=(n + 1) * V)
    pval = _chi2_pvalue(counts, law.ravel() * N)
    assert pval > 1e-3, pval


# ------------------------------------------------------------- race
def test_exponential_race_frequencies():
    r = np.array([0.1, 0.0, 0.35, 0.05, 0.5, 1e-3, 0.0, 0.2])
    N = 200_000
    counts = np.zeros(r.size, np.int64)
    for b in range(N):
        y, _ = oracle.race(r, seed=5, b=b, j=3)
        counts[y] += 1
    assert counts[1] == 0 and counts[6] == 0  # zero weight never wins
    pos = r > 0
    pval = _chi2_pvalue(counts[pos], r[pos] / r.sum() * N)
    assert pval > 1e-3, pval


def test_bonus_token_follows_target_distribution():
    # n = 0: the step is plain sampling of the target's row 0.
    rng = np.random.default_rng(12)
    V, N, T = 9, 400_000, 0.75
    row = rng.normal(0, 1.2, size=(1, 1, V)).astype(np.float32)
    t = np.ascontiguousarray(np.broadcast_to(row, (N, 1, V)))
    res = oracle.spec_verify(t, np.zeros((N, 0, V), np.float32), np.zeros((N, 0), np.int32),
                             np.zeros(N, np.int32), np.full(N, T, np.float32), seed=8,
                             want_stats=False)
    assert (res["accepted_len"] == 0).all()
    counts = np.bincount(res["out_tokens"][:, 0], minlength=V)
    p = _softmax(row[0, 0].astype(np.float64) / np.float64(np.float32(T)))
    assert _chi2_pvalue(counts, p * N) > 1e-3


def test_no_drafts_needs_no_draft_logits():
    # A request without drafts samples its only token from the target row:
    # no draft logits enter, so none need be given, and nothing is flagged.
    # Requests that do have drafts still need them: without, they fall back
    # to greedy and set the temperature bit.
    rng = np.random.default_rng(14)
    V, N, T = 7, 300_000, 1.3
    row = rng.normal(0, 1.0, size=(1, 1, V)).astype(np.float32)
    t = np.ascontiguousarray(np.broadcast_to(row, (N, 1, V)))
    res = oracle.spec_verify(t, None, np.zeros((N, 0), np.int32), np.zeros(N, np.int32),
                             np.full(N, T, np.float32), seed=21, want_stats=False)
    assert res["err"] == 0 and (res["accepted_len"] == 0).all()
    counts = np.bincount(res["out_tokens"][:, 0], minlength=V)
    p = _softmax(row[0, 0].astype(np.float64) / np.float64(np.float32(T)))
    assert _chi2_pvalue(counts, p * N) > 1e-3

    t2, d2, x2, L2 = _random_batch(rng, 6, 2, 12, np.full(6, 0.9, np.float32))
    L2[:3] = 0
    T2 = np.full(6, 0.9, np.float32)
    r = oracle.spec_verify(t2, None, x2, L2, T2, seed=3, want_stats=False)
    assert r["err"] == oracle.ERR_TEMPERATURE
    g = oracle.spec_verify(t2[3:], None, x2[3:], L2[3:], np.zeros(3, np.float32), seed=3, want_stats=False)
    assert (r["accepted_len"][3:] == g["accepted_len"]).all()
    assert (r["out_tokens"][3:] == g["out_tokens"]).all()
    # the first three sampled from p: with any draft tensor given, the same draws
    w = oracle.spec_verify(t2, d2, x2, L2, T2, seed=3, want_stats=False)
    assert (r["out_tokens"][:3] == w["out_tokens"][:3]).all()


# ----------------------------------------------------- invalid device data
def test_invalid_inputs_set_error_bits_and_stay_defined():
    rng = np.random.default_rng(13)
    B, n, V = 6, 3, 10
    T = np.array([1.0, 1.0, -1.0, np.nan, 1e-9, 1.0], np.float32)
    t, d, x, L = _random_batch(rng, B, n, V, np.where(np.isfinite(T) & (T > 0), T, 0).astype(np.float32))
    x[0, 0] = V + 3  # out-of-range token rejects row 0
    L[1] = n + 2  # clamped to n
    res = oracle.spec_verify(t, d, x, L, T, seed=1)
    assert res["err"] == oracle.ERR_TOKEN | oracle.ERR_DRAFT_LEN | oracle.ERR_TEMPERATURE
    assert res["accepted_len"][0] == 0
    assert 0 <= res["accepted_len"][1] <= n
    # negative / NaN / tiny T behave as greedy
    g = oracle.spec_verify(t[2:5], d[2:5], x[2:5], L[2:5], np.zeros(3, np.float32), seed=1)
    assert (res["accepted_len"][2:5] == g["accepted_len"]).all()
    assert (res["out_tokens"][2:5] == g["out_tokens"]).all()
