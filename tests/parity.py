"""Helpers shared by the GPU parity tests: run the CPU oracle on (a sample of)
a workload and compare the CUDA path's outputs with it.

Tolerances (from the verify step's definition of parity):
  * accepted_len and every emitted token bit-exact, except requests whose
    oracle decision margin is below 1e-5 relative (|u - min(1, p/q)| / u on a
    scored row, or the race's top-2 key gap); such near-tie rows are counted
    and must be at most 1e-4 of all rows (at least one allowed per case);
  * per-row log-sum-exp within 1e-5 * max(|LSE|, 1).
"""
from __future__ import annotations

import concurrent.futures
import os

import numpy as np
import torch

import oracle
from workloads.gen import logits_numpy

NEAR_TIE = 1e-5
LSE_TOL = 1e-5


def wait_gpu(timeout_s: float = 120.0):
    """Wait for the current stream like torch.cuda.synchronize(), but fail the
    test instead of blocking forever if the device does not finish."""
    import time

    ev = torch.cuda.Event()
    ev.record()
    t0 = time.monotonic()
    while not ev.query():
        if time.monotonic() - t0 > timeout_s:
            raise TimeoutError(f"GPU work did not finish within {timeout_s} s")
        time.sleep(0.001)
    torch.cuda.synchronize()


def _host(t):
    return None if t is None else t.detach().cpu()


def oracle_on(w, req=None, threads=None, want_lse=True, pos_off=None):
    """Oracle outputs for requests `req` (indices into the batch; None = all).

    Only the selected requests' rows are copied to the host.  Work is split
    across threads (the C oracle runs without the GIL).  pos_off: optional
    [B] position offsets of the random counter's row word."""
    B = w.B
    idx = np.arange(B) if req is None else np.asarray(sorted(req))
    ti = torch.as_tensor(idx, device=w.target.device)
    t = logits_numpy(w.target.index_select(0, ti))
    d = None if w.draft is None else logits_numpy(w.draft.index_select(0, ti))
    x = _host(w.draft_tokens).numpy()[idx]
    L = _host(w.draft_len).numpy()[idx]
    T = _host(w.temperature).numpy()[idx]
    po = None if pos_off is None else np.asarray(_host(pos_off) if hasattr(pos_off, "cpu") else pos_off,
                                                  dtype=np.int32)[idx]
    n = len(idx)
    threads = threads or min(16, os.cpu_count() or 1, max(1, n))
    parts = np.array_split(np.arange(n), threads)

    def run(p):
        if len(p) == 0:
            return None
        sl = slice(p[0], p[-1] + 1)
        r = oracle.spec_verify(t[sl], None if d is None else d[sl], x[sl], L[sl], T[sl], w.seed,
                               req_ids=idx[sl].astype(np.int32),
                               pos_off=None if po is None else po[sl])
        if want_lse:
            r["row_lse_all"] = oracle.row_lse_all(t[sl], None if d is None else d[sl], L[sl], T[sl])
        return r

    with concurrent.futures.ThreadPoolExecutor(max_workers=threads) as ex:
        outs = [o for o in ex.map(run, parts) if o is not None]
    res = {"req": idx, "err": 0}
    for key in ("accepted_len", "out_tokens", "accept_margin", "race_gap", "row_lse_all"):
        if key in outs[0]:
            res[key] = np.concatenate([o[key] for o in outs], axis=0)
    for o in outs:
        res["err"] |= o["err"]
    return res


def compare(w, acc_gpu, out_gpu, ref, row_lse_gpu=None, label=""):
    """Assert parity of the CUDA outputs with the oracle's on ref['req']."""
    idx = ref["req"]
    acc = _host(acc_gpu).numpy()[idx]
    out = _host(out_gpu).numpy()[idx]
    L = _host(w.draft_len).numpy()[idx]
    margin = ref["accept_margin"]
    gap = ref["race_gap"]
    near_rows = np.zeros(len(idx), dtype=np.int64)
    for i in range(len(idx)):
        m = margin[i][~np.isnan(margin[i])]
        near_rows[i] = int((m < NEAR_TIE).sum()) + int(np.isfinite(gap[i]) and gap[i] < NEAR_TIE)
    mism = np.where((acc != ref["accepted_len"]) | (out != ref["out_tokens"]).any(axis=1))[0]
    # a request may differ only where the oracle itself found a near tie
    unexplained = [int(idx[i]) for i in mism if near_rows[i] == 0]
    total_rows = int((L + 1).sum())
    n_near = int(near_rows.sum())
    assert not unexplained, (
        f"{label}: {len(unexplained)} requests differ from the oracle without a near tie, "
        f"e.g. b={unexplained[:5]}: gpu acc={acc[np.isin(idx, unexplained[:5])]}, "
        f"oracle acc={ref['accepted_len'][np.isin(idx, unexplained[:5])]}")
    # A case may hold more near-tie rows than 1e-4 of its rows only when it is
    # small: at most one then (rows whose decision margin is below 1e-5, so
    # the fp32 kernel and the fp64 oracle may decide them differently).
    assert n_near <= max(1, int(1e-4 * total_rows)), f"{label}: {n_near} near-tie rows"
    stats = {"requests": len(idx), "mismatch": len(mism), "near_tie_rows": n_near,
             "rows": total_rows}
    if row_lse_gpu is not None and "row_lse_all" in ref:
        got = _host(row_lse_gpu).double().numpy()[idx]
        exp = ref["row_lse_all"]
        mask = ~np.isnan(exp)
        assert not np.isnan(got[mask]).any(), f"{label}: a scored row has no LSE"
        err = np.abs(got[mask] - exp[mask]) / np.maximum(np.abs(exp[mask]), 1.0)
        stats["lse_max_rel_err"] = float(err.max()) if err.size else 0.0
        assert stats["lse_max_rel_err"] <= LSE_TOL, f"{label}: LSE error {stats['lse_max_rel_err']}"
    return stats
