"""An fp64 numpy restatement of the three per-shard calls of the
vocabulary-sharded verify step, with its exchange records held in float64,
for CPU tests of the exchange between ranks (test infrastructure; the random
numbers come from the oracle's Philox).

It follows the decomposition the GPU calls use: per row and shard the
statistics (K = c max x, S = sum 2^(c x - K), the logit at the draft token;
greedy rows: the max and its first global index), merged over shards into
P = K + log2 S; the acceptance tests u_j < p_j(x_j) / q_j(x_j); per shard
the best race keys r_v / E_v over the shard's entries (global index v), on
r = max(0, p - q) or p for the bonus row, and on p as the fallback; the best
key over shards wins, the lower index on a tie.
"""
import math

import numpy as np
import torch

import oracle

LOG2E = 1.0 / math.log(2.0)
ERR_TOKEN, ERR_DRAFT_LEN, ERR_TEMPERATURE = 1, 2, 4


def _req(T, L_raw, n_max, has_draft):
    L = min(max(int(L_raw), 0), n_max)
    T = float(T)
    greedy = (not T > 0.0) or T < 1e-6 or (not has_draft and L > 0)
    err = (ERR_DRAFT_LEN if L != int(L_raw) else 0) | (ERR_TEMPERATURE if greedy and T != 0.0 else 0)
    return L, T, greedy, err


def _merge(recs):
    """P and the draft-token logit from one row's records of every shard."""
    K = max(r[0] for r in recs)
    S = sum(r[1] * 2.0 ** (r[0] - K) for r in recs if r[1] > 0.0)
    xl = next((r[2] for r in recs if r[3] != 0.0), 0.0)
    return K + math.log2(S), xl


def _better(key, idx, best):
    return key > best[0] or (key == best[0] and idx < best[1])


class NumpyShardOps:
    def stats_buffer(self, B, n_max, device=None):
        return torch.zeros(B * (n_max + 1) * 2, 4, dtype=torch.float64)

    def race_buffer(self, B, device=None):
        return torch.zeros(B, 4, dtype=torch.float64)

    def stats(self, target, draft, V, v0, draft_tokens, draft_len, temperature, out, stream=None):
        t = target.double().numpy()
        d = None if draft is None else draft.double().numpy()
        x = draft_tokens.numpy()
        B, rows, Vs = t.shape
        o = out.numpy()
        for b in range(B):
            L, T, greedy, _ = _req(temperature[b], draft_len[b], rows - 1, d is not None)
            for j in range(L + 1):
                rec = (b * rows + j) * 2
                if greedy:
                    k = int(np.argmax(t[b, j]))  # the first index holding the maximum
                    o[rec] = (t[b, j, k], v0 + k, 0.0, 0.0)
                    continue
                c = LOG2E / T
                for tensor, row in ((0, t[b, j]), (1, None if j >= L else d[b, j])):
                    if row is None:
                        continue
                    K = c * row.max()
                    S = float(np.sum(2.0 ** (c * row - K)))
                    tok = int(x[b, j]) if j < L else -1
                    has = v0 <= tok < v0 + Vs
                    o[rec + tensor] = (K, S, row[tok - v0] if has else 0.0, 1.0 if has else 0.0)

    def race(self, target, draft, V, v0, draft_tokens, draft_len, temperature, seed, stats_all, accepted_len, out,
             error_word=None, stream=None):
        t = target.double().numpy()
        d = None if draft is None else draft.double().numpy()
        x = draft_tokens.numpy()
        st = stats_all.numpy()
        B, rows, Vs = t.shape
        o = out.numpy()
        err_all = 0
        for b in range(B):
            L, T, greedy, err = _req(temperature[b], draft_len[b], rows - 1, d is not None)
            a, tok = L, -1
            for j in range(L + 1):
                rec = (b * rows + j) * 2
                if greedy:
                    M, idx = -math.inf, -1
                    for s in range(st.shape[0]):  # shards in vocabulary order
                        if idx < 0 or st[s, rec, 0] > M:
                            M, idx = st[s, rec, 0], int(st[s, rec, 1])
                    if j == L:
                        tok = idx
                        break
                    if not 0 <= x[b, j] < V:
                        err |= ERR_TOKEN
                    if x[b, j] != idx:
                        a, tok = j, idx
                        break
                    continue
                if j == L:
                    break
                c = LOG2E / T
                Pt, xt = _merge(st[:, rec])
                Pd, xd = _merge(st[:, rec + 1])
                if not 0 <= x[b, j] < V:
                    err |= ERR_TOKEN
                    a = j
                    break
                ratio = 2.0 ** ((c * xt - Pt) - (c * xd - Pd))
                if not oracle.uniform(oracle.draw(seed, b, j, 0, 0)) < ratio:
                    a = j
                    break
            accepted_len[b] = a
            err_all |= err
            if greedy:
                o[b] = (math.inf, tok, math.inf, tok)
                continue
            c = LOG2E / T
            residual = a < L
            rec = (b * rows + a) * 2
            Pt, _ = _merge(st[:, rec])
            Pd = _merge(st[:, rec + 1])[0] if residual else 0.0
            best_r, best_p = (0.0, -1), (0.0, -1)
            for vl in range(Vs):
                v = v0 + vl
                p = 2.0 ** (c * t[b, a, vl] - Pt)
                r = p - 2.0 ** (c * d[b, a, vl] - Pd) if residual else p
                E = -math.log(oracle.uniform(oracle.draw(seed, b, a, v, 1)))
                if r > 0.0 and _better(r / E, v, best_r):
                    best_r = (r / E, v)
                if residual and p > 0.0 and _better(p / E, v, best_p):
                    best_p = (p / E, v)
            o[b] = (best_r[0], best_r[1], best_p[0], best_p[1])
        if error_word is not None:
            error_word[0] = int(error_word[0]) | err_all

    def finish(self, race_all, draft_tokens, accepted_len, out_tokens, stream=None):
        ra = race_all.numpy()
        x = draft_tokens.numpy()
        B, rows = out_tokens.shape
        for b in range(B):
            best_r, best_p = (0.0, -1), (0.0, -1)
            for s in range(ra.shape[0]):
                kr, ir, kp, ip = ra[s, b]
                if ir >= 0 and _better(kr, int(ir), best_r):
                    best_r = (kr, int(ir))
                if ip >= 0 and _better(kp, int(ip), best_p):
                    best_p = (kp, int(ip))
            y = best_r[1] if best_r[1] >= 0 else best_p[1]  # all residual weights vanished: race on p
            a = int(accepted_len[b])
            out_tokens[b] = torch.tensor([int(x[b, k]) if k < a else (y if k == a else -1) for k in range(rows)],
                                         dtype=torch.int32)
