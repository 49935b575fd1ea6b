"""Seeded generators for the five synthetic workloads and for random test shapes.

Every tensor comes from ``torch.Generator(device).manual_seed(...)``; the same
(config, seed, device) always gives the same tensors.  The CPU and CUDA
generators are different streams, so a test draws once on one device and
copies to the other.

Workloads (logits layout: target [B, n_max+1, V], draft [B, n_max, V],
row-major, contiguous V):

1. tiny:      B=4, n=3, V=1024, fp32; t ~ N(0, 2^2); d = t + N(0, 0.5^2);
              T = 1; drafts drawn from softmax(d/T).
2. linear:    B=64, n=4, V=128256, bf16; t ~ N(0, 3^2) plus +8 at one seeded
              index per row; d = bf16(t + N(0, 1)); T = 0.7; drafts drawn
              from softmax(d/T).
3. mtp:       B=256, n=1, V=129280, bf16, logits as in 2; T = 1; plus MTP
              buffers: tokens int32 [512] uniform in [0, V), hidden bf16
              [512, 7168] ~ N(0, 1).
4. greedy:    B=512, n=4, V=128256, bf16, t as in 2; T = 0; draft token is
              the target argmax with probability 0.75, else the second-best
              index; draft logits are nudged so their argmax is that token.
5. ragged:    B=1024, n_b ~ U{1..7}, n_max=7, V=152064, bf16;
              t ~ N(0, 3^2) + bias_v, bias_v = -1.1 ln(v + 1) (softmax of the
              bias alone is Zipf(1.1) over rank v + 1); d = t + N(0, 0.8^2);
              T_b ~ U[0.3, 1.3]; drafts drawn from softmax(d/T_b).

Rows beyond a request's draft length are filled with NaN and their draft
tokens with -1, so a kernel that reads them produces visibly wrong results.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

BF16_NAN = float("nan")


@dataclasses.dataclass
class Workload:
    name: str
    B: int
    n_max: int
    V: int
    dtype: str  # "f32" | "bf16"
    target: torch.Tensor  # [B, n_max+1, V]
    draft: Optional[torch.Tensor]  # [B, n_max, V]
    draft_tokens: torch.Tensor  # int32 [B, n_max]
    draft_len: torch.Tensor  # int32 [B]
    temperature: torch.Tensor  # float32 [B]
    seed: int = 0  # Philox seed of the verify step
    mtp_tokens: Optional[torch.Tensor] = None  # int32 [R]
    hidden: Optional[torch.Tensor] = None  # bf16 [R, H]

    @property
    def rows_target(self) -> int:
        return int(self.draft_len.sum().item()) + self.B

    @property
    def rows_draft(self) -> int:
        """Draft rows a stochastic request must score (greedy requests read none)."""
        L = self.draft_len.to(torch.int64)
        stochastic = (self.temperature > 0).to(torch.int64)
        return int((L * stochastic).sum().item())

    def to(self, device) -> "Workload":
        f = lambda t: None if t is None else t.to(device)
        return dataclasses.replace(
            self, target=f(self.target), draft=f(self.draft), draft_tokens=f(self.draft_tokens),
            draft_len=f(self.draft_len), temperature=f(self.temperature),
            mtp_tokens=f(self.mtp_tokens), hidden=f(self.hidden))


CONFIGS = {
    1: dict(name="tiny B=4 n=3 V=1024 fp32 T=1", B=4, n=3, V=1024, dtype="f32"),
    2: dict(name="draft-target linear B=64 n=4 V=128256 bf16 T=0.7", B=64, n=4, V=128256, dtype="bf16"),
    3: dict(name="MTP single-token B=256 n=1 V=129280 bf16 T=1 (+tokens[512], hidden[512,7168])",
            B=256, n=1, V=129280, dtype="bf16"),
    4: dict(name="greedy B=512 n=4 V=128256 bf16 T=0", B=512, n=4, V=128256, dtype="bf16"),
    5: dict(name="ragged B=1024 n_b~U{1..7} V=152064 bf16 T~U[0.3,1.3]", B=1024, n=7, V=152064,
            dtype="bf16"),
}


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _sample_rows(logits_f32: torch.Tensor, temperature: torch.Tensor, g) -> torch.Tensor:
    """Draft tokens drawn from softmax(logits / T) row by row (T > 0), argmax for T == 0.

    This stands in for the draft model's own sampling; it is not the verify
    method.  logits_f32 [B, n, V], temperature [B].
    """
    B, n, V = logits_f32.shape
    out = torch.empty(B, n, dtype=torch.int64, device=logits_f32.device)
    for b in range(B):
        T = float(temperature[b])
        rows = logits_f32[b]
        if T > 0:
            probs = torch.softmax(rows.double() / T, dim=-1)
            out[b] = torch.multinomial(probs, 1, generator=g).squeeze(-1)
        else:
            out[b] = rows.argmax(dim=-1)
    return out


def _sample_rows_batched(logits_f32: torch.Tensor, temperature: torch.Tensor, g,
                         chunk: int = 64) -> torch.Tensor:
    """Same draw as ``_sample_rows`` but batched over requests (all T > 0)."""
    B, n, V = logits_f32.shape
    out = torch.empty(B, n, dtype=torch.int64, device=logits_f32.device)
    for b0 in range(0, B, chunk):
        b1 = min(B, b0 + chunk)
        T = temperature[b0:b1].double().view(-1, 1, 1)
        probs = torch.softmax(logits_f32[b0:b1].double() / T, dim=-1)
        out[b0:b1] = torch.multinomial(probs.view(-1, V), 1, generator=g).view(b1 - b0, n)
    return out


def _fill_padding(w: Workload) -> Workload:
    """NaN logits and -1 tokens in rows beyond each request's draft length."""
    L = w.draft_len.to(torch.int64)
    j = torch.arange(w.n_max + 1, device=L.device).view(1, -1)
    pad_t = j > L.view(-1, 1)
    w.target[pad_t] = BF16_NAN
    if w.n_max > 0:
        pad_d = j[:, : w.n_max] >= L.view(-1, 1)
        if w.draft is not None:
            w.draft[pad_d] = BF16_NAN
        w.draft_tokens[pad_d] = -1
    return w


def make_config(k: int, device="cpu", seed: Optional[int] = None, B: Optional[int] = None) -> Workload:
    """Workload k (1..5).  ``B`` overrides the request count (same recipe)."""
    c = CONFIGS[k]
    B = c["B"] if B is None else B
    n, V = c["n"], c["V"]
    g = _gen(device, 1000 + k if seed is None else seed)
    dt = torch.float32 if c["dtype"] == "f32" else torch.bfloat16

    if k == 1:
        t = torch.randn(B, n + 1, V, generator=g, device=device) * 2.0
        d = t[:, :n] + torch.randn(B, n, V, generator=g, device=device) * 0.5
        T = torch.ones(B, device=device)
        L = torch.full((B,), n, dtype=torch.int32, device=device)
        x = _sample_rows_batched(d, T, g)
        w = Workload(c["name"], B, n, V, "f32", t.contiguous(), d.contiguous(),
                     x.to(torch.int32), L, T.float())
        return w

    if k in (2, 3, 4):
        t = torch.empty(B, n + 1, V, dtype=dt, device=device)
        d = torch.empty(B, n, V, dtype=dt, device=device)
        T = torch.full((B,), {2: 0.7, 3: 1.0, 4: 0.0}[k], dtype=torch.float32, device=device)
        L = torch.full((B,), n, dtype=torch.int32, device=device)
        x = torch.empty(B, n, dtype=torch.int64, device=device)
        chunk = 32
        for b0 in range(0, B, chunk):
            b1 = min(B, b0 + chunk)
            tf = torch.randn(b1 - b0, n + 1, V, generator=g, device=device) * 3.0
            spike = torch.randint(0, V, (b1 - b0, n + 1, 1), generator=g, device=device)
            tf.scatter_add_(2, spike, torch.full((b1 - b0, n + 1, 1), 8.0, device=device))
            df = tf[:, :n] + torch.randn(b1 - b0, n, V, generator=g, device=device)
            t[b0:b1] = tf.to(dt)
            if k == 4:
                tb = t[b0:b1, :n].float()
                top2 = tb.topk(2, dim=-1).indices  # [b, n, 2]
                take_first = torch.rand(b1 - b0, n, generator=g, device=device) < 0.75
                xx = torch.where(take_first, top2[..., 0], top2[..., 1])
                # draft logits whose argmax is the chosen draft token
                df = df.clone()
                mx = df.max(dim=-1, keepdim=True).values
                df.scatter_(2, xx.unsqueeze(-1), mx + 1.0)
                x[b0:b1] = xx
            d[b0:b1] = df.to(dt)
            if k != 4:
                x[b0:b1] = _sample_rows_batched(d[b0:b1].float(), T[b0:b1], g)
        w = Workload(c["name"], B, n, V, "bf16", t, d, x.to(torch.int32), L, T)
        if k == 3:
            w.mtp_tokens, w.hidden = make_mtp(B * (n + 1), 7168, V, device=device, g=g)
        return w

    if k == 5:
        t = torch.empty(B, n + 1, V, dtype=dt, device=device)
        d = torch.empty(B, n, V, dtype=dt, device=device)
        L = torch.randint(1, n + 1, (B,), generator=g, device=device).to(torch.int32)
        T = (0.3 + torch.rand(B, generator=g, device=device)).float()
        bias = -1.1 * torch.log(torch.arange(V, device=device, dtype=torch.float32) + 1.0)
        x = torch.empty(B, n, dtype=torch.int64, device=device)
        chunk = 32
        for b0 in range(0, B, chunk):
            b1 = min(B, b0 + chunk)
            tf = torch.randn(b1 - b0, n + 1, V, generator=g, device=device) * 3.0 + bias
            df = tf[:, :n] + torch.randn(b1 - b0, n, V, generator=g, device=device) * 0.8
            t[b0:b1] = tf.to(dt)
            d[b0:b1] = df.to(dt)
            x[b0:b1] = _sample_rows_batched(d[b0:b1].float(), T[b0:b1], g)
        w = Workload(c["name"], B, n, V, "bf16", t, d, x.to(torch.int32), L, T)
        return _fill_padding(w)

    raise KeyError(k)


def make_random(B: int, n_max: int, V: int, dtype: str = "bf16", device="cpu", seed: int = 0,
                temperatures=(0.7,), ragged: bool = False, draft_noise: float = 1.0,
                scale: float = 3.0, philox_seed: int = 0) -> Workload:
    """A small random batch for parity tests.

    ``temperatures`` is cycled over requests (0 gives greedy requests);
    ``ragged`` draws draft_len uniformly in [0, n_max].
    """
    g = _gen(device, seed)
    dt = torch.float32 if dtype == "f32" else torch.bfloat16
    tf = torch.randn(B, n_max + 1, V, generator=g, device=device) * scale
    df = tf[:, :n_max] + torch.randn(B, n_max, V, generator=g, device=device) * draft_noise
    t = tf.to(dt)
    d = df.to(dt)
    T = torch.tensor([temperatures[i % len(temperatures)] for i in range(B)],
                     dtype=torch.float32, device=device)
    if ragged:
        L = torch.randint(0, n_max + 1, (B,), generator=g, device=device).to(torch.int32)
    else:
        L = torch.full((B,), n_max, dtype=torch.int32, device=device)
    x = _sample_rows(d.float(), T, g) if n_max > 0 else torch.empty(B, 0, dtype=torch.int64,
                                                                    device=device)
    w = Workload(f"random B={B} n={n_max} V={V} {dtype}", B, n_max, V, dtype, t.contiguous(),
                 d.contiguous(), x.to(torch.int32), L, T, seed=philox_seed)
    return _fill_padding(w)


def make_mtp(R: int, H: int, V: int, device="cpu", g=None, seed: int = 7):
    """MTP buffers: tokens int32 [R] uniform in [0, V), hidden bf16 [R, H] ~ N(0, 1)."""
    if g is None:
        g = _gen(device, seed)
    tokens = torch.randint(0, V, (R,), generator=g, device=device).to(torch.int32)
    hidden = torch.randn(R, H, generator=g, device=device).to(torch.bfloat16)
    return tokens, hidden


def bf16_bits(t: torch.Tensor):
    """A bf16 tensor as a numpy uint16 array of its raw bits (for the oracle)."""
    import numpy as np

    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def logits_numpy(t: Optional[torch.Tensor]):
    """Logits as the oracle takes them: float32 array, or uint16 bits for bf16."""
    if t is None:
        return None
    if t.dtype == torch.bfloat16:
        return bf16_bits(t)
    return t.detach().cpu().contiguous().float().numpy()


def algorithmic_bytes(w: Workload) -> int:
    """Logit bytes the verify step must read: every valid target row, and the
    draft rows of requests with T > 0 (greedy requests read target rows only)."""
    elt = 4 if w.dtype == "f32" else 2
    return (w.rows_target + w.rows_draft) * w.V * elt


def isclose_ratio(a, b):
    return math.isclose(a, b, rel_tol=1e-9)


def pack(w: Workload):
    """The same batch in the packed ragged layout: request b's n_b + 1 target
    rows at cu_rows[b], its n_b draft rows and draft tokens at cu_rows[b] - b.

    Returns (target [R, V], draft [R - B, V] or None, draft_tokens [R - B],
    cu_rows [B + 1] int32), R = sum of (n_b + 1), on the workload's device."""
    L = [int(v) for v in w.draft_len.cpu().tolist()]
    dev = w.target.device
    cu = [0]
    for n in L:
        cu.append(cu[-1] + n + 1)
    t = torch.cat([w.target[b, : L[b] + 1] for b in range(w.B)], dim=0).contiguous()
    d = None
    if w.draft is not None:
        rows = [w.draft[b, : L[b]] for b in range(w.B)]
        d = torch.cat(rows, dim=0).contiguous() if sum(L) > 0 else w.draft.new_empty(0, w.V)
    x = torch.cat([w.draft_tokens[b, : L[b]] for b in range(w.B)], dim=0).contiguous() if sum(L) > 0 \
        else torch.empty(0, dtype=torch.int32, device=dev)
    return t, d, x, torch.tensor(cu, dtype=torch.int32, device=dev)


def unpack_rows(packed: torch.Tensor, cu_rows, n_max: int, fill):
    """Packed per-target-row values [R, ...] back to [B, n_max + 1, ...],
    slots past a request's rows set to `fill`."""
    cu = [int(v) for v in (cu_rows.cpu().tolist() if hasattr(cu_rows, "cpu") else cu_rows)]
    B = len(cu) - 1
    out = packed.new_full((B, n_max + 1) + tuple(packed.shape[1:]), fill)
    for b in range(B):
        n = cu[b + 1] - cu[b]
        out[b, :n] = packed[cu[b]: cu[b + 1]]
    return out
