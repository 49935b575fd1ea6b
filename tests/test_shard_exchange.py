"""The exchange of the vocabulary-sharded step between ranks, on CPU: world
size 2 and 3 gloo ranks each hold one vocabulary range of the same batch and
run spec_verify_shard_rank (its two all-gathers over the group) with an fp64
numpy restatement of the per-shard calls; every rank must end with the
oracle's accepted lengths, tokens and error bits on the whole vocabulary."""
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _batch():
    import torch

    from workloads import make_random

    w = make_random(9, 3, 41, dtype="f32", device="cpu", seed=5, temperatures=(0.0, 0.8, 1.3), ragged=True,
                    philox_seed=77)
    g = torch.Generator().manual_seed(3)
    for b in (4, 7):  # every row filled, all drafts in play
        w.target[b] = torch.randn(w.n_max + 1, w.V, generator=g) * 2
        w.draft[b] = w.target[b, : w.n_max] + torch.randn(w.n_max, w.V, generator=g)
        w.draft_tokens[b] = torch.randint(0, w.V, (w.n_max,), generator=g, dtype=torch.int32)
        w.draft_len[b] = w.n_max
    w.draft_tokens[4, 0] = w.V + 2  # out of range: rejects row 0, sets the token bit
    w.draft_len[7] = 6               # clamped to n_max, sets the draft-length bit
    return w


def _worker(rank, world, port, cuts, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch
    import torch.distributed as dist

    import speculative_decoding_verification_80_gb300 as sd
    from tests.shard_ops_numpy import NumpyShardOps

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = _batch()
        lo, hi = cuts[rank], cuts[rank + 1]
        err = torch.zeros(1, dtype=torch.int32)
        acc, out = sd.spec_verify_shard_rank(w.target[..., lo:hi].contiguous(), w.draft[..., lo:hi].contiguous(), lo,
                                             w.V, w.draft_tokens, w.draft_len, w.temperature, seed=w.seed,
                                             error_word=err, ops=NumpyShardOps())
        q.put((rank, acc.numpy().tolist(), out.numpy().tolist(), int(err.item())))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("cuts", [(0, 20, 41), (0, 1, 30, 41)])
def test_ranks_agree_with_the_oracle(cuts):
    import oracle
    from workloads.gen import logits_numpy

    world = len(cuts) - 1
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, cuts, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
    assert all(p.exitcode == 0 for p in procs)
    res = sorted(q.get(timeout=5) for _ in range(world))

    w = _batch()
    ref = oracle.spec_verify(logits_numpy(w.target), logits_numpy(w.draft), w.draft_tokens.numpy(),
                             w.draft_len.numpy(), w.temperature.numpy(), seed=w.seed, want_stats=False)
    assert ref["err"] == oracle.ERR_TOKEN | oracle.ERR_DRAFT_LEN
    for _, acc, out, err in res:
        assert np.array_equal(np.asarray(acc), ref["accepted_len"])
        assert np.array_equal(np.asarray(out), ref["out_tokens"])
        assert err == ref["err"]
