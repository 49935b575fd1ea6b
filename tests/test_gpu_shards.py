"""GPU parity of the vocabulary-sharded verify (three calls per shard, the
exchange between ranks done in place on one GPU) against the CPU oracle on
the unsharded batch, through the C ABI."""
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


def _split(w, bounds):
    cuts = [0] + list(bounds) + [w.V]
    ts = [w.target[:, :, cuts[i]:cuts[i + 1]].contiguous() for i in range(len(cuts) - 1)]
    ds = None if w.draft is None else [w.draft[:, :, cuts[i]:cuts[i + 1]].contiguous() for i in range(len(cuts) - 1)]
    return ts, ds


@pytest.mark.parametrize("V,dtype,bounds", [(1000, "f32", (499,)), (5003, "bf16", (1701, 3400)),
                                            (50001, "bf16", (25000,)), (40000, "f32", (8, 39000))])
def test_sharded_matches_oracle(V, dtype, bounds):
    w = make_random(32, 4, V, dtype=dtype, device="cuda", seed=V % 101, temperatures=(0.0, 0.7, 1.0, 1.5),
                    ragged=True, philox_seed=V * 3)
    ts, ds = _split(w, bounds)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    acc, out = sd.spec_verify_sharded(ts, ds, w.draft_tokens, w.draft_len, w.temperature, seed=w.seed,
                                      error_word=err)
    wait_gpu()
    ref = oracle_on(w, want_lse=False)
    compare(w, acc, out, ref, None, f"sharded V={V} {dtype} {bounds}")
    assert int(err.item()) == 0


def test_sharded_greedy_without_draft_shards():
    w = make_random(24, 3, 7000, dtype="bf16", device="cuda", seed=4, temperatures=(0.0,), ragged=True)
    w.draft = None
    ts, _ = _split(w, (3500,))
    acc, out = sd.spec_verify_sharded(ts, None, w.draft_tokens, w.draft_len, w.temperature, seed=w.seed)
    wait_gpu()
    ref = oracle_on(w, want_lse=False)
    st = compare(w, acc, out, ref, None, "sharded greedy")
    assert st["mismatch"] == 0


def test_sharded_tokens_on_shard_boundaries():
    # Draft tokens exactly at the first and last entry of each shard, so the
    # logit at x must come from the right shard.
    w = make_random(16, 4, 9000, dtype="bf16", device="cuda", seed=8, temperatures=(0.9,), philox_seed=5)
    bounds = (3000, 6000)
    edges = torch.tensor([0, 2999, 3000, 5999, 6000, 8999], dtype=torch.int32)
    x = edges[torch.arange(w.B * w.n_max) % len(edges)].view(w.B, w.n_max).to("cuda")
    w.draft_tokens = x.contiguous()
    ts, ds = _split(w, bounds)
    acc, out = sd.spec_verify_sharded(ts, ds, w.draft_tokens, w.draft_len, w.temperature, seed=w.seed)
    wait_gpu()
    ref = oracle_on(w, want_lse=False)
    compare(w, acc, out, ref, None, "shard edges")


def test_sharded_config2_two_shards():
    w = make_config(2, device="cuda")
    ts, ds = _split(w, (w.V // 2 + 8,))
    acc, out = sd.spec_verify_sharded(ts, ds, w.draft_tokens, w.draft_len, w.temperature, seed=w.seed)
    wait_gpu()
    ref = oracle_on(w, want_lse=False)
    compare(w, acc, out, ref, None, "sharded config2")
    acc_f, out_f = sd.spec_verify(w.target, w.draft, w.draft_tokens, w.draft_len, w.temperature, seed=w.seed)
    wait_gpu()
    # the fused call and the sharded calls agree except where the oracle's
    # margin is a near tie (already allowed by compare above)
    same = (acc_f == acc) & (out_f == out).all(dim=1)
    assert same.float().mean().item() >= 0.95


def test_sharded_long_drafts_span_two_acceptance_rounds():
    # n_max > 32: one warp tests 32 rows per round, so later rows take a
    # second round; near-identical draft and target keep most rows accepted.
    w = make_random(12, 40, 2000, dtype="f32", device="cuda", seed=21, temperatures=(0.8, 0.0, 1.2),
                    draft_noise=0.05, philox_seed=8)
    ts, ds = _split(w, (977,))
    acc, out = sd.spec_verify_sharded(ts, ds, w.draft_tokens, w.draft_len, w.temperature, seed=w.seed)
    wait_gpu()
    ref = oracle_on(w, want_lse=False)
    compare(w, acc, out, ref, None, "sharded n=40")
    assert (acc.cpu().numpy() > 32).any()


def test_sharded_bad_device_data_sets_the_oracles_error_bits():
    w = make_random(8, 3, 3001, dtype="bf16", device="cuda", seed=2, temperatures=(0.9, 0.0), philox_seed=1)
    w.draft_tokens[1, 0] = w.V + 5     # out of range: rejects row 0
    w.draft_tokens[2, 0] = -3          # negative: rejects row 0
    w.draft_len[3] = 9                 # clamped to n_max
    w.temperature[4] = float("nan")    # greedy
    ts, ds = _split(w, (1500,))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    acc, out = sd.spec_verify_sharded(ts, ds, w.draft_tokens, w.draft_len, w.temperature, seed=w.seed,
                                      error_word=err)
    wait_gpu()
    ref = oracle_on(w, want_lse=False)
    compare(w, acc, out, ref, None, "sharded bad data")
    assert int(err.item()) == ref["err"] == sd.DEV_ERR_TOKEN | sd.DEV_ERR_DRAFT_LEN | sd.DEV_ERR_TEMPERATURE


def _one_rank_worker(root, port, q):
    import sys

    sys.path.insert(0, root)
    import torch
    import torch.distributed as dist

    import speculative_decoding_verification_80_gb300 as sd
    from tests.parity import compare, oracle_on
    from workloads import make_random

    torch.cuda.set_device(0)
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1)
    try:
        w = make_random(16, 3, 5003, dtype="bf16", device="cuda", seed=12, temperatures=(0.0, 0.9),
                        ragged=True, philox_seed=6)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        acc, out = sd.spec_verify_shard_rank(w.target, w.draft, 0, w.V, w.draft_tokens, w.draft_len,
                                             w.temperature, seed=w.seed, error_word=err)
        acc1, out1 = sd.spec_verify_sharded([w.target], [w.draft], w.draft_tokens, w.draft_len, w.temperature,
                                            seed=w.seed)
        torch.cuda.synchronize()
        compare(w, acc, out, oracle_on(w, want_lse=False), None, "one-rank group")
        q.put((torch.equal(acc, acc1) and torch.equal(out, out1), int(err.item())))
    finally:
        dist.destroy_process_group()


def test_shard_rank_one_rank_group_over_nccl():
    # The multi-rank entry with the library's calls and real all-gathers, in
    # a group of one rank (this machine's GPU): the same outputs as the
    # single-GPU sharded call and the oracle's tokens.
    import os
    import socket

    import torch.multiprocessing as mp

    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    p = ctx.Process(target=_one_rank_worker, args=(root, port, q))
    p.start()
    p.join(timeout=300)
    assert p.exitcode == 0
    same, err = q.get(timeout=5)
    assert same and err == 0
