"""GB300 speculative-decoding verify/accept and MTP shift/insert.

A thin ctypes binding over libspecdec.so (include/specdec.h).  The functions
keep the C names; they only marshal torch tensors into device pointers, sizes
and the current CUDA stream.  Every step of the computation runs in the
library's kernels; there is no fallback: if the library is missing or no GPU
is present, the calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

__all__ = [
    "SpecDecError", "load_library", "workspace_bytes", "new_workspace", "workspace_init",
    "spec_verify", "spec_verify_packed", "spec_verify_early_exit", "spec_verify_sharded",
    "spec_verify_shard_rank", "ShardOps", "shard_exchange_buffers", "bytes_read", "mtp_shift_insert", "get_error", "launch_shape", "F32", "BF16",
    "DEV_ERR_TOKEN", "DEV_ERR_DRAFT_LEN", "DEV_ERR_TEMPERATURE", "DEV_ERR_TIMEOUT", "DEV_ERR_SEGMENT",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libspecdec.so")

F32, BF16 = 0, 1
DEV_ERR_TOKEN, DEV_ERR_DRAFT_LEN, DEV_ERR_TEMPERATURE, DEV_ERR_TIMEOUT, DEV_ERR_SEGMENT = 1, 2, 4, 8, 16
_STATUS = {0: "SPECDEC_OK", 1: "SPECDEC_ERR_INVALID_ARG", 2: "SPECDEC_ERR_UNSUPPORTED",
           3: "SPECDEC_ERR_WORKSPACE", 4: "SPECDEC_ERR_CUDA", 5: "SPECDEC_ERR_DEVICE_DATA",
           6: "SPECDEC_ERR_TIMEOUT"}

# Every symbol the header declares (checked by the CPU test-suite).
EXPORTS = ("spec_verify", "mtp_shift_insert", "specdec_verify_workspace_bytes",
           "specdec_workspace_init", "specdec_get_error", "specdec_status_string",
           "specdec_verify_launch_shape", "spec_verify_no_alloc", "spec_verify_packed",
           "spec_verify_early_exit", "specdec_get_bytes_read", "specdec_shard_stats_records",
           "specdec_shard_race_records", "spec_verify_shard_stats", "spec_verify_shard_race", "spec_verify_shard_finish")
EARLY_EXIT_MAX_DRAFT = 31

_lock = threading.Lock()
_lib = None


class SpecDecError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {_STATUS.get(status, status)}")
        self.status = status


def load_library(path: Optional[str] = None):
    """Load libspecdec.so (building it first if it is absent)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        # SPECDEC_LIBRARY points at another build of the same ABI (to compare
        # builds side by side); by default the in-tree library is used.
        p = path or os.environ.get("SPECDEC_LIBRARY") or LIB_PATH
        if not os.path.exists(p):
            from . import build as _build

            _build.build()
        L = ctypes.CDLL(p)
        P, i32, u64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint64, ctypes.c_size_t
        L.specdec_verify_workspace_bytes.argtypes = [i32, i32, i32]
        L.specdec_verify_workspace_bytes.restype = sz
        L.specdec_workspace_init.argtypes = [P, sz, P]
        L.specdec_workspace_init.restype = ctypes.c_int
        L.spec_verify.argtypes = [P, P, ctypes.c_int, i32, i32, i32, P, P, P, u64, P, P, P, P, sz, P]
        L.spec_verify.restype = ctypes.c_int
        if hasattr(L, "spec_verify_early_exit"):
            L.spec_verify_early_exit.argtypes = [P, P, ctypes.c_int, i32, i32, i32, P, P, P, u64, P, P, P, sz, P]
            L.spec_verify_early_exit.restype = ctypes.c_int
            L.specdec_get_bytes_read.argtypes = [P, ctypes.POINTER(ctypes.c_uint64)]
            L.specdec_get_bytes_read.restype = ctypes.c_int
        if hasattr(L, "spec_verify_shard_stats"):
            L.specdec_shard_stats_records.argtypes = [i32, i32]
            L.specdec_shard_stats_records.restype = sz
            L.specdec_shard_race_records.argtypes = [i32]
            L.specdec_shard_race_records.restype = sz
            L.spec_verify_shard_stats.argtypes = [P, P, ctypes.c_int, i32, i32, i32, i32, i32, P, P, P, P, P]
            L.spec_verify_shard_stats.restype = ctypes.c_int
            L.spec_verify_shard_race.argtypes = [P, P, ctypes.c_int, i32, i32, i32, i32, i32, P, P, P, u64, P, i32,
                                                 P, P, P, P]
            L.spec_verify_shard_race.restype = ctypes.c_int
            L.spec_verify_shard_finish.argtypes = [P, i32, i32, i32, P, P, P, P]
            L.spec_verify_shard_finish.restype = ctypes.c_int
        if hasattr(L, "spec_verify_packed"):
            L.spec_verify_packed.argtypes = [P, P, ctypes.c_int, i32, i32, i32, P, i32, P, P, P, u64,
                                             P, P, P, P, sz, P]
            L.spec_verify_packed.restype = ctypes.c_int
        L.mtp_shift_insert.argtypes = [P, P, P, P, i32, i32, i32, P, P, P, P, i32, i32, P, P]
        L.mtp_shift_insert.restype = ctypes.c_int
        L.specdec_get_error.argtypes = [P, ctypes.POINTER(ctypes.c_uint32)]
        L.specdec_get_error.restype = ctypes.c_int
        L.specdec_status_string.argtypes = [ctypes.c_int]
        L.specdec_status_string.restype = ctypes.c_char_p
        L.specdec_verify_launch_shape.argtypes = [i32, i32, i32, ctypes.c_int, ctypes.POINTER(i32),
                                                  ctypes.POINTER(i32)]
        L.specdec_verify_launch_shape.restype = ctypes.c_int
        if hasattr(L, "spec_verify_no_alloc"):
            L.spec_verify_no_alloc.argtypes = [P, P, ctypes.c_int, i32, i32, i32, P, P, P, u64, P, P, P, P]
            L.spec_verify_no_alloc.restype = ctypes.c_int
        if path is None:
            _lib = L
        return L


def _check(status: int, what: str):
    if status != 0:
        raise SpecDecError(status, what)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("spec-decode tensors must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("spec-decode tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _one_device(*tensors, stream=None) -> None:
    """The CUDA tensors of one call share a device, which is the current one
    (where the library launches), and so does the stream when one is given:
    a pointer to another GPU's memory never reaches a kernel."""
    devs = {t.device for t in tensors if t is not None}
    if len(devs) > 1:
        raise ValueError(f"the tensors of one call must share a device, got {sorted(map(str, devs))}")
    if not devs:
        return
    dev = devs.pop()
    if dev.type != "cuda":
        return  # _ptr rejects it
    cur = torch.cuda.current_device()
    if dev.index != cur:
        raise ValueError(f"the tensors are on {dev} but the current device is cuda:{cur}; "
                         f"call under torch.cuda.device({dev.index})")
    sdev = getattr(stream, "device", None)
    if sdev is not None and torch.device(sdev) != dev:
        raise ValueError(f"the stream is on {sdev}, the tensors on {dev}")


def _on(stream):
    """Context in which a call's temporaries (default outputs, workspace) are
    allocated and zeroed: the caller's stream when one is given, so the
    caching allocator ties them to the stream the kernels run on."""
    import contextlib

    if stream is None:
        return contextlib.nullcontext()
    if not isinstance(stream, torch.cuda.Stream):  # a raw cudaStream_t handle
        stream = torch.cuda.ExternalStream(int(stream.cuda_stream if hasattr(stream, "cuda_stream") else stream))
    return torch.cuda.stream(stream)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _need(t: Optional[torch.Tensor], n: int, what: str, dtype=None):
    """Host-side size (and dtype) check, so a wrong buffer never reaches the device."""
    if t is None:
        return
    if t.numel() != n:
        raise ValueError(f"{what} must hold {n} elements, got {t.numel()}")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{what} must be {dtype}, got {t.dtype}")


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"logits must be float32 or bfloat16, got {t.dtype}")


def workspace_bytes(B: int, n_max: int, V: int) -> int:
    return int(load_library().specdec_verify_workspace_bytes(B, n_max, V))


def workspace_init(ws: torch.Tensor, stream=None):
    _one_device(ws, stream=stream)
    _check(load_library().specdec_workspace_init(_ptr(ws), ws.numel(), _stream(stream)),
           "specdec_workspace_init")


def new_workspace(B: int, n_max: int, V: int, device=None, stream=None) -> torch.Tensor:
    """A zero-filled workspace (uint8 tensor) for spec_verify, allocated and
    zeroed on `stream` (default: the current stream)."""
    n = workspace_bytes(B, n_max, V)
    if n == 0:
        raise SpecDecError(1, "specdec_verify_workspace_bytes")
    with _on(stream):
        ws = torch.empty(n, dtype=torch.uint8, device=device or "cuda")
        workspace_init(ws, stream=stream)
    return ws


def launch_shape(B: int, n_max: int, V: int, dtype=torch.bfloat16):
    """(chunks per row, elements per chunk) spec_verify uses for this batch shape."""
    c, s = ctypes.c_int32(0), ctypes.c_int32(0)
    code = F32 if dtype == torch.float32 else BF16
    _check(load_library().specdec_verify_launch_shape(B, n_max, V, code, ctypes.byref(c), ctypes.byref(s)),
           "specdec_verify_launch_shape")
    return c.value, s.value


def spec_verify(target_logits: torch.Tensor, draft_logits: Optional[torch.Tensor],
                draft_tokens: torch.Tensor, draft_len: torch.Tensor, temperature: torch.Tensor,
                seed: int = 0, accepted_len: Optional[torch.Tensor] = None,
                out_tokens: Optional[torch.Tensor] = None, row_lse: Optional[torch.Tensor] = None,
                workspace: Optional[torch.Tensor] = None, stream=None):
    """Batched verify/accept (see include/specdec.h).  Returns (accepted_len, out_tokens)."""
    B, rows, V = target_logits.shape
    n_max = rows - 1
    dev = target_logits.device
    if draft_logits is not None:
        if draft_logits.dtype != target_logits.dtype or tuple(draft_logits.shape) != (B, n_max, V):
            raise ValueError("draft_logits must be [B, n_max, V] of the target's dtype")
    _need(draft_tokens, B * n_max, "draft_tokens", torch.int32)
    _need(draft_len, B, "draft_len", torch.int32)
    _need(temperature, B, "temperature", torch.float32)
    _need(accepted_len, B, "accepted_len", torch.int32)
    _need(out_tokens, B * rows, "out_tokens", torch.int32)
    with _on(stream):
        if accepted_len is None:
            accepted_len = torch.empty(B, dtype=torch.int32, device=dev)
        if out_tokens is None:
            out_tokens = torch.empty(B, rows, dtype=torch.int32, device=dev)
    _need(row_lse, B * rows * 2, "row_lse", torch.float32)
    if workspace is None:
        workspace = new_workspace(B, n_max, V, device=dev, stream=stream)
    _one_device(target_logits, draft_logits, draft_tokens, draft_len, temperature, accepted_len, out_tokens, row_lse,
                workspace, stream=stream)
    st = load_library().spec_verify(
        _ptr(target_logits), _ptr(draft_logits), _dtype_code(target_logits), B, n_max, V,
        _ptr(draft_tokens), _ptr(draft_len), _ptr(temperature), int(seed) & (2**64 - 1),
        _ptr(accepted_len), _ptr(out_tokens), _ptr(row_lse), _ptr(workspace), workspace.numel(),
        _stream(stream))
    _check(st, "spec_verify")
    return accepted_len, out_tokens


def spec_verify_early_exit(target_logits: torch.Tensor, draft_logits: Optional[torch.Tensor],
                           draft_tokens: torch.Tensor, draft_len: torch.Tensor, temperature: torch.Tensor,
                           seed: int = 0, accepted_len: Optional[torch.Tensor] = None,
                           out_tokens: Optional[torch.Tensor] = None,
                           workspace: Optional[torch.Tensor] = None, stream=None):
    """spec_verify without reading the rows after a request's first rejection
    (see include/specdec.h); identical outputs.  Returns (accepted_len, out_tokens)."""
    B, rows, V = target_logits.shape
    n_max = rows - 1
    dev = target_logits.device
    if n_max > EARLY_EXIT_MAX_DRAFT:
        raise ValueError(f"early exit supports n_max <= {EARLY_EXIT_MAX_DRAFT}")
    if draft_logits is not None:
        if draft_logits.dtype != target_logits.dtype or tuple(draft_logits.shape) != (B, n_max, V):
            raise ValueError("draft_logits must be [B, n_max, V] of the target's dtype")
    _need(draft_tokens, B * n_max, "draft_tokens", torch.int32)
    _need(draft_len, B, "draft_len", torch.int32)
    _need(temperature, B, "temperature", torch.float32)
    _need(accepted_len, B, "accepted_len", torch.int32)
    _need(out_tokens, B * rows, "out_tokens", torch.int32)
    with _on(stream):
        if accepted_len is None:
            accepted_len = torch.empty(B, dtype=torch.int32, device=dev)
        if out_tokens is None:
            out_tokens = torch.empty(B, rows, dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = new_workspace(B, n_max, V, device=dev, stream=stream)
    _one_device(target_logits, draft_logits, draft_tokens, draft_len, temperature, accepted_len, out_tokens,
                workspace, stream=stream)
    st = load_library().spec_verify_early_exit(
        _ptr(target_logits), _ptr(draft_logits), _dtype_code(target_logits), B, n_max, V,
        _ptr(draft_tokens), _ptr(draft_len), _ptr(temperature), int(seed) & (2**64 - 1),
        _ptr(accepted_len), _ptr(out_tokens), _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "spec_verify_early_exit")
    return accepted_len, out_tokens


def shard_exchange_buffers(S: int, B: int, n_max: int, device=None):
    """The two gathered buffers of the sharded step for S shards: the row
    statistics (float32 [S, records, 4]) and the race records (int64
    [S, race records, 2])."""
    L = load_library()
    nrec = L.specdec_shard_stats_records(B, n_max)
    nrace = L.specdec_shard_race_records(B)
    dev = device if device is not None else torch.device("cuda")
    return (torch.empty(S, nrec, 4, dtype=torch.float32, device=dev),
            torch.empty(S, nrace, 2, dtype=torch.int64, device=dev))


def spec_verify_sharded(target_shards, draft_shards, draft_tokens: torch.Tensor, draft_len: torch.Tensor,
                        temperature: torch.Tensor, seed: int = 0, error_word: Optional[torch.Tensor] = None,
                        accepted_len: Optional[torch.Tensor] = None, out_tokens: Optional[torch.Tensor] = None,
                        exchange: Optional[tuple] = None, stream=None):
    """The vocabulary-sharded step on one GPU: `target_shards` / `draft_shards`
    are lists of [B, n_max+1, Vs] / [B, n_max, Vs] tensors covering the
    vocabulary in order (draft_shards may be None when every request is
    greedy).  Runs the three per-shard calls of include/specdec_shard.h, each shard
    writing its slice of the gathered buffers in place of the exchange
    between ranks.  `exchange` = shard_exchange_buffers(S, B, n_max) reuses
    the gathered buffers across calls.  Returns (accepted_len, out_tokens)."""
    L = load_library()
    S = len(target_shards)
    B, rows, _ = target_shards[0].shape
    n_max = rows - 1
    V = sum(t.shape[2] for t in target_shards)
    dev = target_shards[0].device
    _need(draft_tokens, B * n_max, "draft_tokens", torch.int32)
    _need(draft_len, B, "draft_len", torch.int32)
    _need(temperature, B, "temperature", torch.float32)
    _need(error_word, 1, "error_word", torch.int32)
    with _on(stream):
        stats, race = exchange if exchange is not None else shard_exchange_buffers(S, B, n_max, device=dev)
    _need(stats, S * L.specdec_shard_stats_records(B, n_max) * 4, "exchange[0]", torch.float32)
    _need(race, S * L.specdec_shard_race_records(B) * 2, "exchange[1]", torch.int64)
    with _on(stream):
        if accepted_len is None:
            accepted_len = torch.empty(B, dtype=torch.int32, device=dev)
        if out_tokens is None:
            out_tokens = torch.empty(B, rows, dtype=torch.int32, device=dev)
    _need(accepted_len, B, "accepted_len", torch.int32)
    _need(out_tokens, B * rows, "out_tokens", torch.int32)
    code = _dtype_code(target_shards[0])
    v0s, v0 = [], 0
    for t in target_shards:
        if t.shape[:2] != (B, rows) or t.dtype != target_shards[0].dtype:
            raise ValueError("every target shard must be [B, n_max+1, Vs] of one dtype")
        v0s.append(v0)
        v0 += t.shape[2]
    if draft_shards is not None:
        if len(draft_shards) != S:
            raise ValueError("one draft shard per target shard")
        for dsh, t in zip(draft_shards, target_shards):
            if tuple(dsh.shape) != (B, n_max, t.shape[2]) or dsh.dtype != t.dtype:
                raise ValueError("draft shard s must be [B, n_max, Vs_s] of the target's dtype")
    _one_device(*target_shards, *(draft_shards or ()), draft_tokens, draft_len, temperature, error_word, stats,
                race, accepted_len, out_tokens, stream=stream)
    st = _stream(stream)
    for s in range(S):
        d = None if draft_shards is None else draft_shards[s]
        _check(L.spec_verify_shard_stats(_ptr(target_shards[s]), _ptr(d), code, B, n_max, V, v0s[s],
                                         target_shards[s].shape[2], _ptr(draft_tokens), _ptr(draft_len),
                                         _ptr(temperature), _ptr(stats[s]), st), "spec_verify_shard_stats")
    for s in range(S):
        d = None if draft_shards is None else draft_shards[s]
        _check(L.spec_verify_shard_race(_ptr(target_shards[s]), _ptr(d), code, B, n_max, V, v0s[s],
                                        target_shards[s].shape[2], _ptr(draft_tokens), _ptr(draft_len),
                                        _ptr(temperature), int(seed) & (2**64 - 1), _ptr(stats), S,
                                        _ptr(accepted_len), _ptr(race[s]), _ptr(error_word), st),
               "spec_verify_shard_race")
    _check(L.spec_verify_shard_finish(_ptr(race), S, B, n_max, _ptr(draft_tokens), _ptr(accepted_len),
                                      _ptr(out_tokens), st), "spec_verify_shard_finish")
    return accepted_len, out_tokens


class ShardOps:
    """The three per-shard calls of the vocabulary-sharded step through the C
    ABI (include/specdec_shard.h), for spec_verify_shard_rank.  A shard's
    exchange records are stats_buffer() and race_buffer(); the all-gathers
    stack one of each per rank."""

    def __init__(self):
        self.L = load_library()

    def stats_buffer(self, B: int, n_max: int, device) -> torch.Tensor:
        return torch.empty(self.L.specdec_shard_stats_records(B, n_max), 4, dtype=torch.float32, device=device)

    def race_buffer(self, B: int, device) -> torch.Tensor:
        return torch.empty(self.L.specdec_shard_race_records(B), 2, dtype=torch.int64, device=device)

    def stats(self, target, draft, V, v0, draft_tokens, draft_len, temperature, out, stream=None):
        B, rows, Vs = target.shape
        _one_device(target, draft, draft_tokens, draft_len, temperature, out, stream=stream)
        _check(self.L.spec_verify_shard_stats(_ptr(target), _ptr(draft), _dtype_code(target), B, rows - 1, V, v0, Vs,
                                              _ptr(draft_tokens), _ptr(draft_len), _ptr(temperature), _ptr(out),
                                              _stream(stream)), "spec_verify_shard_stats")

    def race(self, target, draft, V, v0, draft_tokens, draft_len, temperature, seed, stats_all, accepted_len, out,
             error_word=None, stream=None):
        B, rows, Vs = target.shape
        _one_device(target, draft, draft_tokens, draft_len, temperature, stats_all, accepted_len, out, error_word,
                    stream=stream)
        _check(self.L.spec_verify_shard_race(_ptr(target), _ptr(draft), _dtype_code(target), B, rows - 1, V, v0, Vs,
                                             _ptr(draft_tokens), _ptr(draft_len), _ptr(temperature),
                                             int(seed) & (2**64 - 1), _ptr(stats_all), stats_all.shape[0],
                                             _ptr(accepted_len), _ptr(out), _ptr(error_word), _stream(stream)),
               "spec_verify_shard_race")

    def finish(self, race_all, draft_tokens, accepted_len, out_tokens, stream=None):
        B, rows = out_tokens.shape
        _one_device(race_all, draft_tokens, accepted_len, out_tokens, stream=stream)
        _check(self.L.spec_verify_shard_finish(_ptr(race_all), race_all.shape[0], B, rows - 1, _ptr(draft_tokens),
                                               _ptr(accepted_len), _ptr(out_tokens), _stream(stream)),
               "spec_verify_shard_finish")


def spec_verify_shard_rank(target_shard: torch.Tensor, draft_shard: Optional[torch.Tensor], v0: int, V: int,
                           draft_tokens: torch.Tensor, draft_len: torch.Tensor, temperature: torch.Tensor,
                           seed: int = 0, group=None, error_word: Optional[torch.Tensor] = None,
                           accepted_len: Optional[torch.Tensor] = None, out_tokens: Optional[torch.Tensor] = None,
                           stream=None, ops=None):
    """One rank of a tensor-parallel group: this rank holds the vocabulary
    range [v0, v0 + Vs) of every row (target_shard [B, n_max+1, Vs],
    draft_shard [B, n_max, Vs] or None), ranks of `group` hold consecutive
    ranges in rank order, and every rank passes the same requests
    (draft_tokens, draft_len, temperature, seed).  The step's two exchanges
    are all-gathers over `group` (NCCL on GPUs); every rank ends with the
    same accepted_len [B] and out_tokens [B, n_max+1] as spec_verify on the
    whole vocabulary.  `ops` (default ShardOps()) runs the per-shard calls."""
    import contextlib

    import torch.distributed as dist

    ops = ops if ops is not None else ShardOps()
    S = dist.get_world_size(group)
    B, rows, _ = target_shard.shape
    n_max = rows - 1
    dev = target_shard.device
    _need(draft_tokens, B * n_max, "draft_tokens", torch.int32)
    _need(draft_len, B, "draft_len", torch.int32)
    _need(temperature, B, "temperature", torch.float32)
    if draft_shard is not None and (tuple(draft_shard.shape) != (B, n_max, target_shard.shape[2])
                                    or draft_shard.dtype != target_shard.dtype):
        raise ValueError("draft_shard must be [B, n_max, Vs] of the target shard's dtype")
    if accepted_len is None:
        accepted_len = torch.empty(B, dtype=torch.int32, device=dev)
    if out_tokens is None:
        out_tokens = torch.empty(B, rows, dtype=torch.int32, device=dev)
    _need(accepted_len, B, "accepted_len", torch.int32)
    _need(out_tokens, B * rows, "out_tokens", torch.int32)
    ctx = torch.cuda.stream(stream) if stream is not None else contextlib.nullcontext()
    with ctx:
        mine = ops.stats_buffer(B, n_max, dev)
        ops.stats(target_shard, draft_shard, V, v0, draft_tokens, draft_len, temperature, mine)
        stats_all = mine.new_empty((S,) + tuple(mine.shape))
        dist.all_gather(list(stats_all.unbind(0)), mine, group=group)
        mine_race = ops.race_buffer(B, dev)
        ops.race(target_shard, draft_shard, V, v0, draft_tokens, draft_len, temperature, seed, stats_all,
                 accepted_len, mine_race, error_word)
        race_all = mine_race.new_empty((S,) + tuple(mine_race.shape))
        dist.all_gather(list(race_all.unbind(0)), mine_race, group=group)
        ops.finish(race_all, draft_tokens, accepted_len, out_tokens)
    return accepted_len, out_tokens


def bytes_read(workspace: torch.Tensor) -> int:
    """Logits bytes read by early-exit calls on `workspace` since the last
    read (clears the count; synchronises the device)."""
    v = ctypes.c_uint64(0)
    _check(load_library().specdec_get_bytes_read(_ptr(workspace), ctypes.byref(v)), "specdec_get_bytes_read")
    return int(v.value)


def spec_verify_packed(target_logits: torch.Tensor, draft_logits: Optional[torch.Tensor],
                       cu_rows: torch.Tensor, draft_tokens: torch.Tensor, temperature: torch.Tensor,
                       n_max: int, seed: int = 0, pos_offset: Optional[torch.Tensor] = None,
                       accepted_len: Optional[torch.Tensor] = None,
                       out_tokens: Optional[torch.Tensor] = None, row_lse: Optional[torch.Tensor] = None,
                       workspace: Optional[torch.Tensor] = None, stream=None):
    """Verify/accept on packed ragged rows (see include/specdec.h).

    target_logits [total_rows, V]; draft_logits [total_rows - B, V] or None;
    cu_rows [B + 1] int32 (request b owns target rows cu_rows[b] ..
    cu_rows[b+1]-1, its draft rows and tokens start at cu_rows[b] - b);
    draft_tokens [total_rows - B] int32; n_max an upper bound of the draft
    lengths.  Returns (accepted_len [B], out_tokens [total_rows])."""
    total_rows, V = target_logits.shape
    B = cu_rows.numel() - 1
    dev = target_logits.device
    if B < 1 or total_rows < B:
        raise ValueError("cu_rows must hold B + 1 offsets with B <= total_rows")
    if cu_rows.dtype != torch.int32 or draft_tokens.dtype != torch.int32:
        raise TypeError("cu_rows and draft_tokens must be int32")
    if draft_logits is not None:
        if draft_logits.dtype != target_logits.dtype or tuple(draft_logits.shape) != (total_rows - B, V):
            raise ValueError("draft_logits must be [total_rows - B, V] of the target's dtype")
    _need(draft_tokens, total_rows - B, "draft_tokens", torch.int32)
    _need(temperature, B, "temperature", torch.float32)
    _need(pos_offset, B, "pos_offset", torch.int32)
    _need(accepted_len, B, "accepted_len", torch.int32)
    _need(out_tokens, total_rows, "out_tokens", torch.int32)
    _need(row_lse, total_rows * 2, "row_lse", torch.float32)
    with _on(stream):
        if accepted_len is None:
            accepted_len = torch.empty(B, dtype=torch.int32, device=dev)
        if out_tokens is None:
            out_tokens = torch.empty(total_rows, dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = new_workspace(B, n_max, V, device=dev, stream=stream)
    _one_device(target_logits, draft_logits, cu_rows, draft_tokens, temperature, pos_offset, accepted_len,
                out_tokens, row_lse, workspace, stream=stream)
    st = load_library().spec_verify_packed(
        _ptr(target_logits), _ptr(draft_logits), _dtype_code(target_logits), B, n_max, V,
        _ptr(cu_rows), total_rows, _ptr(draft_tokens), _ptr(temperature), _ptr(pos_offset),
        int(seed) & (2**64 - 1), _ptr(accepted_len), _ptr(out_tokens), _ptr(row_lse), _ptr(workspace),
        workspace.numel(), _stream(stream))
    _check(st, "spec_verify_packed")
    return accepted_len, out_tokens


def mtp_shift_insert(tokens_in: torch.Tensor, tokens_out: torch.Tensor, draft_len: torch.Tensor,
                     accepted_len: torch.Tensor, next_token: torch.Tensor,
                     next_token_stride: int = 0, seg_start: Optional[torch.Tensor] = None,
                     hidden_in: Optional[torch.Tensor] = None,
                     hidden_out: Optional[torch.Tensor] = None, error_word: Optional[torch.Tensor] = None,
                     stream=None):
    """MTP shift + insert on the device (see include/specdec.h).  error_word:
    optional device word (e.g. a spec_verify workspace, whose first word is its
    error word) that receives DEV_ERR_SEGMENT for a segment it could not move."""
    R = tokens_in.numel()
    B = draft_len.numel()
    _need(tokens_in, R, "tokens_in", torch.int32)
    _need(tokens_out, R, "tokens_out", torch.int32)
    _need(draft_len, B, "draft_len", torch.int32)
    _need(accepted_len, B, "accepted_len", torch.int32)
    _need(seg_start, B, "seg_start", torch.int32)
    if next_token.dtype != torch.int32:
        raise TypeError("next_token must be int32")
    if next_token.numel() < (B * next_token_stride if next_token_stride > 0 else B):
        raise ValueError("next_token is smaller than B rows of next_token_stride (or B)")
    H, eb = 0, 0
    if hidden_in is not None:
        if hidden_in.dim() != 2 or hidden_in.shape[0] != R:
            raise ValueError("hidden_in must be [R, H]")
        if hidden_out is not None and (hidden_out.shape != hidden_in.shape or hidden_out.dtype != hidden_in.dtype):
            raise ValueError("hidden_out must match hidden_in")
        H = hidden_in.shape[1]
        eb = hidden_in.element_size()
    if error_word is not None and (error_word.numel() * error_word.element_size() < 4):
        raise ValueError("error_word must hold at least 4 bytes")
    _one_device(tokens_in, tokens_out, draft_len, accepted_len, next_token, seg_start, hidden_in, hidden_out,
                error_word, stream=stream)
    st = load_library().mtp_shift_insert(
        _ptr(tokens_in), _ptr(tokens_out), _ptr(hidden_in), _ptr(hidden_out), R, H, eb,
        _ptr(seg_start), _ptr(draft_len), _ptr(accepted_len), _ptr(next_token),
        int(next_token_stride), B, _ptr(error_word), _stream(stream))
    _check(st, "mtp_shift_insert")
    return tokens_out


def get_error(workspace: torch.Tensor) -> int:
    """Read and clear the sticky device error word (synchronises the device)."""
    bits = ctypes.c_uint32(0)
    st = load_library().specdec_get_error(_ptr(workspace), ctypes.byref(bits))
    if st not in (0, 5, 6):
        _check(st, "specdec_get_error")
    return bits.value
