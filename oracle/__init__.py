"""CPU oracle for the speculative-decoding verify/accept step and the MTP
shift/insert step.

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the
benchmark's CPU-baseline leg are the only callers.  The product library never
imports this module.  The arithmetic lives in ``specdec_oracle.c`` (plain C,
fp64, scalar loops); this file only compiles it with gcc and marshals numpy
arrays through ctypes.  It shares no code with the CUDA path.

Parity pins (what ties this oracle to something other than itself) are the
``-m "not gpu"`` tests in ``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "specdec_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libspecdec_oracle.so")
_lock = threading.Lock()
_lib = None

F32 = 0
BF16 = 1

ERR_TOKEN = 1
ERR_DRAFT_LEN = 2
ERR_TEMPERATURE = 4


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/libspecdec_oracle.so``.

    ``-ffp-contract=off`` keeps a*b+c as two roundings on every host, so the
    x86 build and the aarch64 build give the same doubles.
    """
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            P = ctypes.c_void_p
            i32, u32, u64, dbl = ctypes.c_int32, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_double
            L.oracle_philox4x32_10.argtypes = [P, P, P]
            L.oracle_philox4x32_10.restype = None
            L.oracle_uniform.argtypes = [u32]
            L.oracle_uniform.restype = dbl
            L.oracle_draw.argtypes = [u64, u32, u32, u32, u32]
            L.oracle_draw.restype = u32
            L.oracle_race.argtypes = [P, ctypes.c_int, u64, u32, u32, P]
            L.oracle_race.restype = ctypes.c_int
            L.oracle_spec_verify.argtypes = [P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int, P, P, P, u64, P, P, P, P, P, P, P]
            L.oracle_spec_verify.restype = u32
            L.oracle_row_lse_all.argtypes = [P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int, P, P, P]
            L.oracle_row_lse_all.restype = None
            L.oracle_mtp_shift_insert.argtypes = [P, P, P, P, ctypes.c_int, ctypes.c_int,
                                                  ctypes.c_int, P, P, P, P, ctypes.c_int,
                                                  ctypes.c_int]
            L.oracle_mtp_shift_insert.restype = ctypes.c_int
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def philox4x32_10(ctr, key):
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    lib().oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def uniform(w: int) -> float:
    return lib().oracle_uniform(int(w) & 0xFFFFFFFF)


def draw(seed: int, b: int, j: int, v: int, purpose: int) -> int:
    return int(lib().oracle_draw(seed, b, j, v, purpose))


def race(r, seed: int, b: int, j: int):
    """Exponential race over weights r; returns (winner, top-2 relative gap)."""
    rr = np.ascontiguousarray(r, dtype=np.float64)
    gap = ctypes.c_double(0.0)
    y = lib().oracle_race(_ptr(rr), rr.size, seed, b, j, ctypes.byref(gap))
    return int(y), gap.value


def _as_logits(x):
    """numpy float32 -> (array, F32); numpy uint16 (raw bf16 bits) -> (array, BF16)."""
    if x is None:
        return None, None
    x = np.ascontiguousarray(x)
    if x.dtype == np.float32:
        return x, F32
    if x.dtype == np.uint16:
        return x, BF16
    raise TypeError(f"oracle logits must be float32 or uint16 (bf16 bits), got {x.dtype}")


def spec_verify(target, draft, draft_tokens, draft_len, temperature, seed: int,
                req_ids=None, pos_off=None, want_stats: bool = True):
    """Run the oracle on a dense batch.

    target [B, n_max+1, V], draft [B, n_max, V] or None; float32 or uint16
    (bf16 bits).  Returns a dict with accepted_len [B], out_tokens [B, n_max+1],
    row_lse [B, n_max+1, 2], accept_margin [B, n_max], race_gap [B], err.
    """
    t, dt = _as_logits(target)
    d, dd = _as_logits(draft)
    if d is not None and dd != dt:
        raise TypeError("target and draft dtypes differ")
    B, rows, V = t.shape
    n_max = rows - 1
    if d is not None and d.shape != (B, n_max, V):
        raise ValueError("draft shape mismatch")
    x = np.ascontiguousarray(draft_tokens, dtype=np.int32).reshape(B, n_max)
    L = np.ascontiguousarray(draft_len, dtype=np.int32).reshape(B)
    T = np.ascontiguousarray(temperature, dtype=np.float32).reshape(B)
    rid = None if req_ids is None else np.ascontiguousarray(req_ids, dtype=np.int32).reshape(B)
    pof = None if pos_off is None else np.ascontiguousarray(pos_off, dtype=np.int32).reshape(B)
    acc = np.zeros(B, dtype=np.int32)
    out = np.zeros((B, rows), dtype=np.int32)
    lse = np.zeros((B, rows, 2), dtype=np.float64) if want_stats else None
    margin = np.zeros((B, max(n_max, 1)), dtype=np.float64) if want_stats else None
    gap = np.zeros(B, dtype=np.float64) if want_stats else None
    err = lib().oracle_spec_verify(_ptr(t), _ptr(d), dt, B, n_max, V, _ptr(x), _ptr(L),
                                   _ptr(T), int(seed) & 0xFFFFFFFFFFFFFFFF, _ptr(rid), _ptr(pof),
                                   _ptr(acc), _ptr(out), _ptr(lse), _ptr(margin), _ptr(gap))
    res = {"accepted_len": acc, "out_tokens": out, "err": int(err)}
    if want_stats:
        res.update(row_lse=lse, accept_margin=margin[:, :n_max], race_gap=gap)
    return res


def row_lse_all(target, draft, draft_len, temperature):
    """LSE of s*row for every valid target and draft row: [B, n_max+1, 2]."""
    t, dt = _as_logits(target)
    d, _ = _as_logits(draft)
    B, rows, V = t.shape
    L = np.ascontiguousarray(draft_len, dtype=np.int32).reshape(B)
    T = np.ascontiguousarray(temperature, dtype=np.float32).reshape(B)
    out = np.zeros((B, rows, 2), dtype=np.float64)
    lib().oracle_row_lse_all(_ptr(t), _ptr(d), dt, B, rows - 1, V, _ptr(L), _ptr(T), _ptr(out))
    return out


def mtp_shift_insert(tokens_in, tokens_out, draft_len, accepted_len, next_token,
                     next_token_stride: int, seg_start=None, hidden_in=None,
                     hidden_out=None):
    """In-place on ``tokens_out`` (and ``hidden_out``); returns the bad-segment flag."""
    tin = np.ascontiguousarray(tokens_in, dtype=np.int32)
    assert tokens_out.dtype == np.int32 and tokens_out.flags.c_contiguous
    R = tin.size
    B = int(np.asarray(draft_len).size)
    n = np.ascontiguousarray(draft_len, dtype=np.int32)
    a = np.ascontiguousarray(accepted_len, dtype=np.int32)
    nt = np.ascontiguousarray(next_token, dtype=np.int32)
    ss = None if seg_start is None else np.ascontiguousarray(seg_start, dtype=np.int32)
    H, eb = 0, 0
    if hidden_in is not None:
        assert hidden_out is not None and hidden_out.flags.c_contiguous
        H = hidden_in.shape[1]
        eb = hidden_in.dtype.itemsize
        hidden_in = np.ascontiguousarray(hidden_in)
    return lib().oracle_mtp_shift_insert(_ptr(tin), _ptr(tokens_out), _ptr(hidden_in),
                                         _ptr(hidden_out), R, H, eb, _ptr(ss), _ptr(n), _ptr(a),
                                         _ptr(nt), int(next_token_stride), B)
