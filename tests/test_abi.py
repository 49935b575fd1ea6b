"""The C ABI library loads and exports every function include/*.h
declares; host-side argument checks return their status codes before any
device work (CPU only: no kernel is launched here)."""
import ctypes
import os
import re

import pytest

import speculative_decoding_verification_80_gb300 as sd

INCLUDE = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include")
HEADERS = [os.path.join(INCLUDE, h) for h in ("specdec.h", "specdec_shard.h")]


def _declared_functions():
    text = "".join(open(h).read() for h in HEADERS)
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_\s\*]*?\b([A-Za-z_][A-Za-z0-9_]*)\s*\(",
                       text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "defined")))


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_verification_80_gb300 import build

    build.build()
    return sd.load_library()


def test_header_declares_the_binding_exports():
    assert sorted(sd.EXPORTS) == _declared_functions()


def test_every_declared_symbol_is_exported(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    assert lib.specdec_status_string(0) == b"SPECDEC_OK"
    assert lib.specdec_status_string(3) == b"SPECDEC_ERR_WORKSPACE"
    assert lib.specdec_status_string(6) == b"SPECDEC_ERR_TIMEOUT"
    assert lib.specdec_status_string(7) == b"SPECDEC_UNKNOWN_STATUS"


def test_status_and_error_bits_match_the_header():
    text = open(HEADERS[0]).read()
    for name, value in (("SPECDEC_ERR_DEVICE_DATA", 5), ("SPECDEC_ERR_TIMEOUT", 6)):
        assert re.search(rf"\b{name}\s*=\s*{value}\b", text), name
    for name, value in (("SPECDEC_DEV_ERR_TOKEN", sd.DEV_ERR_TOKEN), ("SPECDEC_DEV_ERR_DRAFT_LEN", sd.DEV_ERR_DRAFT_LEN),
                        ("SPECDEC_DEV_ERR_TEMPERATURE", sd.DEV_ERR_TEMPERATURE),
                        ("SPECDEC_DEV_ERR_TIMEOUT", sd.DEV_ERR_TIMEOUT), ("SPECDEC_DEV_ERR_SEGMENT", sd.DEV_ERR_SEGMENT)):
        assert re.search(rf"#define\s+{name}\s+{value}u\b", text), name


def test_no_alloc_rejects_bad_arguments_before_enqueueing(lib):
    # a bad dtype, a null pointer: the status comes back with no workspace clear
    # enqueued (no device needed: the call never reaches CUDA)
    P = ctypes.c_void_p
    fake = P(0x1000)
    assert lib.spec_verify_no_alloc(fake, fake, 7, 4, 3, 1024, fake, fake, fake, 0, fake, fake, None, None) == 1
    assert lib.spec_verify_no_alloc(None, fake, 0, 4, 3, 1024, fake, fake, fake, 0, fake, fake, None, None) == 1
    assert lib.spec_verify_no_alloc(fake, fake, 0, 4, 3, 1024, fake, None, fake, 0, fake, fake, None, None) == 1


def test_workspace_size_is_host_only(lib):
    n = lib.specdec_verify_workspace_bytes(64, 4, 128256)
    assert n >= 64 * 5 * 12 and n % 256 == 0
    assert lib.specdec_verify_workspace_bytes(64, 4, 0) == 0
    assert lib.specdec_verify_workspace_bytes(0, 4, 10) == 0
    assert lib.specdec_verify_workspace_bytes(4, -1, 10) == 0


@pytest.mark.parametrize("V,dtype", [(1024, sd.F32), (128256, sd.BF16), (129280, sd.BF16),
                                     (152064, sd.BF16), (7, sd.BF16), (4097, sd.BF16), (262144, sd.F32)])
@pytest.mark.parametrize("B,n_max", [(64, 4), (1, 0), (512, 4), (1024, 7)])
def test_launch_shapes(lib, B, n_max, V, dtype):
    n, ch = ctypes.c_int32(0), ctypes.c_int32(0)
    assert lib.specdec_verify_launch_shape(B, n_max, V, dtype, ctypes.byref(n), ctypes.byref(ch)) == 0
    elt = 4 if dtype == sd.F32 else 2
    upper = B * (2 * n_max + 1) * V * elt  # bytes if every row is read
    assert ch.value * elt == (28 if upper >= 300e6 else 24) * 1024  # chunk bytes, at most one stage
    assert n.value * ch.value >= V and (n.value - 1) * ch.value < V


def test_launch_shape_rejects_bad_shapes(lib):
    n, ch = ctypes.c_int32(0), ctypes.c_int32(0)
    for args in [(0, 4, 1024, sd.BF16), (4, -1, 1024, sd.BF16), (4, 4, 0, sd.BF16), (4, 4, 1024, 9)]:
        assert lib.specdec_verify_launch_shape(*args, ctypes.byref(n), ctypes.byref(ch)) == 1


def test_argument_errors_return_codes_without_device_work(lib):
    P = ctypes.c_void_p
    fake = P(0x1000)
    # bad dtype
    assert lib.spec_verify(fake, fake, 7, 4, 3, 1024, fake, fake, fake, 0, fake, fake, None, fake,
                           1 << 20, None) == 1
    # null target
    assert lib.spec_verify(None, fake, 0, 4, 3, 1024, fake, fake, fake, 0, fake, fake, None, fake,
                           1 << 20, None) == 1
    # V <= 0, vocab too large
    assert lib.spec_verify(fake, fake, 0, 4, 3, 0, fake, fake, fake, 0, fake, fake, None, fake,
                           1 << 20, None) == 1
    assert lib.spec_verify(fake, fake, 0, 4, 3, 1 << 20, fake, fake, fake, 0, fake, fake, None,
                           fake, 1 << 20, None) == 2
    # workspace missing / too small / misaligned
    assert lib.spec_verify(fake, fake, 0, 4, 3, 1024, fake, fake, fake, 0, fake, fake, None, None,
                           1 << 20, None) == 3
    assert lib.spec_verify(fake, fake, 0, 4, 3, 1024, fake, fake, fake, 0, fake, fake, None, fake,
                           16, None) == 3
    assert lib.spec_verify(fake, fake, 0, 4, 3, 1024, fake, fake, fake, 0, fake, fake, None,
                           P(0x1001), 1 << 20, None) == 3
    # empty batch is a no-op
    assert lib.spec_verify(None, None, 0, 0, 3, 1024, None, None, None, 0, None, None, None, None,
                           0, None) == 0
    # mtp: null buffers, R not divisible by B without seg_start
    assert lib.mtp_shift_insert(None, fake, None, None, 8, 0, 0, None, fake, fake, fake, 0, 2,
                                None, None) == 1
    assert lib.mtp_shift_insert(fake, fake, None, None, 7, 0, 0, None, fake, fake, fake, 0, 2,
                                None, None) == 1
    assert lib.mtp_shift_insert(fake, fake, None, fake, 8, 4, 2, None, fake, fake, fake, 0, 2,
                                None, None) == 1


def test_packed_argument_errors_return_codes_without_device_work(lib):
    P = ctypes.c_void_p
    fake = P(0x1000)

    def call(target=fake, dtype=0, B=4, n_max=3, V=1024, cu=fake, total=10, tokens=fake, ws=fake,
             ws_bytes=1 << 20):
        return lib.spec_verify_packed(target, fake, dtype, B, n_max, V, cu, total, tokens, fake, None, 0,
                                      fake, fake, None, ws, ws_bytes, None)

    assert call(dtype=7) == 1            # bad dtype
    assert call(target=None) == 1        # null target
    assert call(cu=None) == 1            # no offsets
    assert call(total=3) == 1            # fewer rows than requests
    assert call(tokens=None) == 1        # drafts present but no tokens
    assert call(V=0) == 1
    assert call(V=1 << 20) == 2          # vocabulary too large
    assert call(n_max=1 << 20) == 2      # draft bound too large
    assert call(ws=None) == 3            # workspace missing / too small / misaligned
    assert call(ws_bytes=16) == 3
    assert call(ws=P(0x1001)) == 3
    assert call(B=0, total=0, target=None, cu=None, tokens=None) == 0  # empty batch: no-op


def test_early_exit_argument_errors_return_codes_without_device_work(lib):
    P = ctypes.c_void_p
    fake = P(0x1000)

    def call(dtype=0, B=4, n_max=3, V=1024, target=fake, ws=fake, ws_bytes=1 << 20):
        return lib.spec_verify_early_exit(target, fake, dtype, B, n_max, V, fake, fake, fake, 0, fake, fake,
                                          ws, ws_bytes, None)

    assert call(dtype=7) == 1
    assert call(target=None) == 1
    assert call(n_max=sd.EARLY_EXIT_MAX_DRAFT + 1) == 2  # beyond the done-row mask
    assert call(V=1 << 20) == 2
    assert call(ws=None) == 3
    assert call(ws_bytes=16) == 3
    assert call(B=0, target=None) == 0
    v = ctypes.c_uint64(0)
    assert lib.specdec_get_bytes_read(None, ctypes.byref(v)) == 1


def test_binding_rejects_wrong_sizes_on_the_host():
    # Size and dtype mismatches are caught before any pointer reaches the
    # library (no device needed: the checks run first).
    import torch

    t = torch.zeros(4, 3, 16)
    d = torch.zeros(4, 2, 16)
    x = torch.zeros(4, 2, dtype=torch.int32)
    L = torch.zeros(4, dtype=torch.int32)
    T = torch.zeros(4)
    with pytest.raises(ValueError):
        sd.spec_verify(t, d, torch.zeros(4, 3, dtype=torch.int32), L, T)
    with pytest.raises(ValueError):
        sd.spec_verify(t, d, x, torch.zeros(5, dtype=torch.int32), T)
    with pytest.raises(TypeError):
        sd.spec_verify(t, d, x, L, torch.zeros(4, dtype=torch.float64))
    with pytest.raises(ValueError):
        sd.spec_verify(t, d, x, L, T, out_tokens=torch.zeros(4, 2, dtype=torch.int32))
    with pytest.raises(ValueError):
        sd.spec_verify_early_exit(t, d, x, L, torch.zeros(3))
    tok = torch.zeros(12, dtype=torch.int32)
    with pytest.raises(ValueError):
        sd.mtp_shift_insert(tok, torch.zeros(11, dtype=torch.int32), L, L, L, 0)
    with pytest.raises(ValueError):
        sd.mtp_shift_insert(tok, tok, L, L, torch.zeros(8, dtype=torch.int32), 3)


def test_shard_argument_errors_return_codes_without_device_work(lib):
    P = ctypes.c_void_p
    fake = P(0x1000)

    def stats(dtype=0, B=4, n_max=3, V=1000, v0=0, Vs=500, target=fake, out=fake):
        return lib.spec_verify_shard_stats(target, fake, dtype, B, n_max, V, v0, Vs, fake, fake, fake, out, None)

    assert stats(dtype=7) == 1
    assert stats(target=None) == 1
    assert stats(out=None) == 1
    assert stats(v0=-1) == 1
    assert stats(Vs=0) == 1
    assert stats(v0=600) == 1            # v0 + Vs > V
    assert stats(V=1 << 20, Vs=10) == 2
    assert stats(B=0, target=None) == 0
    assert lib.spec_verify_shard_race(fake, fake, 0, 4, 3, 1000, 0, 500, fake, fake, fake, 0, fake, 0,
                                      fake, fake, None, None) == 1  # S = 0
    assert lib.spec_verify_shard_race(fake, fake, 0, 4, 3, 1000, 0, 500, fake, fake, fake, 0, None, 2,
                                      fake, fake, None, None) == 1  # no gathered records
    assert lib.spec_verify_shard_finish(fake, 0, 4, 3, fake, fake, fake, None) == 1
    assert lib.spec_verify_shard_finish(None, 2, 4, 3, fake, fake, fake, None) == 1
    assert lib.specdec_shard_stats_records(4, 3) == 4 * 4 * 2
    assert lib.specdec_shard_stats_records(0, 3) == 0
    # race records: a few per request, depending on B alone
    for B in (1, 4, 64, 100, 512, 1024, 4096):
        n = lib.specdec_shard_race_records(B)
        assert n % B == 0 and 1 <= n // B <= 16 and (B < 512 or n == B)
    assert lib.specdec_shard_race_records(0) == 0


def test_tensors_of_one_call_must_share_a_device():
    # Host check before any pointer is taken: a tensor on another device
    # never reaches the library.
    import torch

    sd._one_device(torch.zeros(2), None, torch.zeros(3))  # one device: no error (CPU is rejected later)
    with pytest.raises(ValueError, match="share a device"):
        sd._one_device(torch.zeros(2), torch.empty(2, device="meta"))
