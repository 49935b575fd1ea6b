"""Pins of the oracle's MTP shift/insert step against hand-written cases.

Source: "Accelerating Sonar through speculation", §MTP and §Single-token MTP
scheduling; the cases and their citation live in
tests/golden/mtp_shift_insert_cases.json.
"""
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "mtp_shift_insert_cases.json")


def _cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c["name"])
@pytest.mark.parametrize("in_place", [False, True])
def test_mtp_hand_cases(case, in_place):
    tin = np.array(case["tokens_in"], np.int32)
    fill = -7 if case["name"].startswith("segment not covering") else None
    if in_place:
        if fill is not None:
            pytest.skip("the uncovered-slot case is defined for a distinct output buffer")
        out = tin.copy()
        src = out
    else:
        out = np.full_like(tin, -7 if fill is not None else -1)
        src = tin
        if fill is None:
            out[:] = tin  # slots outside segments keep their contents
    bad = oracle.mtp_shift_insert(src, out, case["draft_len"], case["accepted_len"],
                                  case["next_token"], 0, seg_start=case["seg_start"])
    assert bad == 0
    assert out.tolist() == case["expected"]


def test_mtp_next_token_from_out_tokens_layout():
    # next token read as out_tokens[b, a_b] (stride n_max + 1).
    out_tokens = np.array([[11, 12, 13], [21, -1, -1]], np.int32)
    tin = np.array([1, 2, 3, 4, 5, 6], np.int32)
    out = tin.copy()
    oracle.mtp_shift_insert(tin, out, [2, 2], [2, 0], out_tokens.ravel(), 3)
    assert out.tolist() == [2, 3, 13, 21, 6, 6]


def test_mtp_hidden_copy_is_bitwise():
    rng = np.random.default_rng(0)
    hin = rng.integers(0, 2**16, size=(4, 9), dtype=np.uint16)
    hout = np.zeros_like(hin)
    tin = np.arange(4, dtype=np.int32)
    out = tin.copy()
    oracle.mtp_shift_insert(tin, out, [1, 1], [0, 1], [7, 8], 0, hidden_in=hin, hidden_out=hout)
    assert (hout == hin).all()
    assert out.tolist() == [7, 1, 3, 8]


def test_mtp_rejects_segments_outside_the_buffer():
    tin = np.arange(4, dtype=np.int32)
    out = tin.copy()
    assert oracle.mtp_shift_insert(tin, out, [3], [0], [9], 0, seg_start=[2]) == 1
