"""Seeded synthetic inputs for the verify/accept step and the MTP step.

This module is shared by the CPU oracle's tests and by the CUDA path's tests
and benchmark.  It holds none of the verify method's arithmetic: it only draws
logits, draft tokens (the stand-in for a draft model's own sampling), draft
lengths, temperatures and MTP buffers from torch's seeded generators.
"""
from .gen import CONFIGS, Workload, make_config, make_random, make_mtp, pack, unpack_rows  # noqa: F401
