"""libssmverify: the Mamba-layer verify / commit / step of speculative
decoding as hand-written CUDA for B300 (sm_103a), behind a C ABI.

``from ssm_recurrence_verify_b300 import verify, commit, verify_commit, commit_verify, step``
calls the C library on torch CUDA tensors; ``synth`` draws the seeded
synthetic workloads. The CUDA library is loaded on first use and its absence
is an error (there is no CPU fallback).
"""
from .ssmverify import (  # noqa: F401
    SsmError, commit, commit_verify, load_library, step, strerror, verify, verify_commit,
)
