"""libssmverify: the Mamba-layer verify / commit / step of speculative
decoding as hand-written CUDA for B300 (sm_103a), behind a C ABI.

``from ssm_recurrence_verify_b300 import verify, commit, verify_commit, commit_verify, step``
calls the C library on torch CUDA tensors; ``accept_greedy`` / ``accept_sample``
decide accept_len on the device from the verifier's (and draft's) logits;
``*_pool`` run on slots of a state pool and ``prefill`` builds the cached state from a prompt; ``synth`` draws the seeded
synthetic workloads. The CUDA library is loaded on first use and its absence
is an error (there is no CPU fallback).
"""
from .ssmverify import (  # noqa: F401
    SsmError, accept_greedy, accept_sample, commit, commit_pool, commit_verify, commit_verify_pool, load_library,
    prefill, prefill_workspace_bytes, step, step_pool, strerror, verify, verify_commit, verify_commit_pool,
    verify_pool,
)
