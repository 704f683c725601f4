"""Bit-exact identities between the CUDA entry points (GPU, through the C ABI).

The accepted-prefix selection must be exact: the state committed by the fused
kernel after K drafted tokens with j accepted is, bit for bit, the state of
  * ssm_commit with the same j,
  * a fused run drafting only the j accepted tokens,
and j = 0 leaves the cached state bitwise unchanged. y does not depend on the
entry point (verify and verify_commit) nor on j. j plain single-token steps
reach the same state up to fp32 rounding: at N <= 128 the kernels advance the
state by one rank-m tensor-core update over the m tokens of a chunk, and m
rank-1 updates round differently.
"""
import pytest
import torch

import ssm_recurrence_verify_b300 as ssm
from gpu_helpers import np64, rel_err, to_dev
from ssm_recurrence_verify_b300 import synth

pytestmark = pytest.mark.gpu

STEP_RTOL = 1e-5  # j rank-1 updates against one rank-j update: a few fp32 roundings per element

CASES = [
    (8, 4, 128, 128, 2, 8, synth.BF16),
    (6, 3, 70, 64, 1, 17, synth.F32),
    (4, 2, 16, 16, 2, 5, synth.F32),
    (3, 2, 40, 256, 2, 6, synth.BF16),
]


def _inputs(case, dev):
    wl = synth.custom_workload(*case, seed=1000 + case[5])
    d = synth.draw_layer_round(wl)
    K = case[5]
    d["accept_len"] = (torch.arange(case[0], dtype=torch.int32) * 3) % (K + 1)  # covers 0 and K
    if case[0] > 1:
        d["accept_len"][-1] = K
    return to_dev(d, dev), K


@pytest.mark.parametrize("case", CASES, ids=lambda s: "b{}h{}p{}n{}g{}k{}{}".format(*s))
def test_fused_commit_step_agree(cuda_device, case):
    d, K = _inputs(case, cuda_device)
    acc = d["accept_len"]
    s_fused = d["state0"].clone()
    y_fused = ssm.verify_commit(s_fused, d["x"], d["B"], d["C"], d["dt"], d["A"], d["D"], acc)

    s_commit = d["state0"].clone()
    ssm.commit(s_commit, d["x"], d["B"], d["dt"], d["A"], acc)

    y_ver = ssm.verify(d["state0"], d["x"], d["B"], d["C"], d["dt"], d["A"], d["D"])
    torch.cuda.synchronize()
    assert torch.equal(s_fused, s_commit)
    assert torch.equal(y_fused, y_ver)

    for b in range(case[0]):
        j = int(acc[b])
        s_step = d["state0"][b:b + 1].clone()
        for t in range(j):
            ssm.step(s_step, d["x"][b:b + 1, t:t + 1].contiguous(), d["B"][b:b + 1, t:t + 1].contiguous(),
                     d["C"][b:b + 1, t:t + 1].contiguous(), d["dt"][b:b + 1, t:t + 1].contiguous(), d["A"], d["D"])
        torch.cuda.synchronize()
        if case[3] > 128:  # token-by-token recurrence in every entry point
            assert torch.equal(s_step[0], s_fused[b]), (b, j)
        else:
            assert rel_err(np64(s_step[0]), np64(s_fused[b])) <= STEP_RTOL, (b, j)
        if j == 0:
            assert torch.equal(s_fused[b], d["state0"][b])
        else:
            s_short = d["state0"][b:b + 1].clone()
            y_short = ssm.verify_commit(s_short, d["x"][b:b + 1, :j].contiguous(), d["B"][b:b + 1, :j].contiguous(),
                                        d["C"][b:b + 1, :j].contiguous(), d["dt"][b:b + 1, :j].contiguous(), d["A"],
                                        d["D"], torch.full((1,), j, dtype=torch.int32, device=cuda_device))
            torch.cuda.synchronize()
            assert torch.equal(s_short[0], s_fused[b]), (b, j)
            assert torch.equal(y_short[0], y_fused[b, :j]), (b, j)


def test_y_independent_of_accept_len(cuda_device):
    d, K = _inputs(CASES[0], cuda_device)
    ys = []
    for j in (0, 3, K):
        s = d["state0"].clone()
        acc = torch.full_like(d["accept_len"], j)
        ys.append(ssm.verify_commit(s, d["x"], d["B"], d["C"], d["dt"], d["A"], d["D"], acc))
    torch.cuda.synchronize()
    assert torch.equal(ys[0], ys[1]) and torch.equal(ys[0], ys[2])


def test_bad_accept_len_sets_status_and_keeps_state(cuda_device):
    d, K = _inputs(CASES[0], cuda_device)
    acc = d["accept_len"].clone()
    acc[1] = -1
    acc[2] = K + 1
    good = d["accept_len"].clone()
    good[1] = 0
    good[2] = 0
    for fn in ("verify_commit", "commit"):
        s = d["state0"].clone()
        s_ref = d["state0"].clone()
        status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
        if fn == "verify_commit":
            ssm.verify_commit(s, d["x"], d["B"], d["C"], d["dt"], d["A"], d["D"], acc, dev_status=status)
            ssm.verify_commit(s_ref, d["x"], d["B"], d["C"], d["dt"], d["A"], d["D"], good)
        else:
            ssm.commit(s, d["x"], d["B"], d["dt"], d["A"], acc, dev_status=status)
            ssm.commit(s_ref, d["x"], d["B"], d["dt"], d["A"], good)
        torch.cuda.synchronize()
        assert int(status.item()) & ssm.ssmverify.SSM_STATUS_BAD_ACCEPT_LEN, fn
        assert torch.equal(s, s_ref), fn
        assert torch.equal(s[1], d["state0"][1]) and torch.equal(s[2], d["state0"][2])


def test_repeat_is_deterministic(cuda_device):
    d, K = _inputs(CASES[1], cuda_device)
    outs = []
    for _ in range(2):
        s = d["state0"].clone()
        y = ssm.verify_commit(s, d["x"], d["B"], d["C"], d["dt"], d["A"], d["D"], d["accept_len"])
        outs.append((s, y))
    torch.cuda.synchronize()
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


@pytest.mark.parametrize("case", CASES, ids=lambda s: "b{}h{}p{}n{}g{}k{}{}".format(*s))
def test_commit_verify_equals_commit_then_verify(cuda_device, case):
    """The deferred-commit kernel gives bit for bit the state of ssm_commit on
    the previous block and the y of ssm_verify from that state."""
    d, K = _inputs(case, cuda_device)
    new = synth.custom_workload(case[0], case[1], case[2], case[3], case[4], max(1, K // 2 + 1), case[6],
                                seed=3000 + K)
    n = to_dev(synth.draw_tokens(new, 1), cuda_device)
    s1 = d["state0"].clone()
    y1 = ssm.commit_verify(s1, d["x"], d["B"], d["dt"], d["accept_len"], n["x"], n["B"], n["C"], n["dt"], d["A"],
                           d["D"])
    s2 = d["state0"].clone()
    ssm.commit(s2, d["x"], d["B"], d["dt"], d["A"], d["accept_len"])
    y2 = ssm.verify(s2, n["x"], n["B"], n["C"], n["dt"], d["A"], d["D"])
    torch.cuda.synchronize()
    assert torch.equal(s1, s2)
    assert torch.equal(y1, y2)
