"""ssm_prefill_scratch (the prefill that runs its chunked form in the
library's fixed device scratch) against ssm_prefill with a caller workspace,
on two consecutive calls: the same chunk length is chosen, so the results
agree bit for bit. The entry point serves callers that cannot allocate
device memory: a host runtime that owns every device allocation and passes
the library only tensor pointers, or a serving loop that must not call
cudaMalloc (it can synchronise the device) between steps. Collected last on
purpose: it must also pass after every other test has run in the same
process."""
import pytest
import torch

import ssm_recurrence_verify_b300 as ssm
from ssm_recurrence_verify_b300 import ssmverify as sv
from ssm_recurrence_verify_b300 import synth

pytestmark = pytest.mark.gpu


def _case(seed, dev, T=1024):
    wl = synth.custom_workload(2, 8, 64, 128, 2, T, synth.BF16, seed=seed)
    p = synth.draw_params(wl)
    t = {k: v.to(dev) for k, v in synth.draw_tokens(wl, 0).items()}
    return p, t


def test_scratch_prefill_equals_workspace_prefill(cuda_device):
    dev = cuda_device
    for call in range(2):  # two consecutive calls: the scratch is reused
        p, t = _case(600 + call, dev)
        A, D = p["A"].to(dev), p["D"].to(dev)
        slot = torch.tensor([2, 0], dtype=torch.int32, device=dev)
        pool0 = torch.zeros(3, 8, 64, 128)
        pool0[[2, 0]] = p["state0"]
        need = ssm.prefill_workspace_bytes(pool0.to(dev), t["x"], t["B"], t["C"], t["dt"], A, D)
        assert 0 < need <= sv.SSM_PREFILL_SCRATCH_BYTES
        pool_a, pool_b = pool0.clone().to(dev), pool0.clone().to(dev)
        st = torch.zeros(2, dtype=torch.int32, device=dev)
        y_a = ssm.prefill(pool_a, slot, t["x"], t["B"], t["C"], t["dt"], A, D, dev_status=st[:1])
        y_b = sv.prefill_scratch(pool_b, slot, t["x"], t["B"], t["C"], t["dt"], A, D, dev_status=st[1:])
        torch.cuda.synchronize()
        assert st.tolist() == [0, 0]
        assert torch.equal(y_a, y_b) and torch.equal(pool_a, pool_b), call


def test_scratch_prefill_beyond_the_scratch(cuda_device):
    """A 4096-token prompt of a Llama-3-8B-shaped layer needs more chunk
    states than the scratch holds (32 chunks of 2 MiB and a slot map): the
    scratch form then takes a chunk length that fits, or the one-pass form,
    and its results equal ssm_prefill's given a workspace of the scratch's
    size."""
    dev = cuda_device
    T, H, P, N, G = 4096, 32, 128, 128, 8
    wl = synth.custom_workload(1, H, P, N, G, T, synth.BF16, seed=990)
    t = {k: v.to(dev) for k, v in synth.draw_tokens(wl, 0).items()}
    p = synth.draw_params(wl)
    A, D = p["A"].to(dev), p["D"].to(dev)
    pool1 = torch.zeros(1, H, P, N, device=dev)
    assert ssm.prefill_workspace_bytes(pool1, t["x"], t["B"], t["C"], t["dt"], A, D) > sv.SSM_PREFILL_SCRATCH_BYTES
    y1 = sv.prefill_scratch(pool1, None, t["x"], t["B"], t["C"], t["dt"], A, D)
    pool2 = torch.zeros(1, H, P, N, device=dev)
    ws = torch.empty(sv.SSM_PREFILL_SCRATCH_BYTES // 4, device=dev)
    y2 = ssm.prefill(pool2, None, t["x"], t["B"], t["C"], t["dt"], A, D, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2) and torch.equal(pool1, pool2)
