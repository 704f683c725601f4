"""ssm_prefill_scratch (the prefill that runs its chunked form in the
library's fixed device scratch) against ssm_prefill with a caller workspace,
on two consecutive calls: the same chunk length is chosen, so the results
agree bit for bit. Collected last on purpose: it must also pass after every
other test has run in the same process."""
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


def test_scratch_prefill_rejects_oversize_shapes(cuda_device):
    """A 8192-token prompt of a Llama-3-8B-shaped layer needs more chunk
    states than the scratch holds: refused before anything is launched."""
    dev = cuda_device
    T, H, P, N, G = 8192, 32, 128, 128, 8
    pool = torch.zeros(1, H, P, N, device=dev)
    x = torch.zeros(1, T, H, P, dtype=torch.bfloat16, device=dev)
    B = torch.zeros(1, T, G, N, dtype=torch.bfloat16, device=dev)
    dt = torch.zeros(1, T, H, dtype=torch.bfloat16, device=dev)
    A, D = torch.zeros(H, device=dev), torch.zeros(H, device=dev)
    assert ssm.prefill_workspace_bytes(pool, x, B, B, dt, A, D) > sv.SSM_PREFILL_SCRATCH_BYTES
    y = torch.full((1, T, H, P), 3.0, device=dev)
    with pytest.raises(sv.SsmError) as e:
        sv.prefill_scratch(pool, None, x, B, B, dt, A, D, y=y)
    assert e.value.code == sv.SSM_ERR_SHAPE
    torch.cuda.synchronize()
    assert (y == 3.0).all() and (pool == 0).all()
