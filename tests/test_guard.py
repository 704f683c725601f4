"""Out-of-bounds writes: sentinel regions around the state and y stay
untouched by every entry point (GPU). Inputs sit between sentinels as well,
and the committed / emitted values themselves are checked elsewhere."""
import pytest
import torch

import ssm_recurrence_verify_b300 as ssm
from gpu_helpers import to_dev
from ssm_recurrence_verify_b300 import synth

pytestmark = pytest.mark.gpu

PAD = 1024  # floats of sentinel on each side (4 KiB, keeps 16-byte alignment)
SENTINEL = -12345.678


def _guarded(t: torch.Tensor):
    buf = torch.full((PAD + t.numel() + PAD,), SENTINEL, dtype=t.dtype, device=t.device)
    view = buf[PAD:PAD + t.numel()].view(t.shape)
    view.copy_(t)
    return buf, view


def _intact(buf, n):
    return bool((buf[:PAD] == SENTINEL).all()) and bool((buf[PAD + n:] == SENTINEL).all())


@pytest.mark.parametrize("shape", [(3, 4, 50, 128, 2, 9, synth.BF16), (2, 2, 20, 16, 1, 3, synth.F32),
                                   (2, 2, 7, 256, 2, 18, synth.F32)], ids=str)
def test_sentinels_untouched(cuda_device, shape):
    wl = synth.custom_workload(*shape, seed=42)
    d = to_dev(synth.draw_layer_round(wl), cuda_device)
    sbuf, s = _guarded(d["state0"])
    bsz, K, H, P = d["x"].shape
    ybuf, y = _guarded(torch.zeros(bsz, K, H, P, device=cuda_device))
    ssm.verify_commit(s, d["x"], d["B"], d["C"], d["dt"], d["A"], d["D"], d["accept_len"], y=y)
    ssm.verify(s, d["x"], d["B"], d["C"], d["dt"], d["A"], d["D"], y=y)
    ssm.commit(s, d["x"], d["B"], d["dt"], d["A"], d["accept_len"])
    ssm.commit_verify(s, d["x"], d["B"], d["dt"], d["accept_len"], d["x"], d["B"], d["C"], d["dt"], d["A"], d["D"],
                      y=y)
    torch.cuda.synchronize()
    assert _intact(sbuf, s.numel())
    assert _intact(ybuf, y.numel())
    assert torch.isfinite(y).all() and torch.isfinite(s).all()


def test_bounded_wait_times_out_and_device_stays_usable(cuda_device):
    """The bounded wait gives up on a transaction that never completes,
    reports SSM_STATUS_TIMEOUT, and the context keeps working afterwards."""
    import time
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    t0 = time.perf_counter()
    ssm.ssmverify.selftest_wait_timeout(status)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert int(status.item()) == ssm.ssmverify.SSM_STATUS_TIMEOUT
    assert 0.5 < waited < 30.0, waited
    wl = synth.custom_workload(2, 2, 20, 16, 1, 3, synth.F32, seed=43)
    d = to_dev(synth.draw_layer_round(wl), cuda_device)
    st = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    y = ssm.verify_commit(d["state0"], d["x"], d["B"], d["C"], d["dt"], d["A"], d["D"], d["accept_len"], dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and torch.isfinite(y).all()
