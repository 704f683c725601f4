"""The host-buffer front end gives bitwise the results of the device-side
verify_commit: y in host memory and the state updated in place, over several
rounds and with chunk counts that do not divide the batch."""
import pytest
import torch

import ssm_recurrence_verify_b300 as ssm
from gpu_helpers import to_dev
from ssm_recurrence_verify_b300 import synth
from ssm_recurrence_verify_b300.hostpipe import HostPipeline

pytestmark = pytest.mark.gpu


# fewer slots than chunks, as many, the default (twice the chunks), and more slots than that: chunks take
# the slots in turn across calls, wrapping around over the rounds
@pytest.mark.parametrize("chunks,slots", [(1, 1), (3, 2), (5, 3), (2, None), (3, 7)])
def test_pipeline_equals_device_calls(cuda_device, chunks, slots):
    wl = synth.custom_workload(11, 8, 64, 128, 2, 6, synth.BF16, seed=91)
    p = synth.draw_params(wl)
    st_ref = p["state0"].to(cuda_device)
    st = st_ref.clone()
    A, D = p["A"].to(cuda_device), p["D"].to(cuda_device)
    pipe = HostPipeline(st, A, D, wl.ntok, wl.ngroups, torch.bfloat16, chunks=chunks, slots=slots)
    for rnd in range(4):
        t = synth.draw_tokens(wl, rnd)
        acc = synth.draw_accept_len(wl, rnd)
        td = to_dev(t, cuda_device)
        y_ref = ssm.verify_commit(st_ref, td["x"], td["B"], td["C"], td["dt"], A, D, acc.to(cuda_device))
        h = {k: v.pin_memory() for k, v in t.items()}
        y = torch.full((wl.batch, wl.ntok, wl.nheads, wl.headdim), float("nan")).pin_memory()
        pipe.run(h["x"], h["B"], h["C"], h["dt"], acc.pin_memory(), y)
        torch.cuda.synchronize()
        assert torch.equal(y, y_ref.cpu()), rnd
        assert torch.equal(st, st_ref), rnd
    assert int(pipe.status.item()) == 0
    assert pipe.nslots == (2 * pipe.chunks if slots is None else slots)


def test_captured_step_equals_device_calls(cuda_device):
    """Two layers' pipelines captured as one graph; three replays with new
    inputs written into the same pinned buffers each time."""
    from ssm_recurrence_verify_b300.hostpipe import capture_step
    wl = synth.custom_workload(9, 4, 64, 64, 2, 5, synth.BF16, seed=92)
    streams = tuple(torch.cuda.Stream(device=cuda_device) for _ in range(3))
    refs, pipes, bufs = [], [], []
    for layer in range(2):
        p = synth.draw_params(wl, layer)
        A, D = p["A"].to(cuda_device), p["D"].to(cuda_device)
        st = p["state0"].to(cuda_device)
        refs.append((st.clone(), A, D))
        pipes.append(HostPipeline(st, A, D, wl.ntok, wl.ngroups, torch.bfloat16, chunks=4, slots=2,
                                  streams=streams))
        t = synth.draw_tokens(wl, 0, layer)
        h = {k: v.pin_memory() for k, v in t.items()}
        h["accept_len"] = synth.draw_accept_len(wl, 0).pin_memory()
        h["y"] = torch.zeros((wl.batch, wl.ntok, wl.nheads, wl.headdim)).pin_memory()
        bufs.append(h)
    g = capture_step(pipes, [(h["x"], h["B"], h["C"], h["dt"], h["accept_len"], h["y"]) for h in bufs])
    for rnd in range(1, 4):
        for layer, h in enumerate(bufs):
            t = synth.draw_tokens(wl, rnd, layer)
            for k in ("x", "B", "C", "dt"):
                h[k].copy_(t[k])
            h["accept_len"].copy_(synth.draw_accept_len(wl, rnd))
        g.replay()
        torch.cuda.synchronize()
        for layer, h in enumerate(bufs):
            st_ref, A, D = refs[layer]
            td = to_dev({k: h[k] for k in ("x", "B", "C", "dt", "accept_len")}, cuda_device)
            y_ref = ssm.verify_commit(st_ref, td["x"], td["B"], td["C"], td["dt"], A, D, td["accept_len"])
            torch.cuda.synchronize()
            assert torch.equal(h["y"], y_ref.cpu()), (rnd, layer)
            assert torch.equal(pipes[layer].state, st_ref), (rnd, layer)



@pytest.mark.parametrize("chunks,slots", [(3, None), (2, 5)])
def test_deferred_pipeline_equals_device_calls(cuda_device, chunks, slots):
    """run_deferred over five rounds equals, bit for bit, the device calls of
    the serving order: verify the first block, then commit_verify (previous
    block up to its accept_len, new block) each round, and finish() the same
    as a final commit."""
    dev = cuda_device
    wl = synth.custom_workload(11, 8, 64, 128, 2, 6, synth.BF16, seed=93)
    p = synth.draw_params(wl)
    st_ref = p["state0"].to(dev)
    st = st_ref.clone()
    A, D = p["A"].to(dev), p["D"].to(dev)
    pipe = HostPipeline(st, A, D, wl.ntok, wl.ngroups, torch.bfloat16, chunks=chunks, slots=slots)
    rounds = 5
    toks = [synth.draw_tokens(wl, r) for r in range(rounds)]
    accs = [synth.draw_accept_len(wl, r) for r in range(rounds)]
    for r in range(rounds):
        td = to_dev(toks[r], dev)
        if r == 0:
            y_ref = ssm.verify(st_ref, td["x"], td["B"], td["C"], td["dt"], A, D)
        else:
            pd = to_dev(toks[r - 1], dev)
            y_ref = ssm.commit_verify(st_ref, pd["x"], pd["B"], pd["dt"], accs[r - 1].to(dev), td["x"], td["B"],
                                      td["C"], td["dt"], A, D)
        h = {k: v.pin_memory() for k, v in toks[r].items()}
        prev_acc = (accs[r - 1] if r > 0 else torch.zeros(wl.batch, dtype=torch.int32)).pin_memory()
        y = torch.full((wl.batch, wl.ntok, wl.nheads, wl.headdim), float("nan")).pin_memory()
        pipe.run_deferred(prev_acc, h["x"], h["B"], h["C"], h["dt"], y)
        torch.cuda.synchronize()
        assert torch.equal(y, y_ref.cpu()), r
        assert torch.equal(st, st_ref), r
    last = to_dev(toks[-1], dev)
    ssm.commit(st_ref, last["x"], last["B"], last["dt"], A, accs[-1].to(dev))
    pipe.finish(accs[-1].pin_memory())
    torch.cuda.synchronize()
    assert torch.equal(st, st_ref)
    assert int(pipe.status.item()) == 0


def test_deferred_pipeline_needs_two_slots_per_chunk(cuda_device):
    wl = synth.custom_workload(4, 2, 64, 64, 1, 3, synth.BF16, seed=94)
    p = synth.draw_params(wl)
    pipe = HostPipeline(p["state0"].to(cuda_device), p["A"].to(cuda_device), p["D"].to(cuda_device), wl.ntok,
                        wl.ngroups, torch.bfloat16, chunks=2, slots=3)
    t = {k: v.pin_memory() for k, v in synth.draw_tokens(wl, 0).items()}
    y = torch.zeros(wl.batch, wl.ntok, wl.nheads, wl.headdim).pin_memory()
    with pytest.raises(ValueError):
        pipe.run_deferred(torch.zeros(wl.batch, dtype=torch.int32).pin_memory(), t["x"], t["B"], t["C"], t["dt"], y)

@pytest.mark.parametrize("nbytes,offset", [(1, 0), (15, 0), (16, 0), (4096 + 7, 0), (6 << 20, 0), (100003, 3)])
def test_copy_from_host(cuda_device, nbytes, offset):
    """SM-driven copies from page-locked memory: exact bytes for aligned and
    unaligned ranges with ragged tails."""
    from ssm_recurrence_verify_b300 import ssmverify as sv
    g = torch.Generator().manual_seed(nbytes)
    h = torch.randint(0, 256, (nbytes + offset,), dtype=torch.uint8, generator=g).pin_memory()
    d = torch.full((nbytes + offset,), 7, dtype=torch.uint8, device=cuda_device)
    sv.copy_from_host(d[offset:], h[offset:])
    torch.cuda.synchronize()
    assert torch.equal(d[offset:].cpu(), h[offset:])
    if offset:
        assert (d[:offset] == 7).all()


def test_copy_from_host_refuses_pageable_memory(cuda_device):
    from ssm_recurrence_verify_b300 import ssmverify as sv
    h = torch.zeros(64, dtype=torch.uint8)  # not page-locked
    d = torch.empty(64, dtype=torch.uint8, device=cuda_device)
    with pytest.raises(ValueError):
        sv.copy_from_host(d, h)
    lib = sv.load_library()
    import ctypes
    rc = lib.ssm_copy_from_host(ctypes.c_void_p(d.data_ptr()), ctypes.c_void_p(h.data_ptr()), 64, None)
    assert rc == sv.SSM_ERR_UNSUPPORTED


@pytest.mark.parametrize("offset", [0, 3])
def test_copy_from_host_n(cuda_device, offset):
    """Several copies in one call: segments of 5 MB, 16 KB + 9 bytes, 0 bytes,
    7 bytes and 4 KB are exact (offset 0: one kernel over all segments;
    offset 3: unaligned, each segment on its own); bytes around them stay."""
    from ssm_recurrence_verify_b300 import ssmverify as sv
    sizes = [5 << 20, (16 << 10) + 9, 0, 7, 4096]
    g = torch.Generator().manual_seed(11)
    hs = [torch.randint(0, 256, (n + offset,), dtype=torch.uint8, generator=g).pin_memory() for n in sizes]
    ds = [torch.full((n + offset + 16,), 7, dtype=torch.uint8, device=cuda_device) for n in sizes]
    sv.copy_from_host_n([(d[offset:offset + n], h[offset:]) for d, h, n in zip(ds, hs, sizes)])
    torch.cuda.synchronize()
    for d, h, n in zip(ds, hs, sizes):
        assert torch.equal(d[offset:offset + n].cpu(), h[offset:])
        assert (d[:offset] == 7).all() and (d[offset + n:] == 7).all()


def test_copy_from_host_n_refuses_pageable_memory(cuda_device):
    """One pageable source among page-locked ones: the call is refused before
    anything is copied (the binding raises; the C entry returns UNSUPPORTED)."""
    from ssm_recurrence_verify_b300 import ssmverify as sv
    good = torch.arange(64, dtype=torch.uint8).pin_memory()
    bad = torch.zeros(64, dtype=torch.uint8)  # not page-locked
    d1 = torch.full((64,), 7, dtype=torch.uint8, device=cuda_device)
    d2 = torch.full((64,), 7, dtype=torch.uint8, device=cuda_device)
    with pytest.raises(ValueError):
        sv.copy_from_host_n([(d1, good), (d2, bad)])
    segs = (sv.CopySegment * 2)(sv.CopySegment(d1.data_ptr(), good.data_ptr(), 64),
                                sv.CopySegment(d2.data_ptr(), bad.data_ptr(), 64))
    assert sv.load_library().ssm_copy_from_host_n(segs, 2, None) == sv.SSM_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert (d1 == 7).all() and (d2 == 7).all()
