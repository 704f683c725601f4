"""Host-buffer front end: verify + commit with the draft inputs in host memory.

A serving loop whose draft-token inputs arrive in (pinned) host memory and
whose y goes back to the host pays for two PCIe transfers per layer-call, each
larger than the kernel's own time. ``HostPipeline`` hides them behind each
other: the batch is cut into sequence chunks, and three CUDA streams run
chunk c's host-to-device copy, chunk c-1's kernel and chunk c-2's copy of y
back to the host at the same time, through a ring of device staging slots.
Host-to-device copies of page-locked inputs are read by the SMs
(``ssm_copy_from_host``), which is about three times the copy engines' rate
for step-sized transfers on B300 machines.
Every sequence's state, inputs and outputs are contiguous slices of the batch
dimension, so chunks need no gathering. A whole step (one or several layers)
can be captured once into a CUDA graph, so that issuing it costs one graph
launch instead of dozens of copy, event and kernel calls. ``run_deferred``
runs the serving order instead (``ssm_commit_verify``: commit the previous
block, whose inputs stay in the device staging slots, then verify the new
one). The kernels are the library's (through the C ABI); this module only
orders copies and launches.
"""
from __future__ import annotations

from typing import List, Optional

import torch

from . import ssmverify as sv


class HostPipeline:
    """``verify_commit`` for one layer with host-resident x, B, C, dt,
    accept_len and y, on a device-resident state updated in place.

    ``state`` is the device state ``[batch][H][P][N]`` (float32); ``A``, ``D``
    are device ``[H]`` float32. Inputs given to :meth:`run` are host tensors
    with the layouts of ``ssmverify`` (pinned memory for asynchronous copies).
    ``chunks`` sequence chunks are processed per call; ``slots`` device staging
    slots (default: twice the chunks, so that the next chunks' copies need not
    wait for earlier read-backs) rotate between them. ``streams`` (copy-in,
    kernel, copy-out) may be shared by the pipelines of several layers; each
    pipeline orders only its own slots.
    """

    def __init__(self, state: torch.Tensor, A: torch.Tensor, D: torch.Tensor, ntok: int, ngroups: int,
                 in_dtype: torch.dtype = torch.bfloat16, chunks: int = 2, slots: Optional[int] = None, streams=None):
        if not state.is_cuda:
            raise ValueError("state must be a CUDA tensor")
        self.state, self.A, self.D = state, A, D
        self.dev = state.device
        bsz, H, P, N = state.shape
        self.bsz, self.H, self.P, self.N, self.K, self.G = bsz, H, P, N, ntok, ngroups
        self.chunks = max(1, min(chunks, bsz))
        self.bounds = [(bsz * i) // self.chunks for i in range(self.chunks + 1)]
        cmax = max(self.bounds[i + 1] - self.bounds[i] for i in range(self.chunks))
        self.nslots = max(1, 2 * self.chunks if slots is None else slots)

        def dev(*shape, dtype=in_dtype):
            return torch.empty(shape, dtype=dtype, device=self.dev)

        self.slot_x = [dev(cmax, ntok, H, P) for _ in range(self.nslots)]
        self.slot_B = [dev(cmax, ntok, ngroups, N) for _ in range(self.nslots)]
        self.slot_C = [dev(cmax, ntok, ngroups, N) for _ in range(self.nslots)]
        self.slot_dt = [dev(cmax, ntok, H) for _ in range(self.nslots)]
        self.slot_acc = [dev(cmax, dtype=torch.int32) for _ in range(self.nslots)]
        self.slot_y = [dev(cmax, ntok, H, P, dtype=torch.float32) for _ in range(self.nslots)]
        self.status = torch.zeros(1, dtype=torch.int32, device=self.dev)
        if streams is None:
            streams = tuple(torch.cuda.Stream(device=self.dev) for _ in range(3))
        self.s_in, self.s_k, self.s_out = streams
        # slot free again once its y has been copied out
        self.freed: List[Optional[torch.cuda.Event]] = [None] * self.nslots
        # slots are taken in turn across calls, so that with more slots than chunks a call's
        # copies in need not wait for the previous call's read-backs from the same slots
        self.next_slot = 0
        # run_deferred: the slot holding each chunk's previous block (None before the first call), and
        # per slot the event after which no later kernel reads it as a previous block
        self.prev_slot: List[Optional[int]] = [None] * self.chunks
        self.prev_read: List[Optional[torch.cuda.Event]] = [None] * self.nslots

    def _h2d(self, dst: torch.Tensor, src: torch.Tensor) -> None:
        """Host -> device on the copy-in stream: page-locked sources are read
        by the SMs (ssm_copy_from_host, about 3x the copy engines' rate for
        step-sized transfers on B300 machines); others take an ordinary copy."""
        if src.is_pinned() and src.is_contiguous():
            sv.copy_from_host(dst, src, stream=self.s_in)
        else:
            dst.copy_(src, non_blocking=True)

    def run(self, x: torch.Tensor, B: torch.Tensor, C: torch.Tensor, dt: torch.Tensor, accept_len: torch.Tensor,
            y: torch.Tensor) -> None:
        """Enqueue one layer-call: copies in, fused verify + commit per chunk,
        y copied out. Asynchronous; synchronise on :attr:`s_out` (or the
        device) before reading ``y`` or :attr:`status`."""
        for c in range(self.chunks):
            lo, hi = self.bounds[c], self.bounds[c + 1]
            n = hi - lo
            if n == 0:
                continue
            k = self.next_slot
            self.next_slot = (self.next_slot + 1) % self.nslots
            with torch.cuda.stream(self.s_in):
                if self.freed[k] is not None:
                    self.s_in.wait_event(self.freed[k])
                pairs = ((self.slot_x[k][:n], x[lo:hi]), (self.slot_B[k][:n], B[lo:hi]),
                         (self.slot_C[k][:n], C[lo:hi]), (self.slot_dt[k][:n], dt[lo:hi]),
                         (self.slot_acc[k][:n], accept_len[lo:hi]))
                if all(src.is_pinned() and src.is_contiguous() for _, src in pairs):
                    sv.copy_from_host_n(pairs, stream=self.s_in)  # the chunk's inputs in one launch
                else:
                    for dst, src in pairs:
                        self._h2d(dst, src)
                arrived = torch.cuda.Event()
                arrived.record(self.s_in)
            with torch.cuda.stream(self.s_k):
                self.s_k.wait_event(arrived)
                sv.verify_commit(self.state[lo:hi], self.slot_x[k][:n], self.slot_B[k][:n], self.slot_C[k][:n],
                                 self.slot_dt[k][:n], self.A, self.D, self.slot_acc[k][:n], y=self.slot_y[k][:n],
                                 dev_status=self.status, stream=self.s_k)
                done = torch.cuda.Event()
                done.record(self.s_k)
            with torch.cuda.stream(self.s_out):
                self.s_out.wait_event(done)
                y[lo:hi].copy_(self.slot_y[k][:n], non_blocking=True)
                freed = torch.cuda.Event()
                freed.record(self.s_out)
                self.freed[k] = freed


    def run_deferred(self, accept_len_prev: torch.Tensor, x: torch.Tensor, B: torch.Tensor, C: torch.Tensor,
                     dt: torch.Tensor, y: torch.Tensor) -> None:
        """Enqueue one layer-call in the serving order (``ssm_commit_verify``):
        commit the previous call's block up to ``accept_len_prev`` (host
        int32 [batch]; ignored on the first call, which only verifies), then
        verify the new block (host x, B, C, dt) from the committed state and
        copy its y to the host. The previous block's x, B and dt are not sent
        again: they stay in the device staging slots the previous call filled,
        which needs at least twice as many slots as chunks. Asynchronous, like
        :meth:`run`; :meth:`finish` commits the last block. Do not interleave
        :meth:`run` calls before :meth:`finish`: they take the slots in turn
        and would overwrite the kept block."""
        if self.nslots < 2 * self.chunks:
            raise ValueError("run_deferred needs at least twice as many staging slots as chunks")
        for c in range(self.chunks):
            lo, hi = self.bounds[c], self.bounds[c + 1]
            n = hi - lo
            if n == 0:
                continue
            k = self.next_slot
            self.next_slot = (self.next_slot + 1) % self.nslots
            kp = self.prev_slot[c]
            with torch.cuda.stream(self.s_in):
                for ev in (self.freed[k], self.prev_read[k]):  # its y is out, and no kernel still reads it
                    if ev is not None:
                        self.s_in.wait_event(ev)
                pairs = ((self.slot_x[k][:n], x[lo:hi]), (self.slot_B[k][:n], B[lo:hi]),
                         (self.slot_C[k][:n], C[lo:hi]), (self.slot_dt[k][:n], dt[lo:hi]),
                         (self.slot_acc[k][:n], accept_len_prev[lo:hi]))
                if all(src.is_pinned() and src.is_contiguous() for _, src in pairs):
                    sv.copy_from_host_n(pairs, stream=self.s_in)
                else:
                    for dst, src in pairs:
                        self._h2d(dst, src)
                arrived = torch.cuda.Event()
                arrived.record(self.s_in)
            with torch.cuda.stream(self.s_k):
                self.s_k.wait_event(arrived)
                if kp is None:
                    sv.verify(self.state[lo:hi], self.slot_x[k][:n], self.slot_B[k][:n], self.slot_C[k][:n],
                              self.slot_dt[k][:n], self.A, self.D, y=self.slot_y[k][:n], dev_status=self.status,
                              stream=self.s_k)
                else:
                    sv.commit_verify(self.state[lo:hi], self.slot_x[kp][:n], self.slot_B[kp][:n],
                                     self.slot_dt[kp][:n], self.slot_acc[k][:n], self.slot_x[k][:n],
                                     self.slot_B[k][:n], self.slot_C[k][:n], self.slot_dt[k][:n], self.A, self.D,
                                     y=self.slot_y[k][:n], dev_status=self.status, stream=self.s_k)
                done = torch.cuda.Event()
                done.record(self.s_k)
                if kp is not None:
                    self.prev_read[kp] = done
            with torch.cuda.stream(self.s_out):
                self.s_out.wait_event(done)
                y[lo:hi].copy_(self.slot_y[k][:n], non_blocking=True)
                freed = torch.cuda.Event()
                freed.record(self.s_out)
                self.freed[k] = freed
            self.prev_slot[c] = k

    def finish(self, accept_len_last: torch.Tensor) -> None:
        """Commit the last block enqueued by :meth:`run_deferred` up to
        ``accept_len_last`` (host int32 [batch]) and forget it: the next
        :meth:`run_deferred` starts with a verify only."""
        for c in range(self.chunks):
            lo, hi = self.bounds[c], self.bounds[c + 1]
            n, kp = hi - lo, self.prev_slot[c]
            if n == 0 or kp is None:
                continue
            acc = self.slot_acc[kp][:n]
            with torch.cuda.stream(self.s_k):
                acc.copy_(accept_len_last[lo:hi], non_blocking=True)
                sv.commit(self.state[lo:hi], self.slot_x[kp][:n], self.slot_B[kp][:n], self.slot_dt[kp][:n],
                          self.A, acc, dev_status=self.status, stream=self.s_k)
                done = torch.cuda.Event()
                done.record(self.s_k)
                self.prev_read[kp] = done
            self.prev_slot[c] = None


def capture_step(pipelines, inputs, device=None, repeat: int = 1) -> torch.cuda.CUDAGraph:
    """Capture ``repeat`` consecutive steps -- each ``pipelines[i].run(*inputs[i])``
    for every i -- into a CUDA graph and return it. The host and device
    buffers are fixed: replay the graph after writing the next steps' inputs
    into the same pinned host tensors. The pipelines' streams fork from the
    capturing stream and join back into it, so one replay covers all its
    steps and replays on one stream run one after another; within a replay,
    step s + 1's copies in overlap step s's copies out (the state still
    passes from step to step in kernel order)."""
    device = pipelines[0].dev if device is None else device
    streams = []
    for p in pipelines:
        for s in (p.s_in, p.s_k, p.s_out):
            if all(s is not t for t in streams):
                streams.append(s)
    g = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(device=device)
    for p in pipelines:
        p.freed = [None] * p.nslots
        p.next_slot = 0
    with torch.cuda.graph(g, stream=cap):
        fork = torch.cuda.Event()
        fork.record(cap)
        for s in streams:
            s.wait_event(fork)
        for _ in range(repeat):
            for p, args in zip(pipelines, inputs):
                p.run(*args)
        for s in streams:
            e = torch.cuda.Event()
            e.record(s)
            cap.wait_event(e)
    for p in pipelines:
        p.freed = [None] * p.nslots
        p.next_slot = 0
    return g
