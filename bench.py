"""Benchmark: draft tokens verified per second per SSM layer, and achieved HBM
bandwidth of the fused verify/commit kernel against the B300 roofline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload 3] [--cpu-seconds 10] [--no-cpu-baseline]

A step is one pass of the whole path over one batch: every layer of the
workload through the fused verify+commit (plain decode: the step), as one
launch over the layer stack (nlayers) or, with --per-layer-launches, one
launch per layer. The value counts draft tokens x layers per second.
The default workload is the batched speculative-serving load (64 sequences,
one Llama-3-8B-shaped layer: H 32, P 128, N 128, G 8, K 8, bf16 inputs, fp32
state). Inputs are seeded synthetic data drawn on the CPU and resident in HBM
before the timed region; steps rotate over several independent input sets
whose total exceeds twice the L2, so no step reads another step's data from
L2. The K timed steps are captured as CUDA graphs (up to 4096 launches each)
and replayed back to back, as a serving loop runs its layers; CUDA events on
the launching stream time the whole region, and the average launch duration
is that time over the launches.

With --gpus N, N ranks run, one per GPU: started by an outside launcher
(torchrun sets RANK / WORLD_SIZE / LOCAL_RANK / MASTER_*), or else spawned by
this script itself. Rank r owns sequences [r B, (r + 1) B) of a global batch
of N B (weak scaling: B sequences per GPU, drawn from the same seeded streams
as a single-process run of N B sequences); the data path has no collective.
The elapsed time is the maximum over ranks, and the value counts every
rank's sequences.

--impl reference times the fp64 CPU oracle (the only reference there is) on
bounded samples of the same workload, on rank 0 only.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from ssm_recurrence_verify_b300 import synth  # noqa: E402

L2_BYTES = 126 * 1000 * 1000
NSETS_CAP = 1024  # input sets rotated at most (a workload of a few KB per step cannot outgrow the L2 this way)
MAX_GRAPH_LAUNCHES = 4096  # kernel launches captured per CUDA graph in the timed region
# --path values that time the verify/commit workload, and the entry points each launches (launch_layer)
PATH_MODES = {"ssm": "fused", "commit_verify": "deferred", "unfused": "unfused"}
E2E_STEPS_PER_GRAPH = 16   # consecutive host-buffer steps per CUDA graph in the end-to-end measurement
HBM_SPEC_GBS = 8000.0
FALLBACK_HBM_GBS = 6400.0
METRIC = "draft tokens verified/s per SSM layer; achieved HBM GB/s vs B300 peak"
KERNEL_SRC = os.path.join(ROOT, "ssm_recurrence_verify_b300", "csrc", "ssmverify.cu")
PROFILES = os.path.join(ROOT, "profiles")


# ----------------------------------------------------------------------------- distributed host logic

def dist_env():
    """(rank, world_size, local_rank) from the torchrun environment."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def shard(batch_per_rank: int, rank: int):
    """Weak scaling: rank r owns sequences [r * batch, (r + 1) * batch)."""
    return batch_per_rank, rank * batch_per_rank


def max_over_ranks(value: float, world: int) -> float:
    if world == 1:
        return value
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def free_port() -> int:
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_entry(rank: int, world: int, port: int, argv, entry):
    """One spawned rank: the environment torchrun would set, then the bench."""
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world), LOCAL_WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    rc = (main if entry is None else entry)(list(argv))
    if rc:
        raise SystemExit(rc)


def launch_ranks(argv, world: int, entry=None) -> int:
    """`--gpus N` without an outside launcher: start N ranks on this node, one
    process per GPU (rank r on GPU r), by spawn (a fresh interpreter each, so
    no CUDA state is forked), with the rendezvous on 127.0.0.1. Rank 0 prints
    the JSON line. `entry` replaces main in the ranks (tests)."""
    import torch.multiprocessing as mp
    mp.spawn(_rank_entry, args=(world, free_port(), list(argv), entry), nprocs=world, join=True)
    return 0


def init_ranks(world: int, local_rank: int):
    """The process group of a multi-rank run: NCCL on GPUs; gloo where no GPU
    is visible (host-side runs of the timing logic). Only the max-over-ranks
    reduction and the barriers use it: the data path has no collective."""
    import torch.distributed as dist
    if torch.cuda.is_available():
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    else:
        dist.init_process_group("gloo")


# ----------------------------------------------------------------------------- bytes per launch

def algorithmic_bytes(wl: synth.Workload, batch: int, accepted_nonzero: int) -> int:
    """What one layer-call must move: the state read once, written only for
    sequences with j > 0, x/B/C/dt read once (B/C once per group), y written
    once in fp32, accept_len read."""
    H, P, N, G, K = wl.nheads, wl.headdim, wl.dstate, wl.ngroups, wl.ntok
    eb = wl.in_elem_bytes()
    slice_b = H * P * N * 4
    return (batch * slice_b + accepted_nonzero * slice_b + batch * K * (H * P * eb + 2 * G * N * eb + H * eb)
            + batch * K * H * P * 4 + (0 if wl.accept == "all" else batch * 4))


def algorithmic_bytes_commit_verify(wl: synth.Workload, batch: int, accept_len) -> int:
    """What one deferred-commit layer-call (ssm_commit_verify) must move: the
    state read once and written for sequences with j_prev > 0, the previous
    block's x / B / dt for its j_prev accepted tokens only (B once per group),
    the new block's x / B / C / dt, y of the new block in fp32, and
    accept_len_prev."""
    H, P, N, G, K = wl.nheads, wl.headdim, wl.dstate, wl.ngroups, wl.ntok
    eb = wl.in_elem_bytes()
    slice_b = H * P * N * 4
    js = [int(j) for j in accept_len]
    replay = sum(js) * (H * P * eb + G * N * eb + H * eb)
    return (batch * slice_b + sum(1 for j in js if j > 0) * slice_b + replay
            + batch * K * (H * P * eb + 2 * G * N * eb + H * eb) + batch * K * H * P * 4 + batch * 4)


def algorithmic_bytes_unfused(wl: synth.Workload, batch: int, accept_len) -> int:
    """What the unfused pair ssm_verify + ssm_commit must move for one
    layer-call: verify reads every state, x / B / C / dt and writes y; commit
    reads the state of each sequence with j > 0 again, its j accepted tokens'
    x / B / dt and accept_len, and writes that state back."""
    H, P, N, G, K = wl.nheads, wl.headdim, wl.dstate, wl.ngroups, wl.ntok
    eb = wl.in_elem_bytes()
    slice_b = H * P * N * 4
    js = [int(j) for j in accept_len]
    nnz = sum(1 for j in js if j > 0)
    verify = batch * slice_b + batch * K * (H * P * eb + 2 * G * N * eb + H * eb) + batch * K * H * P * 4
    commit = 2 * nnz * slice_b + sum(js) * (H * P * eb + G * N * eb + H * eb) + batch * 4
    return verify + commit


def tile_tensor_macs(wl: synth.Workload, accept_len, layers: int) -> int:
    """Multiply-adds one fused verify+commit launch issues on the tensor cores
    (mma.sync m16n8k8 tf32, 1024 each), at N <= 128 (one warp per 16-row band):
    per warp and 8-token chunk, y = h C^T over N / 8 k-blocks (2 products for
    bf16 inputs, 3 for fp32), the Gram C B^T (1 or 3) and the intra-chunk term
    (3); per state update (N / 8 n-blocks, 2 or 3 products) as the kernel
    takes them: through a chunk that more chunks follow, plus the committed
    state inside it when j falls there, and up to j in the last chunk."""
    H, P, N, K = wl.nheads, wl.headdim, wl.dstate, wl.ntok
    if N > 128:
        return 0
    bf16 = wl.in_dtype != synth.F32
    py, pg, pa = (2, 1, 2) if bf16 else (3, 3, 3)
    warps = -(-P // 16)  # 16-row bands per (sequence, head)
    per_y = (N // 8) * py + (N // 8) * pg + 3
    per_upd = (N // 8) * pa
    total = 0
    for j in accept_len:
        j = int(j) if wl.accept != "all" else K
        mma = 0
        for t0 in range(0, K, 8):
            tc = min(8, K - t0)
            mma += per_y
            more = t0 + tc < K
            jc = j - t0 if 0 < j - t0 <= tc else 0  # committed state after token jc - 1 of this chunk
            if more:
                mma += per_upd * (2 if 0 < jc < tc else 1)
            elif jc > 0:
                mma += per_upd
        total += mma
    return total * H * warps * layers * 1024


# ----------------------------------------------------------------------------- clocks

def physical_gpu(local_rank: int) -> str:
    """The nvidia-smi / NVML id of this process's GPU (CUDA_VISIBLE_DEVICES aware)."""
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        if local_rank < len(ids):
            return ids[local_rank]
    return str(local_rank)


class NvmlCtypes:
    """The few NVML calls the clock sampler makes, straight from the
    driver's libnvidia-ml through ctypes (for hosts without the pynvml
    package). Same names and return values as pynvml; raises on an error."""

    NVML_CLOCK_SM = 1

    def __init__(self):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        self._call("nvmlInit_v2")

    def _call(self, name, *args):
        rc = getattr(self.lib, name)(*args)
        if rc != 0:
            raise RuntimeError(f"{name} returned NVML error {rc}")

    def nvmlDeviceGetHandleByIndex(self, index):
        h = self.ct.c_void_p()
        self._call("nvmlDeviceGetHandleByIndex_v2", self.ct.c_uint(index), self.ct.byref(h))
        return h

    def nvmlDeviceGetHandleByUUID(self, uuid):
        h = self.ct.c_void_p()
        self._call("nvmlDeviceGetHandleByUUID", self.ct.c_char_p(uuid.encode()), self.ct.byref(h))
        return h

    def _clock(self, name, h, kind):
        v = self.ct.c_uint()
        self._call(name, h, self.ct.c_int(kind), self.ct.byref(v))
        return v.value

    def nvmlDeviceGetClockInfo(self, h, kind):
        return self._clock("nvmlDeviceGetClockInfo", h, kind)

    def nvmlDeviceGetMaxClockInfo(self, h, kind):
        return self._clock("nvmlDeviceGetMaxClockInfo", h, kind)

    def nvmlDeviceGetCurrentClocksEventReasons(self, h):
        v = self.ct.c_ulonglong()
        name = ("nvmlDeviceGetCurrentClocksEventReasons" if hasattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons")
                else "nvmlDeviceGetCurrentClocksThrottleReasons")
        self._call(name, h, self.ct.byref(v))
        return v.value


class ClockSampler:
    """Samples the SM clock and clock-event reasons during a window, through
    NVML in a thread (the pynvml package, else the driver's libnvidia-ml via
    ctypes), or through a `nvidia-smi -lms` subprocess where neither loads.
    A polling nvidia-smi subprocess measurably slowed the timed kernels
    (about 2 % at a 20 ms period); the in-process NVML thread is preferred."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x40: "sw_thermal_slowdown",
               0x80: "hw_thermal_slowdown", 0x100: "hw_power_brake_slowdown", 0x2: "applications_clocks_setting"}

    def __init__(self, local_rank: int, period_s: float = 0.02):
        self.samples = []  # (perf_counter, sm_mhz, reason bits)
        self.period = period_s
        self.gpu = physical_gpu(local_rank)
        self.max_mhz = None
        self.err = ""
        self.mode = None
        self._stop = threading.Event()
        errs = []
        for opener in (self._pynvml, NvmlCtypes):
            try:
                nv = opener()
                self.h = (nv.nvmlDeviceGetHandleByUUID(self.gpu) if self.gpu.startswith(("GPU-", "MIG-"))
                          else nv.nvmlDeviceGetHandleByIndex(int(self.gpu)))
                self.max_mhz = nv.nvmlDeviceGetMaxClockInfo(self.h, nv.NVML_CLOCK_SM)
                self.nv = nv
                self.mode = "nvml" if opener is not NvmlCtypes else "nvml-ctypes"
                break
            except Exception as e:
                errs.append(f"{getattr(opener, '__name__', 'nvml')}: {e}")
        if self.mode is None:
            self.err = "; ".join(errs)
            import shutil
            if shutil.which("nvidia-smi"):
                self.mode = "nvidia-smi"

    @staticmethod
    def _pynvml():
        import pynvml
        pynvml.nvmlInit()
        return pynvml

    def _nvml_loop(self):
        f = getattr(self.nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.nv.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self._stop.is_set():
            try:
                self.samples.append((time.perf_counter(), self.nv.nvmlDeviceGetClockInfo(self.h, self.nv.NVML_CLOCK_SM),
                                     int(f(self.h))))
            except Exception:
                pass
            time.sleep(self.period)

    def _smi_loop(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 3:
                continue
            try:
                self.samples.append((time.perf_counter(), float(parts[0]), int(parts[2], 16)))
                self.max_mhz = float(parts[1])
            except ValueError:
                continue

    def start(self):
        if self.mode in ("nvml", "nvml-ctypes"):
            self.t = threading.Thread(target=self._nvml_loop, daemon=True)
            self.t.start()
        elif self.mode == "nvidia-smi":
            import subprocess
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu, "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active",
                 "--format=csv,noheader,nounits", "-lms", str(int(self.period * 1000))],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True, bufsize=1)
            self.t = threading.Thread(target=self._smi_loop, daemon=True)
            self.t.start()
            time.sleep(0.3)  # let the first samples arrive

    def stop(self):
        if self.mode in ("nvml", "nvml-ctypes"):
            self._stop.set()
            self.t.join()
        elif self.mode == "nvidia-smi":
            time.sleep(0.1)
            self.proc.terminate()
            self.proc.wait()
            self.t.join(timeout=2)

    def summary(self, t0: float, t1: float):
        if self.mode is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "note": f"no clock source: {self.err}"}
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        note = f"{self.mode}, sampled during the timed region"
        if not inside:
            inside = self.samples
            note = f"{self.mode}: timed region shorter than the sampling period; samples span warm-up and timed region"
        mhz = [s[1] for s in inside]
        bits = 0
        for s in inside:
            bits |= s[2]
        reasons = sorted(name for bit, name in self.REASONS.items() if bits & bit)
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": self.max_mhz, "reasons": reasons,
                "samples": len(inside), "note": note}


# ----------------------------------------------------------------------------- measured peaks / traffic

def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


HOST_MARKER = "// ----------------------------------------------------------------------------- host side"
PREFILL_MARKER = "// ----------------------------------------------------------------------------- prefill kernels"


def kernel_source_hash(path: str = KERNEL_SRC) -> str:
    """sha256 of the tile kernel's device code: the text before the source's
    prefill kernels (or its host-side section), with #include lines left out,
    so that host-only and prefill-only edits keep a recorded capture valid
    while any edit of the tile kernel voids it."""
    with open(path) as f:
        text = f.read()
    dev = text.split(PREFILL_MARKER)[0].split(HOST_MARKER)[0]
    dev = "\n".join(line for line in dev.splitlines() if not line.startswith("#include"))
    return hashlib.sha256(dev.encode()).hexdigest()


def recorded_traffic(workload_name: str):
    """DRAM bytes per launch from a committed ncu capture of this kernel on
    this workload, or None if absent or taken on different kernel source."""
    path = os.path.join(PROFILES, f"ssm_tile_kernel_{workload_name}.traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except Exception:
        return None
    if rec.get("kernel_source_sha256") != kernel_source_hash():
        return None
    return rec.get("dram_bytes_per_launch")


# ----------------------------------------------------------------------------- GPU arm

def upload_graphs(graphs, stream):
    """Upload each instantiated graph to the device (cudaGraphUpload) without
    running it, so that the first replay inside a timed region does not also
    pay the graph's upload: with a 20-step region that one-time cost moved the
    mean step time by about 2 %."""
    from cuda.bindings import runtime as cudart
    for g in graphs:
        err, = cudart.cudaGraphUpload(g.raw_cuda_graph_exec(), stream.cuda_stream)
        if int(err) != 0:
            raise RuntimeError(f"cudaGraphUpload failed: {err}")
    torch.cuda.synchronize()



class LayerSet:
    """One independent input set of a round: the layer stack's state, inputs,
    y and status as [L]-leading slabs (`stack`; accept_len [batch] is shared
    by the layers), and per layer views of them (`layers`)."""

    def __init__(self, wl, batch, offset, rnd, dev, layers, next_round=False):
        ds = [synth.draw_layer_round(wl, rnd=rnd, layer=layer, batch=batch, batch_offset=offset)
              for layer in range(layers)]
        self.stack = {k: torch.stack([d[k] for d in ds]).to(dev) for k in ("state0", "x", "B", "C", "dt", "A", "D")}
        if next_round:  # the next round's drafts: the new block of a deferred commit (this round's is the previous)
            nx = [synth.draw_tokens(wl, rnd + 1, layer, batch, offset) for layer in range(layers)]
            for k in ("x", "B", "C", "dt"):
                self.stack[k + "2"] = torch.stack([d[k] for d in nx]).to(dev)
        self.stack["accept_len"] = ds[0]["accept_len"].to(dev)  # one accepted prefix per sequence, every layer
        self.stack["y"] = torch.empty((layers, batch, wl.ntok, wl.nheads, wl.headdim), dtype=torch.float32,
                                      device=dev)
        self.stack["status"] = torch.zeros(1, dtype=torch.int32, device=dev)
        self.layers = []
        for layer, d in enumerate(ds):
            e = {k: v[layer] for k, v in self.stack.items() if k not in ("accept_len", "status")}
            e["accept_len"] = self.stack["accept_len"]
            e["status"] = self.stack["status"]
            e["host"] = d
            e["accepted_nonzero"] = int((d["accept_len"] > 0).sum())
            self.layers.append(e)


def launch_layer(ssm, wl, e, mode="fused"):
    """One layer-call (per-layer tensors), or one call over the whole stack
    (the [L]-leading slabs of LayerSet.stack). mode "fused": ssm_verify_commit
    (ssm_step for plain decode); "deferred": the serving order's
    ssm_commit_verify, which commits this set's round (its drafts and
    accept_len) and verifies the next round's drafts from the committed state;
    "unfused": ssm_verify then ssm_commit, two launches."""
    if mode == "unfused":
        ssm.verify(e["state0"], e["x"], e["B"], e["C"], e["dt"], e["A"], e["D"], y=e["y"], dev_status=e["status"])
        ssm.commit(e["state0"], e["x"], e["B"], e["dt"], e["A"], e["accept_len"], dev_status=e["status"])
    elif mode == "deferred":
        ssm.commit_verify(e["state0"], e["x"], e["B"], e["dt"], e["accept_len"], e["x2"], e["B2"], e["C2"], e["dt2"],
                          e["A"], e["D"], y=e["y"], dev_status=e["status"])
    elif wl.accept == "all" and wl.ntok == 1:
        ssm.step(e["state0"], e["x"], e["B"], e["C"], e["dt"], e["A"], e["D"], y=e["y"])
    else:
        ssm.verify_commit(e["state0"], e["x"], e["B"], e["C"], e["dt"], e["A"], e["D"], e["accept_len"], y=e["y"],
                          dev_status=e["status"])


def device_leg(args, wl, rank, world, local_rank):
    """This rank's share of the timed region on its own GPU: W warm-up
    steps, then K steps replayed from CUDA graphs between a barrier and a
    synchronize on each side. Returns this rank's elapsed time and what the
    summary needs; run_ours takes the maximum over ranks."""
    import ssm_recurrence_verify_b300 as ssm
    from ssm_recurrence_verify_b300 import build as libbuild
    if not os.path.exists(libbuild.LIB):
        libbuild.build()
    ssm.load_library()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    batch, offset = shard(wl.batch, rank)
    nl = wl.nlayers
    step_bytes_est = nl * (2 * batch * wl.nheads * wl.headdim * wl.dstate * 4)
    nsets = 1 if step_bytes_est >= 4 * L2_BYTES else max(3, math.ceil(2 * L2_BYTES / step_bytes_est) + 1)
    nsets = min(nsets, NSETS_CAP)
    mode = PATH_MODES.get(getattr(args, "path", "ssm"), "fused")
    sets = [LayerSet(wl, batch, offset, rnd, dev, nl, next_round=mode == "deferred") for rnd in range(nsets)]
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()
    # a layer stack runs as one launch per step (nlayers = L), unless asked per layer
    per_step = 1 if (nl > 1 and not args.per_layer_launches) else nl
    units = (lambda s: [s.stack]) if per_step == 1 and nl > 1 else (lambda s: s.layers)

    # eager warm-up of every set
    with torch.cuda.stream(stream):
        for s in sets:
            for e in units(s):
                launch_layer(ssm, wl, e, mode)
    torch.cuda.synchronize()

    # The warm-up steps and the K timed steps are captured as CUDA graphs
    # (step i uses input set i mod nsets; at most MAX_GRAPH_LAUNCHES launches
    # per graph) and replayed back to back, as a serving loop runs its layers.
    def capture(step_sets):
        per = max(1, MAX_GRAPH_LAUNCHES // (per_step * (2 if mode == "unfused" else 1)))
        out = []
        for i in range(0, len(step_sets), per):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for si in step_sets[i:i + per]:
                    for e in units(sets[si]):
                        launch_layer(ssm, wl, e, mode)
            out.append(g)
        return out

    K = args.steps
    warm_graphs = capture([i % nsets for i in range(args.warmup)])
    timed_sets = [(args.warmup + i) % nsets for i in range(K)]
    timed_graphs = capture(timed_sets)
    torch.cuda.synchronize()
    upload_graphs(warm_graphs + timed_graphs, stream)

    sampler = ClockSampler(local_rank)
    sampler.start()
    with torch.cuda.stream(stream):
        for g in warm_graphs:
            g.replay()
    torch.cuda.synchronize()
    t_all0, t_all1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    with torch.cuda.stream(stream):
        t_all0.record(stream)
        for g in timed_graphs:
            g.replay()
        t_all1.record(stream)
    torch.cuda.synchronize()
    wall1 = time.perf_counter()
    barrier(world)
    sampler.stop()
    elapsed_ms = t_all0.elapsed_time(t_all1)
    for s in sets:
        for e in s.layers:
            assert int(e["status"].item()) == 0, "device reported a bad accept_len"
    # per-step algorithmic bytes, averaged over the sets the timed steps used
    if mode == "deferred":
        step_bytes = [sum(algorithmic_bytes_commit_verify(wl, batch, e["host"]["accept_len"]) for e in s.layers)
                      for s in sets]
    elif mode == "unfused":
        step_bytes = [sum(algorithmic_bytes_unfused(wl, batch, e["host"]["accept_len"]) for e in s.layers)
                      for s in sets]
    else:
        step_bytes = [sum(algorithmic_bytes(wl, batch, e["accepted_nonzero"]) for e in s.layers) for s in sets]
    used = [step_bytes[si] for si in timed_sets]
    step_macs = [tile_tensor_macs(wl, s.layers[0]["host"]["accept_len"], nl) if mode == "fused" else 0 for s in sets]
    e2e = run_e2e(ssm, args, wl, sets[0], stream, dev, world) if args.e2e_steps > 0 and mode == "fused" else None
    return {"elapsed_ms": elapsed_ms, "steps": K, "per_step": per_step, "batch": batch, "nsets": nsets,
            "reread_bytes": (nsets - 1) * step_bytes_est,
            "launch_bytes": statistics.fmean(used) / per_step,
            "launch_macs": statistics.fmean(step_macs[si] for si in timed_sets) / per_step,
            "wall_s": wall1 - wall0, "graphs": len(timed_graphs), "kernels_per_call": 2 if mode == "unfused" else 1,
            "clocks": sampler.summary(wall0, wall1), "e2e": e2e}


def run_ours(args, wl, rank, world, local_rank):
    """The device leg on this rank, then the whole-job figures: the elapsed
    time is the maximum over ranks, and the value counts every rank's
    sequences (weak scaling: each rank owns `batch` sequences)."""
    leg = device_leg(args, wl, rank, world, local_rank)
    K, per_step, nl = leg["steps"], leg["per_step"], wl.nlayers
    max_ms = max_over_ranks(leg["elapsed_ms"], world)
    mean_launch_ms = leg["elapsed_ms"] / (K * per_step)  # this rank's average launch duration over the timed region
    achieved = leg["launch_bytes"] / (mean_launch_ms * 1e-3) / 1e9
    peak, peak_kind = hbm_peak()
    # per SSM layer: Bsz K / t_layer, i.e. every rank's sequences x draft tokens x layers per step time
    tokens_per_step = leg["batch"] * wl.ntok * world * nl
    value = tokens_per_step * K / (max_ms * 1e-3)
    return {
        "value": value, "ms_per_step": max_ms / K, "elapsed_ms": max_ms, "wall_s": leg["wall_s"],
        "launch_ms_mean": mean_launch_ms, "graphs": leg["graphs"],
        "achieved_gbs": achieved, "peak": peak, "peak_kind": peak_kind, "bytes_per_launch": leg["launch_bytes"],
        "macs_per_launch": leg.get("launch_macs", 0),
        "clocks": leg["clocks"], "nsets": leg["nsets"], "reread_bytes": leg.get("reread_bytes"), "e2e": leg["e2e"],
        "launches": K * per_step * leg.get("kernels_per_call", 1),
        "batch": leg["batch"], "layers_per_launch": nl // per_step,
    }


def run_e2e(ssm, args, wl, s, stream, dev, world):
    """Same metric through the public API with host buffers: every step copies
    its inputs from pinned host memory and reads y back. The library's host
    front end (HostPipeline) overlaps the copies of one sequence chunk with the
    kernel of another and the read-back of a third, across all layers."""
    from ssm_recurrence_verify_b300.hostpipe import HostPipeline
    streams = tuple(torch.cuda.Stream(device=dev) for _ in range(3))
    # 2 sequence chunks and 4 staging slots taken in turn measured best on the serving workload
    # (2 slots: 11 % slower; 4 chunks with 8 slots: 6 % slower)
    chunks = min(2, s.layers[0]["x"].shape[0])
    pipes, host = [], []
    for e in s.layers:
        pipes.append(HostPipeline(e["state0"], e["A"], e["D"], wl.ntok, wl.ngroups, wl.torch_in_dtype,
                                  chunks=chunks, slots=2 * chunks, streams=streams))
        acc = e["host"]["accept_len"] if wl.accept != "all" else torch.full_like(e["host"]["accept_len"], wl.ntok)
        h = {k: e["host"][k].pin_memory() for k in ("x", "B", "C", "dt")}
        h["accept_len"] = acc.pin_memory()
        h["y"] = torch.empty(e["y"].shape, dtype=torch.float32).pin_memory()
        host.append(h)
    keys = ("x", "B", "C", "dt", "accept_len")
    h2d = sum(sum(h[k].numel() * h[k].element_size() for k in keys) for h in host)
    d2h = sum(h["y"].numel() * 4 for h in host)

    from ssm_recurrence_verify_b300.hostpipe import capture_step
    step_args = [(h["x"], h["B"], h["C"], h["dt"], h["accept_len"], h["y"]) for h in host]
    for p, a_ in zip(pipes, step_args):  # eager warm-up
        p.run(*a_)
    torch.cuda.synchronize()
    per_graph = E2E_STEPS_PER_GRAPH
    graph = capture_step(pipes, step_args, dev, repeat=per_graph)
    replay = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(replay):
        for _ in range(3):
            graph.replay()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n = max(per_graph, args.e2e_steps // per_graph * per_graph)
    barrier(world)
    with torch.cuda.stream(replay):
        t0.record(replay)
        for _ in range(n // per_graph):
            graph.replay()
        t1.record(replay)
    torch.cuda.synchronize()
    ms = max_over_ranks(t0.elapsed_time(t1), world)
    for p in pipes:
        assert int(p.status.item()) == 0, "device reported a bad accept_len"
    return {"value": s.layers[0]["x"].shape[0] * wl.ntok * len(s.layers) * world * n / (ms * 1e-3), "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n,
            "path": f"HostPipeline: {chunks} sequence chunks per layer, {2 * chunks} staging slots, copy-in (SM reads "
                    f"of pinned memory) / kernel / copy-out streams overlapped, {per_graph} consecutive steps per "
                    f"CUDA graph"}


def run_e2e_pieces(args, local_rank):
    """The end-to-end step of the serving workload taken apart: each piece of
    one HostPipeline step (2 sequence chunks, 4 staging slots) enqueued as the
    pipeline does it, captured into a CUDA graph of 16 steps and timed per
    step: the SM pulls of the inputs, the copy-engine read-back of y, both at
    once, the chunk kernels, pulls and kernels at once, and the whole step."""
    import ssm_recurrence_verify_b300 as ssm
    from ssm_recurrence_verify_b300 import build as libbuild
    from ssm_recurrence_verify_b300 import ssmverify as sv
    from ssm_recurrence_verify_b300.hostpipe import HostPipeline, capture_step
    if not os.path.exists(libbuild.LIB):
        libbuild.build()
    ssm.load_library()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    wl = synth.WORKLOADS[args.workload]
    e = LayerSet(wl, wl.batch, 0, 0, dev, 1).layers[0]
    h = {k: e["host"][k].pin_memory() for k in ("x", "B", "C", "dt", "accept_len")}
    h["y"] = torch.empty(e["y"].shape, dtype=torch.float32).pin_memory()
    streams = tuple(torch.cuda.Stream(device=dev) for _ in range(3))
    p = HostPipeline(e["state0"], e["A"], e["D"], wl.ntok, wl.ngroups, wl.torch_in_dtype, chunks=2, streams=streams)
    rep = E2E_STEPS_PER_GRAPH
    reps = max(2, args.steps // rep)

    def chunks():
        for c in range(p.chunks):
            lo, hi = p.bounds[c], p.bounds[c + 1]
            yield c, lo, hi, hi - lo

    def pulls():
        for c, lo, hi, n in chunks():
            sv.copy_from_host_n(((p.slot_x[c][:n], h["x"][lo:hi]), (p.slot_B[c][:n], h["B"][lo:hi]),
                                 (p.slot_C[c][:n], h["C"][lo:hi]), (p.slot_dt[c][:n], h["dt"][lo:hi]),
                                 (p.slot_acc[c][:n], h["accept_len"][lo:hi])), stream=p.s_in)

    def readback():
        with torch.cuda.stream(p.s_out):
            for c, lo, hi, n in chunks():
                h["y"][lo:hi].copy_(p.slot_y[c][:n], non_blocking=True)

    def kernels():
        for c, lo, hi, n in chunks():
            sv.verify_commit(p.state[lo:hi], p.slot_x[c][:n], p.slot_B[c][:n], p.slot_C[c][:n], p.slot_dt[c][:n],
                             p.A, p.D, p.slot_acc[c][:n], y=p.slot_y[c][:n], dev_status=p.status, stream=p.s_k)

    def time_graph(fn):
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(device=dev)
        with torch.cuda.graph(g, stream=cap):
            fork = torch.cuda.Event()
            fork.record(cap)
            for st in streams:
                st.wait_event(fork)
            for _ in range(rep):
                fn()
            for st in streams:
                ev = torch.cuda.Event()
                ev.record(st)
                cap.wait_event(ev)
        return g

    args_ = (h["x"], h["B"], h["C"], h["dt"], h["accept_len"], h["y"])
    pulls(), readback(), kernels(), p.run(*args_)
    torch.cuda.synchronize()
    graphs = {"pull_us": time_graph(pulls), "readback_us": time_graph(readback),
              "pull_and_readback_us": time_graph(lambda: (pulls(), readback())),
              "kernels_us": time_graph(kernels), "pull_and_kernels_us": time_graph(lambda: (pulls(), kernels())),
              "step_us": capture_step([p], [args_], dev, repeat=rep)}
    upload_graphs(list(graphs.values()), torch.cuda.current_stream(dev))
    rs = torch.cuda.Stream(device=dev)
    out = {}
    for name, g in graphs.items():
        with torch.cuda.stream(rs):
            for _ in range(2):
                g.replay()
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(rs):
            t0.record(rs)
            for _ in range(reps):
                g.replay()
            t1.record(rs)
        torch.cuda.synchronize()
        out[name] = t0.elapsed_time(t1) * 1e3 / (reps * rep)
    assert int(p.status.item()) == 0, "device reported a bad accept_len"
    bytes_in = sum(t.numel() * t.element_size() for k, t in h.items() if k != "y")
    bytes_out = h["y"].numel() * 4
    return {"path": "e2e_pieces", "workload": wl.name, "steps_per_graph": rep, "graphs_timed": reps,
            "h2d_bytes_per_step": bytes_in, "d2h_bytes_per_step": bytes_out,
            **{k: round(v, 1) for k, v in out.items()},
            "step_tokens_per_s": wl.batch * wl.ntok / (out["step_us"] * 1e-6),
            "transfer_bound_tokens_per_s": wl.batch * wl.ntok / (out["pull_and_readback_us"] * 1e-6)}


# ----------------------------------------------------------------------------- acceptance step

ACCEPT_METRIC = "draft tokens decided/s (acceptance step); achieved HBM GB/s vs B300 peak"


def accept_algorithmic_bytes(aw, accept_len, sample: bool) -> int:
    """Bytes the acceptance rule must read for the given outcomes: per
    sequence the verifier rows 0..j (the rows its decisions and its next token
    depend on) and, for sampling, the draft rows 0..min(j, K-1); plus the draft
    tokens (and uniforms), accept_len and next_token."""
    K, V, es = aw.ntok, aw.vocab, aw.logit_bytes()
    n = 0
    for j in accept_len:
        j = int(j)
        n += (j + 1) * V * es + (min(j + 1, K) * V * es if sample else 0)
    batch = len(accept_len)
    n += batch * K * 4 + batch * 8 + (batch * (K + 1) * 4 if sample else 0)
    return n


def run_accept(args, sample: bool, rank, world, local_rank):
    """Time the device acceptance step (one launch per step) on the batched
    serving workload's logits, with the same graph capture, L2 rotation and
    clock sampling as the main path."""
    import ssm_recurrence_verify_b300 as ssm
    from ssm_recurrence_verify_b300 import build as libbuild
    if not os.path.exists(libbuild.LIB):
        libbuild.build()
    ssm.load_library()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    aw = synth.ACCEPT_WORKLOADS[1]
    batch, offset = shard(aw.batch, rank)
    stream = torch.cuda.Stream(device=dev)
    sets = []

    def launch(e):
        if sample:
            ssm.accept_sample(e["target_logits"], e["draft_logits"], e["draft_tokens"], e["uniform"],
                              accept_len=e["accept_len"], next_token=e["next_token"], dev_status=e["status"],
                              stream=stream)
        else:
            ssm.accept_greedy(e["target_logits"], e["draft_tokens"], accept_len=e["accept_len"],
                              next_token=e["next_token"], dev_status=e["status"], stream=stream)

    # The rule reads only the rows up to each sequence's first rejection, so a
    # launch reads less than its inputs: add independent input sets until every
    # set is read again only after more than 2x the L2 of other sets' reads.
    while True:
        w = synth.custom_accept_workload(aw.batch, aw.ntok, aw.vocab, aw.logit_dtype, seed=aw.seed + 1000 * len(sets))
        d = synth.draw_accept_inputs(w, batch=batch, batch_offset=offset)
        e = {k: v.to(dev) for k, v in d.items()}
        e["accept_len"] = torch.empty(batch, dtype=torch.int32, device=dev)
        e["next_token"] = torch.empty(batch, dtype=torch.int32, device=dev)
        e["status"] = torch.zeros(1, dtype=torch.int32, device=dev)
        with torch.cuda.stream(stream):
            launch(e)
        torch.cuda.synchronize()
        e["bytes"] = accept_algorithmic_bytes(aw, e["accept_len"].cpu().tolist(), sample)
        sets.append(e)
        others = sum(x["bytes"] for x in sets) - max(x["bytes"] for x in sets)
        if len(sets) >= 2 and others > 2 * L2_BYTES:
            break
        if len(sets) >= 12:
            break
    nsets = len(sets)

    def capture(idx):
        out = []
        for i in range(0, len(idx), MAX_GRAPH_LAUNCHES):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for si in idx[i:i + MAX_GRAPH_LAUNCHES]:
                    launch(sets[si])
            out.append(g)
        return out

    K = args.steps
    warm = capture([i % nsets for i in range(args.warmup)])
    timed = capture([(args.warmup + i) % nsets for i in range(K)])
    torch.cuda.synchronize()
    upload_graphs(warm + timed, stream)
    sampler = ClockSampler(local_rank)
    sampler.start()
    with torch.cuda.stream(stream):
        for g in warm:
            g.replay()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    with torch.cuda.stream(stream):
        t0.record(stream)
        for g in timed:
            g.replay()
        t1.record(stream)
    torch.cuda.synchronize()
    wall1 = time.perf_counter()
    barrier(world)
    sampler.stop()
    for e in sets:
        assert int(e["status"].item()) == 0, "device reported a bad draft token"
    ms = max_over_ranks(t0.elapsed_time(t1), world)
    launch_ms = t0.elapsed_time(t1) / K
    set_bytes = statistics.fmean(sets[(args.warmup + i) % nsets]["bytes"] for i in range(K))
    achieved = set_bytes / (launch_ms * 1e-3) / 1e9
    peak, peak_kind = hbm_peak()
    value = batch * world * aw.ntok * K / (ms * 1e-3)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        from oracle import accept as acc
        n_seq = 4
        d = synth.draw_accept_inputs(aw, batch=n_seq)
        reps, c0 = 0, time.perf_counter()
        while True:
            if sample:
                acc.accept_sample(d["target_logits"], d["draft_logits"], d["draft_tokens"], d["uniform"])
            else:
                acc.accept_greedy(d["target_logits"], d["draft_tokens"])
            reps += 1
            if time.perf_counter() - c0 >= args.cpu_seconds:
                break
        el = time.perf_counter() - c0
        cpu = {"value": n_seq * aw.ntok * reps / el, "unit": "tokens/s", "cores": 1, "kind": "oracle",
               "sample": f"{n_seq} of the {aw.batch} sequences, {reps} passes, {el:.1f} s, numpy single thread"}
    rule = "speculative sampling" if sample else "greedy"
    return {
        "metric": ACCEPT_METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded; no dataset)",
        "config": {"workload": aw.name, "rule": rule, "batch_per_gpu": batch, "draft_tokens": aw.ntok,
                   "vocab": aw.vocab, "logit_dtype": aw.logit_dtype,
                   "l2": f"{nsets} independent input sets rotated (each read again after > 2x the L2 of other reads)",
                   "reads": "rows up to each sequence's first rejection (the rows the rule depends on)",
                   "timing": f"timed steps captured as CUDA graphs of up to {MAX_GRAPH_LAUNCHES} launches"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": None, "peak_source": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)",
                     "algorithmic_bytes_per_launch": set_bytes, "launch_us_mean": launch_ms * 1e3},
        "cpu_baseline": cpu, "gpu_launches": K, "clocks": sampler.summary(wall0, wall1),
    }


# ----------------------------------------------------------------------------- prefill

PREFILL_METRIC = "prompt tokens/s per SSM layer (prefill); achieved tensor TFLOP/s vs B300 peak"
FALLBACK_BF16_TFLOPS = 1800.0
TF32_PER_BF16 = 1.1 / 2.25  # nominal dense tensor rates of B300: tf32 1.1, bf16 2.25 PFLOP/s


def bf16_peak():
    """Measured dense bf16 tensor throughput (cuBLAS burst) of the B300s."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


def prefill_tensor_macs(H: int, P: int, N: int, T: int, L: int, bf16: bool):
    """Multiply-adds the chunked prefill issues on the tensor cores for one
    prompt of T tokens in chunks of L, split products counted as issued.
    Returns (MACs, operand kind), or (None, why) for shapes not modelled.

    bf16, N 128, L 128, P a multiple of 64: the tcgen05 passes. Chunk states
    S = (w o U) B with w o U in two bf16 parts (B exact): 2 H P T N. Chunk
    outputs per tile of PR rows (128, or 64 where P is not a multiple of 128):
    G = C B^T (L L N), Yi = C H0^T with H0 in two parts (2 L N PR), Yc = M X
    with M in two parts (2 L L PR).
    Otherwise (mma.sync m16n8k8 tf32, 1024 MACs each): chunk states with w o U
    split, fp32 B split too (2 or 3 products); chunk outputs by the tile
    kernel in 8-token sub-chunks, per warp (16 rows) and sub-chunk: h C^T over
    N / 8 k-blocks (2 or 3 products), the Gram C B^T likewise (1 or 3, every
    warp), the intra-chunk term (3), and the state advance over N / 8 blocks
    (2 or 3) for every sub-chunk but a chunk's last."""
    nch = T // L
    if bf16 and N == 128 and L == 128 and P % 64 == 0:
        pr = 128 if P % 128 == 0 else 64
        states = 2 * H * P * T * N
        outputs = nch * H * (P // pr) * (L * L * N + 2 * L * N * pr + 2 * L * L * pr)
        return states + outputs, "tcgen05 kind::f16 (bf16 operands, fp32 accumulation)"
    if N > 128:
        return None, "not modelled for dstate > 128"
    sp = 2 if bf16 else 3
    states = sp * H * P * T * N
    warps = nch * H * (-(-P // 16))  # 16-row bands of the 64-row tiles
    sub = L // 8
    per_sub = (N // 8) * sp + (N // 8) * (1 if bf16 else 3) + 3
    adv = (N // 8) * sp
    outputs = warps * (sub * per_sub + (sub - 1) * adv) * 1024
    return states + outputs, "mma.sync m16n8k8 tf32 (fp32 accumulation)"


# prompt shapes of the prefill bench: name -> (heads, headdim, dstate, ngroups)
PREFILL_SHAPES = {
    "llama3_8b": (32, 128, 128, 8),   # the distilled Llama-3-8B hybrid's Mamba layer
    "mamba2_2p7b": (80, 64, 128, 1),  # a Mamba-2-2.7B layer
}


def run_prefill(args, rank, world, local_rank):
    """Time ssm_prefill: one layer of the chosen shape (default Llama-3-8B:
    H 32, P 128, N 128, G 8; or Mamba-2-2.7B: H 80, P 64, N 128, G 1), one
    2048-token bf16 prompt per GPU, from a zeroed cache slot. The algorithmic
    work is the recurrence over the prompt: 5 flops per state element and
    token (u B, Abar h + u B, and y = C h)."""
    import ssm_recurrence_verify_b300 as ssm
    from ssm_recurrence_verify_b300 import build as libbuild
    if not os.path.exists(libbuild.LIB):
        libbuild.build()
    ssm.load_library()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    H, P, N, G = PREFILL_SHAPES[args.prefill_shape]
    in_dtype = synth.BF16 if args.prefill_dtype == "bf16" else synth.F32
    wl = synth.custom_workload(1, H, P, N, G, 2048, in_dtype, seed=500, accept="all")
    T = wl.ntok
    # inputs + y + state of one step; the workspace (shared) adds its own traffic
    eb = wl.in_elem_bytes()
    step_bytes = T * (wl.nheads * wl.headdim * (eb + 4) + 2 * wl.ngroups * wl.dstate * eb + wl.nheads * eb) \
        + 2 * wl.nheads * wl.headdim * wl.dstate * 4
    nsets = max(2, math.ceil(2 * L2_BYTES / step_bytes) + 1)  # each set read again after > 2x the L2 of others
    sets = []
    for i in range(nsets):
        d = synth.draw_layer_round(wl, rnd=i)
        e = {k: v.to(dev) for k, v in d.items()}
        e["y"] = torch.empty((1, T, wl.nheads, wl.headdim), dtype=torch.float32, device=dev)
        e["pool"] = torch.zeros(1, wl.nheads, wl.headdim, wl.dstate, device=dev)
        sets.append(e)
    nbytes = ssm.prefill_workspace_bytes(sets[0]["pool"], sets[0]["x"], sets[0]["B"], sets[0]["C"], sets[0]["dt"],
                                         sets[0]["A"], sets[0]["D"])
    ws = torch.empty(max(nbytes, 16) // 4, dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def launch(e, chunked=True):
        ssm.prefill(e["pool"], None, e["x"], e["B"], e["C"], e["dt"], e["A"], e["D"], y=e["y"],
                    workspace=ws if chunked else ws[:0], dev_status=status, stream=stream)

    def timed(chunked, steps):
        with torch.cuda.stream(stream):
            for e in sets:
                launch(e, chunked)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(steps):
                launch(sets[i % nsets], chunked)
        with torch.cuda.stream(stream):
            g.replay()
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            t0.record(stream)
            g.replay()
            t1.record(stream)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1) / steps

    steps = max(3, min(args.steps, 200))
    sampler = ClockSampler(local_rank)
    sampler.start()
    wall0 = time.perf_counter()
    ms = timed(True, steps)
    wall1 = time.perf_counter()
    sampler.stop()
    ms_one_pass = timed(False, max(3, steps // 4))
    assert int(status.item()) == 0, "device reported a problem"
    ms_max = max_over_ranks(ms, world)
    # chunk length the library chose: the workspace holds one state per chunk (+ a small slot map)
    nch = nbytes // (wl.nheads * wl.headdim * wl.dstate * 4) if nbytes > 0 else 0
    L = T // nch if nch > 0 else T
    bf16 = args.prefill_dtype == "bf16"
    macs, kind = prefill_tensor_macs(H, P, N, T, L, bf16) if nch > 0 else (None, "one pass")
    peak, peak_kind = bf16_peak()
    if not bf16:
        peak *= TF32_PER_BF16
    achieved = 2.0 * macs / (ms * 1e-3) / 1e12 if macs else None
    io_bytes = step_bytes
    hbm, hbm_kind = hbm_peak()
    io_gbs = io_bytes / (ms * 1e-3) / 1e9
    return {
        "metric": PREFILL_METRIC, "value": T * world / (ms_max * 1e-3), "unit": "tokens/s", "n_gpus": world,
        "steps": steps, "warmup": 3, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded; no dataset)",
        "config": {"workload": f"prefill_{args.prefill_shape}_layer_b1_t{T}_h{H}_p{P}_n{N}_g{G}"
                               + ("" if args.prefill_dtype == "bf16" else "_f32"), "prompt_tokens": T,
                   "batch_per_gpu": 1, "in_dtype": args.prefill_dtype, "workspace_bytes": nbytes,
                   "timing": f"{steps} launches captured in one CUDA graph",
                   "l2": f"{nsets} independent input sets rotated (each read again after > 2x the L2 of other traffic)"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak if achieved else None, "traffic": None,
                     "peak_source": (f"{peak_kind} bf16 dense (MEASURED_PEAKS.json bf16_tflops)" if bf16 else
                                     f"{peak_kind} bf16 dense x {TF32_PER_BF16:.3f} (nominal tf32 / bf16 ratio)"),
                     "work": f"tensor-core multiply-adds issued by the chunked form ({kind}; chunk length {L}), "
                             "split products counted as issued, x 2 flops, over the whole step (three kernels)",
                     "issued_flops_per_step": 2.0 * macs if macs else None,
                     "hbm_gbs_on_io_bytes": io_gbs, "hbm_frac_on_io_bytes": io_gbs / hbm,
                     "io_bytes_per_step": io_bytes,
                     "io_bytes": "prompt inputs read once, y written once in fp32, the cached state read and written"},
        "one_pass_ms": ms_one_pass,
        # the chunked form is three kernels per prompt (chunk states, scan, outputs); the one pass is one
        "gpu_launches": steps * (3 if nbytes > 0 else 1), "clocks": sampler.summary(wall0, wall1),
    }


# ----------------------------------------------------------------------------- oracle (CPU) legs

def oracle_throughput(wl, seconds: float, max_seqs: int = None):
    """Time the fp64 oracle (single thread, as it stands) on the workload's
    first layer, repeating full passes over `max_seqs` sequences until
    `seconds` have elapsed. Returns (tokens per second, description)."""
    import oracle
    seqs = wl.batch if max_seqs is None else min(wl.batch, max_seqs)
    d = synth.draw_layer_round(wl, batch=seqs)
    args = (d["state0"], d["x"], d["B"], d["C"], d["dt"], d["A"], d["D"],
            None if wl.accept == "all" else d["accept_len"])
    reps = 0
    t0 = time.perf_counter()
    while True:
        oracle.verify_commit(*args)
        reps += 1
        if time.perf_counter() - t0 >= seconds:
            break
    el = time.perf_counter() - t0
    toks = seqs * wl.ntok * reps
    return toks / el, (f"{reps} full oracle pass(es) over {seqs} sequence(s) x {wl.ntok} draft tokens of one layer "
                       f"({wl.nheads} heads, P {wl.headdim}, N {wl.dstate}), fp64, {el:.1f} s")


def oracle_throughput_threads(wl, seconds: float, threads: int):
    """The same fp64 oracle, as it stands, on `threads` host threads at once:
    thread i runs full passes over sequence i (mod the batch) of the
    workload's first layer until `seconds` have elapsed. The C recurrence runs
    outside the GIL (ctypes releases it for the call), so the threads occupy
    that many cores. Returns (tokens per second, description)."""
    import concurrent.futures
    import oracle
    args = []
    for i in range(threads):
        d = synth.draw_layer_round(wl, batch=1, batch_offset=i % wl.batch)
        args.append((d["state0"], d["x"], d["B"], d["C"], d["dt"], d["A"], d["D"],
                     None if wl.accept == "all" else d["accept_len"]))
    oracle.verify_commit(*args[0])  # the library loaded (or built) once, before the threads start
    start = threading.Barrier(threads + 1)

    def work(a):
        start.wait(timeout=120)
        t0, reps = time.perf_counter(), 0
        while True:
            oracle.verify_commit(*a)
            reps += 1
            if time.perf_counter() - t0 >= seconds:
                return reps

    with concurrent.futures.ThreadPoolExecutor(max_workers=threads) as ex:
        futs = [ex.submit(work, a) for a in args]
        start.wait(timeout=120)
        t0 = time.perf_counter()
        reps = [f.result() for f in futs]
        el = time.perf_counter() - t0
    toks = sum(reps) * wl.ntok
    return toks / el, (f"{threads} threads at once, thread i over sequence i mod {wl.batch}: {sum(reps)} full oracle "
                       f"passes of one sequence x {wl.ntok} draft tokens of one layer ({wl.nheads} heads, "
                       f"P {wl.headdim}, N {wl.dstate}), fp64, {el:.1f} s")


def host_cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or "unknown"


def cgroup_cpu_limit(path: str = "/sys/fs/cgroup/cpu.max"):
    """Whole cores a cgroup-v2 CPU quota allows ("quota period"), or None when unlimited or absent."""
    try:
        with open(path) as f:
            quota, period = f.read().split()[:2]
        if quota == "max":
            return None
        return max(1, int(int(quota) // int(period)))
    except (OSError, ValueError):
        return None


def host_threads(cap: int = 64) -> int:
    """Cores this process may run on: its affinity set, within the cgroup's CPU quota, at most `cap`."""
    try:
        n = len(os.sched_getaffinity(0))
    except AttributeError:
        n = os.cpu_count() or 1
    q = cgroup_cpu_limit()
    if q is None:  # cgroup v1: quota and period in two files, -1 = unlimited
        try:
            with open("/sys/fs/cgroup/cpu/cpu.cfs_quota_us") as fq, open("/sys/fs/cgroup/cpu/cpu.cfs_period_us") as fp:
                quota, period = int(fq.read()), int(fp.read())
            q = max(1, quota // period) if quota > 0 and period > 0 else None
        except (OSError, ValueError):
            q = None
    if q is not None:
        n = min(n, q)
    return max(1, min(cap, n))


def reference_sample(wl, per_unit_s: float, steps: int):
    """Pick (sequences, heads) per oracle step so that `steps` steps take
    about two minutes. The smallest unit is one sequence and one B/C group's
    heads; heads are taken as whole groups from head 0."""
    hpg = wl.nheads // wl.ngroups
    units_total = wl.batch * wl.ngroups
    budget_units = 120.0 / max(1, steps) / per_unit_s
    units = int(max(1, min(units_total, budget_units)))
    if units >= wl.ngroups:
        return min(wl.batch, units // wl.ngroups), wl.nheads
    return 1, units * hpg


def run_reference(args, wl, rank, world):
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    hpg = wl.nheads // wl.ngroups

    def inputs(seqs, heads):
        d = synth.draw_layer_round(wl, batch=seqs)
        g = heads // hpg
        return (d["state0"][:, :heads].contiguous(), d["x"][:, :, :heads].contiguous(),
                d["B"][:, :, :g].contiguous(), d["C"][:, :, :g].contiguous(), d["dt"][:, :, :heads].contiguous(),
                d["A"][:heads].contiguous(), d["D"][:heads].contiguous(),
                None if wl.accept == "all" else d["accept_len"])

    a1 = inputs(1, hpg)
    t0 = time.perf_counter()
    oracle.verify_commit(*a1)
    per_unit = max(time.perf_counter() - t0, 1e-5)
    seqs, heads = reference_sample(wl, per_unit, args.steps + args.warmup)
    a = inputs(seqs, heads)
    for _ in range(args.warmup):
        oracle.verify_commit(*a)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.verify_commit(*a)
    el = time.perf_counter() - t0
    # a token of one layer is all heads of one sequence; a head subset counts pro rata
    value = seqs * wl.ntok * (heads / wl.nheads) * args.steps / el
    sample = (f"each step: {seqs} of {wl.batch} sequences x {heads} of {wl.nheads} heads x {wl.ntok} draft tokens "
              f"of one layer, fp64 oracle, single thread; tokens credited pro rata to the heads run")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el * 1e3 / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded; no dataset)",
        "config": workload_config(wl, None, world),
        "cpu_baseline": {"kind": "oracle", "value": value, "unit": "tokens/s", "cores": 1, "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def tensor_line(r, wl):
    """The tensor-pipe side of the roofline (the HBM side is `roofline`): the
    mma.sync tf32 work one launch issues, per its average duration, against
    the tf32 dense peak (the measured bf16 peak x the nominal tf32 / bf16
    ratio). At K = 16 the path sits near the compute / HBM ridge."""
    macs = r.get("macs_per_launch", 0)
    if not macs:
        return None
    bf, kind = bf16_peak()
    peak = bf * TF32_PER_BF16
    achieved = 2.0 * macs / (r["launch_ms_mean"] * 1e-3) / 1e12
    return {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
            "issued_flops_per_launch": 2.0 * macs,
            "work": "mma.sync m16n8k8 tf32 multiply-adds issued (split products counted), x 2 flops",
            "peak_source": f"{kind} bf16 dense x {TF32_PER_BF16:.3f} (nominal tf32 / bf16 ratio)"}


ALT_PATHS = {
    "commit_verify": ("draft tokens verified/s per SSM layer, deferred-commit order (ssm_commit_verify); "
                      "achieved HBM GB/s vs B300 peak",
                      {"previous_block": "the set's own round (its drafts and accept_len)",
                       "new_block": "the next round's drafts"}),
    "unfused": ("draft tokens verified/s per SSM layer, unfused (ssm_verify then ssm_commit, two launches per "
                "layer-call); achieved HBM GB/s vs B300 peak over the pair",
                {"launches_per_layer_call": 2}),
}


def alt_path_line(args, wl, r, world):
    """The JSON line of --path commit_verify / unfused: the verify/commit
    workload through another entry point, device-timed like the default path,
    with the HBM roofline on what those calls must move (for the unfused
    pair: both launches together, per layer-call)."""
    metric, extra = ALT_PATHS[args.path]
    return {
        "metric": metric,
        "value": r["value"], "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": r["ms_per_step"], "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic (seeded; no dataset)", "path": args.path,
        "config": dict(workload_config(wl, r["nsets"], world, r.get("reread_bytes")),
                       layers_per_launch=r["layers_per_launch"], **extra),
        "roofline": {"bound": "hbm", "achieved": r["achieved_gbs"], "peak": r["peak"], "unit": "GB/s",
                     "frac": r["achieved_gbs"] / r["peak"], "traffic": None,
                     "peak_source": f"{r['peak_kind']} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)",
                     "algorithmic_bytes_per_launch": r["bytes_per_launch"],
                     "launch_us_mean": r["launch_ms_mean"] * 1e3,
                     "frac_of_8tbs_spec": r["achieved_gbs"] / HBM_SPEC_GBS},
        "cpu_baseline": None, "e2e": None, "gpu_launches": r["launches"], "clocks": r["clocks"],
    } | ({"note": "roofline.achieved and launch_us_mean are per layer-call: the two launches together"}
         if args.path == "unfused" else {})


def workload_config(wl, nsets, world: int = 1, reread_bytes=None):
    cfg = {"workload": wl.name, "batch_per_gpu": wl.batch, "layers": wl.nlayers, "nheads": wl.nheads,
           "headdim": wl.headdim, "dstate": wl.dstate, "ngroups": wl.ngroups, "draft_tokens": wl.ntok,
           "in_dtype": wl.in_dtype, "state_dtype": "f32", "accept_len": wl.accept,
           # each rank runs its own sequences (a batch shard) with no collective on the data path
           "parallelism": f"dp{world}" if world > 1 else "single GPU"}
    if nsets is not None and reread_bytes is not None and nsets > 1 and reread_bytes < 2 * L2_BYTES:
        cfg["l2"] = (f"{nsets} independent input sets rotated (at most {NSETS_CAP}); each set is read again after "
                     f"{reread_bytes / 1e6:.1f} MB of other traffic, less than 2x the 126 MB L2: the workload is "
                     f"smaller than the cache")
    elif nsets is not None:
        cfg["l2"] = (f"{nsets} independent input sets rotated; each set is read again only after more than "
                     f"2x the 126 MB L2 of other traffic")
        cfg["timing"] = (f"timed steps captured as CUDA graphs of up to {MAX_GRAPH_LAUNCHES} launches, replayed back to "
                         f"back; CUDA events on the launching stream around the whole region")
    return cfg


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=3, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--cpu-threads", type=int, default=0,
                    help="host threads for the second, multi-threaded oracle timing (0: the cores this process "
                         "may use, at most 64; 1: skip it)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--layers", type=int, default=None,
                    help="run only the first N layers of a layer stack (a smaller case for profiling)")
    ap.add_argument("--per-layer-launches", action="store_true",
                    help="run a layer stack as one launch per layer instead of one launch over all layers")
    ap.add_argument("--path", choices=["ssm", "commit_verify", "unfused", "accept_sample", "accept_greedy", "prefill",
                                       "e2e_pieces"],
                    default="ssm",
                    help="ssm: the verify/commit step (default); commit_verify: the same workload in the serving "
                         "order, each call committing the previous round's accepted prefix and verifying the next "
                         "round's drafts (ssm_commit_verify); unfused: the same workload as ssm_verify then "
                         "ssm_commit (two launches per layer-call); accept_*: the acceptance step alone; "
                         "prefill: a 2048-token prompt through one layer; e2e_pieces: the host-buffer step of the "
                         "workload taken apart (copies in, read-back, kernels, each alone and together)")
    ap.add_argument("--prefill-dtype", choices=["bf16", "f32"], default="bf16",
                    help="prompt input dtype of --path prefill (f32 prompts take the mma.sync chunk-state pass and "
                         "the tile kernel's chunk outputs instead of the tcgen05 passes)")
    ap.add_argument("--prefill-shape", choices=sorted(PREFILL_SHAPES), default="llama3_8b",
                    help="layer shape of --path prefill")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    wl = synth.WORKLOADS[args.workload]
    if args.layers is not None:  # the first `layers` layers of the stack (profiling a smaller case)
        if not 1 <= args.layers <= wl.nlayers:
            ap.error(f"--layers must be in [1, {wl.nlayers}]")
        wl = dataclasses.replace(wl, nlayers=args.layers, name=f"{wl.name}_first{args.layers}layers")
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        return launch_ranks(sys.argv[1:] if argv is None else argv, args.gpus)
    rank, world, local_rank = dist_env()
    if world != args.gpus:
        ap.error(f"--gpus {args.gpus} but the launcher started {world} rank(s)")

    if args.impl == "reference":
        return run_reference(args, wl, rank, world)

    if world > 1:
        init_ranks(world, local_rank)
    if args.path not in PATH_MODES:
        if args.path == "prefill":
            line = run_prefill(args, rank, world, local_rank)
        elif args.path == "e2e_pieces":
            line = run_e2e_pieces(args, local_rank)
        else:
            line = run_accept(args, args.path == "accept_sample", rank, world, local_rank)
        if rank == 0:
            print(json.dumps(line), flush=True)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return 0
    r = run_ours(args, wl, rank, world, local_rank)

    if args.path != "ssm":
        if rank == 0:
            print(json.dumps(alt_path_line(args, wl, r, world)), flush=True)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return 0

    cpu = cpu_all = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, sample = oracle_throughput(wl, args.cpu_seconds)
        cpu = {"value": v, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": sample,
               "cpu_model": host_cpu_model()}
        nt = host_threads() if args.cpu_threads == 0 else args.cpu_threads
        if nt > 1:  # a window that keeps the CPU work near 2 x cpu_seconds however many threads run
            v, sample = oracle_throughput_threads(wl, max(0.5, 2.0 * args.cpu_seconds / nt), nt)
            cpu_all = {"value": v, "unit": "tokens/s", "cores": nt, "kind": "oracle", "sample": sample,
                       "cpu_model": cpu["cpu_model"]}

    if rank == 0:
        traffic = recorded_traffic(wl.name)
        line = {
            "metric": METRIC, "value": r["value"], "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": r["ms_per_step"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded; no dataset)",
            "config": dict(workload_config(wl, r["nsets"], world, r.get("reread_bytes")),
                           layers_per_launch=r["layers_per_launch"]),
            "roofline": {"bound": "hbm", "achieved": r["achieved_gbs"], "peak": r["peak"], "unit": "GB/s",
                         "frac": r["achieved_gbs"] / r["peak"], "traffic": traffic,
                         "peak_source": f"{r['peak_kind']} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)",
                         "algorithmic_bytes_per_launch": r["bytes_per_launch"],
                         "launch_us_mean": r["launch_ms_mean"] * 1e3,
                         "frac_of_8tbs_spec": r["achieved_gbs"] / HBM_SPEC_GBS},
            "tensor": tensor_line(r, wl),
            "cpu_baseline": cpu,
            "cpu_baseline_threads": cpu_all,
            "e2e": r["e2e"],
            "gpu_launches": r["launches"],
            "clocks": r["clocks"],
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
