"""bench.py's verify/commit paths end to end on the GPU, a few steps each: the
default fused call, the deferred-commit order (ssm_commit_verify) and the
unfused pair (ssm_verify then ssm_commit). Each prints one JSON line whose
launch count, byte count and roofline fraction must be consistent with the
workload (a fraction far above 1 would mean the timed kernels skip work)."""
import json

import pytest

import bench
from ssm_recurrence_verify_b300 import synth

pytestmark = pytest.mark.gpu


def _line(capsys, argv):
    assert bench.main(argv) == 0
    out = [l for l in capsys.readouterr().out.splitlines() if l.startswith("{")]
    assert len(out) == 1
    return json.loads(out[0])


# the tiny fp32 case, and the 16-layer hybrid (bf16, one call over the layer stack; small enough to draw quickly)
@pytest.mark.parametrize("workload", [0, 2])
@pytest.mark.parametrize("path,kernels", [("ssm", 1), ("commit_verify", 1), ("unfused", 2)])
def test_bench_path_line(cuda_device, capsys, workload, path, kernels):
    steps = 6
    argv = ["--workload", str(workload), "--steps", str(steps), "--warmup", "3", "--path", path]
    if path == "ssm":
        argv += ["--no-cpu-baseline", "--e2e-steps", "0"]
    d = _line(capsys, argv)
    wl = synth.WORKLOADS[workload]
    assert d["n_gpus"] == 1 and d["steps"] == steps and d["warmup"] == 3
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["gpu_launches"] == steps * kernels  # a layer stack runs as one call per step
    assert d["config"]["layers_per_launch"] == wl.nlayers
    assert d["config"]["workload"] == wl.name
    r = d["roofline"]
    assert r["bound"] == "hbm" and 0 < r["frac"] < 1.3
    # the byte count per call is at least the state read once and at most read twice and written once
    # plus every input, y and accept_len
    L = wl.nlayers
    slab = L * wl.batch * wl.nheads * wl.headdim * wl.dstate * 4
    assert slab <= r["algorithmic_bytes_per_launch"] <= 3 * slab + L * wl.batch * wl.ntok * (
        3 * wl.nheads * wl.headdim * 4 + 4 * wl.ngroups * wl.dstate * 4 + 2 * wl.nheads * 4) + L * wl.batch * 4
    if path != "ssm":
        assert d["path"] == path
