"""Host-side pieces of the benchmark on CPU: the algorithmic byte count of
one layer-call, the clock summary's window and reason decoding, the tile
kernel's source hash (which decides whether a recorded traffic capture still
applies), the measured-peak lookup, the layer-stack input sets and the
multi-threaded oracle timing."""
import json
import os

import torch

import bench
from ssm_recurrence_verify_b300 import synth


def test_algorithmic_bytes_by_hand():
    """batch 2, H 3, P 4, N 8, G 1, K 5, bf16: the state read for both
    sequences, written for the one with j > 0; x, B, C, dt read once (B and C
    once per group); y written in fp32; accept_len read."""
    wl = synth.custom_workload(2, 3, 4, 8, 1, 5, synth.BF16, seed=1)
    state = 3 * 4 * 8 * 4                        # one sequence's fp32 state: 384 B
    per_token = 3 * 4 * 2 + 2 * 1 * 8 * 2 + 3 * 2  # x, B and C, dt in bf16: 62 B
    y = 3 * 4 * 4                                # fp32 y per token: 48 B
    want = 2 * state + 1 * state + 2 * 5 * (per_token + y) + 2 * 4
    assert bench.algorithmic_bytes(wl, 2, 1) == want == 2260


def test_algorithmic_bytes_accept_all_reads_no_accept_len():
    wl = synth.custom_workload(1, 1, 8, 16, 1, 4, synth.F32, seed=1, accept="all")
    state = 8 * 16 * 4
    assert bench.algorithmic_bytes(wl, 1, 1) == 2 * state + 4 * (8 * 4 + 2 * 16 * 4 + 4 + 8 * 4)


def _sampler(samples, max_mhz=2032.0, mode="nvml"):
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.samples, s.max_mhz, s.mode, s.err = samples, max_mhz, mode, ""
    return s


def test_clock_summary_window_and_reasons():
    # (time, SM MHz, reason bits): only the samples inside [1, 2] count
    s = _sampler([(0.5, 900.0, 0x8), (1.0, 2032.0, 0x0), (1.5, 2000.0, 0x4), (2.0, 1990.0, 0x0),
                  (2.5, 800.0, 0x80)])
    out = s.summary(1.0, 2.0)
    assert out["sm_mhz"] == 2000.0 and out["samples"] == 3 and out["sm_max_mhz"] == 2032.0
    assert out["reasons"] == ["sw_power_cap"]  # the hw_slowdown and thermal bits fall outside the window
    assert "timed region" in out["note"]


def test_clock_summary_decodes_every_reason_bit():
    s = _sampler([(1.0, 1500.0, 0x4 | 0x8 | 0x40 | 0x80)])
    assert s.summary(0.0, 2.0)["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_power_cap",
                                              "sw_thermal_slowdown"]


def test_clock_summary_short_window_and_no_source():
    s = _sampler([(0.1, 2032.0, 0), (0.3, 2032.0, 0)], mode="nvidia-smi")
    out = s.summary(0.15, 0.2)  # shorter than the sampling period: every sample is used, and says so
    assert out["samples"] == 2 and "shorter than the sampling period" in out["note"]
    none = _sampler([], mode=None)
    none.err = "nvml: missing"
    assert none.summary(0.0, 1.0)["sm_mhz"] is None


def test_kernel_source_hash_covers_the_tile_kernel_only(tmp_path):
    """Edits after the prefill marker, and #include lines, leave the hash
    unchanged; an edit of the tile kernel's code changes it."""
    src = ("#include <a.h>\n__global__ void tile() { int a = 1; }\n" + bench.PREFILL_MARKER +
           "\n__global__ void prefill() {}\n")
    p = tmp_path / "k.cu"
    p.write_text(src)
    h0 = bench.kernel_source_hash(str(p))
    p.write_text(src.replace("#include <a.h>", "#include <b.h>").replace("prefill() {}", "prefill() { x(); }"))
    assert bench.kernel_source_hash(str(p)) == h0
    p.write_text(src.replace("int a = 1", "int a = 2"))
    assert bench.kernel_source_hash(str(p)) != h0


def test_recorded_traffic_matches_the_current_tile_kernel():
    """The committed capture of the headline workload was taken on the tile
    kernel as it stands (otherwise the bench reports traffic as null)."""
    name = "batched_spec_serving_b64_h32_p128_n128_g8_k8"
    with open(os.path.join(bench.PROFILES, f"ssm_tile_kernel_{name}.traffic.json")) as f:
        rec = json.load(f)
    assert rec["kernel_source_sha256"] == bench.kernel_source_hash()
    assert bench.recorded_traffic(name) == rec["dram_bytes_per_launch"] > 0


def test_hbm_peak_reads_the_measured_file():
    value, source = bench.hbm_peak()
    path = os.path.join(bench.ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            assert (value, source) == (float(json.load(f)["hbm_gbs"]), "measured")
    else:
        assert (value, source) == (bench.FALLBACK_HBM_GBS, "fallback")


def test_layer_set_shards_views_and_shared_accept_len():
    """The bench's layer-stack input set on CPU: a rank's shard equals its
    slice of the single-process stack, every layer's draw has the same
    accept_len (the stack shares one per sequence), and the per-layer views
    alias the stacked slabs, so per-layer and stacked launches read the same
    memory."""
    wl = synth.custom_workload(4, 2, 8, 16, 1, 3, synth.BF16, seed=9)
    full = bench.LayerSet(wl, 4, 0, 0, "cpu", 3)
    for rank in (0, 1):
        batch, offset = bench.shard(2, rank)
        part = bench.LayerSet(wl, batch, offset, 0, "cpu", 3)
        for k in ("state0", "x", "B", "C", "dt"):
            assert torch.equal(part.stack[k], full.stack[k][:, offset:offset + batch]), (rank, k)
        for k in ("A", "D"):
            assert torch.equal(part.stack[k], full.stack[k]), (rank, k)
        assert torch.equal(part.stack["accept_len"], full.stack["accept_len"][offset:offset + batch])
    for layer, e in enumerate(full.layers):
        assert torch.equal(e["host"]["accept_len"], full.stack["accept_len"])
        for k in ("state0", "x", "y"):
            assert e[k].data_ptr() == full.stack[k][layer].data_ptr(), (layer, k)
        assert e["accepted_nonzero"] == int((full.stack["accept_len"] > 0).sum())
    # the layers differ in their parameters and inputs
    assert not torch.equal(full.stack["A"][0], full.stack["A"][1])
    assert not torch.equal(full.stack["x"][0], full.stack["x"][1])


def test_oracle_timing_on_several_threads():
    """The multi-threaded oracle baseline runs every thread's passes and
    credits their tokens; the host's thread count is its affinity set, capped."""
    wl = synth.WORKLOADS[0]
    v, sample = bench.oracle_throughput_threads(wl, 0.2, 3)
    assert v > 0 and sample.startswith("3 threads at once")
    assert 1 <= bench.host_threads() <= 64 and bench.host_threads(cap=1) == 1
    assert isinstance(bench.host_cpu_model(), str)


def test_json_line_assembly_with_the_device_leg_stubbed(monkeypatch, capsys):
    """main() on a host without a GPU, its device leg replaced by fixed
    numbers: one JSON line with the contract's keys, both oracle baselines
    (one thread, then several) and the roofline fraction computed from them."""
    fake = {"value": 1.0e6, "ms_per_step": 0.5, "nsets": 3, "layers_per_launch": 1, "achieved_gbs": 4000.0,
            "peak": 6400.0, "peak_kind": "measured", "bytes_per_launch": 2.0e6, "launch_ms_mean": 0.5,
            "e2e": None, "launches": 7, "clocks": {"sm_mhz": 2032.0, "sm_max_mhz": 2032.0, "reasons": []}}
    monkeypatch.setattr(bench, "run_ours", lambda *a: fake)
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    assert bench.main(["--workload", "0", "--cpu-seconds", "0.2", "--cpu-threads", "2"]) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks"):
        assert k in line, k
    assert line["roofline"]["frac"] == 4000.0 / 6400.0 and line["roofline"]["bound"] == "hbm"
    assert line["cpu_baseline"]["cores"] == 1 and line["cpu_baseline"]["value"] > 0
    assert line["cpu_baseline_threads"]["cores"] == 2 and line["cpu_baseline_threads"]["value"] > 0
    assert line["config"]["workload"] == synth.WORKLOADS[0].name and line["gpu_launches"] == 7


def test_reference_arm_line(monkeypatch, capsys):
    """`bench.py --impl reference` (the fp64 oracle on the host cores, no GPU):
    one JSON line on the same metric and config as the device arm, with its
    own cpu_baseline and an e2e that copies nothing."""
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.delenv("RANK", raising=False)
    assert bench.main(["--impl", "reference", "--workload", "0", "--steps", "3", "--warmup", "3"]) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC and line["unit"] == "tokens/s"
    assert line["steps"] == 3 and line["warmup"] == 3 and line["value"] > 0 and line["higher_is_better"]
    assert line["config"]["workload"] == synth.WORKLOADS[0].name
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_do_no_work(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--gpus", "2", "--workload", "0", "--steps", "3", "--warmup", "3"]) == 0
    assert capsys.readouterr().out.strip() == ""


def test_cgroup_cpu_limit(tmp_path):
    f = tmp_path / "cpu.max"
    f.write_text("800000 100000\n")
    assert bench.cgroup_cpu_limit(str(f)) == 8
    f.write_text("150000 100000\n")
    assert bench.cgroup_cpu_limit(str(f)) == 1
    f.write_text("max 100000\n")
    assert bench.cgroup_cpu_limit(str(f)) is None
    assert bench.cgroup_cpu_limit(str(tmp_path / "absent")) is None


def test_prefill_tensor_work_by_hand():
    """Issued tensor-core multiply-adds of a 2048-token Llama-3-8B-layer prompt
    (H 32, P N L 128, bf16): chunk states 2 H P T N = 2^31; chunk outputs, per
    chunk and head, G (128^3) + Yi in two parts (2 x 128^3) + Yc in two parts
    (2 x 128^3) = 5 x 2^21, over 16 chunks x 32 heads = 5 x 2^30."""
    macs, kind = bench.prefill_tensor_macs(32, 128, 128, 2048, 128, True)
    assert macs == 2 ** 31 + 5 * 2 ** 30 and kind.startswith("tcgen05")
    # 64-row output tiles (P 64): G once per tile, the row products at 64 rows
    macs64, _ = bench.prefill_tensor_macs(2, 64, 128, 256, 128, True)
    assert macs64 == 2 * 2 * 64 * 256 * 128 + 2 * 2 * (128 ** 3 + 2 * 128 * 128 * 64 + 2 * 128 * 128 * 64)
    assert bench.prefill_tensor_macs(1, 64, 256, 256, 128, False)[0] is None


def test_commit_verify_bytes_by_hand():
    """The deferred-commit call's algorithmic bytes on the serving shapes
    (H 32, P = N 128, G 8, K 8, bf16), two sequences with j_prev = 0 and 3:
    both states read (2 x 2 MiB), one written (j_prev > 0), the 3 accepted
    previous tokens' x (8192 B), B (one group row, 2048 B) and dt (64 B),
    both sequences' new x / B / C / dt, y in fp32 and accept_len."""
    wl = synth.WORKLOADS[3]
    state = 2 * (32 * 128 * 128 * 4)
    write = 1 * (32 * 128 * 128 * 4)
    replay = 3 * (8192 + 2048 + 64)
    new = 2 * 8 * (8192 + 2 * 2048 + 64)
    y = 2 * 8 * 32 * 128 * 4
    assert bench.algorithmic_bytes_commit_verify(wl, 2, [0, 3]) == state + write + replay + new + y + 2 * 4 == 6782152
    # with every previous token accepted the replay reads the whole previous block
    full = bench.algorithmic_bytes_commit_verify(wl, 2, [8, 8])
    assert full == state + state + 16 * (8192 + 2048 + 64) + new + y + 8  # both read, both written


def test_unfused_bytes_by_hand():
    """The unfused pair on the serving shapes, two sequences with j = 0 and 3:
    verify reads both states and both sequences' x / B / C / dt and writes y;
    commit reads and writes the one state with j > 0 and reads the 3 accepted
    tokens' x / B / dt and accept_len."""
    wl = synth.WORKLOADS[3]
    slice_b = 32 * 128 * 128 * 4
    verify = 2 * slice_b + 2 * 8 * (8192 + 2 * 2048 + 64) + 2 * 8 * 32 * 128 * 4
    commit = 2 * slice_b + 3 * (8192 + 2048 + 64) + 2 * 4
    assert bench.algorithmic_bytes_unfused(wl, 2, [0, 3]) == verify + commit == 8879304
    # against the fused call on the same inputs: one more state read and the accepted tokens' inputs again
    fused = bench.algorithmic_bytes(wl, 2, 1)
    assert verify + commit - fused == slice_b + 3 * (8192 + 2048 + 64)


def test_l2_note_says_when_a_workload_is_smaller_than_the_cache():
    wl = synth.WORKLOADS[3]
    big = bench.workload_config(wl, 3, 1, reread_bytes=2 * 268 * 10**6)
    assert "more than 2x the 126 MB L2" in big["l2"]
    small = bench.workload_config(synth.WORKLOADS[0], bench.NSETS_CAP, 1, reread_bytes=(bench.NSETS_CAP - 1) * 4096)
    assert "smaller than the cache" in small["l2"] and f"{bench.NSETS_CAP} independent" in small["l2"]


def test_tile_tensor_work_by_hand():
    """mma.sync work of one launch, K 16 (two 8-token chunks), N 128, bf16, one
    16-row band: y per chunk 16 x 2 + 16 x 1 + 3 = 51 mma, a state update 16 x 2
    = 32. j = 0: y, y and the advance through chunk 0 (134); j = 5: the
    committed state inside chunk 0 and the advance past it (166); j = 12 and
    j = 16: the advance through chunk 0 and the update up to j in chunk 1 (166)."""
    wl = synth.custom_workload(4, 1, 16, 128, 1, 16, synth.BF16, seed=3)
    assert bench.tile_tensor_macs(wl, [0, 5, 12, 16], 1) == (134 + 166 + 166 + 166) * 1024
    assert bench.tile_tensor_macs(wl, [0], 3) == 3 * 134 * 1024  # layers multiply
    f32 = synth.custom_workload(1, 1, 16, 128, 1, 8, synth.F32, seed=3)
    assert bench.tile_tensor_macs(f32, [8], 1) == (16 * 3 + 16 * 3 + 3 + 16 * 3) * 1024
