"""GPU (through the C ABI) against the fp64 oracle, element by element.

Every workload (the five synthetic configurations at full size; the 64-layer
stack on four of its layers), plus ragged shapes, all dstate variants, chunk
boundaries of the draft length, G = 1 and G = H, and the degenerate cases.
"""
import numpy as np
import pytest
import torch

import oracle
import ssm_recurrence_verify_b300 as ssm
from gpu_helpers import RTOL_STATE, np64, rel_err, to_dev, y_tol
from ssm_recurrence_verify_b300 import synth

pytestmark = pytest.mark.gpu


def _oracle_round(state64, t, p, acc):
    return oracle.verify_commit(state64, t["x"], t["B"], t["C"], t["dt"], p["A"], p["D"], acc)


def _check(y_gpu, st_gpu, ref, in_dtype, what):
    ey = rel_err(np64(y_gpu), ref["y"])
    es = rel_err(np64(st_gpu), ref["state"])
    assert ey <= y_tol(in_dtype), f"{what}: y rel err {ey:.3e}"
    assert es <= RTOL_STATE, f"{what}: state rel err {es:.3e}"


def run_workload(wl, dev, layers=None, rounds=None):
    """verify_commit over rounds x layers with the state carried across rounds;
    each layer-call checked against the oracle fed the same inputs."""
    layers = range(wl.nlayers) if layers is None else layers
    rounds = wl.rounds if rounds is None else rounds
    for layer in layers:
        p = synth.draw_params(wl, layer)
        st = p["state0"].to(dev)
        s64 = p["state0"].double().numpy()
        Ad, Dd = p["A"].to(dev), p["D"].to(dev)
        for rnd in range(rounds):
            t = synth.draw_tokens(wl, rnd, layer)
            acc = synth.draw_accept_len(wl, rnd)
            td = to_dev(t, dev)
            status = torch.zeros(1, dtype=torch.int32, device=dev)
            if wl.accept == "all" and wl.ntok == 1:
                y = ssm.step(st, td["x"], td["B"], td["C"], td["dt"], Ad, Dd)
                ref = oracle.verify_commit(s64, t["x"], t["B"], t["C"], t["dt"], p["A"], p["D"], None)
            else:
                y = ssm.verify_commit(st, td["x"], td["B"], td["C"], td["dt"], Ad, Dd, acc.to(dev),
                                      dev_status=status)
                ref = _oracle_round(s64, t, p, acc)
            torch.cuda.synchronize()
            assert int(status.item()) == 0
            _check(y, st, ref, wl.torch_in_dtype, f"{wl.name} layer {layer} round {rnd}")
            s64 = ref["state"]  # each side carries its own state; the oracle keeps fp64


def test_tiny_fp32_workload(cuda_device):
    run_workload(synth.WORKLOADS[0], cuda_device)


def test_tiny_fp32_workload_groups_equal_heads(cuda_device):
    wl = synth.custom_workload(1, 2, 16, 16, 2, 4, synth.F32, seed=100)
    run_workload(wl, cuda_device, rounds=3)


def test_llama3_layer_decode(cuda_device):
    run_workload(synth.WORKLOADS[1], cuda_device, rounds=4)


def test_hybrid_16_layer_verify(cuda_device):
    run_workload(synth.WORKLOADS[2], cuda_device)


def test_batched_speculative_serving(cuda_device):
    """The benchmark's workload at full size (batch 64, K 8), every output."""
    run_workload(synth.WORKLOADS[3], cuda_device)


def test_mamba2_stack_sampled_layers(cuda_device):
    """The 64-layer stack at full per-layer size, on layers 0, 21, 42, 63."""
    run_workload(synth.WORKLOADS[4], cuda_device, layers=[0, 21, 42, 63])


def test_mamba2_full_stack_one_launch(cuda_device):
    """The 64-layer stack as the benchmark launches it: one verify_commit over
    all 64 layers (2.7 GB of state), every output of layers 0, 21, 42 and 63
    against the oracle, and the other layers bit for bit against their own
    single-layer launches on sampled layers 7 and 50."""
    dev = cuda_device
    wl = synth.WORKLOADS[4]
    L = wl.nlayers
    ds = [synth.draw_layer_round(wl, rnd=0, layer=l) for l in range(L)]
    acc = ds[0]["accept_len"]
    S = {k: torch.stack([d[k] for d in ds]).to(dev) for k in ("state0", "x", "B", "C", "dt", "A", "D")}
    st = S["state0"].clone()
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    y = ssm.verify_commit(st, S["x"], S["B"], S["C"], S["dt"], S["A"], S["D"], acc.to(dev), dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for l in (0, 21, 42, 63):
        d = ds[l]
        ref = oracle.verify_commit(d["state0"], d["x"], d["B"], d["C"], d["dt"], d["A"], d["D"], acc)
        _check(y[l], st[l], ref, wl.torch_in_dtype, f"{wl.name} stacked launch, layer {l}")
    for l in (7, 50):
        s1 = S["state0"][l].clone()
        y1 = ssm.verify_commit(s1, S["x"][l], S["B"][l], S["C"][l], S["dt"][l], S["A"][l], S["D"][l], acc.to(dev))
        torch.cuda.synchronize()
        assert torch.equal(s1, st[l]) and torch.equal(y1, y[l]), l


SHAPES = [
    # batch, H, P, N, G, K, dtype
    (1, 2, 16, 16, 1, 4, synth.F32),
    (2, 4, 50, 16, 4, 7, synth.BF16),       # ragged P, G = H
    (3, 2, 33, 32, 1, 16, synth.F32),       # K exactly one chunk
    (2, 3, 64, 32, 3, 17, synth.BF16),      # K crosses the chunk boundary
    (2, 4, 100, 64, 2, 33, synth.F32),      # three chunks, ragged P
    (1, 8, 128, 128, 8, 1, synth.BF16),
    (5, 4, 129, 128, 1, 9, synth.BF16),     # one row past a tile
    (2, 2, 7, 256, 1, 5, synth.F32),        # tiny P, widest N
    (2, 2, 72, 256, 2, 12, synth.BF16),
    (1, 1, 1, 128, 1, 3, synth.F32),        # a single row
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "b{}h{}p{}n{}g{}k{}{}".format(*s))
def test_shapes(cuda_device, shape):
    wl = synth.custom_workload(*shape, seed=sum(shape[:6]))
    run_workload(wl, cuda_device, rounds=2)


def test_large_headdim(cuda_device):
    """A long ragged head dimension (many row tiles)."""
    wl = synth.custom_workload(1, 1, 4100, 256, 1, 3, synth.BF16, seed=77)
    run_workload(wl, cuda_device, rounds=1)


def test_verify_and_commit_unfused_match_oracle(cuda_device):
    """The serving order: verify (state read only) then commit."""
    wl = synth.custom_workload(4, 8, 128, 128, 2, 8, synth.BF16, seed=3)
    d = synth.draw_layer_round(wl)
    dd = to_dev(d, cuda_device)
    before = dd["state0"].clone()
    y = ssm.verify(dd["state0"], dd["x"], dd["B"], dd["C"], dd["dt"], dd["A"], dd["D"])
    torch.cuda.synchronize()
    assert torch.equal(before, dd["state0"])
    ssm.commit(dd["state0"], dd["x"], dd["B"], dd["dt"], dd["A"], dd["accept_len"])
    ref = oracle.verify_commit(d["state0"], d["x"], d["B"], d["C"], d["dt"], d["A"], d["D"], d["accept_len"])
    _check(y, dd["state0"], ref, torch.bfloat16, "unfused")


def test_zero_and_full_acceptance(cuda_device):
    wl = synth.custom_workload(6, 4, 64, 128, 2, 6, synth.F32, seed=9)
    d = synth.draw_layer_round(wl)
    d["accept_len"] = torch.tensor([0, 6, 0, 6, 3, 1], dtype=torch.int32)
    dd = to_dev(d, cuda_device)
    y = ssm.verify_commit(dd["state0"], dd["x"], dd["B"], dd["C"], dd["dt"], dd["A"], dd["D"], dd["accept_len"])
    ref = oracle.verify_commit(d["state0"], d["x"], d["B"], d["C"], d["dt"], d["A"], d["D"], d["accept_len"])
    _check(y, dd["state0"], ref, torch.float32, "zero/full acceptance")
    got = dd["state0"].cpu()
    for b in (0, 2):
        assert torch.equal(got[b], d["state0"][b])


def test_empty_batch_noop(cuda_device):
    e = torch.empty(0, 2, 16, 16, device=cuda_device)
    x = torch.empty(0, 3, 2, 16, device=cuda_device)
    B = torch.empty(0, 3, 1, 16, device=cuda_device)
    dt = torch.empty(0, 3, 2, device=cuda_device)
    A = torch.zeros(2, device=cuda_device)
    acc = torch.empty(0, dtype=torch.int32, device=cuda_device)
    y = ssm.verify_commit(e, x, B, B.clone(), dt, A, A.clone(), acc)
    torch.cuda.synchronize()
    assert y.shape == (0, 3, 2, 16)


def test_sampled_slices_at_full_size(cuda_device):
    """Property at full size, slice by slice: the benchmark's batch, with the
    oracle run one (sequence, head) at a time on a spread of slices."""
    wl = synth.WORKLOADS[3]
    d = synth.draw_layer_round(wl, rnd=5)
    dd = to_dev(d, cuda_device)
    y = ssm.verify_commit(dd["state0"], dd["x"], dd["B"], dd["C"], dd["dt"], dd["A"], dd["D"], dd["accept_len"])
    torch.cuda.synchronize()
    rng = np.random.default_rng(0)
    pairs = [(int(rng.integers(0, wl.batch)), int(rng.integers(0, wl.nheads))) for _ in range(24)]
    ref = oracle.verify_commit_slices(d, pairs)
    yc, sc = y.cpu(), dd["state0"].cpu()
    for (b, h), r in ref.items():
        assert rel_err(np64(yc[b, :, h]), r["y"]) <= y_tol(torch.bfloat16), (b, h)
        assert rel_err(np64(sc[b, h]), r["state"]) <= RTOL_STATE, (b, h)


def _serving_rounds(dev, wl_of_round, rounds, bad_round=None):
    """The serving order with the commit deferred by one round: round 0 only
    verifies; every later round commit_verify()s the previous round's accepted
    prefix and verifies the new drafts. The oracle commits the previous block
    (fp64), then computes the new drafts' y from that state."""
    wl0 = wl_of_round(0)
    p = synth.draw_params(wl0)
    st = p["state0"].to(dev)
    s64 = p["state0"].double().numpy()
    Ad, Dd = p["A"].to(dev), p["D"].to(dev)
    prev = None
    for rnd in range(rounds):
        wl = wl_of_round(rnd)
        t = synth.draw_tokens(wl, rnd)
        acc = synth.draw_accept_len(wl, rnd)
        td = to_dev(t, dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        if prev is None:
            y = ssm.verify(st, td["x"], td["B"], td["C"], td["dt"], Ad, Dd, dev_status=status)
        else:
            pt, pacc = prev
            if rnd == bad_round:
                pacc = pacc.clone()
                pacc[0] = -3
            ptd = to_dev(pt, dev)
            y = ssm.commit_verify(st, ptd["x"], ptd["B"], ptd["dt"], pacc.to(dev), td["x"], td["B"], td["C"],
                                  td["dt"], Ad, Dd, dev_status=status)
            s64 = oracle.verify_commit(s64, pt["x"], pt["B"], pt["C"], pt["dt"], p["A"], p["D"], pacc)["state"]
        ref = oracle.verify_commit(s64, t["x"], t["B"], t["C"], t["dt"], p["A"], p["D"],
                                   torch.zeros(wl.batch, dtype=torch.int32))
        torch.cuda.synchronize()
        want_status = ssm.ssmverify.SSM_STATUS_BAD_ACCEPT_LEN if rnd == bad_round else 0
        assert int(status.item()) == want_status, rnd
        ey = rel_err(np64(y), ref["y"])
        es = rel_err(np64(st), s64)
        assert ey <= y_tol(wl.torch_in_dtype), f"round {rnd}: y rel err {ey:.3e}"
        assert es <= RTOL_STATE, f"round {rnd}: state rel err {es:.3e}"
        prev = (t, acc)


def test_commit_verify_serving_order(cuda_device):
    """Five rounds of the deferred-commit serving order on the Llama-3-8B layer
    shape (batch 4, K 8)."""
    wl = synth.custom_workload(4, 32, 128, 128, 8, 8, synth.BF16, seed=31)
    _serving_rounds(cuda_device, lambda r: wl, 5)


def test_commit_verify_varying_draft_length(cuda_device):
    """Draft lengths that change between rounds, across the staging chunk
    (12 > 8 tokens), ragged P, fp32 inputs, and a bad accept_len in round 2
    (that sequence replays nothing; status bit set; y still produced)."""
    ks = [12, 3, 9, 1]

    def wl_of(r):
        return synth.custom_workload(3, 4, 50, 64, 2, ks[r], synth.F32, seed=32)
    _serving_rounds(cuda_device, wl_of, len(ks), bad_round=2)


@pytest.mark.parametrize("K", [1, 8])
@pytest.mark.parametrize("dtype", [synth.F32, synth.BF16])
def test_long_decode_slow_decay(cuda_device, K, dtype):
    """2048 tokens through one cached state with decays near 1 (A from -0.1
    down to 0, where the state is a plain running sum), as token-by-token
    steps (K = 1) or as rounds of 8 fully accepted drafts, against the fp64
    oracle over the whole sequence: the rounding of the state update must not
    drift past the state tolerance over a long decode."""
    dev = cuda_device
    T = 2048
    wl = synth.custom_workload(2, 4, 64, 128, 2, T, dtype, seed=77)
    d = synth.draw_layer_round(wl)
    d["A"] = torch.tensor([-0.1, -1e-2, -1e-3, 0.0], dtype=torch.float32)
    ref = oracle.verify_commit(d["state0"], d["x"], d["B"], d["C"], d["dt"], d["A"], d["D"], None)
    dd = to_dev(d, dev)
    st = dd["state0"].clone()
    full = torch.full((2,), K, dtype=torch.int32, device=dev)
    ys = []
    for t0 in range(0, T, K):
        blk = [dd[k][:, t0:t0 + K].contiguous() for k in ("x", "B", "C", "dt")]
        if K == 1:
            ys.append(ssm.step(st, *blk, dd["A"], dd["D"]))
        else:
            ys.append(ssm.verify_commit(st, *blk, dd["A"], dd["D"], full))
    y = torch.cat(ys, dim=1)
    torch.cuda.synchronize()
    _check(y, st, ref, wl.torch_in_dtype, f"long decode K={K}")


def _stack(ds, keys):
    return {k: torch.stack([d[k] for d in ds]) for k in keys}


@pytest.mark.parametrize("K,dtype,P,N", [(8, synth.BF16, 64, 128), (12, synth.F32, 64, 128), (6, synth.F32, 40, 256)])
def test_layer_stack_equals_per_layer_calls(cuda_device, K, dtype, P, N):
    """nlayers = L: one call over [L]-leading slabs (A, D [L][H]; accept_len
    [batch] shared) gives, bit for bit, the L single-layer calls on the
    slices, in every entry point (also N = 256, two warps per band, with a
    ragged last tile)."""
    dev = cuda_device
    L, batch = 3, 5
    wl = synth.custom_workload(batch, 4, P, N, 2, K, dtype, seed=880 + K)
    ds = [synth.draw_layer_round(wl, rnd=0, layer=l) for l in range(L)]
    acc = ds[0]["accept_len"].to(dev)
    S = {k: v.to(dev) for k, v in _stack(ds, ("state0", "x", "B", "C", "dt", "A", "D")).items()}
    nxt = [synth.draw_tokens(wl, 1, l) for l in range(L)]
    N2 = {k: v.to(dev) for k, v in _stack(nxt, ("x", "B", "C", "dt")).items()}

    # verify
    y = ssm.verify(S["state0"], S["x"], S["B"], S["C"], S["dt"], S["A"], S["D"])
    for l in range(L):
        yl = ssm.verify(S["state0"][l], S["x"][l], S["B"][l], S["C"][l], S["dt"][l], S["A"][l], S["D"][l])
        assert torch.equal(y[l], yl), ("verify", l)
    # verify_commit, commit, step, commit_verify: state in place
    for fn in ("verify_commit", "commit", "step", "commit_verify"):
        st = S["state0"].clone()
        per = S["state0"].clone()
        if fn == "verify_commit":
            y = ssm.verify_commit(st, S["x"], S["B"], S["C"], S["dt"], S["A"], S["D"], acc)
            ys = [ssm.verify_commit(per[l], S["x"][l], S["B"][l], S["C"][l], S["dt"][l], S["A"][l], S["D"][l], acc)
                  for l in range(L)]
        elif fn == "commit":
            ssm.commit(st, S["x"], S["B"], S["dt"], S["A"], acc)
            for l in range(L):
                ssm.commit(per[l], S["x"][l], S["B"][l], S["dt"][l], S["A"][l], acc)
            y, ys = None, None
        elif fn == "step":
            one = {k: S[k][:, :, :1].contiguous() for k in ("x", "B", "C", "dt")}
            y = ssm.step(st, one["x"], one["B"], one["C"], one["dt"], S["A"], S["D"])
            ys = [ssm.step(per[l], one["x"][l], one["B"][l], one["C"][l], one["dt"][l], S["A"][l], S["D"][l])
                  for l in range(L)]
        else:
            y = ssm.commit_verify(st, S["x"], S["B"], S["dt"], acc, N2["x"], N2["B"], N2["C"], N2["dt"], S["A"],
                                  S["D"])
            ys = [ssm.commit_verify(per[l], S["x"][l], S["B"][l], S["dt"][l], acc, N2["x"][l], N2["B"][l],
                                    N2["C"][l], N2["dt"][l], S["A"][l], S["D"][l]) for l in range(L)]
        torch.cuda.synchronize()
        assert torch.equal(st, per), fn
        if y is not None:
            for l in range(L):
                assert torch.equal(y[l], ys[l]), (fn, l)
    # against the oracle, layer by layer
    st = S["state0"].clone()
    y = ssm.verify_commit(st, S["x"], S["B"], S["C"], S["dt"], S["A"], S["D"], acc)
    torch.cuda.synchronize()
    for l in range(L):
        d = ds[l]
        ref = oracle.verify_commit(d["state0"], d["x"], d["B"], d["C"], d["dt"], d["A"], d["D"], d["accept_len"])
        _check(y[l], st[l], ref, wl.torch_in_dtype, f"stack layer {l}")


def test_hybrid_16_layer_stack_rounds(cuda_device):
    """The 16-layer hybrid workload as one stacked verify_commit per round
    (every layer shares the round's accept_len), state carried across
    rounds, each layer against the oracle."""
    dev = cuda_device
    wl = synth.WORKLOADS[2]
    L = wl.nlayers
    ps = [synth.draw_params(wl, l) for l in range(L)]
    P_ = {k: torch.stack([p[k] for p in ps]).to(dev) for k in ("state0", "A", "D")}
    st = P_["state0"].clone()
    s64 = [p["state0"].double().numpy() for p in ps]
    for rnd in range(wl.rounds):
        ts = [synth.draw_tokens(wl, rnd, l) for l in range(L)]
        T_ = {k: torch.stack([t[k] for t in ts]).to(dev) for k in ("x", "B", "C", "dt")}
        acc = synth.draw_accept_len(wl, rnd)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        y = ssm.verify_commit(st, T_["x"], T_["B"], T_["C"], T_["dt"], P_["A"], P_["D"], acc.to(dev),
                              dev_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        for l in range(L):
            ref = _oracle_round(s64[l], ts[l], ps[l], acc)
            _check(y[l], st[l], ref, wl.torch_in_dtype, f"{wl.name} layer {l} round {rnd}")
            s64[l] = ref["state"]
