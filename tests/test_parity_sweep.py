"""Seeded random shapes against the fp64 oracle (GPU, through the C ABI).

Each case draws batch, heads, head dimension, dstate, groups, draft length,
input dtype, a layer-stack depth and whether the state lives in a pool with a
permuted slot map, and runs one fused verify+commit launch over every layer,
and one deferred-commit launch (commit the block's accepted prefix, verify a
new block of another length from the committed state).
The tile index of the kernels is decoded by divisions by the head count, the
row tiles per head, the sequences per layer and the heads per group, so odd
values of each (and ragged head dimensions) are what these cases exercise.
Pool slots no sequence maps to must come back bitwise untouched.
"""
import numpy as np
import pytest
import torch

import oracle
import ssm_recurrence_verify_b300 as ssm
from gpu_helpers import RTOL_STATE, np64, rel_err, y_tol
from ssm_recurrence_verify_b300 import synth

pytestmark = pytest.mark.gpu


def _cases(n=14, seed=20261203):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        N = int(rng.choice([16, 32, 64, 128, 256]))
        H = int(rng.integers(1, 8))
        G = int(rng.choice([g for g in range(1, H + 1) if H % g == 0]))
        P = int(rng.integers(1, 200))
        K = int(rng.integers(1, 25))
        batch = int(rng.integers(1, 7))
        layers = int(rng.integers(1, 4))
        dtype = synth.BF16 if rng.random() < 0.5 else synth.F32
        pool = bool(rng.random() < 0.5)
        out.append((batch, H, P, N, G, K, dtype, layers, pool))
    return out


@pytest.mark.parametrize("case", _cases(), ids=lambda c: "b{}h{}p{}n{}g{}k{}{}_l{}{}".format(
    *c[:7], c[7], "_pool" if c[8] else ""))
def test_random_shape_stack(cuda_device, case):
    batch, H, P, N, G, K, dtype, L, pool = case
    dev = cuda_device
    wl = synth.custom_workload(batch, H, P, N, G, K, dtype, seed=sum(case[:6]) + 17 * L)
    acc = synth.draw_accept_len(wl, 0)
    ps = [synth.draw_params(wl, layer) for layer in range(L)]
    ts = [synth.draw_tokens(wl, 0, layer) for layer in range(L)]
    stk = lambda src, k: torch.stack([d[k] for d in src]).to(dev)  # noqa: E731
    X, Bm, Cm, dt = stk(ts, "x"), stk(ts, "B"), stk(ts, "C"), stk(ts, "dt")
    A, D = stk(ps, "A"), stk(ps, "D")
    state0 = torch.stack([p["state0"] for p in ps])  # [L][batch][H][P][N]
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    if pool:
        nslots = batch + 3
        slot = torch.from_numpy(np.random.default_rng(batch * 31 + K).permutation(nslots)[:batch].astype(np.int32))
        states = torch.randn(L, nslots, H, P, N, generator=torch.Generator().manual_seed(5))  # unused slots: sentinels
        states[:, slot.long()] = state0
        before = states.clone()
        states = states.to(dev)
        y = ssm.verify_commit_pool(states, slot.to(dev), X, Bm, Cm, dt, A, D, acc.to(dev), dev_status=status)
        torch.cuda.synchronize()
        out = states.cpu()
        used = torch.zeros(nslots, dtype=torch.bool)
        used[slot.long()] = True
        assert torch.equal(out[:, ~used], before[:, ~used]), "a slot no sequence maps to was written"
        got_state = out[:, slot.long()]
    else:
        st = state0.to(dev)
        y = ssm.verify_commit(st, X, Bm, Cm, dt, A, D, acc.to(dev), dev_status=status)
        torch.cuda.synchronize()
        got_state = st.cpu()
    assert int(status.item()) == 0
    for layer in range(L):
        p, t = ps[layer], ts[layer]
        ref = oracle.verify_commit(p["state0"], t["x"], t["B"], t["C"], t["dt"], p["A"], p["D"], acc)
        ey = rel_err(np64(y[layer]), ref["y"])
        es = rel_err(np64(got_state[layer]), ref["state"])
        assert ey <= y_tol(wl.torch_in_dtype), f"layer {layer}: y rel err {ey:.3e}"
        assert es <= RTOL_STATE, f"layer {layer}: state rel err {es:.3e}"


@pytest.mark.parametrize("case", _cases(), ids=lambda c: "b{}h{}p{}n{}g{}k{}{}".format(*c[:7]) + "_l{}{}".format(
    c[7], "_pool" if c[8] else ""))
def test_random_shape_stack_commit_verify(cuda_device, case):
    """ssm_commit_verify: the state after the previous block's accepted prefix
    (oracle: the recurrence over the first j tokens) and y of the new block
    from that state (oracle: every new token from the committed state)."""
    batch, H, P, N, G, K, dtype, L, pool = case
    dev = cuda_device
    wl = synth.custom_workload(batch, H, P, N, G, K, dtype, seed=sum(case[:6]) + 17 * L + 5)
    kn = max(1, (K * 2) // 3)  # the new block's length differs from the previous one's
    wn = synth.custom_workload(batch, H, P, N, G, kn, dtype, seed=sum(case[:6]) + 17 * L + 6)
    acc = synth.draw_accept_len(wl, 0)
    ps = [synth.draw_params(wl, layer) for layer in range(L)]
    prev = [synth.draw_tokens(wl, 0, layer) for layer in range(L)]
    new = [synth.draw_tokens(wn, 1, layer) for layer in range(L)]
    stk = lambda src, k: torch.stack([d[k] for d in src]).to(dev)  # noqa: E731
    A, D = stk(ps, "A"), stk(ps, "D")
    args = (stk(prev, "x"), stk(prev, "B"), stk(prev, "dt"), acc.to(dev), stk(new, "x"), stk(new, "B"),
            stk(new, "C"), stk(new, "dt"), A, D)
    state0 = torch.stack([p["state0"] for p in ps])
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    if pool:
        nslots = batch + 2
        slot = torch.from_numpy(np.random.default_rng(batch * 7 + K).permutation(nslots)[:batch].astype(np.int32))
        states = torch.randn(L, nslots, H, P, N, generator=torch.Generator().manual_seed(9))
        states[:, slot.long()] = state0
        before = states.clone()
        states = states.to(dev)
        y = ssm.commit_verify_pool(states, slot.to(dev), *args, dev_status=status)
        torch.cuda.synchronize()
        out = states.cpu()
        used = torch.zeros(nslots, dtype=torch.bool)
        used[slot.long()] = True
        assert torch.equal(out[:, ~used], before[:, ~used]), "a slot no sequence maps to was written"
        got_state = out[:, slot.long()]
    else:
        st = state0.to(dev)
        y = ssm.commit_verify(st, *args, dev_status=status)
        torch.cuda.synchronize()
        got_state = st.cpu()
    assert int(status.item()) == 0
    for layer in range(L):
        p, t, n = ps[layer], prev[layer], new[layer]
        committed = oracle.verify_commit(p["state0"], t["x"], t["B"], t["C"], t["dt"], p["A"], p["D"], acc,
                                         want_y=False)["state"]
        ref_y = oracle.verify_commit(committed, n["x"], n["B"], n["C"], n["dt"], p["A"], p["D"])["y"]
        es = rel_err(np64(got_state[layer]), committed)
        ey = rel_err(np64(y[layer]), ref_y)
        assert es <= RTOL_STATE, f"layer {layer}: state rel err {es:.3e}"
        assert ey <= y_tol(wl.torch_in_dtype), f"layer {layer}: y rel err {ey:.3e}"
