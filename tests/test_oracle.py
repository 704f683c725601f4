"""The fp64 oracle against its pins (CPU only)."""
import json
import os

import numpy as np
import pytest

import oracle
from oracle_pins import ALL_PINS, rel_err
from ssm_recurrence_verify_b300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(oracle.verify_commit)


def test_tiny_workload_matches_quadratic_form():
    """The tiny fp32 workload (3 rounds, state carried across rounds) through
    the recurrence and through the independent quadratic form."""
    wl = synth.WORKLOADS[0]
    p = synth.draw_params(wl)
    s_rec = p["state0"].double().numpy()
    s_quad = s_rec.copy()
    for rnd in range(wl.rounds):
        t = synth.draw_tokens(wl, rnd)
        acc = synth.draw_accept_len(wl, rnd)
        r = oracle.verify_commit(s_rec, t["x"], t["B"], t["C"], t["dt"], p["A"], p["D"], acc)
        q = oracle.ssd_quadratic(s_quad, t["x"], t["B"], t["C"], t["dt"], p["A"], p["D"], acc)
        assert rel_err(r["y"], q["y"]) < 1e-12
        assert rel_err(r["state"], q["state"]) < 1e-12
        s_rec, s_quad = r["state"], q["state"]


def test_golden_tiny_workload():
    """Regression fixture written by tests/golden/make_golden.py (which calls
    only the oracle): the tiny workload's y and committed state per round."""
    with open(os.path.join(GOLDEN, "tiny_fp32_oracle.json")) as f:
        g = {k: np.asarray(v) for k, v in json.load(f).items() if k not in ("workload", "generator")}
    wl = synth.WORKLOADS[0]
    p = synth.draw_params(wl)
    s = p["state0"]
    for rnd in range(wl.rounds):
        t = synth.draw_tokens(wl, rnd)
        acc = synth.draw_accept_len(wl, rnd)
        r = oracle.verify_commit(s, t["x"], t["B"], t["C"], t["dt"], p["A"], p["D"], acc)
        assert np.array_equal(acc.numpy(), g[f"accept_len_{rnd}"])
        assert rel_err(r["y"], g[f"y_{rnd}"]) < 1e-15
        assert rel_err(r["state"], g[f"state_{rnd}"]) < 1e-15
        s = r["state"]


def test_slices_match_full_batch():
    wl = synth.custom_workload(3, 4, 8, 16, 2, 5, synth.BF16, seed=5)
    d = synth.draw_layer_round(wl)
    full = oracle.verify_commit(d["state0"], d["x"], d["B"], d["C"], d["dt"], d["A"], d["D"], d["accept_len"])
    pairs = [(0, 0), (1, 3), (2, 2)]
    sl = oracle.verify_commit_slices(d, pairs)
    for b, h in pairs:
        assert np.array_equal(sl[(b, h)]["y"], full["y"][b, :, h])
        assert np.array_equal(sl[(b, h)]["state"], full["state"][b, h])


@pytest.mark.parametrize("L", [16, 12, 48])
def test_chunked_regrouping_equals_recurrence(L):
    """The regrouping the chunked prefill rests on, with the oracle alone:
    every chunk's state from h = 0 (S_c), the chunk decays lambda_c (product
    of the chunk's Abar = exp(dt A)), the carry H_c = lambda_c H_{c-1} + S_c
    from the cached state, and each chunk's y from the state it starts from,
    reproduce the token-by-token recurrence over the whole prompt."""
    wl = synth.custom_workload(2, 3, 4, 8, 1, 48, synth.F32, seed=31)
    d = synth.draw_layer_round(wl)
    x, B, C, dt = (d[k].double().numpy() for k in ("x", "B", "C", "dt"))
    A, D = d["A"].double().numpy(), d["D"].double().numpy()
    h0 = d["state0"].double().numpy()
    whole = oracle.verify_commit(h0, x, B, C, dt, A, D, None)
    H = h0.copy()
    ys = []
    for c0 in range(0, 48, L):
        sl = slice(c0, c0 + L)
        S = oracle.verify_commit(np.zeros_like(h0), x[:, sl], B[:, sl], C[:, sl], dt[:, sl], A, D, None)["state"]
        lam = np.prod(np.exp(dt[:, sl] * A[None, None, :]), axis=1)  # [batch][H]
        ys.append(oracle.verify_commit(H, x[:, sl], B[:, sl], C[:, sl], dt[:, sl], A, D, None)["y"])
        H = lam[:, :, None, None] * H + S
    assert rel_err(np.concatenate(ys, axis=1), whole["y"]) < 1e-12
    assert rel_err(H, whole["state"]) < 1e-12
    # a dropped decay (lambda = 1) is caught
    assert rel_err(sum(oracle.verify_commit(np.zeros_like(h0), x[:, c:c + L], B[:, c:c + L], C[:, c:c + L],
                                            dt[:, c:c + L], A, D, None)["state"] for c in range(0, 48, L)) + h0,
                   whole["state"]) > 1e-3
