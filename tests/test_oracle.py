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
