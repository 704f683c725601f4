"""Writes tiny_fp32_oracle.json: the oracle's y and committed state for the
tiny fp32 workload (batch 1, H 2, P 16, N 16, K 4, three rounds with the state
carried over). Calls only the oracle and the seeded input generator.

    python tests/golden/make_golden.py
"""
import os
import sys

import json

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from ssm_recurrence_verify_b300 import synth  # noqa: E402


def main():
    wl = synth.WORKLOADS[0]
    p = synth.draw_params(wl)
    s = p["state0"]
    out = {}
    for rnd in range(wl.rounds):
        t = synth.draw_tokens(wl, rnd)
        acc = synth.draw_accept_len(wl, rnd)
        r = oracle.verify_commit(s, t["x"], t["B"], t["C"], t["dt"], p["A"], p["D"], acc)
        out[f"accept_len_{rnd}"] = acc.tolist()
        out[f"y_{rnd}"] = r["y"].tolist()
        out[f"state_{rnd}"] = r["state"].tolist()
        s = r["state"]
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_fp32_oracle.json")
    with open(path, "w") as f:
        json.dump({"workload": wl.name, "generator": "ssm_recurrence_verify_b300.synth", **out}, f)
        f.write("\n")


if __name__ == "__main__":
    main()
