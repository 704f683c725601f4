"""The serving loop end to end on the device: prefill of each prompt into a
state pool, then rounds of (commit the previous round's accepted prefix +
verify the new drafts) whose accept_len comes straight from the acceptance
kernel of the previous round (it never visits the host), then a last commit.
Checked against the oracles: every round's y and the final states against the
fp64 recurrence run on the accept_len the device produced, and every
accept_len against the acceptance oracle."""
import numpy as np
import pytest
import torch

import oracle
import ssm_recurrence_verify_b300 as ssm
from gpu_helpers import RTOL_STATE, np64, rel_err, y_tol
from oracle import accept as acc_oracle
from ssm_recurrence_verify_b300 import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("rule", ["greedy", "sample"])
def test_prefill_then_speculative_rounds(cuda_device, rule):
    dev = cuda_device
    batch, H, P, N, G, K, T, V, rounds = 4, 4, 64, 64, 2, 4, 64, 500, 4
    prompt = synth.custom_workload(batch, H, P, N, G, T, synth.BF16, seed=701)
    draft = synth.custom_workload(batch, H, P, N, G, K, synth.BF16, seed=702)
    p = synth.draw_params(prompt)
    A, D = p["A"].to(dev), p["D"].to(dev)
    slot = torch.tensor([3, 0, 5, 1], dtype=torch.int32)
    pool = torch.zeros(6, H, P, N, device=dev)

    # prefill
    tp = synth.draw_tokens(prompt, 0)
    tpd = {k: v.to(dev) for k, v in tp.items()}
    y_prompt = ssm.prefill(pool, slot.to(dev), tpd["x"], tpd["B"], tpd["C"], tpd["dt"], A, D)

    # rounds: the acceptance of round r feeds the commit of round r + 1 on the device
    ys, accs, logits, blocks = [], [], [], []
    prev = None
    for r in range(rounds):
        t = synth.draw_tokens(draft, r)
        td = {k: v.to(dev) for k, v in t.items()}
        if prev is None:
            y = ssm.verify_pool(pool, slot.to(dev), td["x"], td["B"], td["C"], td["dt"], A, D)
        else:
            y = ssm.commit_verify_pool(pool, slot.to(dev), prev["x"], prev["B"], prev["dt"], prev["acc"], td["x"],
                                       td["B"], td["C"], td["dt"], A, D)
        lg = synth.draw_accept_inputs(synth.custom_accept_workload(batch, K, V, synth.F32, seed=800 + r))
        lgd = {k: v.to(dev) for k, v in lg.items()}
        if rule == "greedy":
            a_len, _ = ssm.accept_greedy(lgd["target_logits"], lgd["draft_tokens"])
        else:
            a_len, _ = ssm.accept_sample(lgd["target_logits"], lgd["draft_logits"], lgd["draft_tokens"],
                                         lgd["uniform"])
        ys.append(y)
        accs.append(a_len)
        logits.append(lg)
        blocks.append(t)
        prev = {"x": td["x"], "B": td["B"], "dt": td["dt"], "acc": a_len}
    ssm.commit_pool(pool, slot.to(dev), prev["x"], prev["B"], prev["dt"], A, prev["acc"])
    torch.cuda.synchronize()

    # the oracle chain, on the accept_len the device produced
    ref = oracle.verify_commit(np.zeros((batch, H, P, N)), tp["x"], tp["B"], tp["C"], tp["dt"], p["A"], p["D"], None)
    assert rel_err(np64(y_prompt), ref["y"]) <= y_tol(torch.bfloat16)
    state = ref["state"]
    for r in range(rounds):
        a_dev = accs[r].cpu()
        lg = logits[r]
        if rule == "greedy":
            want = acc_oracle.accept_greedy(lg["target_logits"], lg["draft_tokens"])["accept_len"]
            assert np.array_equal(a_dev.numpy(), want)
        else:
            w = acc_oracle.accept_sample(lg["target_logits"], lg["draft_logits"], lg["draft_tokens"], lg["uniform"])
            ok = ~w["near_accept"]
            assert np.array_equal(a_dev.numpy()[ok], w["accept_len"][ok])
        t = blocks[r]
        out = oracle.verify_commit(state, t["x"], t["B"], t["C"], t["dt"], p["A"], p["D"], a_dev)
        assert rel_err(np64(ys[r]), out["y"]) <= y_tol(torch.bfloat16), r
        state = out["state"]
    got = np64(pool[slot.long().to(dev)])
    assert rel_err(got, state) <= RTOL_STATE
    untouched = [i for i in range(6) if i not in slot.tolist()]
    assert (pool[untouched] == 0).all()
    assert len({int(a) for a_ in accs for a in a_.cpu()}) > 1  # the rounds accept different prefixes


def test_layer_stack_serving_loop(cuda_device):
    """The serving loop of a hybrid model with L Mamba layers: each layer's
    prompt prefilled into its pool states[l]; then every round one stacked
    commit_verify_pool call over all layers (accept_len from the device's
    greedy acceptance of the previous round, shared by the layers); a last
    stacked commit. Every layer against the oracle chain."""
    dev = cuda_device
    L, batch, H, P, N, G, K, T, V, rounds = 3, 3, 4, 64, 128, 2, 4, 40, 300, 3
    prompt = synth.custom_workload(batch, H, P, N, G, T, synth.BF16, seed=711)
    draft = synth.custom_workload(batch, H, P, N, G, K, synth.BF16, seed=712)
    ps = [synth.draw_params(prompt, l) for l in range(L)]
    A = torch.stack([p["A"] for p in ps]).to(dev)
    D = torch.stack([p["D"] for p in ps]).to(dev)
    slot = torch.tensor([2, 4, 0], dtype=torch.int32, device=dev)
    pool = torch.zeros(L, 5, H, P, N, device=dev)

    tps = [synth.draw_tokens(prompt, 0, l) for l in range(L)]
    for l in range(L):
        t = {k: v.to(dev) for k, v in tps[l].items()}
        ssm.prefill(pool[l], slot, t["x"], t["B"], t["C"], t["dt"], A[l], D[l])

    ys, accs, blocks, prev = [], [], [], None
    for r in range(rounds):
        ts = [synth.draw_tokens(draft, r, l) for l in range(L)]
        td = {k: torch.stack([t[k] for t in ts]).to(dev) for k in ("x", "B", "C", "dt")}
        if prev is None:
            y = ssm.verify_pool(pool, slot, td["x"], td["B"], td["C"], td["dt"], A, D)
        else:
            y = ssm.commit_verify_pool(pool, slot, prev["x"], prev["B"], prev["dt"], prev["acc"], td["x"], td["B"],
                                       td["C"], td["dt"], A, D)
        lg = synth.draw_accept_inputs(synth.custom_accept_workload(batch, K, V, synth.F32, seed=820 + r))
        a_len, _ = ssm.accept_greedy(lg["target_logits"].to(dev), lg["draft_tokens"].to(dev))
        ys.append(y)
        accs.append(a_len)
        blocks.append(ts)
        prev = {"x": td["x"], "B": td["B"], "dt": td["dt"], "acc": a_len}
    ssm.commit_pool(pool, slot, prev["x"], prev["B"], prev["dt"], A, prev["acc"])
    torch.cuda.synchronize()

    for l in range(L):
        tp = tps[l]
        ref = oracle.verify_commit(np.zeros((batch, H, P, N)), tp["x"], tp["B"], tp["C"], tp["dt"], ps[l]["A"],
                                   ps[l]["D"], None)
        state = ref["state"]
        for r in range(rounds):
            t = blocks[r][l]
            out = oracle.verify_commit(state, t["x"], t["B"], t["C"], t["dt"], ps[l]["A"], ps[l]["D"],
                                       accs[r].cpu())
            assert rel_err(np64(ys[r][l]), out["y"]) <= y_tol(torch.bfloat16), (l, r)
            state = out["state"]
        assert rel_err(np64(pool[l][slot.long()]), state) <= RTOL_STATE, l
    untouched = [i for i in range(5) if i not in slot.tolist()]
    assert (pool[:, untouched] == 0).all()
