"""The seeded input generator: independent streams per tensor, sequence
slicing that does not change a sequence's values, and the acceptance-step
recipe's structure."""
import torch

from ssm_recurrence_verify_b300 import synth


def test_streams_of_different_tensors_are_independent():
    wl = synth.WORKLOADS[3]
    t = synth.draw_tokens(wl, 0, 0, batch=2)
    # B and C have the same shape; drawn from one stream they would coincide
    assert (t["B"] != t["C"]).float().mean() > 0.99
    other = synth.custom_workload(2, 32, 128, 128, 8, 8, synth.BF16, seed=wl.seed + (1 << 32))
    t2 = synth.draw_tokens(other, 0, 0)
    assert (t["x"] != t2["x"]).float().mean() > 0.99  # seeds differing above bit 32 differ
    a, b = synth.draw_tokens(wl, 1, 0, batch=1), synth.draw_tokens(wl, 0, 1, batch=1)
    assert not torch.equal(a["x"], b["x"]) and not torch.equal(a["x"], t["x"][:1])


def test_sequence_slices_are_stable():
    wl = synth.custom_workload(5, 4, 16, 16, 2, 3, synth.BF16, seed=8)
    full = synth.draw_layer_round(wl, rnd=1)
    part = synth.draw_layer_round(wl, rnd=1, batch=2, batch_offset=3)
    for k in ("x", "B", "C", "dt", "state0", "accept_len"):
        assert torch.equal(full[k][3:5], part[k]), k
    aw = synth.custom_accept_workload(5, 3, 300, synth.BF16)
    fa, pa = synth.draw_accept_inputs(aw), synth.draw_accept_inputs(aw, batch=2, batch_offset=3)
    for k in fa:
        assert torch.equal(fa[k][3:5], pa[k]), k


def test_accept_recipe_structure():
    aw = synth.custom_accept_workload(6, 4, 500, synth.F32, agree=1.0)
    d = synth.draw_accept_inputs(aw)
    K, V = 4, 500
    assert d["target_logits"].shape == (6, K + 1, V) and d["draft_logits"].shape == (6, K, V)
    assert d["draft_tokens"].dtype == torch.int32 and d["uniform"].dtype == torch.float32
    assert int(d["draft_tokens"].min()) >= 0 and int(d["draft_tokens"].max()) < V
    # the draft proposes its own peak; with agree = 1 the verifier peaks there too
    assert torch.equal(d["draft_logits"].argmax(-1).int(), d["draft_tokens"])
    assert torch.equal(d["target_logits"][:, :K].argmax(-1).int(), d["draft_tokens"])
    u = d["uniform"]
    assert float(u.min()) >= 0.0 and float(u.max()) < 1.0
    bf = synth.draw_accept_inputs(synth.custom_accept_workload(2, 4, 500, synth.BF16))
    assert bf["target_logits"].dtype == torch.bfloat16
