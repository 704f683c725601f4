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


def test_draw_recipe_distributions():
    """The stated input recipe: state0 ~ N(0, 0.1) (std 0.1), x, B, C ~ N(0, 1/N),
    dt = softplus(N(-2, 1)) > 0, A = -exp(U(0, ln 16)) in [-16, -1], and
    accept_len = tokens accepted before the first rejection with rejection
    probability 0.3, capped at K (P(0) = 0.3, E = sum_{k=1..K} 0.7^k)."""
    wl = synth.custom_workload(4000, 8, 4, 64, 1, 16, synth.F32, seed=77, accept="geometric")
    acc = synth.draw_accept_len(wl).double()
    assert abs(float((acc == 0).double().mean()) - 0.3) < 0.025
    want_mean = sum(0.7 ** k for k in range(1, 17))
    assert abs(float(acc.mean()) - want_mean) < 0.15  # about 3.4 standard errors at 4000 draws
    assert int(acc.max()) == 16 and int(acc.min()) == 0
    small = synth.custom_workload(64, 8, 4, 64, 1, 16, synth.F32, seed=77)
    p = synth.draw_params(small)
    assert abs(float(p["state0"].std()) - 0.1) < 0.005
    assert float(p["A"].max()) <= -1.0 and float(p["A"].min()) >= -16.0
    t = synth.draw_tokens(small)
    for k in ("x", "B", "C"):
        assert abs(float(t[k].std()) - 1 / 8) < 0.01, k  # 1 / sqrt(N), N = 64
    assert float(t["dt"].min()) > 0.0
    raw = torch.log(torch.expm1(t["dt"].double()))  # the pre-softplus normal
    assert abs(float(raw.mean()) + 2.0) < 0.1 and abs(float(raw.std()) - 1.0) < 0.1
    u = synth.draw_accept_len(synth.custom_workload(4000, 1, 1, 1, 1, 8, seed=3))
    assert int(u.min()) == 0 and int(u.max()) == 8 and abs(float(u.double().mean()) - 4.0) < 0.2
