"""Parity of the device acceptance step (greedy and speculative sampling)
with the acceptance oracle, through the C ABI.

Greedy results are integers decided by exact comparisons of the input logits:
they must match bit for bit. Sampling decisions come from fp32 sums whose
order differs between the two sides: accept_len must match wherever the
oracle reports no near-tie, and next_token must lie in the oracle's
admissible range (and equal its exact answer where that range is a single
index)."""
import numpy as np
import pytest
import torch

import ssm_recurrence_verify_b300 as ssm
from oracle import accept as acc
from ssm_recurrence_verify_b300 import synth

pytestmark = pytest.mark.gpu

F32, BF16 = synth.F32, synth.BF16

# (batch, K, V, logit dtype): 128-bit and scalar paths (V * element size a
# multiple of 16 or not), vocabularies smaller than the cluster's slices,
# the largest K, the Llama-3 vocabulary.
CASES = [
    (3, 4, 1000, F32),
    (5, 8, 1003, F32),
    (4, 8, 32000, BF16),
    (7, 5, 32003, BF16),
    (2, 1, 7, F32),
    (9, 3, 8, BF16),
    (2, 32, 4096, BF16),
    (3, 6, 128256, BF16),
]


def _greedy(d, dev):
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    a, n = ssm.accept_greedy(d["target_logits"].to(dev), d["draft_tokens"].to(dev), dev_status=st)
    torch.cuda.synchronize()
    return a.cpu().numpy(), n.cpu().numpy(), int(st.item())


def _sample(d, dev):
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    a, n = ssm.accept_sample(d["target_logits"].to(dev), d["draft_logits"].to(dev), d["draft_tokens"].to(dev),
                             d["uniform"].to(dev), dev_status=st)
    torch.cuda.synchronize()
    return a.cpu().numpy(), n.cpu().numpy(), int(st.item())


def check_greedy(d, dev):
    want = acc.accept_greedy(d["target_logits"], d["draft_tokens"])
    a, n, st = _greedy(d, dev)
    np.testing.assert_array_equal(a, want["accept_len"])
    np.testing.assert_array_equal(n, want["next_token"])
    assert bool(st & ssm.ssmverify.SSM_STATUS_BAD_TOKEN) == bool(want["bad"].any())
    return want


def check_sample(d, dev, max_near_frac=0.05):
    want = acc.accept_sample(d["target_logits"], d["draft_logits"], d["draft_tokens"], d["uniform"])
    a, n, st = _sample(d, dev)
    K, V = d["draft_tokens"].shape[1], d["target_logits"].shape[2]
    ok = ~want["near_accept"]
    assert ok.sum() >= len(ok) - max(1, int(max_near_frac * len(ok)))
    np.testing.assert_array_equal(a[ok], want["accept_len"][ok])
    lo, hi = want["next_lo"], want["next_hi"]
    inside = (n >= lo) & (n <= hi)
    assert inside[ok].all(), (n[ok][~inside[ok]], lo[ok][~inside[ok]], hi[ok][~inside[ok]])
    unique = ok & (lo == hi)
    np.testing.assert_array_equal(n[unique], want["next_token"][unique])
    assert ((a >= 0) & (a <= K) & (n >= 0) & (n < V)).all()
    assert bool(st & ssm.ssmverify.SSM_STATUS_BAD_TOKEN) == bool(want["bad"].any())
    return want, unique


@pytest.mark.parametrize("batch,K,V,dt", CASES)
def test_greedy_matches_oracle(cuda_device, batch, K, V, dt):
    d = synth.draw_accept_inputs(synth.custom_accept_workload(batch, K, V, dt, seed=10 + K))
    check_greedy(d, cuda_device)


@pytest.mark.parametrize("batch,K,V,dt", CASES)
def test_sample_matches_oracle(cuda_device, batch, K, V, dt):
    d = synth.draw_accept_inputs(synth.custom_accept_workload(batch, K, V, dt, seed=20 + K))
    check_sample(d, cuda_device)


@pytest.mark.parametrize("agree,spike", [(1.0, None), (0.0, None), (0.8, 0.0), (0.5, 3.0)])
def test_sample_acceptance_regimes(cuda_device, agree, spike):
    """High and low agreement, and flat distributions (no peak), whose
    residual mass spreads over the whole vocabulary."""
    d = synth.draw_accept_inputs(synth.custom_accept_workload(16, 8, 50000, BF16, seed=31, agree=agree, spike=spike))
    check_sample(d, cuda_device)
    check_greedy(d, cuda_device)


def test_full_workload_parity(cuda_device):
    """The batched serving workload at full size: 64 sequences, K 8, the
    Llama-3 vocabulary, bf16 logits."""
    aw = synth.ACCEPT_WORKLOADS[1]
    d = synth.draw_accept_inputs(aw)
    g = check_greedy(d, cuda_device)
    s, unique = check_sample(d, cuda_device)
    assert len(set(g["accept_len"].tolist())) > 3 and len(set(s["accept_len"].tolist())) > 3
    assert unique.sum() >= 16  # enough sequences whose next token is pinned exactly


def test_greedy_ties_go_to_the_smallest_index(cuda_device):
    """Equal maxima inside one CTA's slice, across slices, and a constant row."""
    V, K = 8000, 3  # bf16: eight slices of 1000 entries
    tl = torch.zeros(4, K + 1, V)
    tl[0, 0, [999, 1000]] = 5.0        # across the slice boundary
    tl[0, 1, [7999, 3000, 3001]] = 2.0  # across slices and inside one
    tl[1, 0, [17, 12]] = 1.0
    tl[1, 1, :] = 0.0                  # constant row: index 0
    tl[2] = -3.0
    tl[2, :, 5] = -1.0                 # all negative, a tie between 5 and 6000
    tl[2, :, 6000] = -1.0
    tl[3, :, [4096]] = 1e4
    drafts = torch.tensor([[999, 3000, 0], [12, 0, 0], [5, 5, 6000], [4096, 4096, 4096]], dtype=torch.int32)
    for dt in (torch.float32, torch.bfloat16):
        d = {"target_logits": tl.to(dt).contiguous(), "draft_tokens": drafts}
        want = check_greedy(d, cuda_device)
        assert want["accept_len"].tolist() == [3, 3, 2, 3] and want["next_token"].tolist()[2] == 5


def test_bad_draft_tokens(cuda_device):
    d = synth.draw_accept_inputs(synth.custom_accept_workload(4, 5, 3000, F32, seed=41, agree=1.0))
    d["draft_tokens"][0, 2] = -1
    d["draft_tokens"][1, 0] = 3000
    d["draft_tokens"][2, 4] = 1 << 30
    g = check_greedy(d, cuda_device)
    s, _ = check_sample(d, cuda_device)
    assert g["accept_len"][:3].tolist() == [2, 0, 4] and g["bad"][:3].all() and not g["bad"][3]
    assert s["accept_len"][1] == 0 and s["bad"][1]


def test_sample_equal_models_accept_everything(cuda_device):
    """q = p: every ratio is 1, every draft is accepted and the bonus token
    comes from p_K."""
    d = synth.draw_accept_inputs(synth.custom_accept_workload(8, 6, 20000, BF16, seed=51))
    d["draft_logits"] = d["target_logits"][:, :6].contiguous()
    d["uniform"] = torch.clamp(d["uniform"], max=0.999)
    s, _ = check_sample(d, cuda_device)
    assert (s["accept_len"] == 6).all()


@pytest.mark.parametrize("seed", [61, 62, 63])
def test_sample_sparse_residual_draw(cuda_device, seed):
    """The draw's rescan when the residual weight sits on a few isolated
    entries: the draft row equals the verifier row except 10 lower at the
    verifier's 8 most likely entries, which hold most of p. With each draft
    token at its row's least likely entry and u = 0.999 every draft is
    rejected, max(0, p - q) is positive only at those 8
    entries, scattered over the vocabulary, and the draw lands among them by
    u_K: the rescanning thread's run is mostly zero-weight segments around
    one crossing. The oracle pins the token exactly where no rounding near-tie
    leaves a choice."""
    d = synth.draw_accept_inputs(synth.custom_accept_workload(24, 2, 32000, BF16, seed=seed))
    tl = d["target_logits"]
    ql = tl[:, :2].clone().float()
    top = torch.topk(tl[:, :2].float(), 8, dim=-1).indices
    ql.scatter_(-1, top, ql.gather(-1, top) - 10.0)
    d["draft_logits"] = ql.to(tl.dtype).contiguous()
    # each draft token at its row's least likely entry: p/q there is 1 minus most of the top-8 mass
    d["draft_tokens"] = torch.argmin(tl[:, :2].float(), dim=-1).to(d["draft_tokens"].dtype).contiguous()
    u = torch.rand(d["uniform"].shape, generator=torch.Generator().manual_seed(seed))
    u[:, :2] = 0.999
    d["uniform"] = u.to(d["uniform"].dtype).contiguous()
    want, unique = check_sample(d, cuda_device)
    assert (want["accept_len"] == 0).all()
    assert unique.sum() >= 20


def test_deterministic_and_stream_ordered(cuda_device):
    d = synth.draw_accept_inputs(synth.custom_accept_workload(12, 8, 40000, BF16, seed=61))
    dev = cuda_device
    tl, ql = d["target_logits"].to(dev), d["draft_logits"].to(dev)
    dr, u = d["draft_tokens"].to(dev), d["uniform"].to(dev)
    s = torch.cuda.Stream()
    outs = []
    with torch.cuda.stream(s):
        for _ in range(3):
            outs.append(ssm.accept_sample(tl, ql, dr, u, stream=s))
            outs.append(ssm.accept_greedy(tl, dr, stream=s))
    s.synchronize()
    for k in range(2, 6):
        assert torch.equal(outs[k][0], outs[k % 2][0]) and torch.equal(outs[k][1], outs[k % 2][1])


def test_accept_feeds_commit_without_host_round_trip(cuda_device):
    """accept_len written by the acceptance kernel drives ssm_commit_verify
    directly: the committed state equals the oracle's for that accept_len."""
    import oracle
    dev = cuda_device
    wl = synth.custom_workload(4, 4, 32, 64, 2, 5, synth.BF16, seed=71)
    p = synth.draw_params(wl)
    t = synth.draw_tokens(wl, 0)
    d = synth.draw_accept_inputs(synth.custom_accept_workload(4, 5, 1000, F32, seed=72))
    state = p["state0"].to(dev)
    A, D = p["A"].to(dev), p["D"].to(dev)
    ssm.verify(state, t["x"].to(dev), t["B"].to(dev), t["C"].to(dev), t["dt"].to(dev), A, D)
    a, _ = ssm.accept_greedy(d["target_logits"].to(dev), d["draft_tokens"].to(dev))
    t2 = synth.draw_tokens(wl, 1)
    ssm.commit_verify(state, t["x"].to(dev), t["B"].to(dev), t["dt"].to(dev), a, t2["x"].to(dev), t2["B"].to(dev),
                      t2["C"].to(dev), t2["dt"].to(dev), A, D)
    torch.cuda.synchronize()
    want_acc = acc.accept_greedy(d["target_logits"], d["draft_tokens"])["accept_len"]
    ref = oracle.verify_commit(p["state0"].double().numpy(), t["x"], t["B"], t["C"], t["dt"], p["A"], p["D"],
                               torch.from_numpy(want_acc).to(torch.int32))
    got = state.double().cpu().numpy()
    want = ref["state"]
    rms = float(np.sqrt(np.mean(want * want)))
    assert float(np.max(np.abs(got - want) / np.maximum(np.abs(want), rms))) <= 1e-4
