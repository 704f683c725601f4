"""Pins for the acceptance oracle (CPU): hand-derived cases, the exact special
cases of the rules, and the property that makes speculative sampling correct
-- the emitted token is distributed exactly as the verifier's distribution --
checked by Monte Carlo. Copies of the sampling rule with a planted mistake
must each fail at least one pin."""
import numpy as np
import pytest

from oracle import accept as acc


def _logits_from_probs(p):
    return np.log(np.asarray(p, dtype=np.float64)).astype(np.float32)


# --------------------------------------------------------------------------- greedy

def test_greedy_hand_cases():
    V = 5
    tl = np.zeros((4, 4, V), dtype=np.float32)  # [b][K+1][V], K = 3
    best = [[2, 0, 4, 1],   # drafts 2, 0, 4 all match: j = 3, bonus token 1
            [2, 3, 4, 1],   # drafts 2, 0, 4: mismatch at t = 1: j = 1, correction 3
            [1, 0, 4, 1],   # mismatch at t = 0: j = 0, correction 1
            [2, 0, 4, 1]]   # draft token out of range at t = 1: j = 1, correction = best at 1 (0)
    for b in range(4):
        for t in range(4):
            tl[b, t, best[b][t]] = 1.0
    drafts = np.array([[2, 0, 4], [2, 0, 4], [2, 0, 4], [2, 7, 4]])
    r = acc.accept_greedy(tl, drafts)
    assert r["accept_len"].tolist() == [3, 1, 0, 1]
    assert r["next_token"].tolist() == [1, 3, 1, 0]
    assert r["bad"].tolist() == [False, False, False, True]


def test_greedy_ties_go_to_the_smallest_index():
    tl = np.zeros((1, 2, 6), dtype=np.float32)
    tl[0, 0, [1, 4]] = 3.0   # tie between 1 and 4 -> 1
    tl[0, 1, [5, 2]] = 2.0   # tie between 2 and 5 -> 2
    assert acc.accept_greedy(tl, np.array([[4]]))["accept_len"].tolist() == [0]
    r = acc.accept_greedy(tl, np.array([[1]]))
    assert r["accept_len"].tolist() == [1] and r["next_token"].tolist() == [2]


# --------------------------------------------------------------------------- sampling, exact cases

def _sample(p_target, p_draft, drafts, u):
    tl = np.stack([_logits_from_probs(p) for p in p_target])[None]
    ql = np.stack([_logits_from_probs(p) for p in p_draft])[None]
    return acc.accept_sample(tl, ql, np.asarray([drafts]), np.asarray([u], dtype=np.float32))


def test_sample_two_token_hand_cases():
    """p = (3/4, 1/4), q = (1/2, 1/2), K = 1. Token 0 has ratio 3/2: always
    accepted; then the bonus token comes from p with u_K. Token 1 has ratio
    1/2: accepted for u < 1/2; rejected otherwise, and the residual
    max(0, p - q) = (1/4, 0) normalises to token 0."""
    p, q = [0.75, 0.25], [0.5, 0.5]
    r = _sample([p, p], [q], [0], [0.99, 0.70])        # accept; bonus: 0.70 * 1 > 0.75? no -> token 0
    assert r["accept_len"].tolist() == [1] and r["next_token"].tolist() == [0]
    r = _sample([p, p], [q], [0], [0.0, 0.80])         # accept; bonus u = 0.8 > 0.75 -> token 1
    assert r["accept_len"].tolist() == [1] and r["next_token"].tolist() == [1]
    r = _sample([p, p], [q], [1], [0.30, 0.99])        # 0.30 < 0.5: accept
    assert r["accept_len"].tolist() == [1]
    r = _sample([p, p], [q], [1], [0.70, 0.99])        # reject; residual is all on token 0
    assert r["accept_len"].tolist() == [0] and r["next_token"].tolist() == [0]


def test_sample_equal_distributions_accept_everything():
    """q = p: every ratio is 1 and every u < 1 accepts; the bonus token is
    p_K's inverse CDF at u_K."""
    rng = np.random.default_rng(3)
    K, V = 5, 7
    tl = rng.normal(0, 2, (2, K + 1, V)).astype(np.float32)
    ql = tl[:, :K].copy()
    drafts = rng.integers(0, V, (2, K))
    u = rng.uniform(0, 0.999, (2, K + 1)).astype(np.float32)
    r = acc.accept_sample(tl, ql, drafts, u)
    assert r["accept_len"].tolist() == [K, K]
    for b in range(2):
        c = np.cumsum(acc.softmax_f32(tl[b, K]).astype(np.float64))
        assert r["next_token"][b] == int(np.searchsorted(c, float(u[b, K]) * c[-1], side="right"))
        assert r["next_lo"][b] == r["next_token"][b] == r["next_hi"][b]  # 7 well-separated weights


def test_sample_rejects_tokens_the_verifier_rules_out():
    """The verifier puts (almost) no mass on the drafted token: rejected at
    t = 0 for any u > 1e-6, and the residual is (almost) p itself, whose mass
    sits on token 3."""
    V = 6
    p = np.full(V, 1e-9); p[3] = 1.0 - 5e-9
    q = np.full(V, 1.0 / V)
    r = _sample([p, p], [q], [0], [0.5, 0.5])
    assert r["accept_len"].tolist() == [0] and r["next_token"].tolist() == [3]


def test_sample_bad_token_is_a_rejection():
    p = [0.5, 0.5]
    r = _sample([p, p, p], [p, p], [0, 9], [0.1, 0.1, 0.1])
    assert r["accept_len"].tolist() == [1] and bool(r["bad"][0])


# --------------------------------------------------------------------------- the distribution property

def _emitted_first_tokens(sampler, p, q, n, seed):
    """Draw n first tokens with K = 1: the draft token from q (inverse CDF with
    its own uniform), then the acceptance rule; the emitted token is the draft
    token if accepted, else the resampled one."""
    rng = np.random.default_rng(seed)
    V = len(p)
    tl = np.tile(_logits_from_probs(p), (n, 2, 1))
    ql = np.tile(_logits_from_probs(q), (n, 1, 1))
    cq = np.cumsum(np.asarray(q, dtype=np.float64))
    drafts = np.minimum(np.searchsorted(cq, rng.uniform(0, 1, n), side="right"), V - 1)[:, None]
    u = rng.uniform(0, 1, (n, 2)).astype(np.float32)
    r = sampler(tl, ql, drafts, u)
    return np.where(r["accept_len"] == 1, drafts[:, 0], r["next_token"])


def _chi2_ok(tokens, p):
    n = len(tokens)
    obs = np.bincount(tokens, minlength=len(p)).astype(np.float64)
    exp_ = n * np.asarray(p, dtype=np.float64)
    chi2 = float(((obs - exp_) ** 2 / exp_).sum())
    return chi2 < 30.0, chi2  # 4 degrees of freedom: P(chi2 > 30) ~ 5e-6


P_TARGET = [0.10, 0.35, 0.05, 0.30, 0.20]
P_DRAFT = [0.30, 0.10, 0.25, 0.15, 0.20]


def pin_distribution(sampler):
    toks = _emitted_first_tokens(sampler, P_TARGET, P_DRAFT, 40000, seed=11)
    ok, chi2 = _chi2_ok(toks, P_TARGET)
    assert ok, chi2


def pin_hand_two_token(sampler):
    p, q = [0.75, 0.25], [0.5, 0.5]
    tl = np.stack([_logits_from_probs(p)] * 2)[None]
    ql = np.stack([_logits_from_probs(q)])[None]
    r = sampler(tl, ql, np.array([[1]]), np.array([[0.70, 0.99]], dtype=np.float32))
    assert r["accept_len"].tolist() == [0] and r["next_token"].tolist() == [0]
    r = sampler(tl, ql, np.array([[1]]), np.array([[0.30, 0.99]], dtype=np.float32))
    assert r["accept_len"].tolist() == [1]


def test_speculative_sampling_preserves_the_target_distribution():
    pin_distribution(acc.accept_sample)


# --------------------------------------------------------------------------- planted mistakes (CPU copies)

def _mutant(kind):
    """A copy of accept_sample's per-position rule with one planted mistake."""
    def run(tl, ql, drafts, u):
        tl, ql, u = np.asarray(tl, np.float32), np.asarray(ql, np.float32), np.asarray(u, np.float32)
        bsz, K1, V = tl.shape
        K = K1 - 1
        out_acc = np.zeros(bsz, dtype=np.int64)
        out_next = np.zeros(bsz, dtype=np.int64)
        for b in range(bsz):
            j = K
            for t in range(K):
                x = int(drafts[b, t])
                p = acc.softmax_f32(tl[b, t])[x]
                q = acc.softmax_f32(ql[b, t])[x]
                ratio = q / p if kind == "ratio_inverted" else p / q
                if not (u[b, t] < ratio):
                    j = t
                    break
            out_acc[b] = j
            if j < K:
                pt, qt = acc.softmax_f32(tl[b, j]), acc.softmax_f32(ql[b, j])
                if kind == "residual_flipped":
                    w = np.maximum(qt - pt, 0)
                elif kind == "no_residual":
                    w = pt
                else:
                    w = np.maximum(pt - qt, 0)
            else:
                w = acc.softmax_f32(tl[b, j])
            c = np.cumsum(w.astype(np.float32), dtype=np.float32)
            out_next[b] = min(int(np.searchsorted(c, u[b, K] * c[-1], side="right")), V - 1)
        return {"accept_len": out_acc, "next_token": out_next}
    return run


@pytest.mark.parametrize("kind", ["ratio_inverted", "residual_flipped", "no_residual"])
def test_planted_sampling_mistakes_are_caught(kind):
    failed = []
    for pin in (pin_distribution, pin_hand_two_token):
        try:
            pin(_mutant(kind))
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, kind


def test_pins_pass_on_the_committed_oracle():
    pin_hand_two_token(acc.accept_sample)
    pin_distribution(acc.accept_sample)


# --------------------------------------------------------------------------- precision reporting

def test_inverse_cdf_hand_values_and_admissible_range():
    """Weights (1, 2, 3, 4), cumulative (1, 3, 6, 10). u = 0.5 puts the
    threshold at 5: index 2 is the first with C > 5. With a band of 1.5,
    lo = first C > 3.5 = index 2 and hi = first C > 6.5 = index 3."""
    w = np.array([1, 2, 3, 4], dtype=np.float32)
    assert acc.inverse_cdf(w, 0.5, 0.0) == (2, 2, 2)
    assert acc.inverse_cdf(w, 0.5, 1.5) == (2, 2, 3)
    assert acc.inverse_cdf(w, 0.0, 0.0) == (0, 0, 0)
    # zero weights are never chosen: the threshold sits on a flat stretch
    w = np.array([0, 1, 0, 0, 1, 0], dtype=np.float32)
    assert acc.inverse_cdf(w, 0.5, 0.0)[0] == 4
    assert acc.inverse_cdf(w, 0.25, 0.0)[0] == 1
    # a threshold at the very top (rounding) falls back to the last positive weight
    assert acc.inverse_cdf(w, 1.0, 0.0)[0] == 4
    # nothing positive: the last index
    assert acc.inverse_cdf(np.zeros(5, np.float32), 0.3, 0.0)[0] == 4


def test_softmax_flushes_subnormal_exponentials():
    row = np.array([0.0, -100.0, -80.0], dtype=np.float32)
    p = acc.softmax_f32(row)
    assert p[1] == 0.0                       # exp(-100) = 3.7e-44 is subnormal in fp32
    assert p[2] == np.float32(np.exp(np.float32(-80.0)) / (1 + np.exp(np.float32(-80.0))))


def test_near_accept_flags_only_close_calls():
    p, q = [0.75, 0.25], [0.5, 0.5]          # draft token 1: ratio exactly 0.5
    r = _sample([p, p], [q], [1], [0.5 + 1e-6, 0.3])
    assert bool(r["near_accept"][0])
    r = _sample([p, p], [q], [1], [0.49, 0.3])
    assert not bool(r["near_accept"][0]) and r["accept_len"].tolist() == [1]
