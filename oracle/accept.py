"""Acceptance of draft tokens, numpy (TEST INFRASTRUCTURE ONLY).

The step right after the verifier's pass in speculative decoding (news summary
"Llama 3+Mamba强强联手！蒸馏到RNN，推理速度提升1.6倍", speculative-decoding
section: the draft model proposes K tokens; a token the verifier agrees with is
accepted; at the first token it does not, processing stops, the state rolls
back to the last accepted token and decoding restarts from there; if all K are
accepted they are kept and the next round begins). The method overview names
the procedure a speculative *sampling* algorithm. Two rules:

* greedy: draft token t is accepted when it is the verifier's most likely
  token at position t; accept_len = j is the number of leading accepted
  tokens, and the next token is the verifier's most likely token at
  position j (a correction after a rejection, the bonus token when j = K).
* sampling: with p_t = softmax(target logits at t) and q_t = softmax(draft
  logits at t), draft token x_t is accepted when u_t < p_t(x_t) / q_t(x_t); at
  the first rejection j the next token is drawn from the normalised residual
  max(0, p_j - q_j), after j = K from p_K, by inverse CDF with u_K.

Precision. The probabilities are fp32 values (the kernel's precision):
e = exp(l - max) in fp32 with results below 2^-126 flushed to zero, and
p = e / sum(e). The cumulative sums of the inverse CDF accumulate those fp32
weights in fp64 (a sequential fp32 cumsum over a 128K vocabulary would carry
more rounding than the kernel's hierarchical sums). Any fp32 evaluation order
agrees with these values to within a small bound, so the functions also report
what another order may legitimately decide: ``near_accept`` (an acceptance
ratio within ``tie_eps`` of its uniform) and ``[next_lo, next_hi]``, the
indices whose cumulative weight lies within ``tie_eps * scale`` of the
threshold (scale = sum(p) + sum(q) = 2 for a residual, 1 for p itself).
Ties of the most likely token go to the smallest index. Draft tokens outside
[0, V) are rejections; the next token is then drawn from p_t (greedy: its
most likely token).

Shared with nothing on the CUDA side; only ``tests/`` and the benchmark's
CPU baseline may import it.
"""
from __future__ import annotations

from typing import Dict

import numpy as np

FTZ = np.float32(2.0 ** -126)
TIE_EPS = 3e-5


def _f32(a) -> np.ndarray:
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().to("cpu").to(torch.float32).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(a, dtype=np.float32)


def _i64(a) -> np.ndarray:
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().to("cpu").numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(a, dtype=np.int64)


def softmax_f32(row: np.ndarray) -> np.ndarray:
    """Softmax of one logit row in fp32: exp(l - max), subnormal results
    flushed to zero, divided by their sum."""
    row = row.astype(np.float32)
    e = np.exp(row - row.max(), dtype=np.float32)
    e[e < FTZ] = 0.0
    return (e / e.sum(dtype=np.float32)).astype(np.float32)


def accept_greedy(target_logits, draft_tokens) -> Dict[str, np.ndarray]:
    """target_logits [b][K+1][V], draft_tokens [b][K] -> accept_len [b],
    next_token [b] (int64), and ``bad`` [b]: a draft token outside [0, V)
    (counted as a mismatch)."""
    tl = _f32(target_logits)
    dr = _i64(draft_tokens)
    bsz, K1, V = tl.shape
    K = K1 - 1
    assert dr.shape == (bsz, K)
    acc = np.zeros(bsz, dtype=np.int64)
    nxt = np.zeros(bsz, dtype=np.int64)
    bad = np.zeros(bsz, dtype=bool)
    for b in range(bsz):
        best = tl[b].argmax(axis=1)  # numpy argmax: first (smallest) index among ties
        j = 0
        while j < K:
            x = dr[b, j]
            if x < 0 or x >= V:
                bad[b] = True
                break
            if best[j] != x:
                break
            j += 1
        acc[b] = j
        nxt[b] = best[j]
    return {"accept_len": acc, "next_token": nxt, "bad": bad}


def accept_sample(target_logits, draft_logits, draft_tokens, uniform,
                  tie_eps: float = TIE_EPS) -> Dict[str, np.ndarray]:
    """Speculative sampling. target_logits [b][K+1][V], draft_logits [b][K][V],
    draft_tokens [b][K], uniform [b][K+1] in [0, 1). Returns accept_len,
    next_token, bad (draft token outside [0, V): rejected there),
    ``near_accept`` [b] (an acceptance decision within tie_eps, relative, of
    its threshold) and ``next_lo`` / ``next_hi`` [b] (the admissible range of
    the next token for this accept_len, see the module docstring)."""
    tl = _f32(target_logits)
    ql = _f32(draft_logits)
    dr = _i64(draft_tokens)
    u = _f32(uniform)
    bsz, K1, V = tl.shape
    K = K1 - 1
    assert ql.shape == (bsz, K, V) and dr.shape == (bsz, K) and u.shape == (bsz, K1)
    acc = np.zeros(bsz, dtype=np.int64)
    nxt = np.zeros(bsz, dtype=np.int64)
    lo = np.zeros(bsz, dtype=np.int64)
    hi = np.zeros(bsz, dtype=np.int64)
    bad = np.zeros(bsz, dtype=bool)
    near = np.zeros(bsz, dtype=bool)
    for b in range(bsz):
        j = K
        for t in range(K):
            x = dr[b, t]
            if x < 0 or x >= V:
                bad[b] = True
                j = t
                break
            p = softmax_f32(tl[b, t])[x]
            q = softmax_f32(ql[b, t])[x]
            ratio = np.float32(p) / np.float32(q) if q > 0 else np.float32(np.inf)
            if abs(float(u[b, t]) - float(ratio)) <= tie_eps * float(ratio):
                near[b] = True
            if not (u[b, t] < ratio):
                j = t
                break
        acc[b] = j
        if j < K and not bad[b]:
            w = np.maximum(softmax_f32(tl[b, j]) - softmax_f32(ql[b, j]), np.float32(0.0)).astype(np.float32)
            scale = 2.0
        else:
            w = softmax_f32(tl[b, j])
            scale = 1.0
        nxt[b], lo[b], hi[b] = inverse_cdf(w, u[b, K], tie_eps * scale)
    return {"accept_len": acc, "next_token": nxt, "bad": bad, "near_accept": near, "next_lo": lo, "next_hi": hi}


def inverse_cdf(w: np.ndarray, u: float, band: float):
    """Inverse CDF of the weights w >= 0 at u: the smallest index v with
    C(v) > u * C(V-1), C the cumulative sum (fp64 accumulation); if rounding
    leaves none, the last index with w > 0 (V - 1 if there is none). Also
    the admissible range [lo, hi]: lo = smallest v with C(v) > thr - band,
    hi = smallest v with C(v) > thr + band (or the fallback above)."""
    w = np.asarray(w, dtype=np.float32)
    c = np.cumsum(w.astype(np.float64))
    total = c[-1]
    thr = float(np.float32(u)) * total
    pos = np.nonzero(w > 0)[0]
    fallback = int(pos[-1]) if len(pos) else len(w) - 1

    def first_above(level):
        i = int(np.searchsorted(c, level, side="right"))
        return i if i < len(w) else fallback

    return first_above(thr), first_above(thr - band), first_above(thr + band)
