"""The quadratic (attention-like) form of the discretised linear RNN, numpy float64.

TEST INFRASTRUCTURE ONLY: an independent formulation used to pin the C
recurrence in ``ssm_oracle.c`` on tiny inputs. It never runs the recurrence.

The pages motivate the whole distillation by the similarity between attention
and the linear-RNN computation (news summary "Llama 3+Mamba ...", initialisation
section: attention is linearised, and the pretrained projections carry over,
with C, B and x in the roles of query, key and value; the method overview says
the same of the Mamba initialisation). Unrolling the recurrence

    a_t = exp(dt_t A),  h_t = a_t h_{t-1} + (dt_t x_t) B_t^T,  y_t = C_t h_t + D x_t

gives, for one (sequence, head), the masked "attention" form

    y_t = w_t (C_t . h_0) + sum_{s <= t} L[t, s] (C_t . B_s) dt_s x_s + D x_t
    L[t, s] = prod_{r = s+1 .. t} a_r = exp(A * sum_{r = s+1 .. t} dt_r)
    w_t     = prod_{r = 0 .. t} a_r   = exp(A * sum_{r <= t} dt_r)

and the state after the first j tokens

    h_j = W_j h_0 + sum_{s < j} L[j-1, s] dt_s x_s B_s^T,   W_j = exp(A * sum_{r < j} dt_r)

(h_0 for j = 0). The decay products are formed from segment sums of dt, a
different route from the step-by-step products of the recurrence.
"""
from __future__ import annotations

from typing import Dict, Optional

import numpy as np


def _as64(a) -> np.ndarray:
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().to("cpu").to(torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(a, dtype=np.float64)


def ssd_quadratic(state0, x, B, C, dt, A, D, accept_len=None) -> Dict[str, np.ndarray]:
    """y for every token and the committed state h_j, via the quadratic form.

    Same shapes as the recurrence oracle: ``state0[b][H][P][N]``,
    ``x[b][K][H][P]``, ``B``/``C[b][K][G][N]``, ``dt[b][K][H]``, ``A``/``D[H]``,
    ``accept_len[b]`` or ``None`` (all K accepted). Head h reads group
    ``h // (H // G)``. Returns ``y`` and ``state`` (float64). Meant for tiny
    inputs: it materialises K x K matrices per (b, h).
    """
    s0, xx, bb, cc, dd = (_as64(v) for v in (state0, x, B, C, dt))
    aa, DD = _as64(A), _as64(D)
    bsz, H, P, N = s0.shape
    K = xx.shape[1]
    G = bb.shape[2]
    hpg = H // G
    acc: Optional[np.ndarray] = None if accept_len is None else np.asarray(_as64(accept_len), dtype=np.int64)

    y = np.zeros((bsz, K, H, P))
    st = np.zeros((bsz, H, P, N))
    tri = np.tril(np.ones((K, K), dtype=bool))
    for b in range(bsz):
        j = K if acc is None else int(acc[b])
        for h in range(H):
            g = h // hpg
            Xh = xx[b, :, h, :]            # [K][P]
            Bg = bb[b, :, g, :]            # [K][N]
            Cg = cc[b, :, g, :]            # [K][N]
            d = dd[b, :, h]                # [K]
            h0 = s0[b, h]                  # [P][N]
            csum = np.concatenate([[0.0], np.cumsum(d)])   # csum[i] = sum_{r < i} dt_r
            # L[t, s] = exp(A * (csum[t+1] - csum[s+1])) on s <= t
            seg = csum[1:, None] - csum[None, 1:]
            L = np.where(tri, np.exp(aa[h] * np.where(tri, seg, 0.0)), 0.0)
            w = np.exp(aa[h] * csum[1:])                    # [K]
            U = d[:, None] * Xh                             # [K][P]
            scores = L * (Cg @ Bg.T)                        # [K][K], the masked C B^T
            y[b, :, h, :] = w[:, None] * (Cg @ h0.T) + scores @ U + DD[h] * Xh
            if 0 <= j <= K:
                if j == 0:
                    st[b, h] = h0
                else:
                    lj = np.exp(aa[h] * (csum[j] - csum[1:j + 1]))   # L[j-1, s] for s < j
                    st[b, h] = np.exp(aa[h] * csum[j]) * h0 + (U[:j] * lj[:, None]).T @ Bg[:j]
            else:
                st[b, h] = h0
    return {"y": y, "state": st}
