"""Pins for the fp64 oracle: facts fixed by the mathematics and by hand
arithmetic, not by the oracle itself.

Every pin takes ``run`` -- a callable with the signature of
``oracle.verify_commit`` -- so the same pins can be run against the committed
oracle and against copies with a planted mistake (``test_oracle_mutants.py``).
Each pin raises ``AssertionError`` when it fails.
"""
from __future__ import annotations

import math

import numpy as np

from oracle import ssd_quadratic

LN2 = math.log(2.0)


def rel_err(got, ref) -> float:
    """max_i |g_i - r_i| / max(|r_i|, rms(r)) over one tensor."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(ref * ref)))
    den = np.maximum(np.abs(ref), rms if rms > 0 else 1e-300)
    return float(np.max(np.abs(got - ref) / den))


def rand_inputs(rng, bsz, H, P, N, G, K, A_zero=False):
    s0 = rng.normal(0, 0.3, (bsz, H, P, N))
    x = rng.normal(0, 1, (bsz, K, H, P))
    B = rng.normal(0, 1, (bsz, K, G, N))
    C = rng.normal(0, 1, (bsz, K, G, N))
    dt = np.log1p(np.exp(rng.normal(-1, 1, (bsz, K, H))))
    A = np.zeros(H) if A_zero else -np.exp(rng.uniform(0, math.log(16), H))
    D = rng.normal(0, 1, H)
    acc = rng.integers(0, K + 1, bsz).astype(np.int32)
    return dict(state0=s0, x=x, B=B, C=C, dt=dt, A=A, D=D, accept_len=acc)


def call(run, d, **kw):
    return run(d["state0"], d["x"], d["B"], d["C"], d["dt"], d["A"], d["D"], d.get("accept_len"), **kw)


# --------------------------------------------------------------------------- hand-derived values

def pin_hand_scalar(run):
    """P = N = 1, K = 3, A = -ln 2. With dt = (1, 2, 1) the decays are
    (1/2, 1/4, 1/2) and u = dt x = (2, 8, -1); by hand:
      h1 = 0.5*1 + 2*1 = 2.5        y0 = 1*2.5 + 0.25*2 = 3.0
      h2 = 0.25*2.5 + 8*0.5 = 4.625 y1 = 2*4.625 + 0.25*4 = 10.25
      h3 = 0.5*4.625 - 1*2 = 0.3125 y2 = 3*0.3125 + 0.25*(-1) = 0.6875
    y uses D*x, not D*u (the two differ at t = 1)."""
    d = dict(state0=np.ones((1, 1, 1, 1)), x=np.array([2.0, 4.0, -1.0]).reshape(1, 3, 1, 1),
             B=np.array([1.0, 0.5, 2.0]).reshape(1, 3, 1, 1), C=np.array([1.0, 2.0, 3.0]).reshape(1, 3, 1, 1),
             dt=np.array([1.0, 2.0, 1.0]).reshape(1, 3, 1), A=np.array([-LN2]), D=np.array([0.25]))
    traj_ref = [1.0, 2.5, 4.625, 0.3125]
    for j in range(4):
        d["accept_len"] = np.array([j], dtype=np.int32)
        r = call(run, d, want_trajectory=True)
        assert rel_err(r["y"].ravel(), [3.0, 10.25, 0.6875]) < 1e-14, r["y"].ravel()
        assert rel_err(r["trajectory"].ravel(), traj_ref) < 1e-14, r["trajectory"].ravel()
        assert abs(r["state"].item() - traj_ref[j]) < 1e-14, (j, r["state"].item())


def pin_hand_2x3(run):
    """P = 2, N = 3, K = 2, A = -ln 2, dt = 1 (decay 1/2), D = 1/2. State rows
    are head-dim channels p, columns state channels n; by hand:
      h1 = [[1.5, 2, -0.5], [-1, -3.5, 0]]      y0 = [2.0, -4.5]
      h2 = [[0.75, 3, -2.25], [-0.5, -1.75, 0]] y1 = [-2.75, -0.5]"""
    d = dict(state0=np.array([[1.0, 0.0, -1.0], [2.0, 1.0, 0.0]]).reshape(1, 1, 2, 3),
             x=np.array([[1.0, -2.0], [2.0, 0.0]]).reshape(1, 2, 1, 2),
             B=np.array([[1.0, 2.0, 0.0], [0.0, 1.0, -1.0]]).reshape(1, 2, 1, 3),
             C=np.array([[0.0, 1.0, 1.0], [1.0, 0.0, 2.0]]).reshape(1, 2, 1, 3),
             dt=np.ones((1, 2, 1)), A=np.array([-LN2]), D=np.array([0.5]),
             accept_len=np.array([1], dtype=np.int32))
    r = call(run, d, want_trajectory=True)
    assert rel_err(r["y"].reshape(2, 2), [[2.0, -4.5], [-2.75, -0.5]]) < 1e-14, r["y"]
    assert rel_err(r["state"].reshape(2, 3), [[1.5, 2.0, -0.5], [-1.0, -3.5, 0.0]]) < 1e-14, r["state"]
    assert rel_err(r["trajectory"][0, 0, 2], [[0.75, 3.0, -2.25], [-0.5, -1.75, 0.0]]) < 1e-14


# --------------------------------------------------------------------------- closed forms

def pin_closed_form_A_zero(run):
    """A = 0 makes every decay 1: h_t = h_0 + sum_{s<=t} dt_s x_s B_s^T (a
    running sum) and y_t = C_t h_t + D x_t."""
    rng = np.random.default_rng(11)
    for (bsz, H, P, N, G, K) in [(2, 4, 5, 3, 2, 5), (1, 3, 4, 6, 3, 1), (3, 2, 7, 2, 1, 6)]:
        d = rand_inputs(rng, bsz, H, P, N, G, K, A_zero=True)
        r = call(run, d, want_trajectory=True)
        g_of_h = np.arange(H) // (H // G)
        Bh = d["B"][:, :, g_of_h, :]                     # [b][K][H][N]
        Ch = d["C"][:, :, g_of_h, :]
        incr = np.einsum("bkh,bkhp,bkhn->bkhpn", d["dt"], d["x"], Bh)
        hs = d["state0"][:, None] + np.cumsum(incr, axis=1)   # [b][K][H][P][N]: h_1..h_K
        y = np.einsum("bkhn,bkhpn->bkhp", Ch, hs) + d["D"][None, None, :, None] * d["x"]
        assert rel_err(r["y"], y) < 1e-12
        traj = np.concatenate([d["state0"][:, None], hs], axis=1).transpose(0, 2, 1, 3, 4)
        assert rel_err(r["trajectory"], traj) < 1e-12
        for b in range(bsz):
            assert rel_err(r["state"][b], traj[b, :, d["accept_len"][b]]) < 1e-12


def pin_quadratic_form(run):
    """Brute force over random tiny shapes against the materialised
    attention-like form (masked C B^T with segment-sum decays)."""
    rng = np.random.default_rng(12)
    for _ in range(60):
        G = int(rng.integers(1, 3))
        H = G * int(rng.integers(1, 3))
        P, N, K = int(rng.integers(1, 9)), int(rng.integers(1, 9)), int(rng.integers(1, 7))
        bsz = int(rng.integers(1, 4))
        d = rand_inputs(rng, bsz, H, P, N, G, K)
        r = call(run, d)
        q = ssd_quadratic(d["state0"], d["x"], d["B"], d["C"], d["dt"], d["A"], d["D"], d["accept_len"])
        assert rel_err(r["y"], q["y"]) < 1e-12, (bsz, H, P, N, G, K)
        assert rel_err(r["state"], q["state"]) < 1e-12, (bsz, H, P, N, G, K)


def pin_dt_zero(run):
    """dt = 0: the decay is 1 and the input term vanishes, so the state never
    moves and y_t = C_t h_0 + D x_t."""
    rng = np.random.default_rng(13)
    d = rand_inputs(rng, 2, 4, 6, 5, 2, 4)
    d["dt"] = np.zeros_like(d["dt"])
    r = call(run, d)
    g_of_h = np.arange(4) // 2
    Ch = d["C"][:, :, g_of_h, :]
    y = np.einsum("bkhn,bhpn->bkhp", Ch, d["state0"]) + d["D"][None, None, :, None] * d["x"]
    assert rel_err(r["y"], y) < 1e-13
    assert np.array_equal(r["state"], d["state0"])


def pin_memoryless(run):
    """A -> -inf makes the decay exactly 0: h_t = dt_t x_t B_t^T regardless
    of the past, and y_t = C_t h_t + D x_t."""
    rng = np.random.default_rng(14)
    d = rand_inputs(rng, 2, 2, 3, 4, 1, 3)
    d["A"] = np.full(2, -1e300)
    r = call(run, d, want_trajectory=True)
    hs = np.einsum("bkh,bkhp,bkn->bkhpn", d["dt"], d["x"], d["B"][:, :, 0, :])
    assert rel_err(r["trajectory"][:, :, 1:], hs.transpose(0, 2, 1, 3, 4)) < 1e-15
    y = np.einsum("bkn,bkhpn->bkhp", d["C"][:, :, 0, :], hs) + d["D"][None, None, :, None] * d["x"]
    assert rel_err(r["y"], y) < 1e-13


def pin_linearity(run):
    """With dt, A, B, C, D fixed the map (x, h_0) -> (y, h_j) is linear."""
    rng = np.random.default_rng(15)
    d1 = rand_inputs(rng, 2, 2, 4, 3, 1, 4)
    d2 = dict(d1)
    d2["x"] = rng.normal(0, 1, d1["x"].shape)
    d2["state0"] = rng.normal(0, 1, d1["state0"].shape)
    ds = dict(d1)
    ds["x"] = 2.0 * d1["x"] - 3.0 * d2["x"]
    ds["state0"] = 2.0 * d1["state0"] - 3.0 * d2["state0"]
    r1, r2, rs = call(run, d1), call(run, d2), call(run, ds)
    assert rel_err(rs["y"], 2.0 * r1["y"] - 3.0 * r2["y"]) < 1e-12
    assert rel_err(rs["state"], 2.0 * r1["state"] - 3.0 * r2["state"]) < 1e-12


def pin_group_mapping(run):
    """Heads use B/C groups in consecutive blocks, g = h // (H // G): with
    H = 4, G = 2 and group 1's B and C zeroed, heads 2, 3 only decay
    (h_j = exp(A sum dt) h_0, y = D x) while heads 0, 1 move."""
    rng = np.random.default_rng(16)
    d = rand_inputs(rng, 1, 4, 3, 5, 2, 3)
    d["B"][:, :, 1, :] = 0.0
    d["C"][:, :, 1, :] = 0.0
    d["accept_len"] = np.array([3], dtype=np.int32)
    r = call(run, d)
    for h in (2, 3):
        decay = math.exp(d["A"][h] * d["dt"][0, :, h].sum())
        assert rel_err(r["state"][0, h], decay * d["state0"][0, h]) < 1e-13
        assert rel_err(r["y"][0, :, h, :], d["D"][h] * d["x"][0, :, h, :]) < 1e-13
    for h in (0, 1):
        decay = math.exp(d["A"][h] * d["dt"][0, :, h].sum())
        assert rel_err(r["state"][0, h], decay * d["state0"][0, h]) > 1e-3


# --------------------------------------------------------------------------- rollback / prefix selection

def pin_rollback_equals_single_steps(run):
    """K steps then rollback to j give exactly (bitwise, same fp64 operation
    order) the state of j single-token steps each fully accepted."""
    rng = np.random.default_rng(17)
    K = 6
    d = rand_inputs(rng, 2, 4, 5, 6, 2, K)
    for j in range(K + 1):
        d["accept_len"] = np.full(2, j, dtype=np.int32)
        full = call(run, d)["state"]
        s = d["state0"].copy()
        for t in range(j):
            one = dict(state0=s, x=d["x"][:, t:t + 1], B=d["B"][:, t:t + 1], C=d["C"][:, t:t + 1],
                       dt=d["dt"][:, t:t + 1], A=d["A"], D=d["D"], accept_len=None)
            s = call(run, one)["state"]
        assert np.array_equal(full, s), j


def pin_prefix_selection(run):
    """The committed state is h_j, the state after exactly j accepted tokens,
    on inputs where h_{j-1}, h_j and h_{j+1} differ far beyond any tolerance;
    y does not depend on j."""
    rng = np.random.default_rng(18)
    K = 5
    d = rand_inputs(rng, 1, 2, 4, 4, 1, K)
    d["dt"] = np.full_like(d["dt"], 0.7)
    d["A"] = np.array([-0.5, -2.0])
    ys = []
    for j in range(K + 1):
        d["accept_len"] = np.array([j], dtype=np.int32)
        r = call(run, d, want_trajectory=True)
        tr = r["trajectory"][0]                      # [H][K+1][P][N]
        assert np.array_equal(r["state"][0], tr[:, j])
        for jj in (j - 1, j + 1):
            if 0 <= jj <= K:
                assert rel_err(tr[:, jj], tr[:, j]) > 1e-2
        q = ssd_quadratic(d["state0"], d["x"], d["B"], d["C"], d["dt"], d["A"], d["D"], d["accept_len"])
        assert rel_err(r["state"], q["state"]) < 1e-12
        ys.append(r["y"])
    for y in ys[1:]:
        assert np.array_equal(y, ys[0])


def pin_invalid_accept_len(run):
    """accept_len outside [0, K] leaves that sequence's state unchanged and is
    reported; the other sequences commit normally."""
    rng = np.random.default_rng(19)
    d = rand_inputs(rng, 3, 2, 3, 4, 1, 3)
    for bad in (-1, 4, -7, 1 << 30):
        d["accept_len"] = np.array([bad, 2, 3], dtype=np.int32)
        r = call(run, d, want_trajectory=True)
        assert int(r["status"]) & 1, bad
        assert np.array_equal(r["state"][0], d["state0"][0])
        assert np.array_equal(r["state"][1], r["trajectory"][1][:, 2])
        assert np.array_equal(r["state"][2], r["trajectory"][2][:, 3])
    d["accept_len"] = np.array([0, 2, 3], dtype=np.int32)
    assert int(call(run, d)["status"]) == 0


def pin_plain_decode(run):
    """accept_len = None accepts all K tokens: the state is h_K."""
    rng = np.random.default_rng(20)
    d = rand_inputs(rng, 2, 2, 3, 4, 2, 1)
    d["accept_len"] = None
    r = call(run, d, want_trajectory=True)
    assert np.array_equal(r["state"], r["trajectory"][:, :, 1])
    q = ssd_quadratic(d["state0"], d["x"], d["B"], d["C"], d["dt"], d["A"], d["D"], None)
    assert rel_err(r["state"], q["state"]) < 1e-13
    assert int(r["status"]) == 0


ALL_PINS = [pin_hand_scalar, pin_hand_2x3, pin_closed_form_A_zero, pin_quadratic_form, pin_dt_zero,
            pin_memoryless, pin_linearity, pin_group_mapping, pin_rollback_equals_single_steps,
            pin_prefix_selection, pin_invalid_accept_len, pin_plain_decode]
