"""fp64 CPU oracle for the Mamba-layer speculative verify/commit step.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package. It shares no
code with the CUDA library (``ssm_recurrence_verify_b300``) and neither imports
the other; the only common module is the seeded input generator, which holds
none of the method's arithmetic.

Two independent formulations live here:

* ``verify_commit`` -- the sequential recurrence in plain C, fp64 (``ssm_oracle.c``),
  the definition the CUDA kernels are checked against.
* ``ssd_quadratic`` -- the materialised attention-like (quadratic) form of the
  same linear RNN in numpy float64, used to pin the C recurrence on tiny inputs.

Parity pins (see ``tests/test_oracle.py``): the A = 0 closed form (a running
sum), the quadratic form, K-steps-then-rollback-to-j versus j single steps,
hand-derived scalar and 2x3 examples, dt = 0 and a = 0 special cases,
linearity, the B/C group mapping, and prefix selection on inputs whose states
differ far beyond any tolerance.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Dict, Optional, Sequence, Tuple

import numpy as np

from .ssd_quadratic import ssd_quadratic  # noqa: F401  (re-export)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssm_oracle.c")
_LIB = os.path.join(_HERE, "libssm_oracle.so")
_lib = None

ORACLE_BAD_ACCEPT_LEN = 1


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (no contraction, so a*S + u*B is two
    roundings) into ``oracle/libssm_oracle.so``."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class Oracle:
    """A loaded copy of the C recurrence. ``Oracle()`` is the committed one;
    tests may load a separately compiled copy (e.g. one with a planted
    mistake) to show that the pins catch it."""

    def __init__(self, path: Optional[str] = None):
        lib = ctypes.CDLL(path or build())
        f = lib.ssm_oracle_verify_commit
        f.argtypes = [ctypes.c_int64] * 6 + [ctypes.c_void_p] * 11
        f.restype = ctypes.c_int
        self._fn = f
        self.path = path or _LIB

    def verify_commit(self, *args, **kwargs) -> Dict[str, np.ndarray]:
        return _verify_commit(self._fn, *args, **kwargs)


def _default() -> Oracle:
    global _lib
    if _lib is None:
        _lib = Oracle()
    return _lib


def _f64(a) -> np.ndarray:
    """Exact widening of an fp32 / bf16 (torch or numpy) array to float64."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().to("cpu").to(torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _i32(a) -> np.ndarray:
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().to("cpu").numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def verify_commit(state0, x, B, C, dt, A, D, accept_len=None, *, want_y: bool = True,
                  want_state: bool = True, want_trajectory: bool = False) -> Dict[str, np.ndarray]:
    """Run the committed fp64 recurrence (see ``_verify_commit``)."""
    return _default().verify_commit(state0, x, B, C, dt, A, D, accept_len, want_y=want_y,
                                    want_state=want_state, want_trajectory=want_trajectory)


def _verify_commit(fn, state0, x, B, C, dt, A, D, accept_len=None, *, want_y: bool = True,
                   want_state: bool = True, want_trajectory: bool = False) -> Dict[str, np.ndarray]:
    """Run the fp64 recurrence for one layer over a batch.

    Shapes: ``state0[b][H][P][N]``, ``x[b][K][H][P]``, ``B``/``C[b][K][G][N]``,
    ``dt[b][K][H]``, ``A``/``D[H]``, ``accept_len[b]`` (int32) or ``None`` for
    "every token accepted" (plain decode). Inputs may be fp32 or bf16; they are
    widened to float64 exactly. Returns a dict with ``y[b][K][H][P]``,
    ``state[b][H][P][N]`` (the committed h_j), ``trajectory[b][H][K+1][P][N]``
    (h_0..h_K) where asked, and ``status`` (bit 0: an accept_len was out of
    range and that sequence's state was left unchanged).
    """
    s0, xx, bb, cc, dd = (_f64(v) for v in (state0, x, B, C, dt))
    aa, DD = _f64(A), _f64(D)
    bsz, H, P, N = s0.shape
    K = xx.shape[1]
    G = bb.shape[2]
    assert xx.shape == (bsz, K, H, P), xx.shape
    assert bb.shape == (bsz, K, G, N) and cc.shape == bb.shape, (bb.shape, cc.shape)
    assert dd.shape == (bsz, K, H), dd.shape
    assert aa.shape == (H,) and DD.shape == (H,)
    acc = None if accept_len is None else _i32(accept_len)
    if acc is not None:
        assert acc.shape == (bsz,)
    y = np.empty((bsz, K, H, P)) if want_y else None
    st = np.empty((bsz, H, P, N)) if want_state else None
    tr = np.empty((bsz, H, K + 1, P, N)) if want_trajectory else None
    rc = fn(bsz, H, P, N, G, K, _ptr(s0), _ptr(xx), _ptr(bb), _ptr(cc), _ptr(dd), _ptr(aa), _ptr(DD),
            _ptr(acc), _ptr(y), _ptr(st), _ptr(tr))
    if rc < 0:
        raise ValueError(f"oracle rejected the shapes (code {rc})")
    out: Dict[str, np.ndarray] = {"status": np.int32(rc)}
    if want_y:
        out["y"] = y
    if want_state:
        out["state"] = st
    if want_trajectory:
        out["trajectory"] = tr
    return out


def verify_commit_slices(inputs: Dict[str, object], pairs: Sequence[Tuple[int, int]]
                         ) -> Dict[Tuple[int, int], Dict[str, np.ndarray]]:
    """The oracle on selected (sequence b, head h) slices of a large batch.

    Marshalling only: each slice is one call of the same recurrence with
    batch = 1, H = 1, G = 1 and that head's group of B/C. Returns, per pair,
    ``y[K][P]`` and ``state[P][N]``.
    """
    import torch

    def t(name):
        v = inputs[name]
        return v if isinstance(v, torch.Tensor) else torch.as_tensor(v)

    state0, x, B, C, dt, A, D = (t(k) for k in ("state0", "x", "B", "C", "dt", "A", "D"))
    acc = inputs.get("accept_len")
    H = state0.shape[1]
    G = B.shape[2]
    out = {}
    for b, h in pairs:
        g = h // (H // G)
        r = verify_commit(state0[b:b + 1, h:h + 1], x[b:b + 1, :, h:h + 1], B[b:b + 1, :, g:g + 1],
                          C[b:b + 1, :, g:g + 1], dt[b:b + 1, :, h:h + 1], A[h:h + 1], D[h:h + 1],
                          None if acc is None else t("accept_len")[b:b + 1])
        out[(b, h)] = {"y": r["y"][0, :, 0, :], "state": r["state"][0, 0], "status": r["status"]}
    return out
