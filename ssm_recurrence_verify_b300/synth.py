"""Seeded synthetic workloads for the Mamba-layer speculative verify/commit step.

This module only *draws* inputs. It holds none of the method's arithmetic: no
discretisation, no recurrence, no output contraction. It is shared by the GPU
path, the tests, the benchmark and the fp64 oracle, so that every side sees the
identical bits.

Where the inputs come from (the pages print no data for this step):

* The shapes are those of the model families the paper distils
  ("The Mamba in the Llama: Distilling and Accelerating Hybrid Models"):
  a Llama-3-8B-shaped layer whose B/C groups mirror the GQA K/V heads (the
  attention-to-linear-RNN correspondence of the paper's initialisation, where
  C, B and x take the roles of Q, K and V), a 50 % hybrid stack, a batched
  speculative-serving load, and a Mamba-2-2.7B-shaped pure SSM stack.
* The draft length K and the accepted-prefix length follow the speculative
  decoding procedure (draft K tokens, accept a prefix, roll back the rest).
* The value distributions are synthetic stand-ins for activations at those
  shapes: ``x, B, C ~ N(0,1)/sqrt(N)``; ``dt = softplus(N(-2, 1))`` (already
  positive, the kernels apply no softplus); ``A_h = -exp(U(0, ln 16))``;
  ``D ~ N(0, 1)``; initial state ``~ N(0, 0.1^2)``.

Every tensor is drawn on the CPU from its own numpy PCG64 stream, seeded
through a SeedSequence over the whole key (workload seed, tensor kind, round,
layer, sequence), so streams of different tensors are independent and any one
layer, round or sequence can be regenerated without drawing the others. (A
single integer seed is not enough: torch's CPU generator keeps only its low 32
bits.) Values are rounded to bf16 on the CPU (round-to-nearest-even) where the
workload says so.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import numpy as np
import torch

F32 = "f32"
BF16 = "bf16"

_TORCH_DTYPE = {F32: torch.float32, BF16: torch.bfloat16}

# tensor kinds, part of every per-tensor seed
_KIND = {"A": 1, "D": 2, "state0": 3, "x": 4, "B": 5, "C": 6, "dt": 7, "accept": 8,
         "draft": 9, "base": 10, "tnoise": 11, "agree": 12, "peak": 13, "uniform": 14}


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape and draw recipe of one synthetic workload.

    ``accept`` is one of ``"uniform"`` (accept_len ~ U{0..K}), ``"geometric"``
    (tokens accepted before the first rejection with per-token rejection
    probability 0.3, capped at K) or ``"all"`` (plain decode: every token kept).
    """

    name: str
    seed: int
    batch: int
    nlayers: int
    nheads: int
    headdim: int  # P
    dstate: int  # N
    ngroups: int  # G
    ntok: int  # K
    in_dtype: str
    accept: str
    rounds: int = 1
    description: str = ""

    @property
    def torch_in_dtype(self) -> torch.dtype:
        return _TORCH_DTYPE[self.in_dtype]

    def in_elem_bytes(self) -> int:
        return 4 if self.in_dtype == F32 else 2

    def state_elems(self) -> int:
        return self.batch * self.nheads * self.headdim * self.dstate


WORKLOADS: Dict[int, Workload] = {
    0: Workload("tiny_fp32_b1_h2_p16_n16_k4", 0, 1, 1, 2, 16, 16, 1, 4, F32, "uniform", rounds=3,
                description="tiny oracle case, fp32 throughout"),
    1: Workload("llama3_8b_layer_decode_b1_h32_p128_n128_g8_k1", 1, 1, 1, 32, 128, 128, 8, 1, BF16, "all",
                description="Llama-3-8B-shaped single Mamba layer, plain decode (K=1)"),
    2: Workload("hybrid50_16layer_verify_b1_h32_p128_n128_g8_k4", 2, 1, 16, 32, 128, 128, 8, 4, BF16,
                "uniform", rounds=3,
                description="50% hybrid verify pass: 16 Mamba layers of the Llama-3-8B shape, K=4"),
    3: Workload("batched_spec_serving_b64_h32_p128_n128_g8_k8", 3, 64, 1, 32, 128, 128, 8, 8, BF16,
                "uniform",
                description="batched speculative serving: 64 sequences, one Llama-3-8B-shaped layer, K=8"),
    4: Workload("mamba2_2p7b_stack_b16_l64_h80_p64_n128_g1_k16", 4, 16, 64, 80, 64, 128, 1, 16, BF16,
                "geometric",
                description="Mamba-2-2.7B-shaped pure SSM stack: 64 layers, 16 sequences, K=16"),
}


def _rng(seed: int, kind: str, rnd: int = 0, layer: int = 0, seq: int = -1) -> np.random.Generator:
    """The stream of one tensor (``seq = -1``: not per sequence)."""
    key = [seed, _KIND[kind], rnd, layer, seq + 1]
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(key)))


def _normal(shape, rng: np.random.Generator, mean: float = 0.0, std: float = 1.0) -> torch.Tensor:
    z = rng.standard_normal(shape, dtype=np.float32)
    return torch.from_numpy(z * np.float32(std) + np.float32(mean))


def _uniform(shape, rng: np.random.Generator, lo: float = 0.0, hi: float = 1.0) -> torch.Tensor:
    r = rng.random(shape, dtype=np.float32)
    return torch.from_numpy(r * np.float32(hi - lo) + np.float32(lo))


def draw_params(wl: Workload, layer: int = 0, batch: Optional[int] = None,
                batch_offset: int = 0) -> Dict[str, torch.Tensor]:
    """Per-layer parameters and cached state: ``A[H]``, ``D[H]`` (fp32) and
    ``state0[batch][H][P][N]`` (fp32). ``batch``/``batch_offset`` select a
    slice of the sequences; a sequence's state does not depend on them."""
    Bsz = wl.batch if batch is None else batch
    H, P, N = wl.nheads, wl.headdim, wl.dstate
    A = -torch.exp(_uniform((H,), _rng(wl.seed, "A", 0, layer), 0.0, math.log(16.0)))
    D = _normal((H,), _rng(wl.seed, "D", 0, layer))
    state0 = torch.empty((Bsz, H, P, N), dtype=torch.float32)
    for i, b in enumerate(range(batch_offset, batch_offset + Bsz)):
        state0[i] = _normal((H, P, N), _rng(wl.seed, "state0", 0, layer, b), 0.0, 0.1)
    return {"A": A, "D": D, "state0": state0}


def draw_tokens(wl: Workload, rnd: int = 0, layer: int = 0, batch: Optional[int] = None,
                batch_offset: int = 0) -> Dict[str, torch.Tensor]:
    """Per-(round, layer) draft-token inputs, in the workload's input dtype.

    ``x[batch][K][H][P]``, ``B``/``C[batch][K][G][N]``, ``dt[batch][K][H]``.
    ``batch``/``batch_offset`` select a slice of the sequences (used to shard
    the batch over ranks); the values of a sequence do not depend on them.
    """
    Bsz = wl.batch if batch is None else batch
    K, H, P, N, G = wl.ntok, wl.nheads, wl.headdim, wl.dstate, wl.ngroups
    out = {}
    inv_sqrt_n = 1.0 / math.sqrt(N)
    for name, shape in (("x", (K, H, P)), ("B", (K, G, N)), ("C", (K, G, N))):
        rows = []
        for b in range(batch_offset, batch_offset + Bsz):
            rows.append(_normal(shape, _rng(wl.seed, name, rnd, layer, b)) * inv_sqrt_n)
        out[name] = torch.stack(rows).to(wl.torch_in_dtype)
    rows = []
    for b in range(batch_offset, batch_offset + Bsz):
        raw = _normal((K, H), _rng(wl.seed, "dt", rnd, layer, b), -2.0, 1.0)
        rows.append(torch.nn.functional.softplus(raw))
    out["dt"] = torch.stack(rows).to(wl.torch_in_dtype)
    return {k: v.contiguous() for k, v in out.items()}


def draw_accept_len(wl: Workload, rnd: int = 0, batch: Optional[int] = None,
                    batch_offset: int = 0) -> torch.Tensor:
    """Accepted draft tokens per sequence for one round, ``int32[batch]``,
    shared by every layer of that round."""
    Bsz = wl.batch if batch is None else batch
    K = wl.ntok
    rng = _rng(wl.seed, "accept", rnd, 0)
    total = batch_offset + Bsz
    if wl.accept == "all":
        full = torch.full((total,), K, dtype=torch.int32)
    elif wl.accept == "uniform":
        full = torch.from_numpy(rng.integers(0, K + 1, total)).to(torch.int32)
    elif wl.accept == "geometric":
        # trials up to and including the first rejection, minus one = tokens accepted
        t = rng.geometric(0.3, total) - 1
        full = torch.from_numpy(np.minimum(t, K)).to(torch.int32)
    else:
        raise ValueError(f"unknown accept recipe {wl.accept!r}")
    return full[batch_offset:batch_offset + Bsz].contiguous()


def draw_layer_round(wl: Workload, rnd: int = 0, layer: int = 0, batch: Optional[int] = None,
                     batch_offset: int = 0) -> Dict[str, torch.Tensor]:
    """Everything one layer-call of one round needs, as CPU tensors."""
    d = draw_params(wl, layer, batch, batch_offset)
    d.update(draw_tokens(wl, rnd, layer, batch, batch_offset))
    d["accept_len"] = draw_accept_len(wl, rnd, batch, batch_offset)
    return d


def custom_workload(batch: int, nheads: int, headdim: int, dstate: int, ngroups: int, ntok: int,
                    in_dtype: str = F32, seed: int = 1234, accept: str = "uniform") -> Workload:
    """An ad-hoc workload with the standard distributions (for shape sweeps)."""
    return Workload(f"custom_b{batch}_h{nheads}_p{headdim}_n{dstate}_g{ngroups}_k{ntok}_{in_dtype}",
                    seed, batch, 1, nheads, headdim, dstate, ngroups, ntok, in_dtype, accept)


# --------------------------------------------------------------------------- acceptance step inputs

@dataclasses.dataclass(frozen=True)
class AcceptWorkload:
    """Synthetic verifier / draft logits for the acceptance step.

    Per sequence: K draft tokens drawn uniformly from the vocabulary; a shared
    N(0, 1) base over the vocabulary for each position (the two models see
    the same context); draft logits = base + ``spike`` at the draft token (the
    draft proposed its most likely token); verifier logits = base + 0.5 N(0, 1)
    + ``spike`` at a peak token that is the draft token with probability
    ``agree`` and a uniformly drawn token otherwise; the bonus position K has
    a uniformly drawn peak. ``spike`` defaults to ln(V) + 1, which puts about
    two thirds of the probability on the peak token at any vocabulary size.
    Uniforms for the sampling rule are U[0, 1) fp32, K + 1 per sequence.
    """

    name: str
    seed: int
    batch: int
    ntok: int  # K
    vocab: int  # V
    logit_dtype: str
    agree: float = 0.8
    spike: Optional[float] = None
    description: str = ""

    @property
    def torch_logit_dtype(self) -> torch.dtype:
        return _TORCH_DTYPE[self.logit_dtype]

    def logit_bytes(self) -> int:
        return 4 if self.logit_dtype == F32 else 2

    def peak(self) -> float:
        return math.log(self.vocab) + 1.0 if self.spike is None else self.spike


ACCEPT_WORKLOADS: Dict[int, AcceptWorkload] = {
    0: AcceptWorkload("accept_tiny_b3_k4_v1000_fp32", 100, 3, 4, 1000, F32,
                      description="tiny oracle case: 3 sequences, K=4, a 1000-token vocabulary, fp32 logits"),
    1: AcceptWorkload("accept_llama3_vocab_b64_k8_v128256_bf16", 103, 64, 8, 128256, BF16,
                      description="batched speculative serving: 64 sequences, K=8, Llama-3 vocabulary "
                                  "(128256), bf16 logits"),
}


def custom_accept_workload(batch: int, ntok: int, vocab: int, logit_dtype: str = F32, seed: int = 4321,
                           agree: float = 0.8, spike: Optional[float] = None) -> AcceptWorkload:
    """An ad-hoc acceptance workload with the standard recipe."""
    return AcceptWorkload(f"accept_custom_b{batch}_k{ntok}_v{vocab}_{logit_dtype}", seed, batch, ntok, vocab,
                          logit_dtype, agree, spike)


def draw_accept_inputs(aw: AcceptWorkload, batch: Optional[int] = None,
                       batch_offset: int = 0) -> Dict[str, torch.Tensor]:
    """``target_logits[batch][K+1][V]``, ``draft_logits[batch][K][V]`` (the
    workload's logit dtype), ``draft_tokens[batch][K]`` (int32) and
    ``uniform[batch][K+1]`` (fp32), as CPU tensors. A sequence's values do not
    depend on ``batch`` / ``batch_offset``."""
    Bsz = aw.batch if batch is None else batch
    K, V = aw.ntok, aw.vocab
    spike = aw.peak()
    tl, ql, dr, un = [], [], [], []
    for b in range(batch_offset, batch_offset + Bsz):
        drafts = torch.from_numpy(_rng(aw.seed, "draft", 0, 0, b).integers(0, V, K))
        base = _normal((K + 1, V), _rng(aw.seed, "base", 0, 0, b))
        agree = _uniform((K,), _rng(aw.seed, "agree", 0, 0, b))
        other = torch.from_numpy(_rng(aw.seed, "peak", 0, 0, b).integers(0, V, K + 1))
        peak = other.clone()
        peak[:K] = torch.where(agree < aw.agree, drafts, other[:K])
        q = base[:K].clone()
        q[torch.arange(K), drafts] += spike
        p = base + 0.5 * _normal((K + 1, V), _rng(aw.seed, "tnoise", 0, 0, b))
        p[torch.arange(K + 1), peak] += spike
        u = _uniform((K + 1,), _rng(aw.seed, "uniform", 0, 0, b))
        tl.append(p.to(aw.torch_logit_dtype))
        ql.append(q.to(aw.torch_logit_dtype))
        dr.append(drafts.to(torch.int32))
        un.append(u)
    return {"target_logits": torch.stack(tl).contiguous(), "draft_logits": torch.stack(ql).contiguous(),
            "draft_tokens": torch.stack(dr).contiguous(), "uniform": torch.stack(un).contiguous()}
