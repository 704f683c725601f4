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

Every tensor is drawn on the CPU from its own ``torch.Generator`` whose seed is
a fixed function of (workload seed, tensor kind, round, layer), so any one
layer or round can be regenerated without drawing the others. Values are
rounded to bf16 on the CPU (round-to-nearest-even) where the workload says so.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import torch

F32 = "f32"
BF16 = "bf16"

_TORCH_DTYPE = {F32: torch.float32, BF16: torch.bfloat16}

# tensor kinds, part of every per-tensor seed
_KIND = {"A": 1, "D": 2, "state0": 3, "x": 4, "B": 5, "C": 6, "dt": 7, "accept": 8}


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


def _gen(seed: int, kind: str, rnd: int = 0, layer: int = 0) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed((seed << 40) ^ (_KIND[kind] << 32) ^ (rnd << 16) ^ layer)
    return g


def _normal(shape, gen: torch.Generator, mean: float = 0.0, std: float = 1.0) -> torch.Tensor:
    t = torch.empty(shape, dtype=torch.float32)
    t.normal_(mean, std, generator=gen)
    return t


def draw_params(wl: Workload, layer: int = 0, batch: Optional[int] = None,
                batch_offset: int = 0) -> Dict[str, torch.Tensor]:
    """Per-layer parameters and cached state: ``A[H]``, ``D[H]`` (fp32) and
    ``state0[batch][H][P][N]`` (fp32). ``batch``/``batch_offset`` select a
    slice of the sequences; a sequence's state does not depend on them."""
    Bsz = wl.batch if batch is None else batch
    H, P, N = wl.nheads, wl.headdim, wl.dstate
    u = torch.empty(H, dtype=torch.float32)
    u.uniform_(0.0, math.log(16.0), generator=_gen(wl.seed, "A", 0, layer))
    A = -torch.exp(u)
    D = _normal((H,), _gen(wl.seed, "D", 0, layer))
    state0 = torch.empty((Bsz, H, P, N), dtype=torch.float32)
    for i, b in enumerate(range(batch_offset, batch_offset + Bsz)):
        state0[i].normal_(0.0, 0.1, generator=_seq_gen(wl.seed, "state0", 0, layer, b))
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
            rows.append(_normal(shape, _seq_gen(wl.seed, name, rnd, layer, b)) * inv_sqrt_n)
        out[name] = torch.stack(rows).to(wl.torch_in_dtype)
    rows = []
    for b in range(batch_offset, batch_offset + Bsz):
        raw = _normal((K, H), _seq_gen(wl.seed, "dt", rnd, layer, b), -2.0, 1.0)
        rows.append(torch.nn.functional.softplus(raw))
    out["dt"] = torch.stack(rows).to(wl.torch_in_dtype)
    return {k: v.contiguous() for k, v in out.items()}


def _seq_gen(seed: int, kind: str, rnd: int, layer: int, b: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed((seed << 44) ^ (_KIND[kind] << 36) ^ (rnd << 28) ^ (layer << 16) ^ b)
    return g


def draw_accept_len(wl: Workload, rnd: int = 0, batch: Optional[int] = None,
                    batch_offset: int = 0) -> torch.Tensor:
    """Accepted draft tokens per sequence for one round, ``int32[batch]``,
    shared by every layer of that round."""
    Bsz = wl.batch if batch is None else batch
    K = wl.ntok
    g = _gen(wl.seed, "accept", rnd, 0)
    total = batch_offset + Bsz
    if wl.accept == "all":
        full = torch.full((total,), K, dtype=torch.int32)
    elif wl.accept == "uniform":
        full = torch.randint(0, K + 1, (total,), generator=g, dtype=torch.int64).to(torch.int32)
    elif wl.accept == "geometric":
        # trials up to and including the first rejection, minus one = tokens accepted
        t = torch.empty(total, dtype=torch.float64)
        t.geometric_(0.3, generator=g)
        full = torch.clamp(t - 1.0, max=float(K)).to(torch.int32)
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
