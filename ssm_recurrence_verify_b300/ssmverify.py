"""Python binding of libssmverify (ctypes): argument marshalling only.

Every step of the path runs in the CUDA library; this module checks torch
tensors (device, dtype, shape, contiguity), fills the C descriptor and calls
the C ABI on the current CUDA stream. If the library is not built the first
call raises: there is no fallback.

Layouts (see ``include/ssmverify.h``): ``state[b][H][P][N]`` fp32,
``x[b][K][H][P]``, ``B``/``C[b][K][G][N]``, ``dt[b][K][H]`` (fp32 or bf16, all
the same), ``A``/``D[H]`` fp32, ``y[b][K][H][P]`` fp32, ``accept_len[b]`` int32.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libssmverify.so")

SSM_F32 = 0
SSM_BF16 = 1
SSM_OK = 0
SSM_ERR_NULL = 1
SSM_ERR_SHAPE = 2
SSM_ERR_UNSUPPORTED = 3
SSM_ERR_ALIGN = 4
SSM_ERR_ALIAS = 5
SSM_ERR_CUDA = 6
SSM_STATUS_BAD_ACCEPT_LEN = 1
SSM_STATUS_TIMEOUT = 2
SSM_STATUS_BAD_TOKEN = 4
SSM_STATUS_BAD_SLOT = 8
SSM_ACCEPT_MAX_NTOK = 32
SSM_ACCEPT_MAX_VOCAB = 1 << 28
SSM_PREFILL_SCRATCH_BYTES = 64 << 20

EXPORTS = ("ssm_verify", "ssm_commit", "ssm_verify_commit", "ssm_commit_verify", "ssm_step",
           "ssm_verify_pool", "ssm_commit_pool", "ssm_verify_commit_pool", "ssm_commit_verify_pool", "ssm_step_pool",
           "ssm_prefill", "ssm_prefill_workspace_bytes", "ssm_prefill_scratch", "ssm_selftest_wait_timeout", "ssm_accept_greedy",
           "ssm_accept_sample", "ssm_copy_from_host", "ssm_copy_from_host_n", "ssm_strerror", "ssm_last_cuda_error",
           "ssm_version")
SSM_COPY_MAX_SEGMENTS = 8


class SsmDesc(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("nheads", ctypes.c_int32), ("headdim", ctypes.c_int32),
                ("dstate", ctypes.c_int32), ("ngroups", ctypes.c_int32), ("ntok", ctypes.c_int32),
                ("in_dtype", ctypes.c_int32), ("nlayers", ctypes.c_int32)]


class PoolDesc(ctypes.Structure):
    _fields_ = [("states", ctypes.c_void_p), ("slot", ctypes.c_void_p), ("nslots", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class CopySegment(ctypes.Structure):
    _fields_ = [("dst", ctypes.c_void_p), ("src", ctypes.c_void_p), ("bytes", ctypes.c_int64)]


class AcceptDesc(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("ntok", ctypes.c_int32), ("vocab", ctypes.c_int32),
                ("logit_dtype", ctypes.c_int32)]


class SsmError(ValueError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"libssmverify error {code}: {msg}")
        self.code = code


_lib = None


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Load (once) and return the CUDA library; raise if it is missing."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libssmverify is not built ({p} missing); run "
                           "`python -m ssm_recurrence_verify_b300.build`")
    lib = ctypes.CDLL(p)
    vp, dp = ctypes.c_void_p, ctypes.POINTER(SsmDesc)
    lib.ssm_verify.argtypes = [dp] + [vp] * 10
    lib.ssm_commit.argtypes = [dp] + [vp] * 8
    lib.ssm_verify_commit.argtypes = [dp] + [vp] * 11
    lib.ssm_commit_verify.argtypes = [dp, vp, ctypes.c_int32] + [vp] * 13
    lib.ssm_step.argtypes = [dp] + [vp] * 10
    lib.ssm_selftest_wait_timeout.argtypes = [vp, vp]
    ap = ctypes.POINTER(AcceptDesc)
    lib.ssm_accept_greedy.argtypes = [ap] + [vp] * 6
    lib.ssm_accept_sample.argtypes = [ap] + [vp] * 8
    pp = ctypes.POINTER(PoolDesc)
    lib.ssm_verify_pool.argtypes = [dp, pp] + [vp] * 9
    lib.ssm_commit_pool.argtypes = [dp, pp] + [vp] * 7
    lib.ssm_verify_commit_pool.argtypes = [dp, pp] + [vp] * 10
    lib.ssm_commit_verify_pool.argtypes = [dp, pp, ctypes.c_int32] + [vp] * 13
    lib.ssm_step_pool.argtypes = [dp, pp] + [vp] * 9
    lib.ssm_prefill.argtypes = [dp, pp] + [vp] * 8 + [ctypes.c_int64, vp, vp]
    lib.ssm_prefill_scratch.argtypes = [dp, pp] + [vp] * 9
    lib.ssm_copy_from_host.argtypes = [vp, vp, ctypes.c_int64, vp]
    lib.ssm_copy_from_host_n.argtypes = [ctypes.POINTER(CopySegment), ctypes.c_int32, vp]
    lib.ssm_prefill_workspace_bytes.argtypes = [dp]
    lib.ssm_prefill_workspace_bytes.restype = ctypes.c_int64
    for f in ("ssm_verify", "ssm_commit", "ssm_verify_commit", "ssm_commit_verify", "ssm_step",
              "ssm_verify_pool", "ssm_commit_pool", "ssm_verify_commit_pool", "ssm_commit_verify_pool",
              "ssm_step_pool", "ssm_prefill", "ssm_prefill_scratch", "ssm_selftest_wait_timeout", "ssm_accept_greedy", "ssm_accept_sample",
              "ssm_copy_from_host", "ssm_copy_from_host_n", "ssm_last_cuda_error", "ssm_version"):
        getattr(lib, f).restype = ctypes.c_int
    lib.ssm_strerror.argtypes = [ctypes.c_int]
    lib.ssm_strerror.restype = ctypes.c_char_p
    if path is None:
        _lib = lib
    return lib


def strerror(code: int) -> str:
    return load_library().ssm_strerror(code).decode()


def _check(code: int):
    if code != SSM_OK:
        msg = strerror(code)
        if code == SSM_ERR_CUDA:
            msg += f" (cudaError {load_library().ssm_last_cuda_error()})"
        raise SsmError(code, msg)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _in_dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return SSM_F32
    if t.dtype == torch.bfloat16:
        return SSM_BF16
    raise ValueError(f"x/B/C/dt must be float32 or bfloat16, got {t.dtype}")


def make_desc(state_shape, x_shape, B_shape, in_dtype: int) -> SsmDesc:
    bsz, H, P, N = state_shape
    K = x_shape[1]
    G = B_shape[2]
    return SsmDesc(bsz, H, P, N, G, K, in_dtype, 0)


def _validate(state, x, B, C, dt, A, D, accept_len, y, pooled=False):
    """Check the tensors of one call; with `pooled`, `state` is a pool
    [nslots][H][P][N] and the batch comes from x. A 5-D state
    [L][batch][H][P][N] makes the call a layer stack: x, B, C, dt, y then
    carry the same leading [L], A and D are [L][H], accept_len stays [batch]."""
    tensors = {"state": state, "x": x, "B": B, "dt": dt, "A": A}
    for k, v in (("C", C), ("D", D), ("accept_len", accept_len), ("y", y)):
        if v is not None:
            tensors[k] = v
    dev = state.device
    for k, v in tensors.items():
        if not v.is_cuda or v.device != dev:
            raise ValueError(f"{k} must be a CUDA tensor on {dev}")
        if not v.is_contiguous():
            raise ValueError(f"{k} must be contiguous")
    if state.dtype != torch.float32 or state.dim() not in (4, 5):
        raise ValueError("state must be float32 [batch][H][P][N] or [L][batch][H][P][N]"
                         + (" (a pool: [nslots] or [L][nslots] in place of batch)" if pooled else ""))
    lead = tuple(state.shape[:-4])  # (L,) for a layer stack
    H, P, N = state.shape[-3:]
    bsz = x.shape[len(lead)] if pooled else state.shape[-4]
    nd = len(lead) + 4
    if x.dim() != nd or tuple(x.shape[:len(lead)]) != lead or x.shape[-4] != bsz or tuple(x.shape[-2:]) != (H, P):
        raise ValueError(f"x must be {list(lead)}[batch][K][H][P] = {list(lead)}[{bsz}][K][{H}][{P}], "
                         f"got {tuple(x.shape)}")
    K = x.shape[-3]
    if B.dim() != nd or tuple(B.shape[:len(lead)]) != lead or tuple(B.shape[-4:-2]) != (bsz, K) or B.shape[-1] != N:
        raise ValueError(f"B must be {list(lead)}[batch][K][G][N], got {tuple(B.shape)}")
    G = B.shape[-2]
    if C is not None and tuple(C.shape) != tuple(B.shape):
        raise ValueError("C must have B's shape")
    if tuple(dt.shape) != lead + (bsz, K, H):
        raise ValueError(f"dt must be {list(lead)}[batch][K][H] = {list(lead + (bsz, K, H))}, got {tuple(dt.shape)}")
    dts = {x.dtype, B.dtype, dt.dtype} | ({C.dtype} if C is not None else set())
    if len(dts) != 1:
        raise ValueError("x, B, C, dt must share one dtype")
    for k, v in (("A", A), ("D", D)):
        if v is not None and (v.dtype != torch.float32 or tuple(v.shape) != lead + (H,)):
            raise ValueError(f"{k} must be float32 {list(lead)}[H]")
    if accept_len is not None and (accept_len.dtype != torch.int32 or tuple(accept_len.shape) != (bsz,)):
        raise ValueError("accept_len must be int32 [batch]")
    if y is not None and (y.dtype != torch.float32 or tuple(y.shape) != tuple(x.shape)):
        raise ValueError(f"y must be float32 {list(lead)}[batch][K][H][P]")
    return SsmDesc(bsz, H, P, N, G, K, _in_dtype(x), lead[0] if lead else 0), G


def _new_y(state, x):
    return torch.empty(tuple(x.shape), dtype=torch.float32, device=state.device)


def verify(state, x, B, C, dt, A, D, y=None, dev_status=None, stream=None) -> torch.Tensor:
    """y for all K draft tokens from the cached state; the state is only read."""
    y = _new_y(state, x) if y is None else y
    desc, _ = _validate(state, x, B, C, dt, A, D, None, y)
    _check(load_library().ssm_verify(ctypes.byref(desc), _ptr(state), _ptr(x), _ptr(B), _ptr(C), _ptr(dt), _ptr(A),
                                     _ptr(D), _ptr(y), _ptr(dev_status), _stream(stream)))
    return y


def commit(state, x, B, dt, A, accept_len, dev_status=None, stream=None) -> None:
    """Advance the state in place by each sequence's accepted prefix (j = 0: unchanged)."""
    desc, _ = _validate(state, x, B, None, dt, A, None, accept_len, None)
    _check(load_library().ssm_commit(ctypes.byref(desc), _ptr(state), _ptr(x), _ptr(B), _ptr(dt), _ptr(A),
                                     _ptr(accept_len), _ptr(dev_status), _stream(stream)))


def verify_commit(state, x, B, C, dt, A, D, accept_len, y=None, dev_status=None, stream=None) -> torch.Tensor:
    """Fused verify + commit: y for all K tokens, state <- h_j in place."""
    y = _new_y(state, x) if y is None else y
    desc, _ = _validate(state, x, B, C, dt, A, D, accept_len, y)
    _check(load_library().ssm_verify_commit(ctypes.byref(desc), _ptr(state), _ptr(x), _ptr(B), _ptr(C), _ptr(dt),
                                            _ptr(A), _ptr(D), _ptr(accept_len), _ptr(y), _ptr(dev_status),
                                            _stream(stream)))
    return y


def commit_verify(state, x_prev, B_prev, dt_prev, accept_len_prev, x, B, C, dt, A, D, y=None, dev_status=None,
                  stream=None) -> torch.Tensor:
    """Commit the previous round's accepted prefix (x_prev / B_prev / dt_prev,
    accept_len_prev) into the state in place, then verify the new drafts from
    it: y for every new token. Equals commit(...) then verify(...)."""
    y = _new_y(state, x) if y is None else y
    desc, G = _validate(state, x, B, C, dt, A, D, None, y)
    lead = tuple(state.shape[:-4])
    bsz, H, P, N = state.shape[-4:]
    if (x_prev.dim() != len(lead) + 4 or tuple(x_prev.shape[:len(lead)]) != lead or x_prev.shape[-4] != bsz
            or tuple(x_prev.shape[-2:]) != (H, P)):
        raise ValueError(f"x_prev must be {list(lead)}[batch][K_prev][H][P], got {tuple(x_prev.shape)}")
    kp = x_prev.shape[-3]
    for k, v, shape in (("B_prev", B_prev, lead + (bsz, kp, G, N)), ("dt_prev", dt_prev, lead + (bsz, kp, H))):
        if tuple(v.shape) != shape:
            raise ValueError(f"{k} must be {list(shape)}, got {tuple(v.shape)}")
    for k, v in (("x_prev", x_prev), ("B_prev", B_prev), ("dt_prev", dt_prev)):
        if v.dtype != x.dtype or not v.is_cuda or v.device != state.device or not v.is_contiguous():
            raise ValueError(f"{k} must be a contiguous {x.dtype} CUDA tensor on {state.device}")
    if accept_len_prev.dtype != torch.int32 or tuple(accept_len_prev.shape) != (bsz,) or not accept_len_prev.is_cuda:
        raise ValueError("accept_len_prev must be int32 [batch] on the GPU")
    _check(load_library().ssm_commit_verify(ctypes.byref(desc), _ptr(state), kp, _ptr(x_prev), _ptr(B_prev),
                                            _ptr(dt_prev), _ptr(accept_len_prev), _ptr(x), _ptr(B), _ptr(C), _ptr(dt),
                                            _ptr(A), _ptr(D), _ptr(y), _ptr(dev_status), _stream(stream)))
    return y


def selftest_wait_timeout(dev_status, stream=None) -> None:
    """Launch the bounded-wait self-test: after about one second the device
    ORs SSM_STATUS_TIMEOUT into `dev_status` (int32 CUDA tensor, one word)."""
    if not (dev_status.is_cuda and dev_status.dtype == torch.int32 and dev_status.numel() >= 1):
        raise ValueError("dev_status must be an int32 CUDA tensor")
    _check(load_library().ssm_selftest_wait_timeout(_ptr(dev_status), _stream(stream)))


def step(state, x, B, C, dt, A, D, y=None, dev_status=None, stream=None) -> torch.Tensor:
    """Plain decode of one token (K = 1): y, and the state advanced in place."""
    y = _new_y(state, x) if y is None else y
    desc, _ = _validate(state, x, B, C, dt, A, D, None, y)
    _check(load_library().ssm_step(ctypes.byref(desc), _ptr(state), _ptr(x), _ptr(B), _ptr(C), _ptr(dt), _ptr(A),
                                   _ptr(D), _ptr(y), _ptr(dev_status), _stream(stream)))
    return y


# ----------------------------------------------------------------------------- acceptance

def _accept_validate(target_logits, draft_tokens, draft_logits, uniform, accept_len, next_token):
    dev = target_logits.device
    tensors = {"target_logits": target_logits, "draft_tokens": draft_tokens}
    for k, v in (("draft_logits", draft_logits), ("uniform", uniform), ("accept_len", accept_len),
                 ("next_token", next_token)):
        if v is not None:
            tensors[k] = v
    for k, v in tensors.items():
        if not v.is_cuda or v.device != dev:
            raise ValueError(f"{k} must be a CUDA tensor on {dev}")
        if not v.is_contiguous():
            raise ValueError(f"{k} must be contiguous")
    if target_logits.dim() != 3:
        raise ValueError("target_logits must be [batch][K+1][V]")
    bsz, K1, V = target_logits.shape
    K = K1 - 1
    if target_logits.dtype == torch.float32:
        dt = SSM_F32
    elif target_logits.dtype == torch.bfloat16:
        dt = SSM_BF16
    else:
        raise ValueError(f"logits must be float32 or bfloat16, got {target_logits.dtype}")
    if draft_tokens.dtype != torch.int32 or tuple(draft_tokens.shape) != (bsz, K):
        raise ValueError(f"draft_tokens must be int32 [batch][K] = [{bsz}][{K}]")
    if draft_logits is not None and (draft_logits.dtype != target_logits.dtype
                                     or tuple(draft_logits.shape) != (bsz, K, V)):
        raise ValueError(f"draft_logits must be {target_logits.dtype} [batch][K][V] = [{bsz}][{K}][{V}]")
    if uniform is not None and (uniform.dtype != torch.float32 or tuple(uniform.shape) != (bsz, K1)):
        raise ValueError(f"uniform must be float32 [batch][K+1] = [{bsz}][{K1}]")
    for k, v in (("accept_len", accept_len), ("next_token", next_token)):
        if v is not None and (v.dtype != torch.int32 or tuple(v.shape) != (bsz,)):
            raise ValueError(f"{k} must be int32 [batch]")
    return AcceptDesc(bsz, K, V, dt)


def _accept_outputs(target_logits, accept_len, next_token):
    bsz = target_logits.shape[0]
    dev = target_logits.device
    if accept_len is None:
        accept_len = torch.empty(bsz, dtype=torch.int32, device=dev)
    if next_token is None:
        next_token = torch.empty(bsz, dtype=torch.int32, device=dev)
    return accept_len, next_token


def accept_greedy(target_logits, draft_tokens, accept_len=None, next_token=None, dev_status=None,
                  stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Greedy acceptance on the device: ``(accept_len, next_token)``, int32
    [batch] each. target_logits [batch][K+1][V] (fp32 or bf16), draft_tokens
    int32 [batch][K]."""
    accept_len, next_token = _accept_outputs(target_logits, accept_len, next_token)
    desc = _accept_validate(target_logits, draft_tokens, None, None, accept_len, next_token)
    _check(load_library().ssm_accept_greedy(ctypes.byref(desc), _ptr(target_logits), _ptr(draft_tokens),
                                            _ptr(accept_len), _ptr(next_token), _ptr(dev_status), _stream(stream)))
    return accept_len, next_token


def accept_sample(target_logits, draft_logits, draft_tokens, uniform, accept_len=None, next_token=None,
                  dev_status=None, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Speculative sampling on the device: ``(accept_len, next_token)``.
    draft_logits [batch][K][V] (the target's dtype), uniform fp32 [batch][K+1]."""
    accept_len, next_token = _accept_outputs(target_logits, accept_len, next_token)
    desc = _accept_validate(target_logits, draft_tokens, draft_logits, uniform, accept_len, next_token)
    _check(load_library().ssm_accept_sample(ctypes.byref(desc), _ptr(target_logits), _ptr(draft_logits),
                                            _ptr(draft_tokens), _ptr(uniform), _ptr(accept_len), _ptr(next_token),
                                            _ptr(dev_status), _stream(stream)))
    return accept_len, next_token


# ----------------------------------------------------------------------------- state pool and prefill

def _pool(states: torch.Tensor, slot: Optional[torch.Tensor], bsz: int):
    """The C pool descriptor: `states` [nslots][H][P][N] fp32 CUDA (a layer
    stack: [L][nslots][H][P][N]), `slot` int32 [batch] CUDA (None: sequence b
    uses slot b), the same slot in every layer."""
    if not states.is_cuda or states.dtype != torch.float32 or states.dim() not in (4, 5) or \
            not states.is_contiguous():
        raise ValueError("pool states must be a contiguous float32 CUDA tensor [nslots][H][P][N] "
                         "or [L][nslots][H][P][N]")
    if slot is not None:
        if not slot.is_cuda or slot.device != states.device or slot.dtype != torch.int32 or \
                tuple(slot.shape) != (bsz,) or not slot.is_contiguous():
            raise ValueError(f"slot must be a contiguous int32 CUDA tensor [{bsz}] on {states.device}")
    return PoolDesc(states.data_ptr(), None if slot is None else slot.data_ptr(), states.shape[-4], 0)


def verify_pool(states, slot, x, B, C, dt, A, D, y=None, dev_status=None, stream=None) -> torch.Tensor:
    """verify on the pool slots `slot` of `states` (read only)."""
    y = _new_y(states, x) if y is None else y
    desc, _ = _validate(states, x, B, C, dt, A, D, None, y, pooled=True)
    pool = _pool(states, slot, desc.batch)
    _check(load_library().ssm_verify_pool(ctypes.byref(desc), ctypes.byref(pool), _ptr(x), _ptr(B), _ptr(C),
                                          _ptr(dt), _ptr(A), _ptr(D), _ptr(y), _ptr(dev_status), _stream(stream)))
    return y


def commit_pool(states, slot, x, B, dt, A, accept_len, dev_status=None, stream=None) -> None:
    """commit into the pool slots."""
    desc, _ = _validate(states, x, B, None, dt, A, None, accept_len, None, pooled=True)
    pool = _pool(states, slot, desc.batch)
    _check(load_library().ssm_commit_pool(ctypes.byref(desc), ctypes.byref(pool), _ptr(x), _ptr(B), _ptr(dt),
                                          _ptr(A), _ptr(accept_len), _ptr(dev_status), _stream(stream)))


def verify_commit_pool(states, slot, x, B, C, dt, A, D, accept_len, y=None, dev_status=None,
                       stream=None) -> torch.Tensor:
    """verify_commit on the pool slots."""
    y = _new_y(states, x) if y is None else y
    desc, _ = _validate(states, x, B, C, dt, A, D, accept_len, y, pooled=True)
    pool = _pool(states, slot, desc.batch)
    _check(load_library().ssm_verify_commit_pool(ctypes.byref(desc), ctypes.byref(pool), _ptr(x), _ptr(B), _ptr(C),
                                                 _ptr(dt), _ptr(A), _ptr(D), _ptr(accept_len), _ptr(y),
                                                 _ptr(dev_status), _stream(stream)))
    return y


def commit_verify_pool(states, slot, x_prev, B_prev, dt_prev, accept_len_prev, x, B, C, dt, A, D, y=None,
                       dev_status=None, stream=None) -> torch.Tensor:
    """commit_verify on the pool slots."""
    y = _new_y(states, x) if y is None else y
    desc, G = _validate(states, x, B, C, dt, A, D, None, y, pooled=True)
    bsz = desc.batch
    lead = tuple(states.shape[:-4])
    H, P, N = states.shape[-3:]
    kp = x_prev.shape[-3] if x_prev.dim() >= 3 else 0
    for k, v, shape in (("x_prev", x_prev, lead + (bsz, kp, H, P)), ("B_prev", B_prev, lead + (bsz, kp, G, N)),
                        ("dt_prev", dt_prev, lead + (bsz, kp, H))):
        if tuple(v.shape) != shape or v.dtype != x.dtype or not v.is_cuda or not v.is_contiguous():
            raise ValueError(f"{k} must be a contiguous {x.dtype} CUDA tensor {list(shape)}")
    if accept_len_prev.dtype != torch.int32 or tuple(accept_len_prev.shape) != (bsz,) or not accept_len_prev.is_cuda:
        raise ValueError("accept_len_prev must be int32 [batch] on the GPU")
    pool = _pool(states, slot, bsz)
    _check(load_library().ssm_commit_verify_pool(ctypes.byref(desc), ctypes.byref(pool), kp, _ptr(x_prev),
                                                 _ptr(B_prev), _ptr(dt_prev), _ptr(accept_len_prev), _ptr(x), _ptr(B),
                                                 _ptr(C), _ptr(dt), _ptr(A), _ptr(D), _ptr(y), _ptr(dev_status),
                                                 _stream(stream)))
    return y


def step_pool(states, slot, x, B, C, dt, A, D, y=None, dev_status=None, stream=None) -> torch.Tensor:
    """step (K = 1) on the pool slots."""
    y = _new_y(states, x) if y is None else y
    desc, _ = _validate(states, x, B, C, dt, A, D, None, y, pooled=True)
    pool = _pool(states, slot, desc.batch)
    _check(load_library().ssm_step_pool(ctypes.byref(desc), ctypes.byref(pool), _ptr(x), _ptr(B), _ptr(C), _ptr(dt),
                                        _ptr(A), _ptr(D), _ptr(y), _ptr(dev_status), _stream(stream)))
    return y


def prefill_workspace_bytes(states, x, B, C, dt, A, D) -> int:
    """Workspace (bytes) that prefill would use for these shapes (0: none)."""
    desc, _ = _validate(states, x, B, C, dt, A, D, None, None, pooled=True)
    return int(load_library().ssm_prefill_workspace_bytes(ctypes.byref(desc)))


def prefill(states, slot, x, B, C, dt, A, D, y=None, workspace=None, dev_status=None,
            stream=None) -> torch.Tensor:
    """Run the prompt x/B/C/dt [batch][T]... from each sequence's cached
    state (pool slot), write y for every prompt token and leave the final
    state in the slot. `workspace` (a CUDA tensor) enables the chunked form;
    by default it is allocated here at the size the library asks for."""
    y = _new_y(states, x) if y is None else y
    desc, _ = _validate(states, x, B, C, dt, A, D, None, y, pooled=True)
    pool = _pool(states, slot, desc.batch)
    lib = load_library()
    if workspace is None:
        nbytes = int(lib.ssm_prefill_workspace_bytes(ctypes.byref(desc)))
        workspace = torch.empty(max(nbytes, 0) // 4, dtype=torch.float32, device=states.device) if nbytes > 0 else None
    if workspace is not None and (not workspace.is_cuda or not workspace.is_contiguous()):
        raise ValueError("workspace must be a contiguous CUDA tensor")
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.ssm_prefill(ctypes.byref(desc), ctypes.byref(pool), _ptr(x), _ptr(B), _ptr(C), _ptr(dt), _ptr(A),
                           _ptr(D), _ptr(y), _ptr(workspace), wbytes, _ptr(dev_status), _stream(stream)))
    return y


def prefill_scratch(states, slot, x, B, C, dt, A, D, y=None, dev_status=None, stream=None) -> torch.Tensor:
    """prefill with the library's fixed device scratch as the workspace
    (the library allocates nothing for it; y is allocated here only when the
    caller passes none). For callers that cannot allocate device memory.
    Calls in one CUDA context that may overlap on the device share the
    scratch and race: order them on one stream. The chunk length is limited
    to those whose workspace fits in SSM_PREFILL_SCRATCH_BYTES, else the
    one-pass form runs."""
    y = _new_y(states, x) if y is None else y
    desc, _ = _validate(states, x, B, C, dt, A, D, None, y, pooled=True)
    pool = _pool(states, slot, desc.batch)
    _check(load_library().ssm_prefill_scratch(ctypes.byref(desc), ctypes.byref(pool), _ptr(x), _ptr(B), _ptr(C),
                                              _ptr(dt), _ptr(A), _ptr(D), _ptr(y), _ptr(dev_status), _stream(stream)))
    return y


def copy_from_host(dst: torch.Tensor, src: torch.Tensor, stream=None) -> torch.Tensor:
    """dst <- src, from a page-locked host tensor to a CUDA tensor of the same
    size, with the SMs reading the host memory (asynchronous on the stream)."""
    if dst.numel() * dst.element_size() != src.numel() * src.element_size():
        raise ValueError("dst and src must have the same number of bytes")
    if not dst.is_cuda or src.is_cuda or not src.is_pinned():
        raise ValueError("dst must be a CUDA tensor and src a page-locked (pinned) host tensor")
    if not dst.is_contiguous() or not src.is_contiguous():
        raise ValueError("dst and src must be contiguous")
    _check(load_library().ssm_copy_from_host(_ptr(dst), _ptr(src), dst.numel() * dst.element_size(),
                                             _stream(stream)))
    return dst


def copy_from_host_n(pairs, stream=None) -> None:
    """Several copies from page-locked host tensors to CUDA tensors of the same
    size, ``pairs`` = [(dst, src), ...] (at most SSM_COPY_MAX_SEGMENTS), in
    one launch (asynchronous on the stream)."""
    if len(pairs) > SSM_COPY_MAX_SEGMENTS:
        raise ValueError(f"at most {SSM_COPY_MAX_SEGMENTS} segments")
    segs = (CopySegment * max(1, len(pairs)))()
    for i, (dst, src) in enumerate(pairs):
        if dst.numel() * dst.element_size() != src.numel() * src.element_size():
            raise ValueError("dst and src must have the same number of bytes")
        if dst.numel() == 0:  # nothing to copy (an empty tensor reports no page-locked storage)
            segs[i] = CopySegment(None, None, 0)
            continue
        if not dst.is_cuda or src.is_cuda or not src.is_pinned():
            raise ValueError("dst must be a CUDA tensor and src a page-locked (pinned) host tensor")
        if not dst.is_contiguous() or not src.is_contiguous():
            raise ValueError("dst and src must be contiguous")
        segs[i] = CopySegment(dst.data_ptr(), src.data_ptr(), dst.numel() * dst.element_size())
    _check(load_library().ssm_copy_from_host_n(segs, len(pairs), _stream(stream)))
