"""The C ABI on the host: the library loads, exports what the header
declares, and rejects bad arguments before launching anything.

The fake-pointer cases never reach a launch (every one fails host
validation); they still run only where no CUDA device is present, so that a
validation bug could never hand a fake pointer to a GPU."""
import ctypes
import os
import re
import subprocess

import pytest
import torch

from ssm_recurrence_verify_b300 import build as libbuild
from ssm_recurrence_verify_b300 import ssmverify as sv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ssmverify.h")

no_gpu_only = pytest.mark.skipif(torch.cuda.is_available(), reason="fake-pointer checks run on CPU-only hosts")


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return sv.load_library()


def header_functions():
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(ssm_[a-z_]+)\s*\(", txt)))


def header_defines():
    out = {}
    for m in re.finditer(r"#define\s+(SSM_[A-Z0-9_]+)\s+(\d+)u?", open(HEADER).read()):
        out[m.group(1)] = int(m.group(2))
    return out


def test_header_is_plain_c_and_cxx():
    for lang in ("c", "c++"):
        subprocess.check_call(["gcc", "-fsyntax-only", "-Wall", "-Werror", "-x", lang, HEADER])


def test_exports_every_declared_symbol(lib):
    declared = header_functions()
    assert set(declared) == set(sv.EXPORTS), declared
    out = subprocess.run(["nm", "-D", "--defined-only", libbuild.LIB], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (ssm_[a-z_]+)\b", out))
    for name in declared:
        assert name in exported, name
        assert getattr(lib, name) is not None


def test_constants_match_header(lib):
    d = header_defines()
    for k, v in d.items():
        if hasattr(sv, k):
            assert getattr(sv, k) == v, k
    assert lib.ssm_version() == d["SSM_VERSION"]
    assert ctypes.sizeof(sv.SsmDesc) == 32


def test_strerror(lib):
    for code in range(0, 7):
        s = sv.strerror(code)
        assert isinstance(s, str) and s
    assert sv.strerror(99) == "unknown error code"


def test_product_path_fails_loudly_without_library(tmp_path):
    with pytest.raises(RuntimeError, match="not built"):
        sv.load_library(str(tmp_path / "missing.so"))


# ----------------------------------------------------------------------------- host validation

BASE = 1 << 40  # fake, never dereferenced: every call below fails validation


def desc(**kw):
    d = dict(batch=2, nheads=4, headdim=32, dstate=128, ngroups=2, ntok=3, in_dtype=sv.SSM_BF16, nlayers=0)
    d.update(kw)
    return sv.SsmDesc(**d)


def ptrs(n, start=BASE, gap=1 << 30):
    return [ctypes.c_void_p(start + i * gap) for i in range(n)]


def vc(lib, d, p):
    """ssm_verify_commit(desc, state, x, B, C, dt, A, D, accept_len, y, dev_status, stream)."""
    return lib.ssm_verify_commit(ctypes.byref(d) if d is not None else None, *p, None)


def cv(lib, d, prev_ntok, p):
    """ssm_commit_verify(desc, state, prev_ntok, x_prev, B_prev, dt_prev, accept_len_prev, x, B, C, dt, A,
    D, y, dev_status, stream); p holds the 13 pointers, state first (prev_ntok goes after it)."""
    return lib.ssm_commit_verify(ctypes.byref(d) if d is not None else None, p[0], prev_ntok, *p[1:], None)


@no_gpu_only
def test_null_desc_and_pointers(lib):
    assert vc(lib, None, ptrs(10)) == sv.SSM_ERR_NULL
    for i in range(9):  # state, x, B, C, dt, A, D, accept_len, y are required
        p = ptrs(10)
        p[i] = None
        assert vc(lib, desc(), p) == sv.SSM_ERR_NULL, i
    p = ptrs(10)
    p[9] = None  # dev_status is optional
    # every pointer valid and distinct, but one misaligned -> still rejected before launch
    p[0] = ctypes.c_void_p(BASE + 8)
    assert vc(lib, desc(), p) == sv.SSM_ERR_ALIGN


@no_gpu_only
@pytest.mark.parametrize("field,value,code", [
    ("batch", -1, sv.SSM_ERR_SHAPE), ("nheads", 0, sv.SSM_ERR_SHAPE), ("headdim", 0, sv.SSM_ERR_SHAPE),
    ("ngroups", 3, sv.SSM_ERR_SHAPE), ("ngroups", 0, sv.SSM_ERR_SHAPE), ("ntok", 0, sv.SSM_ERR_SHAPE),
    ("nlayers", -1, sv.SSM_ERR_SHAPE), ("dstate", 96, sv.SSM_ERR_UNSUPPORTED), ("dstate", 512, sv.SSM_ERR_UNSUPPORTED),
    ("dstate", 8, sv.SSM_ERR_UNSUPPORTED), ("in_dtype", 7, sv.SSM_ERR_UNSUPPORTED),
])
def test_shape_errors(lib, field, value, code):
    d = desc(**{field: value})
    p = ptrs(10)
    p[0] = ctypes.c_void_p(BASE + 8)  # also misaligned: the shape check must come first
    assert vc(lib, d, p) == code


@no_gpu_only
def test_alignment_errors(lib):
    for i, off in [(0, 4), (1, 1), (2, 1), (3, 1), (4, 1), (5, 2), (6, 2), (7, 2), (8, 2), (9, 2)]:
        p = ptrs(10)
        p[i] = ctypes.c_void_p(p[i].value + off)
        assert vc(lib, desc(), p) == sv.SSM_ERR_ALIGN, i
    p = ptrs(10)
    p[1] = ctypes.c_void_p(p[1].value + 2)  # 2-byte aligned is enough for bf16 ...
    p[0] = ctypes.c_void_p(p[0].value + 16)
    p[8] = ctypes.c_void_p(p[8].value + 4)
    d = desc(in_dtype=sv.SSM_F32)  # ... but not for fp32 inputs
    assert vc(lib, d, p) == sv.SSM_ERR_ALIGN


@no_gpu_only
def test_alias_errors(lib):
    # state (written) overlapping x
    p = ptrs(10)
    p[1] = ctypes.c_void_p(p[0].value + 64)
    assert vc(lib, desc(), p) == sv.SSM_ERR_ALIAS
    # y (written) overlapping C
    p = ptrs(10)
    p[8] = ctypes.c_void_p(p[3].value + 16)
    assert vc(lib, desc(), p) == sv.SSM_ERR_ALIAS
    # two read-only buffers may overlap (B and C the same): validation passes
    # and, with no CUDA device on this host, the launch itself fails
    p = ptrs(10)
    p[3] = p[2]
    assert vc(lib, desc(), p) == sv.SSM_ERR_CUDA
    assert lib.ssm_last_cuda_error() != 0
    # dev_status inside y
    p = ptrs(10)
    p[9] = ctypes.c_void_p(p[8].value + 4)
    assert vc(lib, desc(), p) == sv.SSM_ERR_ALIAS
    # verify: the state is read only, so it may overlap inputs, but not y
    d = desc()
    q = ptrs(9)
    q[7] = ctypes.c_void_p(q[0].value + 128)
    assert lib.ssm_verify(ctypes.byref(d), *q, None) == sv.SSM_ERR_ALIAS
    q = ptrs(9)
    q[1] = ctypes.c_void_p(q[0].value + 128)  # x inside the read-only state: allowed
    assert lib.ssm_verify(ctypes.byref(d), *q, None) == sv.SSM_ERR_CUDA


@no_gpu_only
def test_entry_specific_rules(lib):
    d = desc()
    p = ptrs(10)
    p[7] = None
    assert vc(lib, d, p) == sv.SSM_ERR_NULL        # verify_commit needs accept_len
    q = ptrs(9)                                   # step: ntok must be 1
    assert lib.ssm_step(ctypes.byref(d), *q, None) == sv.SSM_ERR_SHAPE
    c = ptrs(7)                                   # commit: accept_len required
    c[5] = None
    assert lib.ssm_commit(ctypes.byref(d), *c, None) == sv.SSM_ERR_NULL


@no_gpu_only
def test_empty_batch_is_a_noop(lib):
    d = desc(batch=0)
    assert vc(lib, d, [None] * 10) == sv.SSM_OK
    assert lib.ssm_verify(ctypes.byref(d), *([None] * 9), None) == sv.SSM_OK
    assert lib.ssm_commit(ctypes.byref(d), *([None] * 7), None) == sv.SSM_OK
    assert cv(lib, d, 3, [None] * 13) == sv.SSM_OK
    d1 = desc(batch=0, ntok=1)
    assert lib.ssm_step(ctypes.byref(d1), *([None] * 9), None) == sv.SSM_OK


def test_python_shim_rejects_cpu_tensors():
    t = torch.zeros(1, 2, 16, 16)
    x = torch.zeros(1, 1, 2, 16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        sv.verify(t, x, torch.zeros(1, 1, 1, 16), torch.zeros(1, 1, 1, 16), torch.zeros(1, 1, 2), torch.zeros(2),
                  torch.zeros(2), y=torch.zeros(1, 1, 2, 16))


@no_gpu_only
def test_commit_verify_validation(lib):
    d = desc()
    # state, x_prev, B_prev, dt_prev, accept_len_prev, x, B, C, dt, A, D, y, dev_status
    p = ptrs(13)
    for i in range(12):  # all but dev_status are required
        q = list(p)
        q[i] = None
        assert cv(lib, d, 3, q) == sv.SSM_ERR_NULL, i
    assert cv(lib, d, 0, p) == sv.SSM_ERR_SHAPE          # prev_ntok >= 1
    assert cv(lib, d, -2, p) == sv.SSM_ERR_SHAPE
    q = list(p)
    q[1] = ctypes.c_void_p(q[1].value + 1)                # x_prev misaligned for bf16
    assert cv(lib, d, 3, q) == sv.SSM_ERR_ALIGN
    q = list(p)
    q[0] = ctypes.c_void_p(q[0].value + 8)                # state needs 16 bytes
    assert cv(lib, d, 3, q) == sv.SSM_ERR_ALIGN
    q = list(p)
    q[11] = ctypes.c_void_p(q[2].value + 64)              # y inside B_prev
    assert cv(lib, d, 3, q) == sv.SSM_ERR_ALIAS
    q = list(p)
    q[1] = ctypes.c_void_p(q[0].value + 256)              # x_prev inside the written state
    assert cv(lib, d, 3, q) == sv.SSM_ERR_ALIAS
    q = list(p)
    q[5] = q[1]                                           # the two blocks may share read-only buffers
    assert cv(lib, d, 3, q) == sv.SSM_ERR_CUDA


@no_gpu_only
def test_selftest_validation(lib):
    assert lib.ssm_selftest_wait_timeout(None, None) == sv.SSM_ERR_NULL
    assert lib.ssm_selftest_wait_timeout(ctypes.c_void_p(BASE + 2), None) == sv.SSM_ERR_ALIGN


def adesc(**kw):
    d = dict(batch=2, ntok=3, vocab=1000, logit_dtype=sv.SSM_BF16)
    d.update(kw)
    return sv.AcceptDesc(**d)


def ag(lib, d, p):
    """ssm_accept_greedy(desc, target_logits, draft_tokens, accept_len, next_token, dev_status, stream)."""
    return lib.ssm_accept_greedy(ctypes.byref(d) if d is not None else None, *p, None)


def asa(lib, d, p):
    """ssm_accept_sample(desc, target_logits, draft_logits, draft_tokens, uniform, accept_len, next_token,
    dev_status, stream)."""
    return lib.ssm_accept_sample(ctypes.byref(d) if d is not None else None, *p, None)


@no_gpu_only
def test_accept_validation(lib):
    assert ag(lib, None, ptrs(5)) == sv.SSM_ERR_NULL
    assert asa(lib, None, ptrs(7)) == sv.SSM_ERR_NULL
    for i in range(4):  # dev_status alone is optional
        p = ptrs(5)
        p[i] = None
        assert ag(lib, adesc(), p) == sv.SSM_ERR_NULL, i
    for i in range(6):
        p = ptrs(7)
        p[i] = None
        assert asa(lib, adesc(), p) == sv.SSM_ERR_NULL, i
    for kw, code in ((dict(ntok=0), sv.SSM_ERR_SHAPE), (dict(ntok=sv.SSM_ACCEPT_MAX_NTOK + 1), sv.SSM_ERR_SHAPE),
                     (dict(vocab=0), sv.SSM_ERR_SHAPE), (dict(vocab=sv.SSM_ACCEPT_MAX_VOCAB + 1), sv.SSM_ERR_SHAPE),
                     (dict(batch=-1), sv.SSM_ERR_SHAPE), (dict(logit_dtype=5), sv.SSM_ERR_UNSUPPORTED)):
        assert ag(lib, adesc(**kw), ptrs(5)) == code, kw
        assert asa(lib, adesc(**kw), ptrs(7)) == code, kw
    # alignment: logits to their element size, the int32 / float arrays to 4 bytes
    for i, off in [(0, 1), (1, 2), (2, 2), (3, 2), (4, 2)]:
        p = ptrs(5)
        p[i] = ctypes.c_void_p(p[i].value + off)
        assert ag(lib, adesc(), p) == sv.SSM_ERR_ALIGN, i
    for i, off in [(0, 1), (1, 1), (2, 2), (3, 2), (4, 2), (5, 2), (6, 2)]:
        p = ptrs(7)
        p[i] = ctypes.c_void_p(p[i].value + off)
        assert asa(lib, adesc(), p) == sv.SSM_ERR_ALIGN, i
    p = ptrs(5)
    p[0] = ctypes.c_void_p(p[0].value + 2)            # 2 bytes suffice for bf16 logits, not for fp32
    assert ag(lib, adesc(logit_dtype=sv.SSM_F32), p) == sv.SSM_ERR_ALIGN
    assert ag(lib, adesc(), p) == sv.SSM_ERR_CUDA     # valid: with no device here the launch fails
    # aliasing: outputs against inputs and each other
    p = ptrs(5)
    p[2] = ctypes.c_void_p(p[1].value + 4)            # accept_len inside draft_tokens
    assert ag(lib, adesc(), p) == sv.SSM_ERR_ALIAS
    p = ptrs(5)
    p[3] = p[2]                                        # next_token on accept_len
    assert ag(lib, adesc(), p) == sv.SSM_ERR_ALIAS
    p = ptrs(7)
    p[6] = ctypes.c_void_p(p[5].value + 4)            # dev_status inside next_token
    assert asa(lib, adesc(), p) == sv.SSM_ERR_ALIAS
    p = ptrs(7)
    p[4] = ctypes.c_void_p(p[1].value + 64)           # accept_len inside the draft logits
    assert asa(lib, adesc(), p) == sv.SSM_ERR_ALIAS
    p = ptrs(7)
    p[1] = p[0]                                        # read-only inputs may overlap
    assert asa(lib, adesc(), p) == sv.SSM_ERR_CUDA
    # an empty batch inspects no pointer
    assert ag(lib, adesc(batch=0), [None] * 5) == sv.SSM_OK
    assert asa(lib, adesc(batch=0), [None] * 7) == sv.SSM_OK


def test_accept_shim_checks_shapes():
    t = torch.zeros(2, 4, 10)
    with pytest.raises(ValueError, match="CUDA tensor"):
        sv.accept_greedy(t, torch.zeros(2, 3, dtype=torch.int32))


def _arity(name):
    """Parameter count of a header declaration."""
    txt = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    m = re.search(r"\b" + name + r"\s*\(([^)]*)\)", txt)
    return len([a for a in m.group(1).split(",") if a.strip()])


def test_binding_arities_match_header(lib):
    for name in sv.EXPORTS:
        argtypes = getattr(lib, name).argtypes
        if argtypes is not None:
            assert len(argtypes) == _arity(name), name


@no_gpu_only
def test_layer_stack_validation(lib):
    """nlayers = L scales every per-layer buffer (and a pool) by L; accept_len
    and the slot map stay [batch]; prefill takes one layer."""
    xb = 2 * 3 * 4 * 32 * 2  # bytes of one layer's x: batch 2, K 3, H 4, P 32, bf16
    for L, code in ((0, sv.SSM_ERR_CUDA), (1, sv.SSM_ERR_CUDA), (3, sv.SSM_ERR_ALIAS)):
        p = ptrs(10)
        p[8] = ctypes.c_void_p(p[1].value + xb + 64)  # y just past layer 0's x: inside layer 1's
        assert vc(lib, desc(nlayers=L), p) == code, L
    p = ptrs(10)
    assert vc(lib, desc(nlayers=64), p) == sv.SSM_ERR_CUDA  # valid: the launch fails on this host
    st = ptrs(1)[0].value
    args = ptrs(9, start=BASE + (1 << 35))
    # a stacked pool is [L][nslots][H][P][N]: valid (the launch fails on this host) ...
    assert lib.ssm_verify_commit_pool(ctypes.byref(desc(nlayers=2)), ctypes.byref(pool(st)), *args,
                                      None) == sv.SSM_ERR_CUDA
    # ... and y just past layer 0's pool lies inside layer 1's
    pb = 4 * 4 * 32 * 128 * 4  # nslots 4 x H 4 x P 32 x N 128 x fp32
    a2 = list(args)
    a2[7] = ctypes.c_void_p(st + pb + 64)
    assert lib.ssm_verify_commit_pool(ctypes.byref(desc(nlayers=1)), ctypes.byref(pool(st)), *a2,
                                      None) == sv.SSM_ERR_CUDA
    assert lib.ssm_verify_commit_pool(ctypes.byref(desc(nlayers=2)), ctypes.byref(pool(st)), *a2,
                                      None) == sv.SSM_ERR_ALIAS
    pargs = ptrs(7, start=BASE + (1 << 35))
    assert lib.ssm_prefill(ctypes.byref(desc(nlayers=2)), ctypes.byref(pool(st)), *pargs, None, 0, None,
                           None) == sv.SSM_ERR_UNSUPPORTED
    assert lib.ssm_prefill_workspace_bytes(ctypes.byref(desc(nlayers=2, batch=1, ntok=2048))) == 0


@no_gpu_only
def test_prefill_chunk_rule_for_tensor_core_shapes(lib):
    """bf16 prompts with N = 128, headdim a multiple of 64 and at least two
    128-token chunks take 128-token chunks whatever the device: workspace =
    batch * (T / 128) states + the chunks' slot map + each chunk's decay
    product per head (each 16-byte rounded). Other shapes chunk only to fill
    the device, which this host has none of (0)."""
    def ws(**kw):
        return lib.ssm_prefill_workspace_bytes(ctypes.byref(desc(**kw)))

    def r16(n):
        return (n + 15) // 16 * 16

    def want(batch, T, H, P):
        nch = batch * (T // 128)
        return nch * H * P * 128 * 4 + r16(nch * 4) + r16(nch * H * 4)

    for P in (64, 128, 192, 256):
        assert ws(batch=1, nheads=80, headdim=P, ngroups=1, ntok=2048) == want(1, 2048, 80, P), P
    assert ws(batch=3, nheads=4, headdim=64, ngroups=2, ntok=384) == want(3, 384, 4, 64)
    # one 2048-token prompt of a Llama-3-8B or a Mamba-2-2.7B layer fits the library's fixed scratch, so
    # ssm_prefill_scratch takes the same 128-token chunks as a caller workspace would
    for H, P, G in ((32, 128, 8), (80, 64, 1)):
        assert 0 < ws(batch=1, nheads=H, headdim=P, ngroups=G, ntok=2048) <= sv.SSM_PREFILL_SCRATCH_BYTES
    for kw in (dict(headdim=96), dict(dstate=64), dict(in_dtype=sv.SSM_F32), dict(ntok=128), dict(ntok=2000)):
        base = dict(batch=1, nheads=8, headdim=64, dstate=128, ngroups=1, ntok=2048)
        base.update(kw)
        assert ws(**base) == 0, kw



@no_gpu_only
def test_tile_count_limit(lib):
    """A call whose tiles (layers x batch x heads x row tiles) reach 2^31 is a
    shape error found on the host (the kernels decode tile indices in 32
    bits); one tile fewer passes validation and fails only at the launch.
    The fake buffers are spaced 2^47 bytes apart: the state alone is 2^46."""
    P = ptrs(12, gap=1 << 47)
    # 64-row tiles at dstate 128: headdim 64 is one row tile per (sequence, head)
    at = desc(batch=1 << 20, nheads=1 << 11, headdim=64, ngroups=1)
    assert vc(lib, at, P[:10] + [None]) == sv.SSM_ERR_SHAPE
    stacked = desc(batch=1 << 10, nheads=1 << 11, headdim=64, ngroups=1, nlayers=1 << 10)
    assert vc(lib, stacked, P[:10] + [None]) == sv.SSM_ERR_SHAPE
    below = desc(batch=(1 << 20) - 1, nheads=1 << 11, headdim=64, ngroups=1)
    assert vc(lib, below, P[:10] + [None]) == sv.SSM_ERR_CUDA

def pool(states, slot=None, nslots=4, reserved=0):
    return sv.PoolDesc(states, slot, nslots, reserved)


@no_gpu_only
def test_pool_and_prefill_validation(lib):
    d = desc()  # batch 2
    P = ptrs(12)
    st = P[0].value
    vcp = lambda pl, p: lib.ssm_verify_commit_pool(ctypes.byref(d), ctypes.byref(pl) if pl is not None else None, *p,
                                                   None)
    pre = lambda pl, p, ws=None, wsb=0: lib.ssm_prefill(ctypes.byref(d), ctypes.byref(pl) if pl is not None else None,
                                                        *p, ws, wsb, None, None)
    # verify_commit_pool: x, B, C, dt, A, D, accept_len, y, dev_status
    args = P[1:10]
    assert vcp(None, args) == sv.SSM_ERR_NULL
    assert vcp(pool(st, reserved=1), args) == sv.SSM_ERR_SHAPE
    assert vcp(pool(st, nslots=0), args) == sv.SSM_ERR_SHAPE
    assert vcp(pool(st, nslots=1), args) == sv.SSM_ERR_SHAPE          # no slot map: nslots >= batch
    assert vcp(pool(st, slot=P[10].value, nslots=1), args) == sv.SSM_ERR_CUDA  # a slot map: one slot is enough
    assert vcp(pool(st, slot=P[10].value + 2), args) == sv.SSM_ERR_ALIGN
    assert vcp(pool(st + 8), args) == sv.SSM_ERR_ALIGN                # states need 16 bytes
    assert vcp(pool(None), args) == sv.SSM_ERR_NULL
    a2 = list(args)
    a2[7] = ctypes.c_void_p(st + 64)                                   # y inside the pool
    assert vcp(pool(st), a2) == sv.SSM_ERR_ALIAS
    # prefill: x, B, C, dt, A, D, y
    pargs = P[1:7] + [P[8]]
    assert pre(None, pargs) == sv.SSM_ERR_NULL
    assert pre(pool(st), pargs, None, -1) == sv.SSM_ERR_SHAPE          # negative workspace size
    assert pre(pool(st, reserved=1), pargs) == sv.SSM_ERR_SHAPE
    p2 = list(pargs)
    p2[6] = ctypes.c_void_p(st + 64)                                   # y inside the pool
    assert pre(pool(st), p2) == sv.SSM_ERR_ALIAS
    assert pre(pool(st), pargs) == sv.SSM_ERR_CUDA                     # valid: the launch fails on this host
    d0 = desc(batch=0)
    assert lib.ssm_prefill(ctypes.byref(d0), ctypes.byref(pool(None)), *([None] * 8), 0, None, None) == sv.SSM_OK
    assert lib.ssm_prefill_workspace_bytes(ctypes.byref(d0)) == 0
    assert lib.ssm_prefill_scratch(ctypes.byref(d), None, *([None] * 9)) == sv.SSM_ERR_NULL


@no_gpu_only
def test_copy_from_host_n_validation(lib):
    """Segment count, null pointers, negative sizes and overlapping
    destinations are refused before anything else is looked at."""
    Seg = sv.CopySegment
    mk = lambda *t: (Seg * max(1, len(t)))(*t)
    a, b = BASE, BASE + (1 << 30)
    assert lib.ssm_copy_from_host_n(mk(), 0, None) == sv.SSM_OK
    assert lib.ssm_copy_from_host_n(mk(), -1, None) == sv.SSM_ERR_SHAPE
    assert lib.ssm_copy_from_host_n((Seg * 9)(), 9, None) == sv.SSM_ERR_SHAPE
    assert lib.ssm_copy_from_host_n(None, 1, None) == sv.SSM_ERR_NULL
    assert lib.ssm_copy_from_host_n(mk(Seg(a, b, -1)), 1, None) == sv.SSM_ERR_SHAPE
    assert lib.ssm_copy_from_host_n(mk(Seg(None, b, 16)), 1, None) == sv.SSM_ERR_NULL
    assert lib.ssm_copy_from_host_n(mk(Seg(a, b, 64), Seg(a + 32, b + 4096, 64)), 2, None) == sv.SSM_ERR_ALIAS
    assert lib.ssm_copy_from_host_n(mk(Seg(a, b, 64), Seg(b + 32, a + 4096, 64)), 2, None) == sv.SSM_ERR_ALIAS
    assert lib.ssm_copy_from_host_n(mk(Seg(a, b, 0), Seg(a, b, 0)), 2, None) == sv.SSM_OK  # empty: nothing to do


def test_copy_from_host_n_binding_limits():
    """The binding refuses more segments than the library takes, before any
    device or pointer is looked at."""
    pairs = [(torch.zeros(4), torch.zeros(4))] * (sv.SSM_COPY_MAX_SEGMENTS + 1)
    with pytest.raises(ValueError):
        sv.copy_from_host_n(pairs)
