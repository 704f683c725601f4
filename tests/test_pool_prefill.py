"""State-pool entry points and prefill on the GPU, through the C ABI.

Pool variants are the plain entry points with the state reached through a
slot map: on the same data they must give the plain results bit for bit and
leave every other slot untouched. Prefill is the recurrence over a whole
prompt from the cached state: it is compared with the fp64 oracle (every
token accepted), in its one-pass and its chunked form."""
import numpy as np
import pytest
import torch

import oracle
import ssm_recurrence_verify_b300 as ssm
from gpu_helpers import RTOL_STATE, np64, rel_err, y_tol
from ssm_recurrence_verify_b300 import ssmverify as sv
from ssm_recurrence_verify_b300 import synth

pytestmark = pytest.mark.gpu


def _inputs(batch, H, P, N, G, K, dtype, seed, rnd=0):
    wl = synth.custom_workload(batch, H, P, N, G, K, dtype, seed=seed)
    p = synth.draw_params(wl)
    t = synth.draw_tokens(wl, rnd)
    return wl, p, t


def _dev(d, dev):
    return {k: v.to(dev) for k, v in d.items()}


@pytest.mark.parametrize("dtype", [synth.F32, synth.BF16])
def test_pool_variants_equal_plain_calls(cuda_device, dtype):
    dev = cuda_device
    batch, H, P, N, G, K = 4, 4, 64, 128, 2, 5
    wl, p, t = _inputs(batch, H, P, N, G, K, dtype, seed=301)
    nslots = 7
    slot = torch.tensor([5, 0, 3, 6], dtype=torch.int32)
    pool0 = torch.randn(nslots, H, P, N, generator=torch.Generator().manual_seed(3)) * 0.1
    pool0[slot.long()] = p["state0"]
    td = _dev(t, dev)
    A, D = p["A"].to(dev), p["D"].to(dev)
    acc = synth.draw_accept_len(wl, 0).to(dev)
    sl = slot.to(dev)
    others = [i for i in range(nslots) if i not in slot.tolist()]

    def fresh():
        return pool0.clone().to(dev), p["state0"].clone().to(dev)

    # verify
    pool, st = fresh()
    y_p = ssm.verify_pool(pool, sl, td["x"], td["B"], td["C"], td["dt"], A, D)
    y_s = ssm.verify(st, td["x"], td["B"], td["C"], td["dt"], A, D)
    torch.cuda.synchronize()
    assert torch.equal(y_p, y_s) and torch.equal(pool.cpu(), pool0)
    # verify_commit
    pool, st = fresh()
    y_p = ssm.verify_commit_pool(pool, sl, td["x"], td["B"], td["C"], td["dt"], A, D, acc)
    y_s = ssm.verify_commit(st, td["x"], td["B"], td["C"], td["dt"], A, D, acc)
    torch.cuda.synchronize()
    assert torch.equal(y_p, y_s) and torch.equal(pool[sl.long()], st)
    assert torch.equal(pool.cpu()[others], pool0[others])
    # commit
    pool, st = fresh()
    ssm.commit_pool(pool, sl, td["x"], td["B"], td["dt"], A, acc)
    ssm.commit(st, td["x"], td["B"], td["dt"], A, acc)
    torch.cuda.synchronize()
    assert torch.equal(pool[sl.long()], st) and torch.equal(pool.cpu()[others], pool0[others])
    # commit_verify (previous block = this round's, new block = the next round's)
    t2 = _dev(synth.draw_tokens(wl, 1), dev)
    pool, st = fresh()
    y_p = ssm.commit_verify_pool(pool, sl, td["x"], td["B"], td["dt"], acc, t2["x"], t2["B"], t2["C"], t2["dt"], A, D)
    y_s = ssm.commit_verify(st, td["x"], td["B"], td["dt"], acc, t2["x"], t2["B"], t2["C"], t2["dt"], A, D)
    torch.cuda.synchronize()
    assert torch.equal(y_p, y_s) and torch.equal(pool[sl.long()], st)
    assert torch.equal(pool.cpu()[others], pool0[others])
    # step, and the identity map (slot None: sequence b uses slot b)
    w1, p1, t1 = _inputs(batch, H, P, N, G, 1, dtype, seed=302)
    t1 = _dev(t1, dev)
    pool, st = fresh()
    y_p = ssm.step_pool(pool, sl, t1["x"], t1["B"], t1["C"], t1["dt"], A, D)
    y_s = ssm.step(st, t1["x"], t1["B"], t1["C"], t1["dt"], A, D)
    torch.cuda.synchronize()
    assert torch.equal(y_p, y_s) and torch.equal(pool[sl.long()], st)
    pool = p["state0"].clone().to(dev)
    st = p["state0"].clone().to(dev)
    y_p = ssm.verify_commit_pool(pool, None, td["x"], td["B"], td["C"], td["dt"], A, D, acc)
    y_s = ssm.verify_commit(st, td["x"], td["B"], td["C"], td["dt"], A, D, acc)
    torch.cuda.synchronize()
    assert torch.equal(y_p, y_s) and torch.equal(pool, st)


@pytest.mark.parametrize("fn,K", [("verify_commit", 3), ("prefill", 3), ("prefill", 64)])
def test_bad_slots_write_nothing(cuda_device, fn, K):
    """Sequences whose slot is outside [0, nslots): status bit set, their y
    and every slot no valid sequence maps to untouched (prefill with K = 64
    takes the chunked form)."""
    dev = cuda_device
    batch, H, P, N, G = 4, 2, 32, 64, 1
    wl, p, t = _inputs(batch, H, P, N, G, K, synth.F32, seed=303)
    td = _dev(t, dev)
    A, D = p["A"].to(dev), p["D"].to(dev)
    acc = torch.full((batch,), K, dtype=torch.int32, device=dev)
    pool0 = p["state0"].clone()
    slot = torch.tensor([1, 4, -1, 2], dtype=torch.int32, device=dev)  # nslots = 4: 4 and -1 are invalid
    pool = pool0.clone().to(dev)
    y = torch.full((batch, K, H, P), 7.0, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    if fn == "verify_commit":
        ssm.verify_commit_pool(pool, slot, td["x"], td["B"], td["C"], td["dt"], A, D, acc, y=y, dev_status=st)
    else:
        if K == 64:
            assert ssm.prefill_workspace_bytes(pool, td["x"], td["B"], td["C"], td["dt"], A, D) > 0
        ssm.prefill(pool, slot, td["x"], td["B"], td["C"], td["dt"], A, D, y=y, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & sv.SSM_STATUS_BAD_SLOT
    assert torch.equal(pool[0].cpu(), pool0[0]) and torch.equal(pool[3].cpu(), pool0[3])  # no sequence maps here
    assert (y[1] == 7.0).all() and (y[2] == 7.0).all()  # bad slots: y untouched
    assert not (y[0] == 7.0).any() and not (y[3] == 7.0).any()
    # the valid sequences match the plain call on their own states
    ref = oracle.verify_commit(pool0[[1, 2]], t["x"][[0, 3]], t["B"][[0, 3]], t["C"][[0, 3]], t["dt"][[0, 3]],
                               p["A"], p["D"], None)
    assert rel_err(np64(y[[0, 3]]), ref["y"]) <= 1e-4
    assert rel_err(np64(pool[[1, 2]]), ref["state"]) <= 1e-4


def _prefill_case(dev, batch, H, P, N, G, T, dtype, seed, chunked=True):
    wl, p, t = _inputs(batch, H, P, N, G, T, dtype, seed=seed)
    nslots = batch + 2
    slot = torch.randperm(nslots, generator=torch.Generator().manual_seed(seed))[:batch].to(torch.int32)
    pool0 = torch.zeros(nslots, H, P, N)
    pool0[slot.long()] = p["state0"]  # a continuing prompt: start from a nonzero cached state
    pool = pool0.to(dev)
    td = _dev(t, dev)
    A, D = p["A"].to(dev), p["D"].to(dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = None if chunked else torch.empty(0, device=dev)
    y = ssm.prefill(pool, slot.to(dev), td["x"], td["B"], td["C"], td["dt"], A, D, workspace=ws, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = oracle.verify_commit(p["state0"], t["x"], t["B"], t["C"], t["dt"], p["A"], p["D"], None)
    ey = rel_err(np64(y), ref["y"])
    es = rel_err(np64(pool[slot.long().to(dev)]), ref["state"])
    assert ey <= y_tol(wl.torch_in_dtype), (T, dtype, ey)
    assert es <= RTOL_STATE, (T, dtype, es)
    untouched = [i for i in range(nslots) if i not in slot.tolist()]
    assert torch.equal(pool.cpu()[untouched], pool0[untouched])
    return y, pool


@pytest.mark.parametrize("T", [1, 8, 40, 64, 96, 256, 1024])
@pytest.mark.parametrize("dtype", [synth.F32, synth.BF16])
def test_prefill_matches_oracle(cuda_device, T, dtype):
    _prefill_case(cuda_device, 2, 4, 64, 128, 2, T, dtype, seed=400 + T)


@pytest.mark.parametrize("N,P,dtype", [(16, 64, synth.F32), (64, 128, synth.BF16), (256, 64, synth.BF16),
                                         (128, 96, synth.BF16)])
def test_prefill_other_geometries(cuda_device, N, P, dtype):
    """State sizes whose chunk passes take other layouts: N = 16 and 64 (one
    warp per band), N = 256 (two warps per band: the chunk passes use the
    recurrence), and P = 96 (not a multiple of the 64-row tile)."""
    _prefill_case(cuda_device, 2, 4, P, N, 2, 256, dtype, seed=480 + N + P)


def test_prefill_chunked_and_one_pass_agree(cuda_device):
    """The chunked regrouping and the plain recurrence agree to rounding, and
    the small shape really does take the chunked form."""
    dev = cuda_device
    args = dict(batch=1, H=4, P=64, N=128, G=2, T=512, dtype=synth.BF16, seed=451)
    pool = torch.zeros(1, 4, 64, 128, device=dev)
    x = torch.zeros(1, 512, 4, 64, dtype=torch.bfloat16, device=dev)
    Bc = torch.zeros(1, 512, 2, 128, dtype=torch.bfloat16, device=dev)
    dt = torch.zeros(1, 512, 4, dtype=torch.bfloat16, device=dev)
    AD = torch.zeros(4, device=dev)
    assert ssm.prefill_workspace_bytes(pool, x, Bc, Bc, dt, AD, AD) > 0
    y1, s1 = _prefill_case(dev, chunked=True, **args)
    y2, s2 = _prefill_case(dev, chunked=False, **args)
    assert rel_err(np64(y1), np64(y2)) <= 1e-4 and rel_err(np64(s1), np64(s2)) <= 1e-4


def test_prefill_llama_layer_shape(cuda_device):
    """A Llama-3-8B-shaped layer (H 32, P 128, N 128, G 8), one 2048-token prompt."""
    _prefill_case(cuda_device, 1, 32, 128, 128, 8, 2048, synth.BF16, seed=461)


def test_prefill_mamba2_layer_shape(cuda_device):
    """A Mamba-2-2.7B-shaped layer (H 80, P 64, N 128, G 1), one 2048-token
    prompt: the head-pair chunk-state tiles and the 64-row output tiles."""
    _prefill_case(cuda_device, 1, 80, 64, 128, 1, 2048, synth.BF16, seed=464)


def test_prefill_tensor_memory_chunk_states(cuda_device):
    """A shape whose chunk states take the tensor-memory (tcgen05) pass: bf16,
    N = 128, 128-token chunks, two 128-row tiles per head (P = 256)."""
    _prefill_case(cuda_device, 2, 16, 256, 128, 4, 1024, synth.BF16, seed=462)


def test_prefill_then_speculative_round(cuda_device):
    """Prefill a prompt, then verify + commit K drafts from the cached state:
    the same as the oracle over the prompt followed by the drafts."""
    dev = cuda_device
    batch, H, P, N, G, T, K = 2, 4, 64, 64, 2, 256, 6
    wl, p, t = _inputs(batch, H, P, N, G, T, synth.F32, seed=471)
    w2 = synth.custom_workload(batch, H, P, N, G, K, synth.F32, seed=472)
    t2 = synth.draw_tokens(w2, 0)
    acc = synth.draw_accept_len(w2, 0)
    pool = torch.zeros(batch, H, P, N, device=dev)
    td, t2d = _dev(t, dev), _dev(t2, dev)
    A, D = p["A"].to(dev), p["D"].to(dev)
    ssm.prefill(pool, None, td["x"], td["B"], td["C"], td["dt"], A, D)
    y = ssm.verify_commit_pool(pool, None, t2d["x"], t2d["B"], t2d["C"], t2d["dt"], A, D, acc.to(dev))
    torch.cuda.synchronize()
    zero = torch.zeros(batch, H, P, N)
    r1 = oracle.verify_commit(zero, t["x"], t["B"], t["C"], t["dt"], p["A"], p["D"], None)
    r2 = oracle.verify_commit(r1["state"], t2["x"], t2["B"], t2["C"], t2["dt"], p["A"], p["D"], acc)
    assert rel_err(np64(y), r2["y"]) <= 1e-4 and rel_err(np64(pool), r2["state"]) <= 1e-4


@pytest.mark.parametrize("dtype", [synth.F32, synth.BF16])
def test_pool_layer_stack_equals_per_layer_pool_calls(cuda_device, dtype):
    """A stacked pool [L][nslots][H][P][N] with one slot map for every layer:
    each pool entry point over the stack equals, bit for bit, the per-layer
    pool calls on states[l]; a bad slot writes nothing in any layer."""
    dev = cuda_device
    L, batch, nslots, K = 3, 4, 7, 8
    wl = synth.custom_workload(batch, 4, 64, 128, 2, K, dtype, seed=990)
    ds = [synth.draw_layer_round(wl, rnd=0, layer=l) for l in range(L)]
    S = {k: torch.stack([d[k] for d in ds]).to(dev) for k in ("x", "B", "C", "dt", "A", "D")}
    acc = ds[0]["accept_len"].to(dev)
    g = torch.Generator().manual_seed(5)
    pool0 = (0.1 * torch.randn(L, nslots, 4, 64, 128, generator=g)).to(dev)
    slot = torch.tensor([5, 0, 9, 2], dtype=torch.int32, device=dev)  # slot 9: out of range
    nxt = [synth.draw_tokens(wl, 1, l) for l in range(L)]
    N2 = {k: torch.stack([t[k] for t in nxt]).to(dev) for k in ("x", "B", "C", "dt")}
    one = {k: S[k][:, :, :1].contiguous() for k in ("x", "B", "C", "dt")}

    def run(fn, pool, l=None):
        sel = (lambda t: t) if l is None else (lambda t: t[l])
        st = pool if l is None else pool[l]
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        if fn == "verify":
            y = ssm.verify_pool(st, slot, *(sel(S[k]) for k in ("x", "B", "C", "dt", "A", "D")), dev_status=status)
        elif fn == "verify_commit":
            y = ssm.verify_commit_pool(st, slot, *(sel(S[k]) for k in ("x", "B", "C", "dt", "A", "D")), acc,
                                       dev_status=status)
        elif fn == "commit":
            ssm.commit_pool(st, slot, sel(S["x"]), sel(S["B"]), sel(S["dt"]), sel(S["A"]), acc, dev_status=status)
            y = None
        elif fn == "commit_verify":
            y = ssm.commit_verify_pool(st, slot, sel(S["x"]), sel(S["B"]), sel(S["dt"]), acc,
                                       *(sel(N2[k]) for k in ("x", "B", "C", "dt")), sel(S["A"]), sel(S["D"]),
                                       dev_status=status)
        else:
            y = ssm.step_pool(st, slot, *(sel(one[k]) for k in ("x", "B", "C", "dt")), sel(S["A"]), sel(S["D"]),
                              dev_status=status)
        return y, status

    for fn in ("verify", "verify_commit", "commit", "commit_verify", "step"):
        stacked = pool0.clone()
        per = pool0.clone()
        y, status = run(fn, stacked)
        outs = [run(fn, per, l) for l in range(L)]
        torch.cuda.synchronize()
        assert torch.equal(stacked, per), fn
        assert int(status.item()) & ssm.ssmverify.SSM_STATUS_BAD_SLOT, fn
        if y is not None:
            for l in range(L):
                assert torch.equal(y[l][torch.tensor([0, 1, 3])], outs[l][0][torch.tensor([0, 1, 3])]), (fn, l)
        untouched = [i for i in range(nslots) if i not in (5, 0, 2)]
        assert torch.equal(stacked[:, untouched], pool0[:, untouched]), fn


@pytest.mark.parametrize("P", [256, 64])
def test_prefill_tensor_memory_bad_slot(cuda_device, P):
    """The tcgen05 prefill passes (128- and 64-row output tiles) with one
    sequence on an invalid slot: its y stays unwritten, the status bit is set,
    the valid sequence matches the oracle and no other slot changes."""
    dev = cuda_device
    batch, H, N, G, T = 2, 16, 128, 4, 1024
    wl, p, t = _inputs(batch, H, P, N, G, T, synth.BF16, seed=463)
    td = _dev(t, dev)
    A, D = p["A"].to(dev), p["D"].to(dev)
    nslots = 3
    pool0 = torch.zeros(nslots, H, P, N)
    pool0[2] = p["state0"][0]
    pool = pool0.to(dev)
    slot = torch.tensor([2, 7], dtype=torch.int32, device=dev)  # sequence 1: out of range
    y = torch.full((batch, T, H, P), 7.0, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    ssm.prefill(pool, slot, td["x"], td["B"], td["C"], td["dt"], A, D, y=y, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & sv.SSM_STATUS_BAD_SLOT
    assert (y[1] == 7.0).all()
    assert torch.equal(pool[:2].cpu(), pool0[:2])
    ref = oracle.verify_commit(p["state0"][:1], t["x"][:1], t["B"][:1], t["C"][:1], t["dt"][:1], p["A"], p["D"], None)
    assert rel_err(np64(y[:1]), ref["y"]) <= y_tol(torch.bfloat16)
    assert rel_err(np64(pool[2:3]), ref["state"]) <= RTOL_STATE


@pytest.mark.parametrize("T", [256, 384])
def test_prefill_tensor_memory_few_chunks(cuda_device, T):
    """The tcgen05 passes with two and three 128-token chunks (bf16, N = 128,
    P = 128) on a small batch, against the oracle."""
    _prefill_case(cuda_device, 3, 4, 128, 128, 2, T, synth.BF16, seed=470 + T)


@pytest.mark.parametrize("P", [64, 192])
def test_prefill_tensor_memory_64_row_tiles(cuda_device, P):
    """The tcgen05 output pass on 64-row tiles: P a multiple of 64 but not of
    128 (one and three tiles per head; the chunk states come from the mma.sync
    pass), bf16, N = 128, four 128-token chunks, against the oracle."""
    _prefill_case(cuda_device, 2, 4, P, 128, 2, 512, synth.BF16, seed=475 + P)


@pytest.mark.parametrize("H,G", [(8, 1), (6, 2)])
def test_prefill_tensor_memory_p64_head_pairs(cuda_device, H, G):
    """P = 64: the tcgen05 chunk-state pass takes a 128-row tile over two heads
    of one group (H / G even: w and dt differ per half, B is shared); with an
    odd number of heads per group it keeps the mma.sync pass. Both against the
    oracle."""
    _prefill_case(cuda_device, 2, H, 64, 128, G, 384, synth.BF16, seed=480 + 7 * H + G)
