"""ZeRO stage 3 on the GPU: the owner-only step and the gather, against the oracle.

Stage 3 ("Data parallelism and ZeRO stages 1 to 3", section 2, stage 3, and
section 4) keeps only each rank's own chunk of the parameters between steps and
gathers the full parameters when they are needed. Through the C ABI:
  * zero_step_ex(owner_only=1) must write exactly the oracle's owner-only
    chunks (``zero_step(..., all_gather=False)``) into each owner's replica and
    leave every other replica element as it was;
  * zero_gather must then give every replica the oracle's ``gather`` result,
    bit for bit; owner-only steps followed by one gather equal the same number
    of stage-1/2 steps, bit for bit.
"""

import numpy as np
import pytest
import torch

import oracle
from parity_util import assert_bf16_within_one_ulp, exact_fraction, flat
from test_gpu_parity import HP, Case, host_of

pytestmark = pytest.mark.gpu

CASES = [(1, 1), (7, 3), (33, 4), (4099, 5), (100_003, 4), (100_003, 8), (65_537, 13),
         (300_007, 6), (1_000_003, 8)]


def owner_only_step(c):
    """One owner-only step on both sides; returns the oracle's chunks."""
    hg = c.new_grads()
    c.t += 1
    shards, c.o_states = oracle.zero_step(c.o_reps, hg, c.o_states, c.t, precision=c.prec,
                                          mode="fp32", all_gather=False, **c.hp)
    c.abi.zero_step_ex(c.reps, c.grads, c.st, c.t, owner_only=True, **c.hp)
    torch.cuda.synchronize()
    return shards


def check_owner_only(c, shards, before):
    b = oracle.shard_bounds(c.n, c.N) if c.bounds is None else c.bounds
    assert exact_fraction(host_of(c.m), flat(c.o_states, "m")) == 1.0
    assert exact_fraction(host_of(c.v), flat(c.o_states, "v")) == 1.0
    if c.mixed:
        master = flat(c.o_states, "master")
        assert exact_fraction(host_of(c.master), master) == 1.0
    for r in range(c.N):
        got = host_of(c.reps[r])
        lo, hi = b[r], b[r + 1]
        assert np.array_equal(got[lo:hi], shards[r]), f"rank {r}: own chunk"
        if c.mixed:
            assert_bf16_within_one_ulp(got[lo:hi], master[lo:hi], f"rank {r}")
        outside = np.ones(c.n, bool)
        outside[lo:hi] = False
        assert np.array_equal(got[outside], before[r][outside]), f"rank {r}: released part written"


def gather_and_check(c, shards):
    c.abi.zero_gather(c.reps, c.st)
    torch.cuda.synchronize()
    full = oracle.gather(shards, c.prec)
    for r in range(c.N):
        assert np.array_equal(host_of(c.reps[r]), full[r]), f"replica {r} after gather"
    c.o_reps = full


@pytest.mark.parametrize("prec", [oracle.FP32, oracle.BF16_MIXED])
@pytest.mark.parametrize("n,N", CASES)
def test_owner_only_step_then_gather(abi, cuda, n, N, prec):
    c = Case(abi, cuda, n, N, prec, seed=n * 17 + N)
    c.bounds = None
    for _ in range(2):
        before = [host_of(x) for x in c.reps]
        shards = owner_only_step(c)
        check_owner_only(c, shards, before)
        gather_and_check(c, shards)


@pytest.mark.parametrize("prec", [oracle.FP32, oracle.BF16_MIXED])
@pytest.mark.parametrize("layout", ["shifted", "mixed_phase"])
def test_owner_only_unaligned(abi, cuda, prec, layout):
    n, N = 50_011, 4
    if layout == "shifted":
        kw = dict(rep_off=[3] * N, grad_off=[3] * N, state_off=3)
    else:
        kw = dict(rep_off=[1, 2, 3, 0], grad_off=[0, 0, 0, 1], state_off=0)
    c = Case(abi, cuda, n, N, prec, seed=11, **kw)
    c.bounds = None
    for _ in range(2):
        before = [host_of(x) for x in c.reps]
        shards = owner_only_step(c)
        check_owner_only(c, shards, before)
        gather_and_check(c, shards)


@pytest.mark.parametrize("prec", [oracle.FP32, oracle.BF16_MIXED])
def test_owner_only_whole_tensor_shards(abi, cuda, prec):
    rng = np.random.default_rng(31)
    numels = rng.integers(1, 30_000, 23).tolist()
    n, N = int(sum(numels)), 4
    tb = abi.zero_tensor_shard_bounds(numels, N)
    c = Case(abi, cuda, n, N, prec, seed=32)
    init = host_of(c.master) if c.mixed else host_of(c.reps[0])
    c.st = abi.zero_init_states(n, N, prec, c.m, c.v, c.master,
                                c.master.clone() if c.mixed else None, bounds=tb)
    c.o_states = oracle.init_states(n, N, prec, master_init=init, mode="fp32", bounds=tb)
    c.bounds = tb
    for _ in range(2):
        before = [host_of(x) for x in c.reps]
        hg = c.new_grads()
        c.t += 1
        shards, c.o_states = oracle.zero_step(c.o_reps, hg, c.o_states, c.t, precision=prec,
                                              mode="fp32", bounds=tb, all_gather=False, **HP)
        abi.zero_step_ex(c.reps, c.grads, c.st, c.t, owner_only=True, **HP)
        torch.cuda.synchronize()
        check_owner_only(c, shards, before)
        gather_and_check(c, shards)


@pytest.mark.parametrize("prec", [oracle.FP32, oracle.BF16_MIXED])
def test_owner_only_steps_then_one_gather_equal_full_steps(abi, cuda, prec):
    """The step reads a parameter only from its owner's replica (or the master),
    so the gather can wait until the parameters are needed."""
    n, N = 1_000_003, 4
    a = Case(abi, cuda, n, N, prec, seed=5)
    b = Case(abi, cuda, n, N, prec, seed=5)
    for t in range(1, 4):
        a.new_grads()
        for r in range(N):
            b.grads[r].copy_(a.grads[r])
        abi.zero_step_ex(a.reps, a.grads, a.st, t, owner_only=True, **HP)
        abi.zero_step(b.reps, b.grads, b.st, t, **HP)
    abi.zero_gather(a.reps, a.st)
    torch.cuda.synchronize()
    for x, y in [(a.m, b.m), (a.v, b.v)] + list(zip(a.reps, b.reps)):
        assert torch.equal(x, y)
    if a.mixed:
        assert torch.equal(a.master, b.master)


@pytest.mark.parametrize("prec", [oracle.FP32, oracle.BF16_MIXED])
def test_gather_range_touches_only_its_range(abi, cuda, prec):
    n, N = 200_003, 5
    c = Case(abi, cuda, n, N, prec, seed=9)
    dt = c.dt
    # distinct content per replica so every copied element is visible
    for r in range(N):
        src = torch.randn(n, device=cuda).to(dt)
        c.reps[r].copy_(src)
    before = [host_of(x) for x in c.reps]
    lo, hi = 12_345, 150_001
    abi.zero_gather(c.reps, c.st, lo, hi)
    torch.cuda.synchronize()
    b = oracle.shard_bounds(n, N)
    want = [x.copy() for x in before]
    for j0 in range(N):
        a_, b_ = max(b[j0], lo), min(b[j0 + 1], hi)
        if a_ < b_:
            for r in range(N):
                want[r][a_:b_] = before[j0][a_:b_]
    for r in range(N):
        assert np.array_equal(host_of(c.reps[r]), want[r]), f"replica {r}"


def test_gather_rejects_bad_arguments(abi, cuda):
    c = Case(abi, cuda, 1000, 3, oracle.FP32, seed=1)
    with pytest.raises(abi.ZeroError) as e:
        abi.zero_gather(c.reps, c.st, 10, 2000)
    assert e.value.code == abi.ZERO_EINVAL
    with pytest.raises(abi.ZeroError) as e:
        abi.zero_gather([c.reps[0], c.reps[0], c.reps[2]], c.st)
    assert e.value.code == abi.ZERO_EINVAL
    abi.zero_gather(c.reps, c.st, 500, 500)  # empty range: nothing to do


@pytest.mark.parametrize("prec", [oracle.FP32, oracle.BF16_MIXED])
def test_owner_only_with_empty_shards(abi, cuda, prec):
    """Fewer tensors than ranks: whole-tensor shards leave some ranks empty; the
    owner-only step and the gather skip them."""
    numels = [40_003, 17, 90_000]
    n, N = int(sum(numels)), 5
    tb = abi.zero_tensor_shard_bounds(numels, N)
    assert tb == oracle.tensor_shard_bounds(numels, N)
    assert any(tb[r] == tb[r + 1] for r in range(N))
    c = Case(abi, cuda, n, N, prec, seed=41)
    init = host_of(c.master) if c.mixed else host_of(c.reps[0])
    c.st = abi.zero_init_states(n, N, prec, c.m, c.v, c.master,
                                c.master.clone() if c.mixed else None, bounds=tb)
    c.o_states = oracle.init_states(n, N, prec, master_init=init, mode="fp32", bounds=tb)
    c.bounds = tb
    for _ in range(2):
        before = [host_of(x) for x in c.reps]
        hg = c.new_grads()
        c.t += 1
        shards, c.o_states = oracle.zero_step(c.o_reps, hg, c.o_states, c.t, precision=prec,
                                              mode="fp32", bounds=tb, all_gather=False, **HP)
        abi.zero_step_ex(c.reps, c.grads, c.st, c.t, owner_only=True, **HP)
        torch.cuda.synchronize()
        check_owner_only(c, shards, before)
        gather_and_check(c, shards)


def test_owner_only_and_gather_degenerate(abi, cuda):
    # one rank: the owner-only step is the full step, the gather has nothing to do
    a = Case(abi, cuda, 10_007, 1, oracle.FP32, seed=42)
    b = Case(abi, cuda, 10_007, 1, oracle.FP32, seed=42)
    a.new_grads()
    b.grads[0].copy_(a.grads[0])
    abi.zero_step_ex(a.reps, a.grads, a.st, 1, owner_only=True, **HP)
    abi.zero_step(b.reps, b.grads, b.st, 1, **HP)
    abi.zero_gather(a.reps, a.st)
    torch.cuda.synchronize()
    assert torch.equal(a.reps[0], b.reps[0]) and torch.equal(a.m, b.m)
    # n = 0: both calls accept empty buffers and do nothing
    z = Case(abi, cuda, 0, 3, oracle.FP32, seed=43)
    abi.zero_step_ex(z.reps, z.grads, z.st, 1, owner_only=True, **HP)
    abi.zero_gather(z.reps, z.st)
    torch.cuda.synchronize()
