"""Out-of-range writes: every call that works on a sub-range [lo, hi) of the
vector must leave every other index bitwise as it was, in m, v, the master and
every replica, and no call may write outside its buffers.

compute-sanitizer is not available on the GPU pool, so these checks stand in
for it: the ranges are ragged (odd ends, off the 16-byte vector grid and the
2048-element grid, across shard edges), the buffers sit between sentinel
guard regions (parity_util.GUARD, checked after every call here and by the
conftest after every test), and the values inside the range must equal those
of the same step over the whole vector. The update is elementwise ("Data
parallelism and ZeRO stages 1 to 3", section 2), so a range step is the full
step restricted to the range.
"""

import numpy as np
import pytest
import torch

import oracle
from parity_util import check_guards, guarded_empty
from test_gpu_parity import HP, Case, host_of

pytestmark = pytest.mark.gpu

N_ELEMS, N_RANKS = 200_003, 4          # shard edges at 50,001, 100,002, 150,003
RANGES = [(1, 2), (3, 4101), (2047, 6145), (50_000, 50_003), (99_997, 112_347),
          (12_345, 150_001), (N_ELEMS - 5, N_ELEMS), (0, N_ELEMS)]


def snapshot(c):
    bufs = {"m": c.m, "v": c.v}
    if c.mixed:
        bufs["master"] = c.master
    for r in range(c.N):
        bufs[f"replica {r}"] = c.reps[r]
    return {k: host_of(x) for k, x in bufs.items()}


def expect_range(before, full, lo, hi, owner_only_bounds=None):
    """`before` outside [lo, hi), `full` inside it; with owner-only bounds a
    replica takes `full` only over its own shard within the range."""
    want = {}
    for key, b in before.items():
        w = b.copy()
        a_, b_ = lo, hi
        if owner_only_bounds is not None and key.startswith("replica"):
            r = int(key.split()[1])
            a_, b_ = max(lo, owner_only_bounds[r]), min(hi, owner_only_bounds[r + 1])
        if a_ < b_:
            w[a_:b_] = full[key][a_:b_]
        want[key] = w
    return want


def assert_matches(c, want, what):
    check_guards()
    got = snapshot(c)
    for key in want:
        diff = np.flatnonzero(got[key].view(np.uint32 if got[key].dtype == np.float32
                                            else got[key].dtype) !=
                              want[key].view(np.uint32 if want[key].dtype == np.float32
                                             else want[key].dtype))
        assert diff.size == 0, f"{what}: {key} differs at {diff.size} indices, first {diff[:5]}"


def twin_cases(abi, cuda, prec, seed, off):
    kw = dict(rep_off=[off] * N_RANKS, grad_off=[off] * N_RANKS, state_off=off)
    a = Case(abi, cuda, N_ELEMS, N_RANKS, prec, seed=seed, **kw)
    b = Case(abi, cuda, N_ELEMS, N_RANKS, prec, seed=seed, **kw)
    a.new_grads()
    for r in range(N_RANKS):
        b.grads[r].copy_(a.grads[r])
    torch.cuda.synchronize()
    return a, b


@pytest.mark.parametrize("prec", [oracle.FP32, oracle.BF16_MIXED])
@pytest.mark.parametrize("off", [0, 3])
@pytest.mark.parametrize("entry", ["zero_step_range", "zero_step_ex", "zero_step_ex_owner_only",
                                   "zero_step_sgd"])
def test_range_step_leaves_the_rest_untouched(abi, cuda, prec, off, entry):
    a, b = twin_cases(abi, cuda, prec, seed=5 + off, off=off)
    owner_only = entry == "zero_step_ex_owner_only"
    sgd = entry == "zero_step_sgd"
    sgd_kw = dict(lr=0.01, momentum=0.9, dampening=0.1, weight_decay=0.01)
    if sgd:  # momentum SGD keeps its buffer in m; v is left alone by the step
        pass
    bounds = oracle.shard_bounds(N_ELEMS, N_RANKS)
    for t, (lo, hi) in enumerate(RANGES, start=1):
        before = snapshot(a)
        # b: the same step over the whole vector, from the same state
        for key, x in [("m", b.m), ("v", b.v)] + ([("master", b.master)] if b.mixed else []) + \
                [(f"replica {r}", b.reps[r]) for r in range(N_RANKS)]:
            x.copy_(torch.from_numpy(before[key].view(np.int16) if before[key].dtype == np.uint16
                                     else before[key]).view(x.dtype))
        if entry == "zero_step_range":
            abi.zero_step_range(a.reps, a.grads, a.st, t, HP["lr"], HP["beta1"], HP["beta2"],
                                HP["eps"], HP["weight_decay"], lo, hi)
            abi.zero_step(b.reps, b.grads, b.st, t, **HP)
        elif sgd:
            abi.zero_step_sgd(a.reps, a.grads, a.st, t, lo=lo, hi=hi, **sgd_kw)
            abi.zero_step_sgd(b.reps, b.grads, b.st, t, **sgd_kw)
        else:
            abi.zero_step_ex(a.reps, a.grads, a.st, t, grad_scale=0.5, lo=lo, hi=hi,
                             owner_only=owner_only, **HP)
            abi.zero_step_ex(b.reps, b.grads, b.st, t, grad_scale=0.5, owner_only=owner_only,
                             **HP)
        torch.cuda.synchronize()
        full = snapshot(b)
        want = expect_range(before, full, lo, hi, bounds if owner_only else None)
        assert_matches(a, want, f"{entry} [{lo}, {hi})")


@pytest.mark.parametrize("prec", [oracle.FP32, oracle.BF16_MIXED])
def test_single_bucket_leaves_the_rest_untouched(abi, cuda, prec):
    """zero_step_bucket on one bucket at a time, with a bucket size off the
    vector grid (edges at odd indices), in a shuffled order."""
    a, b = twin_cases(abi, cuda, prec, seed=17, off=1)
    bucket_bytes = 24_574
    count = abi.zero_bucket_count(N_ELEMS, prec, bucket_bytes)
    order = np.random.default_rng(3).permutation(count)[:4].tolist() + [count - 1]
    for k in order:
        lo, hi = abi.zero_bucket_range(N_ELEMS, prec, bucket_bytes, k)
        before = snapshot(a)
        abi.zero_step_bucket(a.reps, a.grads, a.st, 1, HP["lr"], HP["beta1"], HP["beta2"],
                             HP["eps"], HP["weight_decay"], bucket_bytes, k, None, None)
        for key, x in [("m", b.m), ("v", b.v)] + ([("master", b.master)] if b.mixed else []) + \
                [(f"replica {r}", b.reps[r]) for r in range(N_RANKS)]:
            x.copy_(torch.from_numpy(before[key].view(np.int16) if before[key].dtype == np.uint16
                                     else before[key]).view(x.dtype))
        abi.zero_step(b.reps, b.grads, b.st, 1, **HP)
        torch.cuda.synchronize()
        want = expect_range(before, snapshot(b), lo, hi)
        assert_matches(a, want, f"bucket {k} [{lo}, {hi})")


@pytest.mark.parametrize("prec", [oracle.FP32, oracle.BF16_MIXED])
@pytest.mark.parametrize("clip", [False, True])
def test_host_input_step_stays_in_bounds(abi, cuda, prec, clip):
    """The chunk-pipelined host-input step with guarded staging, replicas and
    state, chunks that split vector units (40,006 bytes), a staging phase
    shifted by one element: bitwise the device step, nothing written outside a
    buffer, and the host copy of the parameters equal to replica 0."""
    a, b = twin_cases(abi, cuda, prec, seed=23, off=0)
    n, N = N_ELEMS, N_RANKS
    staging = [guarded_empty(n, a.dt, cuda, 1, f"staging {r}") for r in range(N)]
    host = [x.cpu().pin_memory() for x in a.grads]
    out = torch.empty(n, dtype=a.dt).pin_memory()
    norm = guarded_empty(1, torch.float64, cuda, 0, "norm_sq") if clip else None
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    count = abi.zero_grad_norm_scratch_count(n, prec)
    scratch = guarded_empty(count, torch.float64, cuda, 0, "norm scratch")
    ref_norm = guarded_empty(1, torch.float64, cuda, 0, "reference norm_sq")
    host_scratch = guarded_empty(count, torch.float64, cuda, 0, "host-input norm scratch")
    for t in (1, 2):
        o = abi.StepOpts(t, HP["lr"], HP["beta1"], HP["beta2"], HP["eps"], HP["weight_decay"],
                         1.0, 0.05 if clip else 0.0, norm.data_ptr() if clip else None, 0, -1, 0,
                         host_scratch.data_ptr() if clip else None, count if clip else 0)
        abi.zero_step_from_host_ex(a.reps, host, staging, a.st, adamw=o, host_params_out=out,
                                   chunk_bytes=40_006, h2d=h2d, d2h=d2h)
        if clip:
            # the norm of the same buffers (its chunking follows their 16-byte phase)
            abi.zero_grad_norm_sq(staging, prec, scratch, ref_norm, n)
        abi.zero_step_ex(b.reps, b.grads, b.st, t, max_grad_norm=0.05 if clip else 0.0,
                         norm_sq=ref_norm if clip else None, **HP)
        torch.cuda.synchronize()
        check_guards()
        for x, y in [(a.m, b.m), (a.v, b.v)] + list(zip(a.reps, b.reps)):
            assert torch.equal(x, y)
        if clip:
            assert torch.equal(norm, ref_norm)
        assert torch.equal(out, b.reps[0].cpu())
        for s, g in zip(staging, b.grads):
            assert torch.equal(s, g)
