"""GPU parity of sharded global-norm clipping and the accumulation factor.

The squared global norm (zero_grad_norm_sq) against the oracle's squared
shard norms, its bit-reproducibility, and the clipped / scaled step
(zero_step_ex) against the oracle's step with the same options.
"""

import numpy as np
import pytest
import torch

import oracle
from parity_util import assert_fp32_close, flat
from test_gpu_parity import HP, Case, host_of, to_dev

pytestmark = pytest.mark.gpu


def norm_buffers(abi, n, prec, device):
    count = abi.zero_grad_norm_scratch_count(n, prec)
    return (torch.empty(count, dtype=torch.float64, device=device),
            torch.empty(1, dtype=torch.float64, device=device))


@pytest.mark.parametrize("prec", [oracle.FP32, oracle.BF16_MIXED])
@pytest.mark.parametrize("n,N,offset", [(0, 2, 0), (1, 1, 0), (4099, 3, 1), (1_000_003, 4, 0),
                                        (2_000_000, 8, 3), (65_537, 13, 0), (300_007, 5, 2)])
def test_grad_norm_matches_oracle(abi, cuda, n, N, offset, prec):
    rng = np.random.default_rng(n + N)
    mixed = prec == oracle.BF16_MIXED
    dt = torch.bfloat16 if mixed else torch.float32
    hs = []
    for _ in range(N):
        g = rng.normal(0, 1e-2, n).astype(np.float32)
        hs.append(oracle.f32_to_bf16_rne(g) if mixed else g)
    dev = [to_dev(h, dt, cuda, offset) for h in hs]
    scratch, out = norm_buffers(abi, n, prec, cuda)
    abi.zero_grad_norm_sq(dev, prec, scratch, out, n)
    first = out.clone()
    abi.zero_grad_norm_sq(dev, prec, scratch, out, n)
    torch.cuda.synchronize()
    assert torch.equal(first, out)                      # bit-reproducible
    ref = oracle.grad_norm(hs, precision=prec, mode="fp32") ** 2
    assert float(out.item()) == pytest.approx(ref, rel=1e-9, abs=1e-300)


def test_grad_norm_rejects_small_scratch(abi, cuda):
    n = 1_000_000
    dev = [torch.zeros(n, device=cuda) for _ in range(2)]
    scratch = torch.empty(2, dtype=torch.float64, device=cuda)
    out = torch.empty(1, dtype=torch.float64, device=cuda)
    with pytest.raises(abi.ZeroError) as e:
        abi.zero_grad_norm_sq(dev, abi.ZERO_FP32, scratch, out, n)
    assert e.value.code == abi.ZERO_EINVAL


def clipped_step(abi, c, norm_bufs, grad_scale, max_norm):
    scratch, out = norm_bufs
    if max_norm:
        abi.zero_grad_norm_sq(c.grads, c.prec, scratch, out, c.n)
    abi.zero_step_ex(c.reps, c.grads, c.st, c.t, grad_scale=grad_scale,
                     max_grad_norm=max_norm or 0.0, norm_sq=out if max_norm else None, **HP)


@pytest.mark.parametrize("prec", [oracle.FP32, oracle.BF16_MIXED])
@pytest.mark.parametrize("grad_scale,max_norm", [(1.0, 0.05), (0.25, 0.02), (0.5, None),
                                                 (1.0, 1e6)])
def test_clipped_scaled_step_matches_oracle(abi, cuda, prec, grad_scale, max_norm):
    n, N = 1_000_003, 4
    c = Case(abi, cuda, n, N, prec, seed=61)
    bufs = norm_buffers(abi, n, prec, cuda)
    for _ in range(3):
        hg = c.new_grads(scale=1e-3)
        c.t += 1
        c.o_reps, c.o_states = oracle.zero_step(c.o_reps, hg, c.o_states, c.t, precision=prec,
                                                mode="fp32", grad_scale=grad_scale,
                                                max_grad_norm=max_norm, **HP)
        clipped_step(abi, c, bufs, grad_scale, max_norm)
        torch.cuda.synchronize()
        c.compare(exact=False)


def test_step_ex_defaults_equal_zero_step(abi, cuda):
    for prec in (oracle.FP32, oracle.BF16_MIXED):
        a = Case(abi, cuda, 500_009, 8, prec, seed=62)
        b = Case(abi, cuda, 500_009, 8, prec, seed=62)
        a.new_grads()
        for r in range(8):
            b.grads[r].copy_(a.grads[r])
        a.t = b.t = 1
        a.gpu_step()
        abi.zero_step_ex(b.reps, b.grads, b.st, 1, **HP)
        torch.cuda.synchronize()
        for x, y in [(a.m, b.m), (a.v, b.v)] + list(zip(a.reps, b.reps)):
            assert torch.equal(x, y)


def test_step_ex_argument_errors(abi, cuda):
    c = Case(abi, cuda, 1000, 2, oracle.FP32)
    with pytest.raises(abi.ZeroError):      # clipping needs the squared norm
        abi.zero_step_ex(c.reps, c.grads, c.st, 1, max_grad_norm=1.0, **HP)
    with pytest.raises(abi.ZeroError):
        abi.zero_step_ex(c.reps, c.grads, c.st, 1, grad_scale=0.0, **HP)
    with pytest.raises(abi.ZeroError):
        abi.zero_step_ex(c.reps, c.grads, c.st, 1, lo=5, hi=1001, **HP)


def test_optimizer_clipping_host_and_device_agree(abi, cuda):
    from zero_sharded_optimizer_gb300.optimizer import ZeroOptimizer
    n, N = 400_003, 4
    rng = np.random.default_rng(63)
    p0 = torch.from_numpy(rng.normal(0, 0.02, n).astype(np.float32))
    kw = dict(lr=1e-3, weight_decay=0.01, max_grad_norm=0.01, grad_scale=0.5)
    a, b = ZeroOptimizer(n, N, **kw), ZeroOptimizer(n, N, **kw)
    pa = [p0.to(cuda) for _ in range(N)]
    pb = [p0.to(cuda) for _ in range(N)]
    o_reps = [p0.numpy().copy() for _ in range(N)]
    o_st = oracle.init_states(n, N)
    for t in range(1, 3):
        host = [torch.from_numpy(rng.normal(0, 1e-3, n).astype(np.float32)).pin_memory()
                for _ in range(N)]
        a.step(pa, host)
        b.step(pb, [h.to(cuda) for h in host])
        o_reps, o_st = oracle.zero_step(o_reps, [h.numpy() for h in host], o_st, t, lr=1e-3,
                                        weight_decay=0.01, max_grad_norm=0.01, grad_scale=0.5)
        torch.cuda.synchronize()
        assert all(torch.equal(x, y) for x, y in zip(pa, pb))
        assert_fp32_close(host_of(pa[0]), o_reps[0], f"t={t}")
        assert_fp32_close(host_of(a.m), flat(o_st, "m"), f"t={t} m")


@pytest.mark.parametrize("prec", [oracle.FP32, oracle.BF16_MIXED])
@pytest.mark.parametrize("n,N,kind", [(1_000_003, 4, "adamw"), (1_000_003, 8, "adamw"),
                                      (300_007, 2, "adamw"), (300_007, 3, "owner_only"),
                                      (300_007, 1, "adamw"), (65_537, 13, "adamw"),
                                      (500_009, 4, "sgd"), (500_009, 1, "sgd"),
                                      (50_011, 4, "mixed_phase"),
                                      (4099, 3, "adamw"), (2000, 4, "empty_range")])
def test_step_computing_its_own_norm_equals_two_calls(abi, cuda, prec, n, N, kind):
    """zero_step_ex / zero_step_sgd given norm_scratch: the call forms the norm
    itself (its partial sums, their total) and the step follows as a
    programmatic dependent that waits for the norm. Bitwise the same as
    zero_grad_norm_sq followed by the step that reads the norm, over rank
    counts 1-13, both precisions, owner-only, SGD and mixed 16-byte phases
    (the persistent grid), the norm scalar included; for an empty range only
    the norm is written."""
    from test_gpu_sgd import SgdCase
    kw = {}
    if kind == "mixed_phase":
        kw = dict(rep_off=[1, 2, 3, 0], grad_off=[0, 0, 0, 1], state_off=0)
    if kind == "sgd":
        a = SgdCase(abi, cuda, n, N, prec, "damped_wd", seed=81)
        b = SgdCase(abi, cuda, n, N, prec, "damped_wd", seed=81)
    else:
        a = Case(abi, cuda, n, N, prec, seed=81, **kw)
        b = Case(abi, cuda, n, N, prec, seed=81, **kw)
    count = abi.zero_grad_norm_scratch_count(n, prec)
    scratch = torch.empty(count, dtype=torch.float64, device=cuda)
    norm_a = torch.full((1,), -1.0, dtype=torch.float64, device=cuda)
    ref_scratch = torch.empty(count, dtype=torch.float64, device=cuda)
    norm_b = torch.empty(1, dtype=torch.float64, device=cuda)
    lo, hi = (700, 700) if kind == "empty_range" else (0, -1)
    for t in (1, 2):
        a.new_grads(scale=1e-2)
        for r in range(N):
            b.grads[r].copy_(a.grads[r])
        abi.zero_grad_norm_sq(b.grads, prec, ref_scratch, norm_b, n)
        if kind == "sgd":
            abi.zero_step_sgd(a.reps, a.grads, a.st, t, max_grad_norm=0.05, norm_sq=norm_a,
                              norm_scratch=scratch, lo=lo, hi=hi, **a.kw())
            abi.zero_step_sgd(b.reps, b.grads, b.st, t, max_grad_norm=0.05, norm_sq=norm_b,
                              lo=lo, hi=hi, **b.kw())
        else:
            own = kind == "owner_only"
            abi.zero_step_ex(a.reps, a.grads, a.st, t, max_grad_norm=0.05, norm_sq=norm_a,
                             norm_scratch=scratch, grad_scale=0.5, lo=lo, hi=hi, owner_only=own,
                             **HP)
            abi.zero_step_ex(b.reps, b.grads, b.st, t, max_grad_norm=0.05, norm_sq=norm_b,
                             grad_scale=0.5, lo=lo, hi=hi, owner_only=own, **HP)
        torch.cuda.synchronize()
        assert torch.equal(norm_a, norm_b), (float(norm_a), float(norm_b))
        assert float(norm_a) > 0.05 ** 2  # the case clips
        pairs = list(zip(a.reps, b.reps))
        if kind == "sgd":
            pairs.append((a.buf, b.buf))
        else:
            pairs += [(a.m, b.m), (a.v, b.v)]
        if a.mixed:
            pairs.append((a.master, b.master))
        for x, y in pairs:
            assert torch.equal(x, y)


def test_step_computing_its_own_norm_rejects_bad_scratch(abi, cuda):
    n, N = 100_000, 2
    c = Case(abi, cuda, n, N, oracle.FP32, seed=82)
    count = abi.zero_grad_norm_scratch_count(n, oracle.FP32)
    scratch = torch.empty(count, dtype=torch.float64, device=cuda)
    norm = torch.empty(1, dtype=torch.float64, device=cuda)
    with pytest.raises(abi.ZeroError) as e:  # too small
        abi.zero_step_ex(c.reps, c.grads, c.st, 1, max_grad_norm=1.0, norm_sq=norm,
                         norm_scratch=scratch[:count - 1], **HP)
    assert e.value.code == abi.ZERO_EINVAL
    with pytest.raises(abi.ZeroError) as e:  # no output scalar
        abi.zero_step_ex(c.reps, c.grads, c.st, 1, max_grad_norm=1.0, norm_scratch=scratch, **HP)
    assert e.value.code == abi.ZERO_EINVAL
    with pytest.raises(abi.ZeroError) as e:  # the scalar inside the scratch
        abi.zero_step_ex(c.reps, c.grads, c.st, 1, max_grad_norm=1.0, norm_sq=scratch[3:4],
                         norm_scratch=scratch, **HP)
    assert e.value.code == abi.ZERO_EINVAL
    torch.cuda.synchronize()
