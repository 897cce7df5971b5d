"""GPU parity of the fused step with momentum SGD (zero_step_sgd) against the oracle.

The pages name SGD beside AdamW as an elementwise optimizer that ZeRO wraps
unchanged ("Data parallelism and ZeRO stages 1 to 3", section 2, stage 1); the
oracle follows torch.optim.SGD. Same seeded inputs on both sides, compared
element by element: bit-exact in practice, asserted against the parity
tolerances as well.
"""

import numpy as np
import pytest
import torch

import oracle
from parity_util import (assert_bf16_within_one_ulp, assert_fp32_close,
                         assert_same_bits_or_both_nan, check_guards, exact_fraction, flat,
                         guarded_empty)
from test_gpu_parity import host_of, host_tensor, to_dev

pytestmark = pytest.mark.gpu

VARIANTS = {  # momentum, dampening, weight_decay, nesterov
    "plain": (0.0, 0.0, 0.0, False),
    "plain_wd": (0.0, 0.0, 0.05, False),
    "momentum": (0.9, 0.0, 0.0, False),
    "damped_wd": (0.9, 0.1, 0.01, False),
    "nesterov_wd": (0.5, 0.0, 0.1, True),
}


class SgdCase:
    def __init__(self, abi, device, n, N, prec, variant, seed=0, rep_off=None, grad_off=None,
                 state_off=0, lr=0.05, bounds=None):
        self.abi, self.device, self.n, self.N, self.prec = abi, device, n, N, prec
        self.mu, self.damp, self.wd, self.nest = VARIANTS[variant]
        self.lr = lr
        self.rng = np.random.default_rng(seed)
        self.mixed = prec == oracle.BF16_MIXED
        self.dt = torch.bfloat16 if self.mixed else torch.float32
        rep_off = rep_off or [0] * N
        grad_off = grad_off or [0] * N
        init = self.rng.normal(0, 0.5, n).astype(np.float32)
        rep_host = oracle.f32_to_bf16_rne(init) if self.mixed else init
        self.reps = [to_dev(rep_host, self.dt, device, rep_off[r], f"replica {r}")
                     for r in range(N)]
        self.grads = [to_dev(np.zeros(n, np.uint16 if self.mixed else np.float32), self.dt,
                             device, grad_off[r], f"gradient {r}") for r in range(N)]
        f32 = torch.float32
        self.buf = None
        if self.mu:
            self.buf = guarded_empty(n, f32, device, state_off, "momentum buffer").fill_(7.0)
        self.master = None
        master_init = None
        if self.mixed:
            self.master = guarded_empty(n, f32, device, state_off, "master").zero_()
            master_init = to_dev(init, torch.float32, device, state_off, "master_init")
        self.st = abi.zero_init_states(n, N, prec, self.buf, None, self.master, master_init,
                                       bounds=bounds)
        self.bounds = bounds
        self.o_reps = [rep_host.copy() for _ in range(N)]
        self.o_states = oracle.init_states_sgd(n, N, prec, master_init=init, mode="fp32",
                                               bounds=bounds, momentum=self.mu != 0)
        self.t = 0

    def new_grads(self, scale=1.0):
        hs = []
        for r in range(self.N):
            g = self.rng.normal(0, scale, self.n).astype(np.float32)
            if self.mixed:
                g = oracle.f32_to_bf16_rne(g)
            hs.append(g)
            self.grads[r].copy_(host_tensor(g, self.dt))
        return hs

    def kw(self):
        return dict(lr=self.lr, momentum=self.mu, dampening=self.damp,
                    weight_decay=self.wd, nesterov=self.nest)

    def step(self, owner_only=False, **extra):
        hg = self.new_grads()
        self.t += 1
        out, self.o_states = oracle.zero_step_sgd(
            self.o_reps, hg, self.o_states, self.t, precision=self.prec, mode="fp32",
            bounds=self.bounds, all_gather=not owner_only, **self.kw(), **extra)
        self.abi.zero_step_sgd(self.reps, self.grads, self.st, self.t, owner_only=owner_only,
                               **self.kw(), **extra)
        torch.cuda.synchronize()
        if not owner_only:
            self.o_reps = out
        return out

    def compare(self):
        check_guards()  # nothing written outside any buffer
        if self.mu:
            ob = flat(self.o_states, "buf")
            gb = host_of(self.buf)
            assert_fp32_close(gb, ob, "momentum buffer")
            assert exact_fraction(gb, ob) == 1.0
        if self.mixed:
            om = flat(self.o_states, "master")
            gm = host_of(self.master)
            assert_fp32_close(gm, om, "master")
            assert exact_fraction(gm, om) == 1.0
            for r in range(self.N):
                assert_bf16_within_one_ulp(host_of(self.reps[r]), om, f"replica {r}")
        for r in range(self.N):
            got = host_of(self.reps[r])
            if not self.mixed:
                assert_fp32_close(got, self.o_reps[r], f"replica {r}")
            assert np.array_equal(got, self.o_reps[r]), f"replica {r} not bit-exact"


# One rank in fp32 takes two units per thread: 6151 elements leave 1537
# units (one past three blocks' 512) and a 3-element tail; 100_003 and
# 1_000_003 end inside a block's second units.
GRID = [(1, 1), (6151, 1), (100_003, 1), (1_000_003, 1), (7, 3), (33, 4), (4099, 5),
        (100_003, 2), (100_003, 4), (100_003, 8), (65_537, 13), (300_007, 6), (1_000_003, 8)]


@pytest.mark.parametrize("prec", [oracle.FP32, oracle.BF16_MIXED])
@pytest.mark.parametrize("variant", sorted(VARIANTS))
@pytest.mark.parametrize("n,N", GRID)
def test_sgd_step_parity_grid(abi, cuda, n, N, prec, variant):
    c = SgdCase(abi, cuda, n, N, prec, variant, seed=n * 7 + N)
    for _ in range(3):
        c.step()
        c.compare()


@pytest.mark.parametrize("prec", [oracle.FP32, oracle.BF16_MIXED])
@pytest.mark.parametrize("layout", ["shifted", "mixed_phase"])
def test_sgd_unaligned_layouts(abi, cuda, prec, layout):
    n, N = 50_011, 4
    if layout == "shifted":
        kw = dict(rep_off=[3] * N, grad_off=[3] * N, state_off=3)
    else:
        kw = dict(rep_off=[1, 2, 3, 0], grad_off=[0, 0, 0, 1], state_off=0)
    c = SgdCase(abi, cuda, n, N, prec, "damped_wd", seed=21, **kw)
    for _ in range(3):
        c.step()
        c.compare()


@pytest.mark.parametrize("prec", [oracle.FP32, oracle.BF16_MIXED])
def test_sgd_stage3_owner_only_then_gather(abi, cuda, prec):
    n, N = 300_007, 4
    c = SgdCase(abi, cuda, n, N, prec, "nesterov_wd", seed=23)
    b = oracle.shard_bounds(n, N)
    for _ in range(2):
        before = [host_of(x) for x in c.reps]
        shards = c.step(owner_only=True)
        for r in range(N):
            got = host_of(c.reps[r])
            assert np.array_equal(got[b[r]:b[r + 1]], shards[r])
            keep = np.ones(n, bool)
            keep[b[r]:b[r + 1]] = False
            assert np.array_equal(got[keep], before[r][keep])
        abi.zero_gather(c.reps, c.st)
        torch.cuda.synchronize()
        c.o_reps = oracle.gather(shards, prec)
        c.compare()


@pytest.mark.parametrize("prec", [oracle.FP32, oracle.BF16_MIXED])
def test_sgd_whole_tensor_shards(abi, cuda, prec):
    rng = np.random.default_rng(24)
    numels = rng.integers(1, 20_000, 17).tolist()
    n, N = int(sum(numels)), 3
    tb = abi.zero_tensor_shard_bounds(numels, N)
    c = SgdCase(abi, cuda, n, N, prec, "momentum", seed=25, bounds=tb)
    for _ in range(3):
        c.step()
        c.compare()


@pytest.mark.parametrize("prec", [oracle.FP32, oracle.BF16_MIXED])
@pytest.mark.parametrize("N", [4, 1])
def test_sgd_clipped_and_scaled(abi, cuda, prec, N):
    n = 200_003
    c = SgdCase(abi, cuda, n, N, prec, "damped_wd", seed=26)
    norm = torch.empty(1, dtype=torch.float64, device=cuda)
    count = abi.zero_grad_norm_scratch_count(n, prec)
    scratch = torch.empty(count, dtype=torch.float64, device=cuda)
    for max_norm, scale in [(0.5, 1.0), (1e6, 0.25), (0.05, 0.5)]:
        hg = c.new_grads()
        c.t += 1
        c.o_reps, c.o_states = oracle.zero_step_sgd(
            c.o_reps, hg, c.o_states, c.t, precision=prec, mode="fp32", grad_scale=scale,
            max_grad_norm=max_norm, **c.kw())
        abi.zero_grad_norm_sq(c.grads, prec, scratch, norm, n)
        abi.zero_step_sgd(c.reps, c.grads, c.st, c.t, grad_scale=scale, max_grad_norm=max_norm,
                          norm_sq=norm, **c.kw())
        torch.cuda.synchronize()
        # the multiplier comes from a norm summed in another order: within tolerance
        if c.mu:
            assert_fp32_close(host_of(c.buf), flat(c.o_states, "buf"), "buffer")
        for r in range(N):
            if prec == oracle.FP32:
                assert_fp32_close(host_of(c.reps[r]), c.o_reps[r], f"replica {r}")
            else:
                assert_bf16_within_one_ulp(host_of(c.reps[r]), flat(c.o_states, "master"))
        # keep both sides on the same trajectory for the next step
        if c.mu:
            c.buf.copy_(torch.from_numpy(flat(c.o_states, "buf")))
        if c.mixed:
            c.master.copy_(torch.from_numpy(flat(c.o_states, "master")))
        for r in range(N):
            c.reps[r].copy_(host_tensor(c.o_reps[r], c.dt))


@pytest.mark.parametrize("prec", [oracle.FP32, oracle.BF16_MIXED])
@pytest.mark.parametrize("variant,N", [("damped_wd", 4), ("nesterov_wd", 4), ("momentum", 1),
                                       ("plain_wd", 2)])
def test_sgd_nan_and_inf_propagate_like_the_oracle(abi, cuda, prec, variant, N):
    """Momentum SGD with special gradients (NaN in one rank, +Inf, opposite
    infinities, a rank sum that overflows), two steps, one rank included (two
    units per thread): every output equals the oracle bit for bit, NaN
    matching NaN."""
    n = 100_003
    c = SgdCase(abi, cuda, n, N, prec, variant, seed=71)
    rng = np.random.default_rng(72)
    idx = rng.permutation(n)[:4 * 600].reshape(4, 600)
    for _ in range(2):
        hs = []
        for r in range(N):
            g = rng.normal(0, 1e-3, n).astype(np.float32)
            g[idx[0]] = np.nan if r == N - 1 else g[idx[0]]
            g[idx[1]] = np.inf if r == 0 else g[idx[1]]
            if N > 1:
                g[idx[2]] = -np.inf if r == 0 else (np.inf if r == 1 else g[idx[2]])
            g[idx[3]] = 3e38
            hs.append(oracle.f32_to_bf16_rne(g) if c.mixed else g)
            c.grads[r].copy_(host_tensor(hs[-1], c.dt))
        c.t += 1
        with np.errstate(all="ignore"):
            c.o_reps, c.o_states = oracle.zero_step_sgd(c.o_reps, hs, c.o_states, c.t,
                                                        precision=prec, mode="fp32", **c.kw())
        abi.zero_step_sgd(c.reps, c.grads, c.st, c.t, **c.kw())
        torch.cuda.synchronize()
        check_guards()
        if c.mu:
            assert_same_bits_or_both_nan(host_of(c.buf), flat(c.o_states, "buf"), "buffer")
        if c.mixed:
            assert_same_bits_or_both_nan(host_of(c.master), flat(c.o_states, "master"),
                                         "master")
        for r in range(N):
            assert_same_bits_or_both_nan(host_of(c.reps[r]), c.o_reps[r], f"replica {r}")
    assert np.isnan(host_of(c.master if c.mixed else c.reps[0])[idx[0]]).all()


def test_sgd_range_partition_is_bitwise_full_step(abi, cuda):
    n, N = 400_009, 4
    a = SgdCase(abi, cuda, n, N, oracle.FP32, "damped_wd", seed=27)
    b = SgdCase(abi, cuda, n, N, oracle.FP32, "damped_wd", seed=27)
    cuts = [0, 12_345, 200_000, 200_001, n]
    for t in (1, 2):
        a.new_grads()
        for r in range(N):
            b.grads[r].copy_(a.grads[r])
        abi.zero_step_sgd(a.reps, a.grads, a.st, t, **a.kw())
        for lo, hi in zip(cuts, cuts[1:]):
            abi.zero_step_sgd(b.reps, b.grads, b.st, t, lo=lo, hi=hi, **b.kw())
    torch.cuda.synchronize()
    assert torch.equal(a.buf, b.buf)
    for x, y in zip(a.reps, b.reps):
        assert torch.equal(x, y)


def test_sgd_state_and_option_errors(abi, cuda):
    n, N = 1000, 2
    c = SgdCase(abi, cuda, n, N, oracle.FP32, "momentum", seed=1)
    with pytest.raises(abi.ZeroError) as e:   # AdamW needs v
        abi.zero_step(c.reps, c.grads, c.st, 1, lr=1e-3)
    assert e.value.code == abi.ZERO_EINVAL
    with pytest.raises(abi.ZeroError) as e:   # Nesterov with dampening
        abi.zero_step_sgd(c.reps, c.grads, c.st, 1, lr=0.1, momentum=0.9, dampening=0.1,
                          nesterov=True)
    assert e.value.code == abi.ZERO_EINVAL
    with pytest.raises(abi.ZeroError) as e:   # negative momentum
        abi.zero_step_sgd(c.reps, c.grads, c.st, 1, lr=0.1, momentum=-0.5)
    assert e.value.code == abi.ZERO_EINVAL
    plain = SgdCase(abi, cuda, n, N, oracle.FP32, "plain", seed=2)
    with pytest.raises(abi.ZeroError) as e:   # momentum without a buffer
        abi.zero_step_sgd(plain.reps, plain.grads, plain.st, 1, lr=0.1, momentum=0.9)
    assert e.value.code == abi.ZERO_EINVAL
    abi.zero_step_sgd(plain.reps, plain.grads, plain.st, 1, lr=0.1)  # plain SGD is fine
    torch.cuda.synchronize()


@pytest.mark.parametrize("prec", [oracle.FP32, oracle.BF16_MIXED])
def test_sgd_empty_shards_and_empty_vector(abi, cuda, prec):
    numels = [30_011, 9, 70_001]
    n, N = int(sum(numels)), 6
    tb = abi.zero_tensor_shard_bounds(numels, N)
    assert any(tb[r] == tb[r + 1] for r in range(N))
    c = SgdCase(abi, cuda, n, N, prec, "nesterov_wd", seed=51, bounds=tb)
    for _ in range(3):
        c.step()
        c.compare()
    z = SgdCase(abi, cuda, 0, 2, prec, "momentum", seed=52)
    z.abi.zero_step_sgd(z.reps, z.grads, z.st, 1, **z.kw())
    torch.cuda.synchronize()


@pytest.mark.parametrize("prec", [oracle.FP32, oracle.BF16_MIXED])
def test_optimizer_sgd_and_stage3_with_host_gradients(abi, cuda, prec):
    """ZeroOptimizer with host gradients (the chunk-pipelined host-input step)
    equals the same optimizer fed device gradients, bit for bit: momentum SGD,
    stage 3 (owner-only step; the host copy of the parameters takes each shard
    from its owner and the other replica elements stay as they were), both
    together, AdamW with a gradient scale, and clipping (the host-input call
    computes the norm after every chunk has arrived; the device path uses
    zero_grad_norm_sq with its own scratch)."""
    from zero_sharded_optimizer_gb300.optimizer import ZeroOptimizer
    n, N = 200_003, 4
    mixed = prec == oracle.BF16_MIXED
    dt = torch.bfloat16 if mixed else torch.float32
    rng = np.random.default_rng(61)
    init = torch.from_numpy(rng.normal(0, 0.02, n).astype(np.float32))
    bounds = oracle.shard_bounds(n, N)
    for kw in (dict(optimizer="sgd", momentum=0.9, nesterov=True), dict(stage=3),
               dict(stage=3, optimizer="sgd", momentum=0.9), dict(grad_scale=0.25),
               dict(max_grad_norm=0.05), dict(max_grad_norm=0.05, grad_scale=0.5, stage=3),
               dict(optimizer="sgd", momentum=0.9, max_grad_norm=0.05)):
        stage3 = kw.get("stage") == 3
        common = dict(precision=prec, lr=1e-3, weight_decay=0.01,
                      master_init=init if mixed else None, **kw)
        a, b = ZeroOptimizer(n, N, **common), ZeroOptimizer(n, N, **common)
        pa = [init.to(cuda).to(dt) for _ in range(N)]
        pb = [p.clone() for p in pa]
        out = torch.empty(n, dtype=dt).pin_memory()
        for _ in range(3):
            host = [torch.from_numpy(rng.normal(0, 1e-3, n).astype(np.float32)).to(dt)
                    .pin_memory() for _ in range(N)]
            before = [p.clone() for p in pa]
            a.step(pa, host, host_params_out=out, chunk_bytes=1 << 18)
            b.step(pb, [h.to(cuda) for h in host])
            if stage3:
                b.gather(pb)
            torch.cuda.synchronize()
            assert torch.equal(out, pb[0].cpu()), kw
            if stage3:
                for r in range(N):
                    lo, hi = bounds[r], bounds[r + 1]
                    assert torch.equal(pa[r][:lo], before[r][:lo]), (kw, r)
                    assert torch.equal(pa[r][hi:], before[r][hi:]), (kw, r)
                a.gather(pa)
        torch.cuda.synchronize()
        assert all(torch.equal(x, y) for x, y in zip(pa, pb)), kw
        for key in ("m", "v", "master"):
            x, y = getattr(a, key), getattr(b, key)
            assert (x is None and y is None) or torch.equal(x, y)
        if kw.get("max_grad_norm"):
            assert torch.equal(a._norm, b._norm), kw
            assert float(a._norm) > 0.05 ** 2, "the case must clip"


def test_clipped_host_step_checks_norm_sq_before_queuing(abi, cuda):
    """The clipped host-input step refuses a misaligned or overlapping norm_sq,
    and a missing, short, misaligned or overlapping norm scratch, before any
    copy is queued: the staging buffers keep their contents."""
    n, N = 50_000, 2
    reps = [torch.zeros(n, device=cuda) for _ in range(N)]
    m, v = torch.empty(n, device=cuda), torch.empty(n, device=cuda)
    st = abi.zero_init_states(n, N, abi.ZERO_FP32, m, v, None, None)
    staging = [torch.full((n,), 7.0, device=cuda) for _ in range(N)]
    host = [torch.ones(n).pin_memory() for _ in range(N)]
    scalar = torch.empty(2, dtype=torch.float64, device=cuda)
    count = abi.zero_grad_norm_scratch_count(n, abi.ZERO_FP32)
    scratch = torch.empty(count, dtype=torch.float64, device=cuda)
    sp = scratch.data_ptr()
    for ptr, sc, cnt, code in ((scalar.data_ptr() + 4, sp, count, abi.ZERO_EALIGN),
                               (staging[1].data_ptr() + 800, sp, count, abi.ZERO_EINVAL),
                               (scalar.data_ptr(), None, 0, abi.ZERO_EINVAL),      # no scratch
                               (scalar.data_ptr(), sp, count - 1, abi.ZERO_EINVAL),  # too small
                               (scalar.data_ptr(), sp + 4, count - 1, abi.ZERO_EALIGN),
                               (scalar.data_ptr(), staging[0].data_ptr(), count, abi.ZERO_EINVAL)):
        o = abi.StepOpts(1, 1e-3, 0.9, 0.999, 1e-8, 0.0, 1.0, 1.0, ptr, 0, -1, 0, sc, cnt)
        with pytest.raises(abi.ZeroError) as e:
            abi.zero_step_from_host_ex(reps, host, staging, st, adamw=o)
        assert e.value.code == code
    torch.cuda.synchronize()
    assert all(bool((s == 7.0).all()) for s in staging)
    st.close()
