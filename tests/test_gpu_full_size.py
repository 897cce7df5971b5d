"""Parity at the workloads' full sizes, in the benchmark's launch configuration.

Inputs are generated on the device (seeded). Before each step the sampled
indices' inputs are copied back; after it, their outputs. The oracle computes
the sampled outputs one by one (the step is elementwise, so a sample is an
exact sub-problem), and the replicas are checked bitwise equal on the device
over all n. Samples: random indices plus every shard and bucket edge and both
ends of the vector.
"""

import numpy as np
import pytest
import torch

import oracle
from parity_util import assert_bf16_within_one_ulp, assert_fp32_close
from zero_sharded_optimizer_gb300 import inputs

pytestmark = pytest.mark.gpu


def sample_indices(n, N, bucket_ranges=(), k=1 << 15, seed=0):
    rng = np.random.default_rng(seed)
    idx = set(rng.integers(0, n, k).tolist())
    edges = set(oracle.shard_bounds(n, N)) | {0, n}
    for lo, hi in bucket_ranges:
        edges |= {lo, hi}
    for e in edges:
        idx |= {e + d for d in range(-9, 9) if 0 <= e + d < n}
    return np.array(sorted(idx), dtype=np.int64)


def oracle_on_sample(wl, t, g_s, p_s, m_s, v_s, master_s, grad_scale=1.0):
    """The oracle's step on the sampled sub-problem (k indices, N ranks);
    ``grad_scale`` multiplies the mean gradient (a clip multiplier formed from
    the whole vector's norm, since the sample's own norm is not that)."""
    N, k = wl.N, len(m_s)
    b = oracle.shard_bounds(k, N)
    states = []
    for i in range(N):
        st = {"m": m_s[b[i]:b[i + 1]].copy(), "v": v_s[b[i]:b[i + 1]].copy()}
        if master_s is not None:
            st["master"] = master_s[b[i]:b[i + 1]].copy()
        states.append(st)
    reps, new = oracle.zero_step([p_s] * N, g_s, states, t, lr=wl.lr, beta1=wl.beta1,
                                 beta2=wl.beta2, eps=wl.eps, weight_decay=wl.weight_decay,
                                 precision=wl.precision, mode="fp32", grad_scale=grad_scale)
    cat = lambda key: np.concatenate([s[key] for s in new])  # noqa: E731
    return reps[0], cat("m"), cat("v"), (cat("master") if master_s is not None else None)


@pytest.mark.parametrize("name", ["fp32_25m", "gpt2_small", "fp32_320m", "mixed_1p3b"])
def test_full_size_sampled(abi, cuda, name):
    from zero_sharded_optimizer_gb300.optimizer import ZeroOptimizer
    wl = inputs.WORKLOADS[name]
    n, N = wl.n, wl.N
    mixed = wl.precision == inputs.BF16_MIXED
    init = inputs.init_params_fp32(n, wl, seed=0, device=cuda)
    reps = inputs.make_replicas(init, N, wl.precision)
    grads = inputs.make_grads(n, N, wl.precision, device=cuda)
    opt = ZeroOptimizer(n, N, wl.precision, lr=wl.lr, betas=(wl.beta1, wl.beta2), eps=wl.eps,
                        weight_decay=wl.weight_decay, master_init=init if mixed else None)
    del init
    ranges = opt.bucket_ranges(wl.bucket_bytes) if wl.bucket_bytes else []
    idx = sample_indices(n, N, ranges, seed=len(name))
    idx_d = torch.from_numpy(idx).to(cuda)
    take = lambda x: inputs.to_numpy_storage(x[idx_d])  # noqa: E731
    producer, side = torch.cuda.Stream(), torch.cuda.Stream()
    for t in range(1, wl.steps + 1):
        p_before = take(opt.master) if mixed else take(reps[0])
        m_before, v_before = take(opt.m), take(opt.v)
        if wl.bucket_bytes:
            # gradients arrive bucket by bucket, in reverse index order
            ready = []
            producer.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(producer):
                for lo, hi in ranges:
                    inputs.fill_grads(grads, wl, step=t, lo=lo, hi=hi)
                    ev = torch.cuda.Event()
                    ev.record(producer)
                    ready.append(ev)
            side.wait_stream(torch.cuda.current_stream())
            opt.step_bucketed(reps, grads, ready, side, wl.bucket_bytes, timeout_ms=600_000)
        else:
            inputs.fill_grads(grads, wl, step=t)
            opt.step(reps, grads)
        torch.cuda.synchronize()
        g_s = [take(g) for g in grads]
        ref_p, ref_m, ref_v, ref_master = oracle_on_sample(
            wl, t, g_s, p_before, m_before, v_before, p_before if mixed else None)
        assert_fp32_close(take(opt.m), ref_m, f"{name} t={t} m")
        assert_fp32_close(take(opt.v), ref_v, f"{name} t={t} v")
        if mixed:
            assert_fp32_close(take(opt.master), ref_master, f"{name} t={t} master")
            for r in range(N):
                assert_bf16_within_one_ulp(take(reps[r]), ref_master, f"{name} t={t} rep {r}")
        else:
            for r in range(N):
                assert_fp32_close(take(reps[r]), ref_p, f"{name} t={t} rep {r}")
        for r in range(1, N):
            assert torch.equal(reps[r], reps[0])
        if wl.zero_frac:
            # the shared zero mask leaves ~1% of indices with an exact zero mean
            zeros = np.all(np.stack([inputs.to_numpy_storage(g[idx_d]) for g in grads]) == 0, 0)
            assert 0.003 < zeros.mean() < 0.03


def oracle_sgd_on_sample(wl, t, g_s, p_s, buf_s, master_s, momentum):
    N, k = wl.N, len(p_s)
    b = oracle.shard_bounds(k, N)
    states = []
    for i in range(N):
        st = {"buf": buf_s[b[i]:b[i + 1]].copy()}
        if master_s is not None:
            st["master"] = master_s[b[i]:b[i + 1]].copy()
        states.append(st)
    reps, new = oracle.zero_step_sgd([p_s] * N, g_s, states, t, lr=wl.lr, momentum=momentum,
                                     weight_decay=wl.weight_decay, precision=wl.precision,
                                     mode="fp32")
    cat = lambda key: np.concatenate([s[key] for s in new])  # noqa: E731
    return reps[0], cat("buf"), (cat("master") if master_s is not None else None)


@pytest.mark.parametrize("name", ["gpt2_small", "fp32_320m"])
@pytest.mark.parametrize("variant", ["sgd", "stage3"])
def test_full_size_sampled_sgd_and_stage3(abi, cuda, name, variant):
    """Momentum SGD, and the stage-3 owner-only step followed by the gather, at
    full size: sampled outputs against the oracle; after the gather every
    replica equal to the owner's on the device over all n."""
    from zero_sharded_optimizer_gb300.optimizer import ZeroOptimizer
    wl = inputs.WORKLOADS[name]
    n, N = wl.n, wl.N
    mixed = wl.precision == inputs.BF16_MIXED
    sgd = variant == "sgd"
    init = inputs.init_params_fp32(n, wl, seed=1, device=cuda)
    reps = inputs.make_replicas(init, N, wl.precision)
    grads = inputs.make_grads(n, N, wl.precision, device=cuda)
    opt = ZeroOptimizer(n, N, wl.precision, lr=wl.lr, betas=(wl.beta1, wl.beta2), eps=wl.eps,
                        weight_decay=wl.weight_decay, master_init=init if mixed else None,
                        optimizer="sgd" if sgd else "adamw", momentum=0.9 if sgd else 0.0,
                        stage=2 if sgd else 3)
    del init
    idx = sample_indices(n, N, seed=7 + len(name))
    idx_d = torch.from_numpy(idx).to(cuda)
    take = lambda x: inputs.to_numpy_storage(x[idx_d])  # noqa: E731
    bounds = np.array(oracle.shard_bounds(n, N))
    owner = np.searchsorted(bounds, idx, side="right") - 1
    for t in range(1, 4):
        p_before = take(opt.master) if mixed else take(reps[0])
        s_before = [take(opt.m)] if sgd else [take(opt.m), take(opt.v)]
        inputs.fill_grads(grads, wl, step=t, seed=1)
        opt.step(reps, grads)
        torch.cuda.synchronize()
        g_s = [take(g) for g in grads]
        if sgd:
            ref_p, ref_buf, ref_master = oracle_sgd_on_sample(
                wl, t, g_s, p_before, s_before[0], p_before if mixed else None, 0.9)
            assert_fp32_close(take(opt.m), ref_buf, f"{name} t={t} buf")
        else:
            ref_p, ref_m, ref_v, ref_master = oracle_on_sample(
                wl, t, g_s, p_before, s_before[0], s_before[1], p_before if mixed else None)
            assert_fp32_close(take(opt.m), ref_m, f"{name} t={t} m")
            assert_fp32_close(take(opt.v), ref_v, f"{name} t={t} v")
            # released: each replica is current only over its own shard
            own = np.stack([take(reps[r]) for r in range(N)])[owner, np.arange(len(idx))]
            if mixed:
                assert_bf16_within_one_ulp(own, ref_master, f"{name} t={t} own shards")
            else:
                assert_fp32_close(own, ref_p, f"{name} t={t} own shards")
            opt.gather(reps)
            torch.cuda.synchronize()
        if mixed:
            assert_fp32_close(take(opt.master), ref_master, f"{name} t={t} master")
            for r in range(N):
                assert_bf16_within_one_ulp(take(reps[r]), ref_master, f"{name} t={t} rep {r}")
        else:
            for r in range(N):
                assert_fp32_close(take(reps[r]), ref_p, f"{name} t={t} rep {r}")
        for r in range(1, N):
            assert torch.equal(reps[r], reps[0])


def test_indices_beyond_int32(abi, cuda):
    """The largest single buffer: n = 2^31 + 12,345 fp32 parameters over two
    ranks (about 60 GB on the device at the peak), one step, sampled around
    the 2^31 element boundary, the shard edge and both ends."""
    import dataclasses
    from zero_sharded_optimizer_gb300.optimizer import ZeroOptimizer
    wl = dataclasses.replace(inputs.WORKLOADS["fp32_320m"], name="fp32_2g", n=(1 << 31) + 12_345,
                             N=2, steps=1)
    assert wl.zero_frac == 0  # keeps the generator's scratch to one buffer
    n, N = wl.n, wl.N
    init = inputs.init_params_fp32(n, wl, seed=3, device=cuda)
    reps = inputs.make_replicas(init, N, wl.precision)
    del init
    grads = inputs.make_grads(n, N, wl.precision, device=cuda)
    inputs.fill_grads(grads, wl, step=1, seed=3)
    opt = ZeroOptimizer(n, N, wl.precision, lr=wl.lr, betas=(wl.beta1, wl.beta2), eps=wl.eps,
                        weight_decay=wl.weight_decay)
    idx = sample_indices(n, N, [(0, 1 << 31), (1 << 31, n)], k=1 << 14, seed=31)
    idx_d = torch.from_numpy(idx).to(cuda)
    take = lambda x: inputs.to_numpy_storage(x[idx_d])  # noqa: E731
    p_before, m_before, v_before = take(reps[0]), take(opt.m), take(opt.v)
    opt.step(reps, grads)
    torch.cuda.synchronize()
    ref_p, ref_m, ref_v, _ = oracle_on_sample(wl, 1, [take(g) for g in grads], p_before,
                                              m_before, v_before, None)
    assert_fp32_close(take(opt.m), ref_m, "2^31+ m")
    assert_fp32_close(take(opt.v), ref_v, "2^31+ v")
    for r in range(N):
        assert_fp32_close(take(reps[r]), ref_p, f"2^31+ rep {r}")
    assert torch.equal(reps[1], reps[0])
    assert ((1 << 31) + 5) in set(idx.tolist())
    # the gather past 2^31: clear what each replica does not own, then gather
    half = n // 2 + (n % 2)
    want = reps[0].clone()
    reps[0][half:].zero_()
    reps[1][:half].zero_()
    abi.zero_gather(reps, opt.states)
    torch.cuda.synchronize()
    assert torch.equal(reps[0], want) and torch.equal(reps[1], want)
    del want
    # the DDP mean past 2^31, bit for bit on the samples
    g_s = [take(g) for g in grads]
    abi.ddp_allreduce_mean(grads, wl.precision)
    torch.cuda.synchronize()
    ref = oracle.allreduce_mean(g_s, wl.precision, mode="fp32")
    for r in range(N):
        assert np.array_equal(take(grads[r]), ref[r])


def oracle_norm_sq(grads, precision, chunk=1 << 23):
    """The oracle's squared norm of the whole mean gradient, from host copies
    of the device gradients taken chunk by chunk (squared norms add over
    disjoint chunks)."""
    n = grads[0].numel()
    total = 0.0
    for lo in range(0, n, chunk):
        hi = min(n, lo + chunk)
        part = [inputs.to_numpy_storage(g[lo:hi]) for g in grads]
        total += oracle.grad_norm(part, precision=precision, mode="fp32") ** 2
    return total


@pytest.mark.parametrize("name", ["gpt2_small", "fp32_320m"])
def test_full_size_sampled_clipped(abi, cuda, name):
    """Sharded global-norm clipping at full size, as the bench's clipped line
    runs it: ZeroOptimizer with max_grad_norm and device gradients, so
    zero_step_ex forms the norm itself (thousands of 32,768-element partial
    sums, added in the step's prologue). The norm against the oracle's, over
    the whole vector; the sampled outputs against the oracle's step with the
    clip multiplier formed from that whole-vector norm."""
    import math
    from zero_sharded_optimizer_gb300.optimizer import ZeroOptimizer
    wl = inputs.WORKLOADS[name]
    n, N = wl.n, wl.N
    mixed = wl.precision == inputs.BF16_MIXED
    max_norm = 1.0
    init = inputs.init_params_fp32(n, wl, seed=2, device=cuda)
    reps = inputs.make_replicas(init, N, wl.precision)
    grads = inputs.make_grads(n, N, wl.precision, device=cuda)
    opt = ZeroOptimizer(n, N, wl.precision, lr=wl.lr, betas=(wl.beta1, wl.beta2), eps=wl.eps,
                        weight_decay=wl.weight_decay, master_init=init if mixed else None,
                        max_grad_norm=max_norm)
    del init
    idx = sample_indices(n, N, seed=11 + len(name))
    idx_d = torch.from_numpy(idx).to(cuda)
    take = lambda x: inputs.to_numpy_storage(x[idx_d])  # noqa: E731
    assert abi.zero_grad_norm_scratch_count(n, wl.precision) > 3000  # thousands of partials
    for t in (1, 2):
        p_before = take(opt.master) if mixed else take(reps[0])
        m_before, v_before = take(opt.m), take(opt.v)
        inputs.fill_grads(grads, wl, step=t, seed=2)
        opt.step(reps, grads)
        torch.cuda.synchronize()
        ref_nsq = oracle_norm_sq(grads, wl.precision)
        assert float(opt._norm.item()) == pytest.approx(ref_nsq, rel=1e-9)
        mult = oracle.grad_multiplier(math.sqrt(ref_nsq), 1.0, max_norm)
        assert mult < 0.5, "the case must clip"
        g_s = [take(g) for g in grads]
        ref_p, ref_m, ref_v, ref_master = oracle_on_sample(
            wl, t, g_s, p_before, m_before, v_before, p_before if mixed else None,
            grad_scale=mult)
        assert_fp32_close(take(opt.m), ref_m, f"{name} t={t} m")
        assert_fp32_close(take(opt.v), ref_v, f"{name} t={t} v")
        if mixed:
            assert_fp32_close(take(opt.master), ref_master, f"{name} t={t} master")
            for r in range(N):
                assert_bf16_within_one_ulp(take(reps[r]), ref_master, f"{name} t={t} rep {r}")
        else:
            for r in range(N):
                assert_fp32_close(take(reps[r]), ref_p, f"{name} t={t} rep {r}")
        for r in range(1, N):
            assert torch.equal(reps[r], reps[0])
