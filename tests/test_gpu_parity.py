"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Inputs are seeded numpy draws copied to the device; the oracle sees the same
bytes. Sizes span many vector units, several CTAs and ragged heads/tails;
offset views exercise the unaligned and mixed-phase paths. Tolerances are in
parity_util.
"""

import numpy as np
import pytest
import torch

import oracle
from parity_util import (assert_bf16_within_one_ulp, assert_fp32_close,
                         assert_same_bits_or_both_nan, check_guards, exact_fraction, flat,
                         guarded_empty)
from zero_sharded_optimizer_gb300 import inputs

pytestmark = pytest.mark.gpu

HP = dict(lr=3e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.01)


def host_tensor(host, dtype):
    """CPU tensor of `host` (float32, or bf16 bits as uint16) in `dtype`."""
    if dtype == torch.bfloat16:
        return torch.from_numpy(host.view(np.int16).copy()).view(torch.bfloat16)
    return torch.from_numpy(host.copy())


def to_dev(host, dtype, device, offset=0, what="buffer"):
    """Device view of `host` (float32, or bf16 bits as uint16) starting `offset`
    elements into a guarded allocation: every element around the view holds a
    sentinel that the conftest checks after the test (parity_util.GUARD)."""
    view = guarded_empty(host.shape[0], dtype, device, offset, what)
    view.copy_(host_tensor(host, dtype))
    return view


def host_of(t):
    return inputs.to_numpy_storage(t)


class Case:
    """One problem: device buffers, oracle state, and a step that checks both."""

    def __init__(self, abi, device, n, N, prec, seed=0, rep_off=None, grad_off=None,
                 state_off=0, hp=None):
        self.abi, self.device, self.n, self.N, self.prec = abi, device, n, N, prec
        self.hp = dict(HP if hp is None else hp)
        self.rng = np.random.default_rng(seed)
        self.mixed = prec == oracle.BF16_MIXED
        self.dt = torch.bfloat16 if self.mixed else torch.float32
        rep_off = rep_off or [0] * N
        self.grad_off = grad_off or [0] * N
        init = self.rng.normal(0, 0.5, n).astype(np.float32)
        if self.mixed:
            rep_host = oracle.f32_to_bf16_rne(init)    # replicas hold RNE(init)
        else:
            rep_host = init
        self.reps = [to_dev(rep_host, self.dt, device, rep_off[r], f"replica {r}")
                     for r in range(N)]
        self.grads = [to_dev(np.zeros(n, np.uint16 if self.mixed else np.float32), self.dt,
                             device, self.grad_off[r], f"gradient {r}") for r in range(N)]
        f32 = torch.float32
        self.m = guarded_empty(n, f32, device, state_off, "m").fill_(7.0)
        self.v = guarded_empty(n, f32, device, state_off, "v").fill_(7.0)
        self.master = None
        master_init = None
        if self.mixed:
            self.master = guarded_empty(n, f32, device, state_off, "master").zero_()
            master_init = to_dev(init, torch.float32, device, state_off, "master_init")
        self.st = abi.zero_init_states(n, N, prec, self.m, self.v, self.master, master_init)
        self.o_reps = [rep_host.copy() for _ in range(N)]
        self.o_states = oracle.init_states(n, N, prec, master_init=init, mode="fp32")
        self.t = 0

    def new_grads(self, scale=1.0):
        hs = []
        for r in range(self.N):
            g = (self.rng.normal(0, scale, self.n)).astype(np.float32)
            if self.mixed:
                g = oracle.f32_to_bf16_rne(g)
            hs.append(g)
            self.grads[r].copy_(host_tensor(g, self.dt))
        return hs

    def oracle_step(self, host_grads):
        self.t += 1
        self.o_reps, self.o_states = oracle.zero_step(
            self.o_reps, host_grads, self.o_states, self.t, precision=self.prec, mode="fp32",
            **self.hp)

    def gpu_step(self):
        self.abi.zero_step(self.reps, self.grads, self.st, self.t, **self.hp)

    def step(self, scale=1.0):
        hg = self.new_grads(scale)
        self.oracle_step(hg)
        self.gpu_step()
        torch.cuda.synchronize()

    def compare(self, exact=False):
        check_guards()  # nothing written outside any buffer
        om, ov = flat(self.o_states, "m"), flat(self.o_states, "v")
        gm, gv = host_of(self.m), host_of(self.v)
        assert_fp32_close(gm, om, "m")
        assert_fp32_close(gv, ov, "v")
        if self.mixed:
            omaster = flat(self.o_states, "master")
            assert_fp32_close(host_of(self.master), omaster, "master")
            for r in range(self.N):
                assert_bf16_within_one_ulp(host_of(self.reps[r]), omaster, f"replica {r}")
        else:
            for r in range(self.N):
                assert_fp32_close(host_of(self.reps[r]), self.o_reps[r], f"replica {r}")
        # all replicas bitwise equal to each other (the all-gather)
        r0 = host_of(self.reps[0])
        for r in range(1, self.N):
            assert np.array_equal(host_of(self.reps[r]), r0)
        if exact:
            assert exact_fraction(gm, om) == 1.0
            assert exact_fraction(gv, ov) == 1.0
            assert np.array_equal(r0, self.o_reps[0])
            if self.mixed:
                assert exact_fraction(host_of(self.master), flat(self.o_states, "master")) == 1.0


GRID = [(1, 1), (5, 2), (7, 3), (33, 4), (4099, 5), (4099, 8), (100_003, 1), (100_003, 2),
        (100_003, 3), (100_003, 4), (100_003, 8), (65_537, 13), (1_000_003, 4), (1_000_003, 8),
        (300_007, 5), (300_007, 6), (300_007, 7), (2_000_000, 2)]


@pytest.mark.parametrize("prec", [oracle.FP32, oracle.BF16_MIXED])
@pytest.mark.parametrize("n,N", GRID)
def test_step_parity_grid(abi, cuda, n, N, prec):
    c = Case(abi, cuda, n, N, prec, seed=n * 31 + N)
    for _ in range(3):
        c.step()
        c.compare(exact=True)


def test_tiny_adam_workload(abi, cuda):
    """n=10,007 fp32 params, N=2, U(-1,1) params and N(0,1) grads from
    default_rng(0), Adam lr=1e-2 (0.9, 0.999), eps=1e-8, wd=0, t=1..5: every
    element of every output."""
    wl = inputs.WORKLOADS["tiny_adam"]
    params, grads = inputs.tiny_adam_numpy(wl.n, wl.N, wl.steps, seed=0)
    hp = dict(lr=wl.lr, beta1=wl.beta1, beta2=wl.beta2, eps=wl.eps, weight_decay=wl.weight_decay)
    reps = [torch.from_numpy(params.copy()).to(cuda) for _ in range(wl.N)]
    gdev = [torch.empty(wl.n, dtype=torch.float32, device=cuda) for _ in range(wl.N)]
    m = torch.empty(wl.n, dtype=torch.float32, device=cuda)
    v = torch.empty_like(m)
    st = abi.zero_init_states(wl.n, wl.N, abi.ZERO_FP32, m, v)
    o_reps = [params.copy() for _ in range(wl.N)]
    o_st = oracle.init_states(wl.n, wl.N)
    assert abi.zero_shard_bounds(wl.n, wl.N) == [0, 5004, 10007]
    for t in range(1, wl.steps + 1):
        for r in range(wl.N):
            gdev[r].copy_(torch.from_numpy(grads[t - 1][r]))
        abi.zero_step(reps, gdev, st, t, **hp)
        o_reps, o_st = oracle.zero_step(o_reps, grads[t - 1], o_st, t, mode="fp32", **hp)
        torch.cuda.synchronize()
        for r in range(wl.N):
            assert_fp32_close(host_of(reps[r]), o_reps[r], f"t={t} replica {r}")
            assert np.array_equal(host_of(reps[r]), o_reps[r])
        assert np.array_equal(host_of(m), flat(o_st, "m"))
        assert np.array_equal(host_of(v), flat(o_st, "v"))


@pytest.mark.parametrize("prec", [oracle.FP32, oracle.BF16_MIXED])
@pytest.mark.parametrize("layout", ["shifted", "mixed_phase", "per_rank"])
def test_unaligned_layouts(abi, cuda, prec, layout):
    n, N = 50_011, 4
    if layout == "shifted":        # every buffer shifted by the same amount: vector path + head
        kw = dict(rep_off=[3] * N, grad_off=[3] * N, state_off=3)
    elif layout == "mixed_phase":  # phases differ: scalar path
        kw = dict(rep_off=[1, 2, 3, 0], grad_off=[0, 0, 0, 1], state_off=0)
    else:
        kw = dict(rep_off=[5] * N, grad_off=[5] * N, state_off=1)
    c = Case(abi, cuda, n, N, prec, seed=7, **kw)
    for _ in range(2):
        c.step()
        c.compare(exact=True)


def test_hyperparameters_honoured(abi, cuda):
    for hp in [dict(lr=0.1, beta1=0.5, beta2=0.6, eps=1e-3, weight_decay=0.0),
               dict(lr=1e-4, beta1=0.0, beta2=0.0, eps=0.0, weight_decay=0.3),
               dict(lr=0.0, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.5)]:
        c = Case(abi, cuda, 9_999, 3, oracle.FP32, seed=3, hp=hp)
        for _ in range(3):
            c.step()
            c.compare(exact=True)


def test_tiny_and_zero_gradients(abi, cuda):
    # gradients ~1e-7 (the eps term matters) and exact zeros (no movement)
    c = Case(abi, cuda, 20_000, 4, oracle.FP32, seed=4)
    c.step(scale=1e-7)
    c.compare(exact=True)
    before = host_of(c.reps[0]).copy()
    for g in c.grads:
        g.zero_()
    c.oracle_step([np.zeros(c.n, np.float32)] * c.N)
    c.gpu_step()
    torch.cuda.synchronize()
    c.compare(exact=True)
    assert not np.array_equal(host_of(c.reps[0]), before)   # decay still applies


def test_empty_and_degenerate(abi, cuda):
    for n, N in [(0, 1), (0, 4), (3, 5), (1, 64), (1000, 64)]:
        for prec in (oracle.FP32, oracle.BF16_MIXED):
            c = Case(abi, cuda, n, N, prec, seed=n + N)
            c.step()
            c.compare(exact=True)
    with pytest.raises(abi.ZeroError):
        Case(abi, cuda, 10, 65, oracle.FP32)


def test_state_views_and_init(abi, cuda):
    n, N = 10_007, 3
    c = Case(abi, cuda, n, N, oracle.BF16_MIXED, seed=5)
    torch.cuda.synchronize()
    assert np.all(host_of(c.m) == 0) and np.all(host_of(c.v) == 0)
    b = abi.zero_shard_bounds(n, N)
    for r in range(N):
        view = c.st.view(r)
        assert (view["lo"], view["hi"]) == (b[r], b[r + 1])
        assert view["m"] == c.m.data_ptr() + 4 * b[r]
        assert view["v"] == c.v.data_ptr() + 4 * b[r]
        assert view["master"] == c.master.data_ptr() + 4 * b[r]
    assert c.st.info() == (n, N, oracle.BF16_MIXED)


@pytest.mark.parametrize("prec", [oracle.FP32, oracle.BF16_MIXED])
def test_range_partition_is_bitwise_full_step(abi, cuda, prec):
    n, N = 200_003, 4
    a = Case(abi, cuda, n, N, prec, seed=9)
    b = Case(abi, cuda, n, N, prec, seed=9)
    cuts = [0, 1, 17, 4096, 99_999, 100_001, 150_000, n]
    for t in range(1, 3):
        hg = a.new_grads()
        for r in range(N):
            b.grads[r].copy_(a.grads[r])
        a.t = b.t = t
        a.gpu_step()
        for lo, hi in zip(cuts, cuts[1:]):
            abi.zero_step_range(b.reps, b.grads, b.st, t, HP["lr"], HP["beta1"], HP["beta2"],
                                HP["eps"], HP["weight_decay"], lo, hi)
        torch.cuda.synchronize()
        for x, y in [(a.m, b.m), (a.v, b.v)] + list(zip(a.reps, b.reps)):
            assert torch.equal(x, y)
    with pytest.raises(abi.ZeroError):
        abi.zero_step_range(b.reps, b.grads, b.st, 1, 1e-3, 0.9, 0.9, 1e-8, 0.0, 5, n + 1)


@pytest.mark.parametrize("prec", [oracle.FP32, oracle.BF16_MIXED])
def test_bucketed_equals_monolithic(abi, cuda, prec):
    n, N = 300_007, 8
    bucket_bytes = 24_574          # not a multiple of 16 bytes: bucket edges off the vector grid
    a = Case(abi, cuda, n, N, prec, seed=11)
    b = Case(abi, cuda, n, N, prec, seed=11)
    es = 2 if prec == oracle.BF16_MIXED else 4
    ranges = [abi.zero_bucket_range(n, prec, bucket_bytes, k)
              for k in range(abi.zero_bucket_count(n, prec, bucket_bytes))]
    assert ranges == oracle.bucket_bounds(n, es, bucket_bytes)
    producer = torch.cuda.Stream()
    side = torch.cuda.Stream()
    for t in range(1, 4):
        a.new_grads()
        a.t = b.t = t
        a.gpu_step()
        # the producer writes each bucket (reverse index order), then marks it ready
        ready = []
        producer.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(producer):
            for lo, hi in ranges:
                for r in range(N):
                    b.grads[r][lo:hi].copy_(a.grads[r][lo:hi])
                ev = torch.cuda.Event()
                ev.record(producer)
                ready.append(ev)
        side.wait_stream(torch.cuda.current_stream())
        done = torch.cuda.Event()
        abi.zero_step_bucketed(b.reps, b.grads, b.st, t, HP["lr"], HP["beta1"], HP["beta2"],
                               HP["eps"], HP["weight_decay"], bucket_bytes, ready, side, done,
                               timeout_ms=60_000)
        torch.cuda.synchronize()
        for x, y in [(a.m, b.m), (a.v, b.v)] + list(zip(a.reps, b.reps)):
            assert torch.equal(x, y)
    # one bucket at a time, hook style
    c = Case(abi, cuda, n, N, prec, seed=12)
    d = Case(abi, cuda, n, N, prec, seed=12)
    c.new_grads()
    for r in range(N):
        d.grads[r].copy_(c.grads[r])
    c.t = 1
    c.gpu_step()
    for k in range(len(ranges)):
        ev = torch.cuda.Event()
        ev.record()
        abi.zero_step_bucket(d.reps, d.grads, d.st, 1, HP["lr"], HP["beta1"], HP["beta2"],
                             HP["eps"], HP["weight_decay"], bucket_bytes, k, ev, side)
    torch.cuda.synchronize()
    for x, y in [(c.m, d.m), (c.v, d.v)] + list(zip(c.reps, d.reps)):
        assert torch.equal(x, y)


@pytest.mark.parametrize("prec", [oracle.FP32, oracle.BF16_MIXED])
def test_bucket_chain_completes_in_order(abi, cuda, prec):
    """Bucket launches are programmatic dependents of the one before: a
    bucket's blocks may start while the previous bucket drains, but every
    bucket completes in stream order. Over 1,000+ tiny buckets (down to one
    block each, ragged edges), a copy of every output queued on the side
    stream right after the call -- and the done event -- must see all the
    buckets: bitwise equal to the monolithic step."""
    n, N = 100_003, 4
    bucket_bytes = 390 if prec == oracle.FP32 else 194   # 97 elements: odd, off the vector grid
    a = Case(abi, cuda, n, N, prec, seed=14)
    b = Case(abi, cuda, n, N, prec, seed=14)
    count = abi.zero_bucket_count(n, prec, bucket_bytes)
    assert count > 1000
    side = torch.cuda.Stream()
    for t in (1, 2):
        a.new_grads()
        for r in range(N):
            b.grads[r].copy_(a.grads[r])
        a.t = b.t = t
        a.gpu_step()
        side.wait_stream(torch.cuda.current_stream())
        done = torch.cuda.Event()
        abi.zero_step_bucketed(b.reps, b.grads, b.st, t, HP["lr"], HP["beta1"], HP["beta2"],
                               HP["eps"], HP["weight_decay"], bucket_bytes, None, side, done)
        with torch.cuda.stream(side):  # queued right behind the last bucket
            snap = [x.clone() for x in [b.m, b.v] + list(b.reps)]
        after_done = torch.cuda.Stream()
        after_done.wait_event(done)
        with torch.cuda.stream(after_done):
            snap_done = [x.clone() for x in [b.m, b.v] + list(b.reps)]
        torch.cuda.synchronize()
        want = [a.m, a.v] + list(a.reps)
        for x, y, z in zip(snap, snap_done, want):
            assert torch.equal(x, z) and torch.equal(y, z)


def test_bucketed_deadline_reports_timeout(abi, cuda):
    """A producer that is late: the host deadline passes, the call returns
    ZERO_ETIMEDOUT, and the queued work still completes correctly."""
    n, N = 100_000, 2
    bucket_bytes = 4 * 50_000
    a = Case(abi, cuda, n, N, oracle.FP32, seed=13)
    b = Case(abi, cuda, n, N, oracle.FP32, seed=13)
    a.new_grads()
    for r in range(N):
        b.grads[r].copy_(a.grads[r])
    torch.cuda.synchronize()
    a.t = b.t = 1
    a.gpu_step()
    producer = torch.cuda.Stream()
    side = torch.cuda.Stream()
    ready = []
    with torch.cuda.stream(producer):
        torch.cuda._sleep(400_000_000)          # a bounded busy kernel (~0.2 s)
        for _ in range(2):
            ev = torch.cuda.Event()
            ev.record(producer)
            ready.append(ev)
    with pytest.raises(abi.ZeroError) as e:
        abi.zero_step_bucketed(b.reps, b.grads, b.st, 1, HP["lr"], HP["beta1"], HP["beta2"],
                               HP["eps"], HP["weight_decay"], bucket_bytes, ready, side, None,
                               timeout_ms=5)
    assert e.value.code == abi.ZERO_ETIMEDOUT
    torch.cuda.synchronize()
    for x, y in [(a.m, b.m), (a.v, b.v)] + list(zip(a.reps, b.reps)):
        assert torch.equal(x, y)


@pytest.mark.parametrize("prec", [oracle.FP32, oracle.BF16_MIXED])
@pytest.mark.parametrize("n,N", [(1, 1), (9, 2), (4099, 3), (100_003, 4), (100_003, 8),
                                 (65_537, 13), (1_000_003, 5), (1_000_003, 6), (1_000_003, 7)])
def test_ddp_allreduce_mean(abi, cuda, n, N, prec):
    rng = np.random.default_rng(n + N)
    mixed = prec == oracle.BF16_MIXED
    dt = torch.bfloat16 if mixed else torch.float32
    hs = []
    for _ in range(N):
        g = rng.normal(0, 1, n).astype(np.float32)
        hs.append(oracle.f32_to_bf16_rne(g) if mixed else g)
    dev = [to_dev(h, dt, cuda, offset=1 if n % 2 else 0) for h in hs]
    abi.ddp_allreduce_mean(dev, prec)
    torch.cuda.synchronize()
    ref = oracle.allreduce_mean(hs, precision=prec, mode="fp32")
    for r in range(N):
        assert np.array_equal(host_of(dev[r]), ref[r])


def _pinned_host(h, dt):
    """A pinned host tensor holding `h` (float32, or bf16 bits as uint16)."""
    if dt == torch.bfloat16:
        t = torch.from_numpy(h.view(np.int16).copy()).view(torch.bfloat16)
    else:
        t = torch.from_numpy(h.copy())
    return t.pin_memory()


@pytest.mark.parametrize("prec", [oracle.FP32, oracle.BF16_MIXED])
@pytest.mark.parametrize("n,N,chunk_bytes", [(1, 1, 64), (4099, 3, 1000), (100_003, 4, 1 << 16),
                                             (100_003, 8, 25 << 20), (1_000_003, 5, 1 << 20),
                                             (65_537, 13, 4094)])
def test_ddp_mean_from_host(abi, cuda, n, N, chunk_bytes, prec):
    """The chunk-pipelined DDP mean of host gradients: every staging buffer and
    the host copy equal the oracle's mean bit for bit, with chunks that split
    vectors (1000 and 4094 bytes) and a staging offset that shifts the phase."""
    rng = np.random.default_rng(n * 3 + N)
    mixed = prec == oracle.BF16_MIXED
    dt = torch.bfloat16 if mixed else torch.float32
    hs = []
    for _ in range(N):
        g = rng.normal(0, 1, n).astype(np.float32)
        hs.append(oracle.f32_to_bf16_rne(g) if mixed else g)
    host = [_pinned_host(h, dt) for h in hs]
    staging = [to_dev(np.zeros(n, np.uint16 if mixed else np.float32), dt, cuda,
                      offset=1 if n % 2 else 0) for _ in range(N)]
    out = torch.empty(n, dtype=dt).pin_memory()
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    abi.ddp_allreduce_mean_from_host(host, staging, prec, n, out, chunk_bytes, None, h2d, d2h)
    torch.cuda.synchronize()
    ref = oracle.allreduce_mean(hs, precision=prec, mode="fp32")
    for r in range(N):
        assert np.array_equal(host_of(staging[r]), ref[r]), f"staging {r}"
    assert np.array_equal(inputs.to_numpy_storage(out), ref[0])


@pytest.mark.parametrize("prec", [oracle.FP32, oracle.BF16_MIXED])
def test_ddp_mean_from_host_back_to_back(abi, cuda, prec):
    """Calls queued back to back on the same buffers, with no synchronisation
    between them: each host copy holds its own call's mean."""
    n, N = 300_007, 4
    mixed = prec == oracle.BF16_MIXED
    dt = torch.bfloat16 if mixed else torch.float32
    rng = np.random.default_rng(77)
    staging = [guarded_empty(n, dt, cuda, 1 + r, f"staging {r}") for r in range(N)]
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    calls = []
    for _ in range(3):
        hs = []
        for _ in range(N):
            g = rng.normal(0, 1, n).astype(np.float32)
            hs.append(oracle.f32_to_bf16_rne(g) if mixed else g)
        host = [_pinned_host(h, dt) for h in hs]
        out = torch.empty(n, dtype=dt).pin_memory()
        abi.ddp_allreduce_mean_from_host(host, staging, prec, n, out, 1 << 18, None, h2d, d2h)
        calls.append((hs, host, out))
    torch.cuda.synchronize()
    for hs, _, out in calls:
        ref = oracle.allreduce_mean(hs, precision=prec, mode="fp32")
        assert np.array_equal(inputs.to_numpy_storage(out), ref[0])
    for r in range(N):
        assert np.array_equal(host_of(staging[r]), ref[r])


@pytest.mark.parametrize("prec", [oracle.FP32, oracle.BF16_MIXED])
def test_ddp_mean_from_host_chained_on_a_handle(abi, cuda, prec):
    """Calls on a DdpHost handle, queued back to back with no synchronisation:
    chunk k of each call waits only for the previous call's mean and copy back
    of chunk k. Every host copy holds its own call's mean, bit for bit; a reset
    in the middle (after device work that reads the staging buffers) and a
    change of chunk size both fall back to waiting for the compute stream. The
    staging buffers sit between guard regions."""
    n, N = 300_007, 4
    mixed = prec == oracle.BF16_MIXED
    dt = torch.bfloat16 if mixed else torch.float32
    rng = np.random.default_rng(78)
    staging = [guarded_empty(n, dt, cuda, 1 + r, f"staging {r}") for r in range(N)]
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    ddp = abi.DdpHost()
    calls = []
    for i in range(6):
        hs = []
        for _ in range(N):
            g = rng.normal(0, 1, n).astype(np.float32)
            hs.append(oracle.f32_to_bf16_rne(g) if mixed else g)
        host = [_pinned_host(h, dt) for h in hs]
        out = torch.empty(n, dtype=dt).pin_memory()
        if i == 3:  # device work on the staging buffers between calls, then a reset
            calls.append(("seen", staging[0].clone()))
            ddp.reset()
        chunk = 1 << 18 if i != 4 else 3 * (1 << 16) + 6
        ddp.mean_from_host(host, staging, prec, n, out, chunk, None, h2d, d2h)
        calls.append((hs, out))
    torch.cuda.synchronize()
    last_ref = None
    for entry in calls:
        if isinstance(entry[0], str):  # the clone saw the mean of the call before it
            assert np.array_equal(host_of(entry[1]), last_ref[0])
            continue
        hs, out = entry
        last_ref = oracle.allreduce_mean(hs, precision=prec, mode="fp32")
        assert np.array_equal(inputs.to_numpy_storage(out), last_ref[0])
    for r in range(N):
        assert np.array_equal(host_of(staging[r]), last_ref[r])
    ddp.close()


def test_ddp_mean_from_host_rejects_bad_arguments(abi, cuda):
    n, N = 1000, 3
    staging = [torch.empty(n, device=cuda) for _ in range(N)]
    host = [torch.zeros(n).pin_memory() for _ in range(N)]
    with pytest.raises(abi.ZeroError) as e:  # the same staging buffer twice
        abi.ddp_allreduce_mean_from_host(host, [staging[0], staging[0], staging[2]], abi.ZERO_FP32)
    assert e.value.code == abi.ZERO_EINVAL
    with pytest.raises(abi.ZeroError) as e:  # a chunk below one element
        abi.ddp_allreduce_mean_from_host(host, staging, abi.ZERO_FP32, chunk_bytes=2)
    assert e.value.code == abi.ZERO_EINVAL
    with pytest.raises(TypeError):  # device tensors where host ones are expected
        abi.ddp_allreduce_mean_from_host(staging, staging, abi.ZERO_FP32)
    abi.ddp_allreduce_mean_from_host([h[:0] for h in host], [s[:0] for s in staging],
                                     abi.ZERO_FP32, 0)  # n = 0: nothing to do
    torch.cuda.synchronize()


def test_checkpoint_resume_is_bitwise(abi, cuda):
    from zero_sharded_optimizer_gb300.optimizer import ZeroOptimizer
    n, N = 123_457, 4
    rng = np.random.default_rng(21)
    init = torch.from_numpy(rng.normal(0, 0.02, n).astype(np.float32)).to(cuda)
    gs = [[torch.from_numpy(rng.normal(0, 1e-3, n).astype(np.float32)).to(cuda).to(torch.bfloat16)
           for _ in range(N)] for _ in range(6)]
    kw = dict(precision=abi.ZERO_BF16_MIXED, lr=6e-4, betas=(0.9, 0.999), weight_decay=0.1,
              master_init=init)
    ref = ZeroOptimizer(n, N, **kw)
    ref_p = [init.to(torch.bfloat16) for _ in range(N)]
    for g in gs:
        ref.step(ref_p, g)
    a = ZeroOptimizer(n, N, **kw)
    a_p = [init.to(torch.bfloat16) for _ in range(N)]
    for g in gs[:3]:
        a.step(a_p, g)
    ckpt = a.state_dict()
    ckpt_p = [p.clone() for p in a_p]
    b = ZeroOptimizer(n, N, **kw)
    b.load_state_dict(ckpt)
    for g in gs[3:]:
        b.step(ckpt_p, g)
    torch.cuda.synchronize()
    assert b.t == ref.t == 6
    assert torch.equal(b.master, ref.master) and torch.equal(b.m, ref.m)
    assert all(torch.equal(x, y) for x, y in zip(ckpt_p, ref_p))


def test_optimizer_host_gradients_match_device(abi, cuda):
    from zero_sharded_optimizer_gb300.optimizer import ZeroOptimizer
    n, N = 77_777, 4
    rng = np.random.default_rng(22)
    p0 = torch.from_numpy(rng.normal(0, 0.02, n).astype(np.float32))
    host = [torch.from_numpy(rng.normal(0, 1e-3, n).astype(np.float32)).pin_memory()
            for _ in range(N)]
    a = ZeroOptimizer(n, N, lr=1e-3, weight_decay=0.01)
    b = ZeroOptimizer(n, N, lr=1e-3, weight_decay=0.01)
    pa = [p0.to(cuda) for _ in range(N)]
    pb = [p0.to(cuda) for _ in range(N)]
    out = torch.empty(n, dtype=torch.float32).pin_memory()
    for _ in range(3):
        # chunks of 10,001 elements: chunk edges fall off the 16-byte vector grid
        a.step(pa, host, host_params_out=out, chunk_bytes=40_004)
        b.step(pb, [h.to(cuda) for h in host])
        torch.cuda.synchronize()
        assert all(torch.equal(x, y) for x, y in zip(pa, pb))
        assert torch.equal(out, pb[0].cpu())


def test_step_from_host_mixed_matches_device(abi, cuda):
    from zero_sharded_optimizer_gb300.optimizer import ZeroOptimizer
    n, N = 1_000_003, 8
    rng = np.random.default_rng(23)
    init = torch.from_numpy(rng.normal(0, 0.02, n).astype(np.float32))
    kw = dict(precision=abi.ZERO_BF16_MIXED, lr=6e-4, weight_decay=0.1, master_init=init)
    a, b = ZeroOptimizer(n, N, **kw), ZeroOptimizer(n, N, **kw)
    pa = [init.to(cuda).to(torch.bfloat16) for _ in range(N)]
    pb = [p.clone() for p in pa]
    out = torch.empty(n, dtype=torch.bfloat16).pin_memory()
    for _ in range(2):
        host = [torch.from_numpy(rng.normal(0, 1e-3, n).astype(np.float32)).to(torch.bfloat16)
                .pin_memory() for _ in range(N)]
        a.step(pa, host, host_params_out=out, chunk_bytes=1 << 20)
        b.step(pb, [h.to(cuda) for h in host])
        torch.cuda.synchronize()
        assert torch.equal(a.master, b.master) and all(torch.equal(x, y) for x, y in zip(pa, pb))
        assert torch.equal(out, pb[0].cpu())


@pytest.mark.parametrize("prec", [oracle.FP32, oracle.BF16_MIXED])
def test_host_steps_back_to_back_match_device(abi, cuda, prec):
    """Host-input steps queued without synchronizing: each chunk's copy of the
    next call overlaps the previous call's tail, waiting only for that call's
    step on the chunk. A device step in between breaks the chain (the copies
    then wait for everything on the stream). Bitwise equal to device steps."""
    from zero_sharded_optimizer_gb300.optimizer import ZeroOptimizer
    n, N = 300_007, 4
    mixed = prec == oracle.BF16_MIXED
    dt = torch.bfloat16 if mixed else torch.float32
    rng = np.random.default_rng(24)
    init = torch.from_numpy(rng.normal(0, 0.02, n).astype(np.float32))
    kw = dict(precision=prec, lr=1e-3, weight_decay=0.01, master_init=init if mixed else None)
    a, b = ZeroOptimizer(n, N, **kw), ZeroOptimizer(n, N, **kw)
    pa = [init.to(cuda).to(dt) for _ in range(N)]
    pb = [p.clone() for p in pa]
    hosts = [[torch.from_numpy(rng.normal(0, 1e-3, n).astype(np.float32)).to(dt).pin_memory()
              for _ in range(N)] for _ in range(6)]
    outs = [torch.empty(n, dtype=dt).pin_memory() for _ in range(6)]
    for k, host in enumerate(hosts):
        if k == 3:  # a device step between host steps
            a.step(pa, [h.to(cuda) for h in host])
        else:
            a.step(pa, host, host_params_out=outs[k], chunk_bytes=64 * 1024)
        b.step(pb, [h.to(cuda) for h in host])
        if k != 3:
            outs[k] = (outs[k], pb[0].clone())  # expected value, kept on the device
    torch.cuda.synchronize()
    assert all(torch.equal(x, y) for x, y in zip(pa, pb))
    for k in range(6):
        if k != 3:
            got, ref = outs[k]
            assert torch.equal(got, ref.cpu()), f"host copy of step {k}"


@pytest.mark.parametrize("prec", [oracle.FP32, oracle.BF16_MIXED])
def test_zero_and_subnormal_state_bitwise(abi, cuda, prec):
    """m and v at exact zero, in the subnormal range and just above it (what
    zero gradients decay them into), stepped with zero and tiny gradients:
    bit-exact against the oracle."""
    n, N = 300_007, 4
    c = Case(abi, cuda, n, N, prec, seed=51)
    rng = np.random.default_rng(52)
    kind = rng.integers(0, 4, n)
    u = rng.uniform(-1, 1, n)
    m = np.select([kind == 0, kind == 1, kind == 2], [0.0, u * 1e-40, u * 1e-37],
                  rng.normal(0, 1e-3, n)).astype(np.float32)
    v = np.select([kind == 0, kind == 1, kind == 2], [0.0, np.abs(u) * 1e-40, np.abs(u) * 1e-37],
                  rng.uniform(0, 1e-6, n)).astype(np.float32)
    assert np.any((m != 0) & (np.abs(m) < np.finfo(np.float32).tiny))
    c.m.copy_(torch.from_numpy(m))
    c.v.copy_(torch.from_numpy(v))
    b = oracle.shard_bounds(n, N)
    for i in range(N):
        c.o_states[i]["m"] = m[b[i]:b[i + 1]].copy()
        c.o_states[i]["v"] = v[b[i]:b[i + 1]].copy()
    for t in range(2):
        hs = []
        for r in range(N):
            g = np.where(kind < 2, 0.0, rng.normal(0, 1e-20, n)).astype(np.float32)
            if c.mixed:
                g = oracle.f32_to_bf16_rne(g)
            hs.append(g)
            c.grads[r].copy_(host_tensor(g, c.dt))
        c.oracle_step(hs)
        c.gpu_step()
        torch.cuda.synchronize()
        c.compare(exact=True)


def _special_grads(rng, n, N, mixed, idx):
    """Gradients N(0, 1e-3) with special values at the index sets of idx: a NaN
    in one rank, +Inf, opposite infinities (a NaN sum), a rank sum that
    overflows float32 (3e38 in every rank) and a square that overflows
    (1e20: v becomes +Inf)."""
    hs = []
    for r in range(N):
        g = rng.normal(0, 1e-3, n).astype(np.float32)
        if r == 1:
            g[idx[0]] = np.nan
        if r == 0:
            g[idx[1]] = np.inf
        if r == 2:
            g[idx[2]] = -np.inf
        if r == 3:
            g[idx[2]] = np.inf
        g[idx[3]] = 3e38
        g[idx[4]] = 1e20
        hs.append(oracle.f32_to_bf16_rne(g) if mixed else g)
    return hs


@pytest.mark.parametrize("prec", [oracle.FP32, oracle.BF16_MIXED])
def test_nan_and_inf_propagate_like_the_oracle(abi, cuda, prec):
    """NaN and Inf propagate as IEEE arithmetic gives them, nothing skipped: two
    steps with special gradients (and the NaN and infinite state they leave),
    then the DDP mean of special gradients, and clipping with a NaN norm (the
    coefficient min(1, NaN) stays 1) and with an infinite one (coefficient 0).
    Every output equals the oracle bit for bit, NaN matching NaN."""
    n, N = 100_003, 4
    c = Case(abi, cuda, n, N, prec, seed=61)
    rng = np.random.default_rng(62)
    idx = rng.permutation(n)[:5 * 700].reshape(5, 700)

    def compare(case):
        check_guards()
        for key, buf in [("m", case.m), ("v", case.v)] + ([("master", case.master)]
                                                         if case.mixed else []):
            assert_same_bits_or_both_nan(host_of(buf), flat(case.o_states, key), key)
        for r in range(N):
            want = oracle.f32_to_bf16_rne(flat(case.o_states, "master")) if case.mixed \
                else case.o_reps[r]
            assert_same_bits_or_both_nan(host_of(case.reps[r]), want, f"replica {r}")

    for _ in range(2):
        hs = _special_grads(rng, n, N, c.mixed, idx)
        for r in range(N):
            c.grads[r].copy_(host_tensor(hs[r], c.dt))
        with np.errstate(all="ignore"):
            c.oracle_step(hs)
        c.gpu_step()
        torch.cuda.synchronize()
        compare(c)
    m = host_of(c.m)
    assert np.isnan(m[idx[0]]).all() and np.isinf(host_of(c.v)[idx[4]]).all()

    # the DDP mean
    hs = _special_grads(rng, n, N, c.mixed, idx)
    dev = [to_dev(h, c.dt, cuda) for h in hs]
    abi.ddp_allreduce_mean(dev, prec)
    torch.cuda.synchronize()
    with np.errstate(all="ignore"):
        ref = oracle.allreduce_mean(hs, precision=prec, mode="fp32")
    for r in range(N):
        assert_same_bits_or_both_nan(host_of(dev[r]), ref[r], f"mean {r}")

    # clipping: a NaN norm, then an infinite one (no NaN gradient)
    count = abi.zero_grad_norm_scratch_count(n, prec)
    scratch = torch.empty(count, dtype=torch.float64, device=cuda)
    norm = torch.empty(1, dtype=torch.float64, device=cuda)
    for with_nan in (True, False):
        d = Case(abi, cuda, n, N, prec, seed=63)
        hs = _special_grads(rng, n, N, d.mixed, idx)
        if not with_nan:
            nan_free = [np.where(np.isin(np.arange(n), idx[0]), 0, h).astype(h.dtype)
                        for h in hs]
            hs = [h.copy() for h in nan_free]
            hs[2][idx[2]] = hs[3][idx[2]]       # +Inf + +Inf: no NaN sum either
        for r in range(N):
            d.grads[r].copy_(host_tensor(hs[r], d.dt))
        d.t = 1
        with np.errstate(all="ignore"):
            d.o_reps, d.o_states = oracle.zero_step(d.o_reps, hs, d.o_states, 1, precision=prec,
                                                    mode="fp32", max_grad_norm=1.0, **d.hp)
        abi.zero_step_ex(d.reps, d.grads, d.st, 1, max_grad_norm=1.0, norm_sq=norm,
                         norm_scratch=scratch, **d.hp)
        torch.cuda.synchronize()
        assert np.isnan(float(norm)) if with_nan else np.isinf(float(norm))
        compare(d)


@pytest.mark.parametrize("prec", [oracle.FP32, oracle.BF16_MIXED])
def test_whole_tensor_shards(abi, cuda, prec):
    """Shards made of whole tensors: bit-exact against the oracle with the same
    bounds, and bit-identical to the array_split shards (ownership only)."""
    rng = np.random.default_rng(92)
    numels = rng.integers(1, 40_000, 29).tolist()
    n, N = int(sum(numels)), 4
    tb = abi.zero_tensor_shard_bounds(numels, N)
    assert tb == oracle.tensor_shard_bounds(numels, N) != oracle.shard_bounds(n, N)
    a = Case(abi, cuda, n, N, prec, seed=93)
    b = Case(abi, cuda, n, N, prec, seed=93)
    # rebuild a's state with whole-tensor shards (same fp32 initial weights as b)
    init = host_of(b.master) if a.mixed else host_of(b.reps[0])
    a.st = abi.zero_init_states(n, N, prec, a.m, a.v, a.master,
                                b.master.clone() if a.mixed else None, bounds=tb)
    a.o_states = oracle.init_states(n, N, prec, master_init=init, mode="fp32", bounds=tb)
    assert a.st.view(1)["lo"] == tb[1]
    for _ in range(2):
        hg = a.new_grads()
        for r in range(N):
            b.grads[r].copy_(a.grads[r])
        a.t += 1
        a.o_reps, a.o_states = oracle.zero_step(a.o_reps, hg, a.o_states, a.t, precision=prec,
                                                mode="fp32", bounds=tb, **HP)
        a.gpu_step()
        b.t = a.t
        b.gpu_step()
        torch.cuda.synchronize()
        a.compare(exact=True)
        for x, y in [(a.m, b.m), (a.v, b.v)] + list(zip(a.reps, b.reps)):
            assert torch.equal(x, y)


@pytest.mark.parametrize("prec", [oracle.FP32, oracle.BF16_MIXED])
def test_maximum_rank_count(abi, cuda, prec):
    """N = ZERO_MAX_RANKS (64): the step, the owner-only step with its gather,
    and the DDP mean, each against the oracle."""
    n, N = 10_007, abi.ZERO_MAX_RANKS
    c = Case(abi, cuda, n, N, prec, seed=64)
    for _ in range(2):
        c.step()
        c.compare(exact=True)
    hg = c.new_grads()
    c.t += 1
    shards, c.o_states = oracle.zero_step(c.o_reps, hg, c.o_states, c.t, precision=prec,
                                          mode="fp32", all_gather=False, **c.hp)
    abi.zero_step_ex(c.reps, c.grads, c.st, c.t, owner_only=True, **c.hp)
    abi.zero_gather(c.reps, c.st)
    torch.cuda.synchronize()
    full = oracle.gather(shards, prec)
    for r in range(N):
        assert np.array_equal(host_of(c.reps[r]), full[r])
    g = [x.clone() for x in c.grads]
    abi.ddp_allreduce_mean(g, prec)
    torch.cuda.synchronize()
    ref = oracle.allreduce_mean(hg, prec, mode="fp32")
    for r in range(N):
        assert np.array_equal(host_of(g[r]), ref[r])
