"""Pins of the CPU oracle to facts fixed outside the oracle itself.

Each test compares the oracle with a value the pages print (fixtures under
tests/golden/, each with its source), a closed form, an invariant, or a library
routine (np.array_split, np.mean, torch.optim.Adam/AdamW, torch's bf16 cast).
The mutation tests at the end plant one plausible mistake at a time in the
oracle (on the CPU) and check that some pin catches it.
"""

import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import zero_oracle as zo

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def flat_state(states, key):
    return np.concatenate([s[key] for s in states])


# ---------------------------------------------------------------------------
# Shard bounds
# ---------------------------------------------------------------------------

def test_shard_bounds_equal_array_split():
    for n in range(0, 201):
        for N in range(1, 18):
            pieces = np.array_split(np.arange(n), N)
            b = oracle.shard_bounds(n, N)
            assert len(b) == N + 1 and b[0] == 0 and b[-1] == n
            for i, piece in enumerate(pieces):
                assert b[i + 1] - b[i] == len(piece)
                if len(piece):
                    assert piece[0] == b[i]


@pytest.mark.parametrize("n,N", [(10_007, 2), (10_007, 3), (1_000_003, 7), (6_250_001, 8)])
def test_shard_bounds_equal_array_split_large(n, N):
    pieces = np.array_split(np.arange(n, dtype=np.int64), N)
    starts = [int(p[0]) for p in pieces] + [n]
    assert oracle.shard_bounds(n, N) == starts


def test_shard_bounds_page_examples():
    for ex in golden("shard_examples.json")["examples"]:
        assert oracle.shard_bounds(ex["n"], ex["N"]) == ex["bounds"], ex["source"]


def test_shard_bounds_rejects():
    with pytest.raises(ValueError):
        oracle.shard_bounds(5, 0)
    with pytest.raises(ValueError):
        oracle.shard_bounds(-1, 2)
    assert oracle.shard_bounds(3, 5) == [0, 1, 2, 3, 3, 3]   # n < N: empty shards


# ---------------------------------------------------------------------------
# Worked examples
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("mode", ["fp64", "fp32"])
def test_p2_worked_example(mode):
    ex = golden("p2_worked_example.json")
    n, N = ex["n"], ex["N"]
    params = [np.array(ex["params"], np.float32) for _ in range(N)]
    grads = [np.array(g, np.float32) for g in ex["grads"]]
    states = oracle.init_states(n, N, mode=mode)
    assert [len(s["m"]) for s in states] == [len(s) for s in ex["shards"]]
    new_p, new_states = oracle.zero_step(params, grads, states, ex["t"], lr=ex["lr"], mode=mode)
    for rep in new_p:
        np.testing.assert_allclose(rep, ex["expected_params"], rtol=0, atol=1e-7)
    # the page's per-worker mean gradients: on the first step m = (1-b1) g_bar and
    # v = (1-b2) g_bar^2 (course page, section 3)
    for i, gb in enumerate(ex["mean_grad_per_worker"]):
        gb = np.array(gb)
        tol = 1e-15 if mode == "fp64" else 2e-7
        np.testing.assert_allclose(new_states[i]["m"], 0.1 * gb, rtol=1e-6, atol=tol)
        np.testing.assert_allclose(new_states[i]["v"], 0.001 * gb * gb, rtol=1e-5, atol=tol)
    # parameter 3 has a zero mean gradient and does not move at all
    assert new_p[0][3] == np.float32(1.0)


@pytest.mark.parametrize("mode", ["fp64", "fp32"])
def test_p1_worked_example(mode):
    ex = golden("p1_worked_example.json")
    w = np.array(ex["w"], np.float32)
    p = ex["p"]
    grads = [w - np.float32(r) for r in range(p)]
    bounds = oracle.shard_bounds(len(w), p)
    assert np.diff(bounds).tolist() == ex["chunk_sizes"]
    np.testing.assert_allclose(np.mean(np.stack(grads), 0), w - 1.5)
    states = oracle.init_states(len(w), p, mode=mode)
    new_p, _ = oracle.zero_step([w.copy() for _ in range(p)], grads, states, 1, lr=ex["lr"],
                                weight_decay=ex["weight_decay"], mode=mode)
    for rep in new_p:
        np.testing.assert_allclose(rep, ex["expected_w"], rtol=0, atol=1e-6)


# ---------------------------------------------------------------------------
# Closed forms
# ---------------------------------------------------------------------------

def test_first_step_moves_lr_times_sign():
    # course page section 3: at t=1, m_hat = g_bar and sqrt(v_hat) = |g_bar|, so each
    # entry moves by lr * g_bar / (|g_bar| + eps)
    rng = np.random.default_rng(1)
    n, N, lr, eps = 1001, 3, 0.05, 1e-8
    p0 = rng.normal(size=n)
    grads = [rng.normal(size=n) for _ in range(N)]
    gbar = np.mean(np.stack(grads), 0)
    new_p, _ = oracle.zero_step([p0.copy() for _ in range(N)], grads,
                                oracle.init_states(n, N, mode="fp64"), 1, lr=lr, eps=eps,
                                mode="fp64")
    np.testing.assert_allclose(new_p[0], p0 - lr * gbar / (np.abs(gbar) + eps), rtol=1e-6,
                               atol=1e-7)


@pytest.mark.parametrize("wd", [0.0, 0.1])
def test_constant_gradient_closed_form(wd):
    # constant g for every step: m_t = (1-b1^t) g and v_t = (1-b2^t) g^2, hence
    # m_hat = g, v_hat = g^2 at every t and p_t = p_{t-1}(1 - lr wd) - lr g/(|g|+eps)
    rng = np.random.default_rng(2)
    n, N, lr, eps, b1, b2 = 257, 4, 1e-2, 1e-8, 0.9, 0.95
    g = rng.normal(size=n)
    p = rng.normal(size=n)
    states = oracle.init_states(n, N, mode="fp64")
    params = [p.copy() for _ in range(N)]
    expect = p.copy()
    for t in range(1, 9):
        params, states = oracle.zero_step(params, [g] * N, states, t, lr=lr, beta1=b1, beta2=b2,
                                          eps=eps, weight_decay=wd, mode="fp64")
        expect = expect * (1 - lr * wd) - lr * g / (np.abs(g) + eps)
        np.testing.assert_allclose(params[0], expect, rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(flat_state(states, "m"), (1 - b1 ** t) * g, rtol=1e-12)
        np.testing.assert_allclose(flat_state(states, "v"), (1 - b2 ** t) * g * g, rtol=1e-12)


# ---------------------------------------------------------------------------
# Library routines: torch.optim on the mean gradient
# ---------------------------------------------------------------------------

def _torch_reference(p0, grad_seq, lr, b1, b2, eps, wd, dtype):
    torch = pytest.importorskip("torch")
    p = torch.tensor(p0, dtype=dtype, requires_grad=True)
    cls = torch.optim.AdamW if wd > 0 else torch.optim.Adam
    opt = cls([p], lr=lr, betas=(b1, b2), eps=eps, weight_decay=wd, foreach=False)
    out = []
    for grads in grad_seq:
        gbar = np.mean(np.stack([np.asarray(g, np.float64) for g in grads]), 0)
        p.grad = torch.tensor(gbar, dtype=dtype)
        opt.step()
        st = opt.state[p]
        out.append((p.detach().numpy().copy(), st["exp_avg"].numpy().copy(),
                    st["exp_avg_sq"].numpy().copy()))
    return out


@pytest.mark.parametrize("N,wd,scale", [(1, 0.0, 1.0), (2, 0.0, 1.0), (4, 0.01, 1e-3),
                                         (3, 0.1, 1e-7), (8, 0.1, 1.0)])
def test_fp64_matches_torch_adamw(N, wd, scale):
    rng = np.random.default_rng(3 + N)
    n, lr, b1, b2, eps = 1003, 3e-3, 0.9, 0.95, 1e-8
    p0 = rng.normal(0, 0.02, size=n)
    seq = [[rng.normal(0, scale, size=n) for _ in range(N)] for _ in range(6)]
    ref = _torch_reference(p0, seq, lr, b1, b2, eps, wd, dtype=__import__("torch").float64)
    params = [p0.copy() for _ in range(N)]
    states = oracle.init_states(n, N, mode="fp64")
    for t, grads in enumerate(seq, start=1):
        params, states = oracle.zero_step(params, grads, states, t, lr=lr, beta1=b1, beta2=b2,
                                          eps=eps, weight_decay=wd, mode="fp64")
        rp, rm, rv = ref[t - 1]
        np.testing.assert_allclose(params[0], rp, rtol=1e-12, atol=1e-18)
        # torch forms m with lerp, a different rounding order: a few ulps of max|m|
        np.testing.assert_allclose(flat_state(states, "m"), rm, rtol=1e-12,
                                   atol=1e-13 * np.abs(rm).max())
        np.testing.assert_allclose(flat_state(states, "v"), rv, rtol=1e-12,
                                   atol=1e-13 * np.abs(rv).max())


def test_special_values_match_torch_adamw():
    """Reading: NaN and Inf propagate as IEEE arithmetic gives them, nothing is
    skipped. One step from zero state against torch.optim.AdamW in float64 on the
    same mean gradient, with a NaN in one rank, +Inf, opposite infinities (a NaN
    sum), a rank sum that overflows and a square that overflows in v: the NaN
    positions of p, m and v are the same and every other value agrees,
    infinities included. Each special value stays at its own index: the other
    indices equal the step with those gradients zeroed. (One step only: torch
    forms m with lerp, m + w*(g - m), which turns an infinite m into NaN on the
    next step where beta1*m + (1 - beta1)*g keeps it infinite.)"""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(41)
    n, N, lr, b1, b2, eps, wd = 64, 4, 1e-3, 0.9, 0.95, 1e-8, 0.1
    p0 = rng.normal(0, 0.02, n)
    grads = [rng.normal(0, 1e-3, n) for _ in range(N)]
    grads[1][0:4] = np.nan
    grads[0][4:8] = np.inf
    grads[2][8:12], grads[3][8:12] = -np.inf, np.inf
    for g in grads:
        g[12:16] = 1.7e308   # the rank sum overflows to +Inf
        g[16:20] = 1e160     # the mean is finite, its square overflows: v = +Inf
    special = np.zeros(n, bool)
    special[:20] = True
    with np.errstate(all="ignore"):
        (rp, rm, rv), = _torch_reference(p0, [grads], lr, b1, b2, eps, wd, dtype=torch.float64)
        params, states = oracle.zero_step([p0.copy() for _ in range(N)], grads,
                                          oracle.init_states(n, N, mode="fp64"), 1, lr=lr,
                                          beta1=b1, beta2=b2, eps=eps, weight_decay=wd,
                                          mode="fp64")
    for got, want in [(params[0], rp), (flat_state(states, "m"), rm),
                      (flat_state(states, "v"), rv)]:
        assert np.array_equal(np.isnan(got), np.isnan(want))
        ok = ~np.isnan(want)
        np.testing.assert_allclose(got[ok], want[ok], rtol=1e-12, atol=1e-18)
    assert np.all(np.isnan(params[0][:16])) and np.all(np.isfinite(params[0][16:]))
    assert np.all(np.isinf(flat_state(states, "v")[16:20]))
    zeroed = [np.where(special, 0.0, g) for g in grads]
    clean, _ = oracle.zero_step([p0.copy() for _ in range(N)], zeroed,
                                oracle.init_states(n, N, mode="fp64"), 1, lr=lr, beta1=b1,
                                beta2=b2, eps=eps, weight_decay=wd, mode="fp64")
    assert np.array_equal(params[0][~special], clean[0][~special])


def test_fp32_mirror_close_to_torch_fp32_and_fp64():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(11)
    n, N, lr, b1, b2, eps, wd = 4099, 4, 3e-4, 0.9, 0.95, 1e-8, 0.01
    p0 = rng.normal(0, 0.02, size=n).astype(np.float32)
    seq = [[rng.normal(0, 1e-3, size=n).astype(np.float32) for _ in range(N)] for _ in range(10)]
    ref32 = _torch_reference(p0, seq, lr, b1, b2, eps, wd, dtype=torch.float32)
    p32 = [p0.copy() for _ in range(N)]
    p64 = [p0.astype(np.float64) for _ in range(N)]
    s32 = oracle.init_states(n, N, mode="fp32")
    s64 = oracle.init_states(n, N, mode="fp64")
    for t, grads in enumerate(seq, start=1):
        p32, s32 = oracle.zero_step(p32, grads, s32, t, lr=lr, beta1=b1, beta2=b2, eps=eps,
                                    weight_decay=wd, mode="fp32")
        p64, s64 = oracle.zero_step(p64, grads, s64, t, lr=lr, beta1=b1, beta2=b2, eps=eps,
                                    weight_decay=wd, mode="fp64")
        for key, ref in (("m", ref32[t - 1][1]), ("v", ref32[t - 1][2])):
            x = flat_state(s32, key)
            assert np.all(np.abs(x - ref) <= 1e-6 * np.abs(ref).max() + 1e-5 * np.abs(ref))
            y = flat_state(s64, key)
            # m and v are sums of terms of size ~max|y|: allow a few fp32 ulps of that
            assert np.all(np.abs(x - y) <= 1e-5 * np.abs(y) + 1e-6 * np.abs(y).max())
        assert np.all(np.abs(p32[0] - ref32[t - 1][0]) <= 1e-6 + 1e-5 * np.abs(ref32[t - 1][0]))
        assert np.all(np.abs(p32[0] - p64[0]) <= 1e-6 + 1e-5 * np.abs(p64[0]))


# ---------------------------------------------------------------------------
# Invariants
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 7, 8])
@pytest.mark.parametrize("mode", ["fp32", "fp64"])
def test_sharded_equals_unsharded(N, mode):
    rng = np.random.default_rng(100 + N)
    n = 1009
    dt = np.float64 if mode == "fp64" else np.float32
    p = rng.normal(size=n).astype(dt)
    params = [p.copy() for _ in range(N)]
    states = oracle.init_states(n, N, mode=mode)
    m = np.zeros(n, dt)
    v = np.zeros(n, dt)
    for t in range(1, 4):
        grads = [rng.normal(size=n).astype(np.float32) for _ in range(N)]
        gbar = zo._mean_over_ranks([g.astype(dt) for g in grads], mode)
        params, states = oracle.zero_step(params, grads, states, t, lr=1e-2, weight_decay=0.05,
                                          mode=mode)
        p, m, v = oracle.adam_full(p, gbar, m, v, t, lr=1e-2, weight_decay=0.05, mode=mode)
        for rep in params:                    # every replica, bitwise
            assert rep.dtype == dt and np.array_equal(rep, p)
        assert np.array_equal(flat_state(states, "m"), m)
        assert np.array_equal(flat_state(states, "v"), v)


def test_state_sizes_are_shards():
    states = oracle.init_states(10_007, 3)
    assert [len(s["m"]) for s in states] == [3336, 3336, 3335]


def test_allreduce_mean_matches_np_mean():
    rng = np.random.default_rng(5)
    for N in (1, 2, 3, 8):
        grads = [rng.normal(size=777) for _ in range(N)]
        out = oracle.allreduce_mean(grads, mode="fp64")
        ref = np.mean(np.stack(grads), 0)
        assert len(out) == N
        for o in out:
            assert np.array_equal(o, out[0])
            np.testing.assert_allclose(o, ref, rtol=1e-14)
        # fp32 mirror of the same mean: exact for power-of-two N on fp32 inputs
        g32 = [g.astype(np.float32) for g in grads]
        m32 = oracle.allreduce_mean(g32, mode="fp32")[0]
        np.testing.assert_allclose(m32, np.mean(np.stack(g32).astype(np.float64), 0),
                                   rtol=1e-5, atol=1e-6)


# ---------------------------------------------------------------------------
# Mixed precision
# ---------------------------------------------------------------------------

def test_bf16_round_trip_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(6)
    x = np.concatenate([
        rng.normal(size=10_000).astype(np.float32),
        (rng.normal(size=1000) * 1e-38).astype(np.float32),           # subnormals
        np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -1.0 - 2.0 ** -8,  # ties
                  np.float32(3.3895314e38), np.inf, -np.inf, 0.0, -0.0], np.float32),
    ])
    ours = oracle.f32_to_bf16_rne(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = oracle.bf16_to_f32(ours)
    assert np.array_equal(back, torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16)
                          .float().numpy())
    assert oracle.f32_to_bf16_rne(np.array([1.0 + 2.0 ** -8], np.float32))[0] == 0x3F80  # tie->even
    assert np.isnan(oracle.bf16_to_f32(oracle.f32_to_bf16_rne(np.array([np.nan], np.float32))))[0]


def test_mixed_step_master_matches_torch_and_replicas_are_rne():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(7)
    n, N, lr, b1, b2, eps, wd = 2053, 8, 6e-4, 0.9, 0.999, 1e-8, 0.1
    init = rng.normal(0, 0.02, size=n).astype(np.float32)
    reps = [oracle.f32_to_bf16_rne(init) for _ in range(N)]
    states = oracle.init_states(n, N, oracle.BF16_MIXED, master_init=init)
    seq = []
    for t in range(1, 5):
        grads = [oracle.f32_to_bf16_rne(rng.normal(0, 1e-3, size=n).astype(np.float32))
                 for _ in range(N)]
        seq.append([oracle.bf16_to_f32(g) for g in grads])
        reps, states = oracle.zero_step(reps, grads, states, t, lr=lr, beta1=b1, beta2=b2,
                                        eps=eps, weight_decay=wd, precision=oracle.BF16_MIXED)
        master = flat_state(states, "master")
        for r in reps:
            assert np.array_equal(r, oracle.f32_to_bf16_rne(master))
    ref = _torch_reference(init, seq, lr, b1, b2, eps, wd, dtype=torch.float64)
    rp = ref[-1][0]
    assert np.all(np.abs(master - rp) <= 1e-6 + 1e-5 * np.abs(rp))


def test_mixed_requires_master_init():
    with pytest.raises(ValueError):
        oracle.init_states(10, 2, oracle.BF16_MIXED)


# ---------------------------------------------------------------------------
# Memory accounting
# ---------------------------------------------------------------------------

def test_memory_course_table():
    tab = golden("p1_memory_table.json")
    for row in tab["rows"]:
        got = oracle.memory_breakdown(tab["n"], tab["p"], row["stage"], oracle.FP64_EMU,
                                      row["rank"])
        assert got == (row["params"], row["grads"], row["optimizer"]), row
    assert sum(oracle.memory_breakdown(10, 4, 3, oracle.FP64_EMU, 0)) == tab["stage3_rank0_total"]
    assert sum(oracle.memory_breakdown(10, 4, 0, oracle.FP64_EMU, 0)) == tab["one_process_total"]


def test_memory_page_figures():
    prec = {"fp32": oracle.FP32, "bf16_mixed": oracle.BF16_MIXED}
    gib = 2.0 ** 30
    for fig in golden("memory_figures.json")["figures"]:
        if "per_param" in fig:
            for k, v in fig["per_param"].items():
                assert oracle.memory_breakdown(1, 1, 0, prec[k], 0) == tuple(v)
            continue
        n, N, pr = fig["n"], fig["N"], prec[fig["precision"]]
        if "by_stage" in fig:
            for st, val in fig["by_stage"].items():
                got = oracle.memory_bytes(n, N, int(st), pr) / gib
                assert abs(got - val) < fig["rounded_to"], (fig["source"], st, got)
        if "less_than" in fig:
            assert oracle.memory_bytes(n, N, fig["stage"], pr) / gib < fig["less_than"]
        if "exact" in fig:
            assert oracle.memory_bytes(n, N, fig["stage"], pr) == fig["exact"]
        if "by_stage_exact" in fig:
            for st, val in fig["by_stage_exact"].items():
                assert oracle.memory_bytes(n, N, int(st), pr) == val, (fig["source"], st)


@pytest.mark.parametrize("N", [1, 2, 4, 8, 64])
def test_memory_stage_formulas(N):
    # 16n, 4n + 12n/N, 2n + 14n/N, 16n/N (mixed) and 16n, 8n + 8n/N, 4n + 12n/N, 16n/N
    # (fp32) when N divides n
    n = 64 * 1000
    assert [oracle.memory_bytes(n, N, s, oracle.BF16_MIXED) for s in range(4)] == \
        [16 * n, 4 * n + 12 * n // N, 2 * n + 14 * n // N, 16 * n // N]
    assert [oracle.memory_bytes(n, N, s, oracle.FP32) for s in range(4)] == \
        [16 * n, 8 * n + 8 * n // N, 4 * n + 12 * n // N, 16 * n // N]


def test_memory_one_over_p_44_params():
    # course test catalogue: a 44-parameter model on 4 ranks has exact 1/p shares
    for prec in (oracle.FP32, oracle.BF16_MIXED):
        per_rank = [sum(oracle.memory_breakdown(44, 4, 3, prec, r)) for r in range(4)]
        assert per_rank == [sum(oracle.memory_breakdown(44, 1, 0, prec, 0)) // 4] * 4
    # shares of the unequal chunks add back up to the whole
    for st in (1, 2, 3):
        opt = sum(oracle.memory_breakdown(10, 4, st, oracle.FP32, r)[2] for r in range(4))
        assert opt == 8 * 10


def test_memory_rejects():
    for args in [(10, 0, 1, 0), (10, 4, 4, 0), (10, 4, -1, 0), (-1, 4, 1, 0), (10, 4, 1, 7)]:
        with pytest.raises(ValueError):
            oracle.memory_bytes(*args)


# ---------------------------------------------------------------------------
# Buckets
# ---------------------------------------------------------------------------

def test_bucket_bounds_25mib():
    cap = 25 * 1024 * 1024            # bucket_cap_mb * 1024 * 1024 bytes
    n = 1_300_000_000
    b = oracle.bucket_bounds(n, 2, cap)
    assert len(b) == 100 == math.ceil(n * 2 / cap)
    assert b[0] == (n - cap // 2, n)                   # first ready: the highest indices
    assert b[-1] == (0, n - 99 * (cap // 2)) and b[-1][1] == 2_387_200
    for (lo, hi), (lo2, hi2) in zip(b, b[1:]):
        assert hi2 == lo and lo2 < lo
    assert oracle.bucket_bounds(0, 4, cap) == []
    assert oracle.bucket_bounds(10, 4, 12) == [(7, 10), (4, 7), (1, 4), (0, 1)]


# ---------------------------------------------------------------------------
# Mutation checks: one planted mistake at a time must fail a pin above
# ---------------------------------------------------------------------------

def _fails(fn):
    try:
        fn()
    except AssertionError:
        return True
    return False


def test_mutant_sum_instead_of_mean(monkeypatch):
    def summed(pieces, mode):
        acc = np.array(pieces[0], dtype=zo._dtype(mode), copy=True)
        for piece in pieces[1:]:
            acc = acc + piece
        return acc
    monkeypatch.setattr(zo, "_mean_over_ranks", summed)
    assert _fails(lambda: test_p2_worked_example("fp64"))


def test_mutant_no_bias_correction(monkeypatch):
    real = zo._adam

    def no_bc(p, g, m, v, t, lr, b1, b2, eps, wd, mode):
        p = np.asarray(p, np.float64) * (1 - lr * wd)
        m = b1 * np.asarray(m, np.float64) + (1 - b1) * g
        v = b2 * np.asarray(v, np.float64) + (1 - b2) * g * g
        return p - lr * m / (np.sqrt(v) + eps), m, v
    monkeypatch.setattr(zo, "_adam", no_bc)
    assert _fails(lambda: test_p2_worked_example("fp64"))
    monkeypatch.setattr(zo, "_adam", real)


def test_mutant_eps_inside_sqrt(monkeypatch):
    def eps_in(p, g, m, v, t, lr, b1, b2, eps, wd, mode):
        p = np.asarray(p, np.float64) * (1 - lr * wd)
        m = b1 * np.asarray(m, np.float64) + (1 - b1) * g
        v = b2 * np.asarray(v, np.float64) + (1 - b2) * g * g
        mh, vh = m / (1 - b1 ** t), v / (1 - b2 ** t)
        return p - lr * mh / np.sqrt(vh + eps), m, v
    monkeypatch.setattr(zo, "_adam", eps_in)
    assert _fails(lambda: test_fp64_matches_torch_adamw(3, 0.1, 1e-7))


def test_mutant_coupled_weight_decay(monkeypatch):
    def l2(p, g, m, v, t, lr, b1, b2, eps, wd, mode):
        p = np.asarray(p, np.float64)
        g = g + wd * p
        m = b1 * np.asarray(m, np.float64) + (1 - b1) * g
        v = b2 * np.asarray(v, np.float64) + (1 - b2) * g * g
        mh, vh = m / (1 - b1 ** t), v / (1 - b2 ** t)
        return p - lr * mh / (np.sqrt(vh) + eps), m, v
    monkeypatch.setattr(zo, "_adam", l2)
    assert _fails(lambda: test_fp64_matches_torch_adamw(4, 0.01, 1e-3))


def test_mutant_wrong_chunk_start(monkeypatch):
    def shifted(n, N):             # remainder given to the last ranks instead
        q, r = divmod(n, N)
        return [i * q + max(0, i - (N - r)) for i in range(N + 1)]
    monkeypatch.setattr(zo, "shard_bounds", shifted)
    monkeypatch.setattr(oracle, "shard_bounds", shifted)
    assert _fails(test_shard_bounds_page_examples)


def test_mutant_no_all_gather(monkeypatch):
    def own_shard_only(new_shards, N, precision, mode):
        reps = []
        for i in range(N):
            parts = [s if j == i else np.full_like(s, 1.0) for j, s in enumerate(new_shards)]
            reps.append(zo._replica_from(np.concatenate(parts), precision, mode))
        return reps
    monkeypatch.setattr(zo, "_all_gather", own_shard_only)
    assert _fails(lambda: test_p1_worked_example("fp64"))


def test_mutant_dropped_hyperparameters(monkeypatch):
    real = zo.zero_step

    def default_lr(params, grads, states, t, lr=1e-2, **kw):
        return real(params, grads, states, t, **kw)
    monkeypatch.setattr(oracle, "zero_step", default_lr)
    assert _fails(lambda: test_p2_worked_example("fp64"))


# ---------------------------------------------------------------------------
# Global-norm clipping and the accumulation factor
# ---------------------------------------------------------------------------

def test_grad_norm_closed_form():
    # a constant mean gradient c on n entries has norm |c| sqrt(n), whatever the shards
    for n, N in [(10, 4), (1001, 3), (64, 8)]:
        grads = [np.full(n, 3.0 * (r + 1), np.float32) for r in range(N)]
        c = 3.0 * (N + 1) / 2
        assert oracle.grad_norm(grads, mode="fp64") == pytest.approx(abs(c) * math.sqrt(n),
                                                                      rel=1e-15)


@pytest.mark.parametrize("max_norm,scale", [(0.5, 1.0), (100.0, 1.0), (0.05, 0.25), (None, 0.5)])
def test_clipped_step_matches_torch(max_norm, scale):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(31)
    n, N, lr, b1, b2, eps, wd = 777, 4, 1e-3, 0.9, 0.95, 1e-8, 0.1
    p0 = rng.normal(0, 0.02, size=n)
    p = torch.tensor(p0, dtype=torch.float64, requires_grad=True)
    opt = torch.optim.AdamW([p], lr=lr, betas=(b1, b2), eps=eps, weight_decay=wd, foreach=False)
    params = [p0.copy() for _ in range(N)]
    states = oracle.init_states(n, N, mode="fp64")
    for t in range(1, 5):
        grads = [rng.normal(0, 0.05, size=n) for _ in range(N)]
        gbar = np.mean(np.stack(grads), 0) * scale
        p.grad = torch.tensor(gbar, dtype=torch.float64)
        if max_norm is not None:
            total = torch.nn.utils.clip_grad_norm_([p], max_norm)
            assert oracle.grad_norm(grads, mode="fp64") * scale == pytest.approx(float(total),
                                                                                  rel=1e-12)
        opt.step()
        params, states = oracle.zero_step(params, grads, states, t, lr=lr, beta1=b1, beta2=b2,
                                          eps=eps, weight_decay=wd, mode="fp64",
                                          grad_scale=scale, max_grad_norm=max_norm)
        np.testing.assert_allclose(params[0], p.detach().numpy(), rtol=1e-11, atol=1e-16)


def test_accumulation_factor_equals_mean_of_micro_batches():
    # k micro-batches summed with factor 1/k is the step on their mean (exact in
    # float64 for k a power of two)
    rng = np.random.default_rng(32)
    n, N, k = 513, 2, 4
    micro = [[rng.normal(size=n) for _ in range(N)] for _ in range(k)]
    summed = [sum(micro[i][r] for i in range(k)) for r in range(N)]
    mean = [summed[r] / k for r in range(N)]
    p0 = rng.normal(size=n)
    a, _ = oracle.zero_step([p0] * N, summed, oracle.init_states(n, N, mode="fp64"), 1,
                            mode="fp64", grad_scale=1.0 / k)
    b, _ = oracle.zero_step([p0] * N, mean, oracle.init_states(n, N, mode="fp64"), 1,
                            mode="fp64")
    assert np.array_equal(a[0], b[0])


def test_mutant_clip_on_sum_of_gradients(monkeypatch):
    real = zo.grad_norm

    def norm_of_sum(grads, precision=oracle.FP32, mode="fp32"):
        return real(grads, precision, mode) * len(grads)
    monkeypatch.setattr(zo, "grad_norm", norm_of_sum)
    assert _fails(lambda: test_clipped_step_matches_torch(0.5, 1.0))


# ---------------------------------------------------------------------------
# Whole-tensor shards
# ---------------------------------------------------------------------------

def test_tensor_shards_page_example():
    # "ZeRO One", "Sharding Parameters": 291 tensors over 4 ranks -> tensors
    # (0,73), (73,146), (146,219), (219,291); with unit sizes the element offsets
    # equal the tensor indices, with other sizes they are the tensors' offsets
    assert oracle.tensor_shard_bounds([1] * 291, 4) == [0, 73, 146, 219, 291]
    rng = np.random.default_rng(81)
    numels = rng.integers(0, 5000, 291).tolist()
    offsets = np.concatenate([[0], np.cumsum(numels)])
    b = oracle.tensor_shard_bounds(numels, 4)
    assert b == [int(offsets[k]) for k in (0, 73, 146, 219, 291)]
    # counts per rank follow array_split over the tensor list
    for T, N in [(148, 8), (5, 8), (13, 3)]:
        sizes = [len(p) for p in np.array_split(np.arange(T), N)]
        b = oracle.tensor_shard_bounds([1] * T, N)
        assert np.diff(b).tolist() == sizes


@pytest.mark.parametrize("mode", ["fp32", "fp64"])
def test_tensor_shards_change_nothing_but_ownership(mode):
    rng = np.random.default_rng(82)
    numels = rng.integers(1, 300, 37).tolist()
    n, N = int(sum(numels)), 4
    dt = np.float64 if mode == "fp64" else np.float32
    p = rng.normal(size=n).astype(dt)
    tb = oracle.tensor_shard_bounds(numels, N)
    assert tb != oracle.shard_bounds(n, N)
    a_p, b_p = [p.copy() for _ in range(N)], [p.copy() for _ in range(N)]
    a_s = oracle.init_states(n, N, mode=mode, bounds=tb)
    b_s = oracle.init_states(n, N, mode=mode)
    assert [len(s["m"]) for s in a_s] == np.diff(tb).tolist()
    for t in range(1, 4):
        grads = [rng.normal(size=n).astype(np.float32) for _ in range(N)]
        a_p, a_s = oracle.zero_step(a_p, grads, a_s, t, weight_decay=0.1, mode=mode, bounds=tb)
        b_p, b_s = oracle.zero_step(b_p, grads, b_s, t, weight_decay=0.1, mode=mode)
        assert all(np.array_equal(x, b_p[0]) for x in a_p)
        assert np.array_equal(flat_state(a_s, "v"), flat_state(b_s, "v"))


def test_tensor_shard_memory():
    numels = [100, 7, 7, 900, 3]
    tb = oracle.tensor_shard_bounds(numels, 2)           # tensors (0..3), (3..5)
    assert tb == [0, 114, 1017]
    assert oracle.memory_breakdown(1017, 2, 1, oracle.BF16_MIXED, 0, bounds=tb) == \
        (2 * 1017, 2 * 1017, 12 * 114)
    assert oracle.memory_breakdown(1017, 2, 3, oracle.FP32, 1, bounds=tb) == \
        (4 * 903, 4 * 903, 8 * 903)
    with pytest.raises(ValueError):
        oracle.memory_breakdown(1017, 2, 1, oracle.FP32, 0, bounds=[0, 2000, 1017])


# ---------------------------------------------------------------------------
# ZeRO-3: release after the step, gather before the forward pass
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("mode", ["fp64", "fp32"])
def test_p1_worked_example_stage3(mode):
    # course page section 3: "every stage gives this on every rank: rank 0 computes
    # entries 0 to 2, rank 3 entries 8 and 9, and ... stage 3's gather() assembles
    # the rest"
    ex = golden("p1_worked_example.json")
    w = np.array(ex["w"], np.float32)
    p = ex["p"]
    grads = [w - np.float32(r) for r in range(p)]
    states = oracle.init_states(len(w), p, mode=mode)
    shards, _ = oracle.zero_step([w.copy() for _ in range(p)], grads, states, 1, lr=ex["lr"],
                                 weight_decay=ex["weight_decay"], mode=mode, all_gather=False)
    assert [len(s) for s in shards] == ex["chunk_sizes"]
    np.testing.assert_allclose(shards[0], ex["expected_w"][:3], atol=1e-6)
    np.testing.assert_allclose(shards[3], ex["expected_w"][8:], atol=1e-6)
    for rep in oracle.gather(shards):
        np.testing.assert_allclose(rep, ex["expected_w"], atol=1e-6)


def test_stage3_gather_equals_all_gather():
    rng = np.random.default_rng(101)
    n, N = 1009, 5
    init = rng.normal(0, 0.02, n).astype(np.float32)
    for prec in (oracle.FP32, oracle.BF16_MIXED):
        reps = [oracle.f32_to_bf16_rne(init) if prec else init.copy() for _ in range(N)]
        a_s = oracle.init_states(n, N, prec, master_init=init)
        b_s = oracle.init_states(n, N, prec, master_init=init)
        g = [rng.normal(size=n).astype(np.float32) for _ in range(N)]
        if prec:
            g = [oracle.f32_to_bf16_rne(x) for x in g]
        full, _ = oracle.zero_step(reps, g, a_s, 1, precision=prec)
        shards, _ = oracle.zero_step(reps, g, b_s, 1, precision=prec, all_gather=False)
        for x, y in zip(oracle.gather(shards), full):
            assert np.array_equal(x, y)


# ---------------------------------------------------------------------------
# Momentum SGD as the wrapped optimizer
# ---------------------------------------------------------------------------

def _torch_sgd(p0, seq, lr, momentum, dampening, wd, nesterov, dtype):
    """torch.optim.SGD stepped on np.mean of each step's gradients."""
    torch = pytest.importorskip("torch")
    w = torch.nn.Parameter(torch.tensor(np.asarray(p0), dtype=dtype))
    opt = torch.optim.SGD([w], lr=lr, momentum=momentum, dampening=dampening, weight_decay=wd,
                          nesterov=nesterov)
    out = []
    for grads in seq:
        w.grad = torch.tensor(np.mean(np.stack([np.asarray(g, np.float64) for g in grads]),
                                      axis=0), dtype=dtype)
        opt.step()
        buf = opt.state[w].get("momentum_buffer")
        out.append((w.detach().numpy().copy(), None if buf is None else buf.numpy().copy()))
    return out


SGD_CASES = [  # (N, momentum, dampening, wd, nesterov)
    (1, 0.0, 0.0, 0.0, False), (2, 0.9, 0.0, 0.0, False), (4, 0.9, 0.1, 0.01, False),
    (3, 0.5, 0.0, 0.1, True), (8, 0.99, 0.0, 0.0, True), (4, 0.0, 0.0, 0.05, False)]


@pytest.mark.parametrize("N,mu,damp,wd,nest", SGD_CASES)
def test_sgd_fp64_matches_torch_sgd(N, mu, damp, wd, nest):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(40 + N)
    n, lr = 1003, 0.05
    p0 = rng.normal(0, 0.5, size=n)
    seq = [[rng.normal(0, 1.0, size=n) for _ in range(N)] for _ in range(5)]
    ref = _torch_sgd(p0, seq, lr, mu, damp, wd, nest, torch.float64)
    params = [p0.copy() for _ in range(N)]
    states = oracle.init_states_sgd(n, N, mode="fp64", momentum=mu != 0)
    for t, grads in enumerate(seq, start=1):
        params, states = oracle.zero_step_sgd(params, grads, states, t, lr=lr, momentum=mu,
                                              dampening=damp, weight_decay=wd, nesterov=nest,
                                              mode="fp64")
        rp, rb = ref[t - 1]
        for rep in params:
            np.testing.assert_allclose(rep, rp, rtol=1e-12, atol=1e-14)
        if mu:
            assert all(s["buf"] is not None for s in states)
            np.testing.assert_allclose(flat_state(states, "buf"), rb, rtol=1e-12, atol=1e-14)
        else:
            assert rb is None and all(s["buf"] is None for s in states)


@pytest.mark.parametrize("N,mu,damp,wd,nest", SGD_CASES[1:4])
def test_sgd_fp32_mirror_close_to_torch_fp32(N, mu, damp, wd, nest):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(50 + N)
    n, lr = 4099, 1e-2
    p0 = rng.normal(0, 0.02, size=n).astype(np.float32)
    seq = [[rng.normal(0, 1e-3, size=n).astype(np.float32) for _ in range(N)] for _ in range(5)]
    ref = _torch_sgd(p0, seq, lr, mu, damp, wd, nest, torch.float32)
    params = [p0.copy() for _ in range(N)]
    states = oracle.init_states_sgd(n, N, mode="fp32")
    for t, grads in enumerate(seq, start=1):
        params, states = oracle.zero_step_sgd(params, grads, states, t, lr=lr, momentum=mu,
                                              dampening=damp, weight_decay=wd, nesterov=nest)
        rp, rb = ref[t - 1]
        assert params[0].dtype == np.float32
        assert np.all(np.abs(params[0] - rp) <= 1e-6 + 1e-5 * np.abs(rp))
        b = flat_state(states, "buf")
        assert np.all(np.abs(b - rb) <= 1e-6 * np.abs(rb).max() + 1e-5 * np.abs(rb))


@pytest.mark.parametrize("nest", [False, True])
def test_sgd_constant_gradient_closed_form(nest):
    # constant g, no decay or dampening: buf_t = g (1 - mu^t) / (1 - mu); the step
    # moves by lr * buf_t, or lr * (g + mu buf_t) with Nesterov
    n, N, lr, mu, t_max = 7, 3, 0.1, 0.9, 6
    g = np.linspace(-2.0, 3.0, n)
    p0 = np.linspace(1.0, -1.0, n)
    params = [p0.copy() for _ in range(N)]
    states = oracle.init_states_sgd(n, N, mode="fp64")
    moved = np.zeros(n)
    for t in range(1, t_max + 1):
        params, states = oracle.zero_step_sgd(params, [g] * N, states, t, lr=lr, momentum=mu,
                                              nesterov=nest, mode="fp64")
        buf = g * (1.0 - mu ** t) / (1.0 - mu)
        moved += lr * (g + mu * buf if nest else buf)
        np.testing.assert_allclose(flat_state(states, "buf"), buf, rtol=1e-13)
        np.testing.assert_allclose(params[1], p0 - moved, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("N", [1, 2, 3, 4, 7, 8])
@pytest.mark.parametrize("mode", ["fp32", "fp64"])
def test_sgd_sharded_equals_unsharded(N, mode):
    rng = np.random.default_rng(200 + N)
    n = 1009
    dt = np.float64 if mode == "fp64" else np.float32
    p = rng.normal(size=n).astype(dt)
    params = [p.copy() for _ in range(N)]
    states = oracle.init_states_sgd(n, N, mode=mode)
    buf = None
    for t in range(1, 5):
        grads = [rng.normal(size=n).astype(np.float32) for _ in range(N)]
        gbar = zo._mean_over_ranks([g.astype(dt) for g in grads], mode)
        params, states = oracle.zero_step_sgd(params, grads, states, t, lr=1e-2, momentum=0.9,
                                              dampening=0.1, weight_decay=0.05, mode=mode)
        p, buf = oracle.sgd_full(p, gbar, buf, t, lr=1e-2, momentum=0.9, dampening=0.1,
                                 weight_decay=0.05, mode=mode)
        for rep in params:
            assert rep.dtype == dt and np.array_equal(rep, p)
        assert np.array_equal(flat_state(states, "buf"), buf)


@pytest.mark.parametrize("N", [2, 4])
def test_sgd_ddp_matches_single_process(N):
    # course page section 4, test_ddp_matches_single_process: 2 and 4 ranks,
    # 5 momentum-SGD steps agree with one process on the whole batch to 1e-10.
    # Least squares: rank r's gradient is that of its slice's mean loss; the
    # single process differentiates the whole batch's mean loss directly.
    rng = np.random.default_rng(300 + N)
    n, B = 12, 6
    X = rng.normal(size=(N * B, n))
    y = rng.normal(size=N * B)
    w0 = rng.normal(size=n)
    params = [w0.copy() for _ in range(N)]
    states = oracle.init_states_sgd(n, N, mode="fp64")
    w = w0.copy()
    buf = np.zeros(n)
    for t in range(1, 6):
        grads = [X[r * B:(r + 1) * B].T @ (X[r * B:(r + 1) * B] @ params[r] - y[r * B:(r + 1) * B])
                 / B for r in range(N)]
        params, states = oracle.zero_step_sgd(params, grads, states, t, lr=0.05, momentum=0.9,
                                              mode="fp64")
        g_full = X.T @ (X @ w - y) / (N * B)
        buf = g_full if t == 1 else 0.9 * buf + g_full
        w = w - 0.05 * buf
        for rep in params:
            np.testing.assert_allclose(rep, w, rtol=0, atol=1e-10)


def test_sgd_stage3_gather_equals_all_gather():
    rng = np.random.default_rng(77)
    n, N = 1009, 4
    init = rng.normal(0, 0.02, n).astype(np.float32)
    for prec in (oracle.FP32, oracle.BF16_MIXED):
        reps = [oracle.f32_to_bf16_rne(init) if prec else init.copy() for _ in range(N)]
        g = [rng.normal(size=n).astype(np.float32) for _ in range(N)]
        if prec:
            g = [oracle.f32_to_bf16_rne(x) for x in g]
        full, a = oracle.zero_step_sgd(reps, g, oracle.init_states_sgd(n, N, prec, init), 1,
                                       momentum=0.9, precision=prec)
        shards, b = oracle.zero_step_sgd(reps, g, oracle.init_states_sgd(n, N, prec, init), 1,
                                         momentum=0.9, precision=prec, all_gather=False)
        for x, y in zip(oracle.gather(shards), full):
            assert np.array_equal(x, y)
        if prec:
            np.testing.assert_array_equal(full[0], oracle.f32_to_bf16_rne(flat_state(a, "master")))


def test_sgd_rejects():
    with pytest.raises(ValueError):
        zo._sgd(np.zeros(3), np.zeros(3), None, 0, 0.1, 0.9, 0.0, 0.0, False, "fp64")
    with pytest.raises(ValueError):
        zo._sgd(np.zeros(3), np.zeros(3), None, 1, 0.1, 0.0, 0.0, 0.0, True, "fp64")
    with pytest.raises(ValueError):
        zo._sgd(np.zeros(3), np.zeros(3), None, 1, 0.1, 0.9, 0.1, 0.0, True, "fp64")


def _sgd_mutant(**override):
    real = zo._sgd

    def mutant(p, g, buf, t, lr, momentum, dampening, weight_decay, nesterov, mode):
        kw = dict(lr=lr, momentum=momentum, dampening=dampening, weight_decay=weight_decay,
                  nesterov=nesterov)
        kw.update(override)
        return real(p, g, buf, t, kw["lr"], kw["momentum"], kw["dampening"],
                    kw["weight_decay"], kw["nesterov"], mode)
    return mutant


@pytest.mark.parametrize("override,case", [
    (dict(dampening=0.0), (4, 0.9, 0.1, 0.01, False)),
    (dict(nesterov=False), (3, 0.5, 0.0, 0.1, True)),
    (dict(momentum=0.0, nesterov=False), (2, 0.9, 0.0, 0.0, False)),
    (dict(weight_decay=0.0), (4, 0.0, 0.0, 0.05, False))])
def test_mutant_sgd_dropped_terms(monkeypatch, override, case):
    monkeypatch.setattr(zo, "_sgd", _sgd_mutant(**override))
    assert _fails(lambda: test_sgd_fp64_matches_torch_sgd(*case))


def test_mutant_sgd_first_step_damped(monkeypatch):
    # the buffer starts as (1 - dampening) g instead of g
    real = zo._sgd

    def mutant(p, g, buf, t, lr, momentum, dampening, weight_decay, nesterov, mode):
        if t == 1 and momentum:
            buf = np.zeros_like(np.asarray(g, dtype=zo._dtype(mode)))
            t = 2
        return real(p, g, buf, t, lr, momentum, dampening, weight_decay, nesterov, mode)
    monkeypatch.setattr(zo, "_sgd", mutant)
    assert _fails(lambda: test_sgd_fp64_matches_torch_sgd(4, 0.9, 0.1, 0.01, False))


# ---------------------------------------------------------------------------
# Brute force on tiny inputs: one entry at a time in Python scalars
# ---------------------------------------------------------------------------

def _brute_adamw(p, gs, m, v, t, lr, b1, b2, eps, wd):
    """One entry, Python floats (IEEE double): mean in rank order, then AdamW."""
    g = 0.0
    for x in gs:
        g = g + x
    g = g / len(gs)
    p = p * (1.0 - lr * wd)
    m = b1 * m + (1.0 - b1) * g
    v = b2 * v + (1.0 - b2) * (g * g)
    m_hat = m / (1.0 - b1 ** t)
    v_hat = v / (1.0 - b2 ** t)
    return p - lr * m_hat / (math.sqrt(v_hat) + eps), m, v


def _brute_adamw_f32(p, gs, m, v, c):
    """One entry in float32 scalars, one rounding per written operation."""
    f = np.float32
    g = f(gs[0])
    for x in gs[1:]:
        g = f(g + f(x))
    g = f(g / f(len(gs)))
    p = f(p * c["decay"])
    m = f(f(c["b1"] * m) + f(c["omb1"] * g))
    v = f(f(c["b2"] * v) + f(c["omb2"] * f(g * g)))
    d = f(f(np.sqrt(v) / c["bc2s"]) + c["eps"])
    return f(p - f(c["step"] * f(m / d))), m, v


@pytest.mark.parametrize("n,N", [(1, 1), (2, 3), (5, 2), (7, 5), (8, 4)])
def test_brute_force_tiny_adamw(n, N):
    rng = np.random.default_rng(500 + 10 * n + N)
    lr, b1, b2, eps, wd = 3e-3, 0.9, 0.95, 1e-8, 0.05
    p0 = rng.normal(size=n)
    params64 = [p0.copy() for _ in range(N)]
    params32 = [p0.astype(np.float32) for _ in range(N)]
    s64 = oracle.init_states(n, N, mode="fp64")
    s32 = oracle.init_states(n, N, mode="fp32")
    bp64 = [(float(x), 0.0, 0.0) for x in p0]
    bp32 = [(np.float32(x), np.float32(0), np.float32(0)) for x in p0.astype(np.float32)]
    for t in range(1, 5):
        grads = [rng.normal(size=n).astype(np.float32) for _ in range(N)]
        params64, s64 = oracle.zero_step(params64, grads, s64, t, lr=lr, beta1=b1, beta2=b2,
                                         eps=eps, weight_decay=wd, mode="fp64")
        params32, s32 = oracle.zero_step(params32, grads, s32, t, lr=lr, beta1=b1, beta2=b2,
                                         eps=eps, weight_decay=wd, mode="fp32")
        c = oracle.mirror_scalars(t, lr, b1, b2, eps, wd)
        bp64 = [_brute_adamw(p, [float(g[j]) for g in grads], m, v, t, lr, b1, b2, eps, wd)
                for j, (p, m, v) in enumerate(bp64)]
        bp32 = [_brute_adamw_f32(p, [g[j] for g in grads], m, v, c)
                for j, (p, m, v) in enumerate(bp32)]
        for rep in params64:   # double: the same values up to the order of the last ops
            np.testing.assert_allclose(rep, [x[0] for x in bp64], rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(flat_state(s64, "m"), [x[1] for x in bp64], rtol=1e-13,
                                   atol=1e-16)
        for rep in params32:   # fp32-mirror: bit for bit
            assert np.array_equal(rep, np.array([x[0] for x in bp32], np.float32))
        assert np.array_equal(flat_state(s32, "v"), np.array([x[2] for x in bp32], np.float32))


@pytest.mark.parametrize("n,N", [(1, 1), (3, 2), (8, 5)])
def test_brute_force_tiny_sgd(n, N):
    rng = np.random.default_rng(600 + 10 * n + N)
    lr, mu, damp, wd = 0.05, 0.9, 0.1, 0.01
    p0 = rng.normal(size=n)
    params = [p0.copy() for _ in range(N)]
    states = oracle.init_states_sgd(n, N, mode="fp64")
    brute = [(float(x), 0.0) for x in p0]
    for t in range(1, 5):
        grads = [rng.normal(size=n) for _ in range(N)]
        params, states = oracle.zero_step_sgd(params, grads, states, t, lr=lr, momentum=mu,
                                              dampening=damp, weight_decay=wd, mode="fp64")
        nxt = []
        for j, (p, b) in enumerate(brute):
            g = 0.0
            for gr in grads:
                g = g + float(gr[j])
            g = g / N + wd * p
            b = g if t == 1 else mu * b + (1.0 - damp) * g
            nxt.append((p - lr * b, b))
        brute = nxt
        for rep in params:
            np.testing.assert_allclose(rep, [x[0] for x in brute], rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(flat_state(states, "buf"), [x[1] for x in brute], rtol=1e-13,
                                   atol=1e-15)
