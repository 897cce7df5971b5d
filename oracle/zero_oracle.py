"""CPU oracle for one ZeRO step over N simulated data-parallel ranks.

TEST INFRASTRUCTURE. Only the test suite, the package's smoke check and the
benchmark's CPU-baseline leg may import this module. The product path (the
CUDA library and its Python binding) never calls it and shares no code with it.

What it computes (plain definitions, written out slowly; numpy with a loop over
ranks and workers only):

* ``shard_bounds``   -- the np.array_split partition of the parameter indices
  ("ZeRO-Sharded Adam Step", section "The shards").
* ``zero_step``      -- reduce-scatter-mean of the N local gradients, Adam/AdamW
  on each worker's shard with that worker's own m and v, all-gather of the
  updated shards into every replica ("ZeRO-Sharded Adam Step", sections
  "The step" and "What to implement"; "Data parallelism and ZeRO stages 1 to 3",
  section 2 "Principles", stages 1 and 2).
* ``adam_full``      -- the same Adam/AdamW step on the whole vector with the mean
  gradient: the unsharded reference that the sharded step must equal
  ("ZeRO-Sharded Adam Step", section "Requirements").
* ``allreduce_mean`` -- the DDP gradient mean, identical on every rank
  ("Data parallelism and ZeRO stages 1 to 3", section 2, "DDP").
* ``memory_bytes`` / ``memory_breakdown`` -- model-state bytes per rank by ZeRO
  stage ("Data Parallelism & ZeRO", section "ZeRO, stage by stage";
  "Data parallelism and ZeRO optimization", sections "Memory Consumption
  Analysis" and "ZeRO-1/2/3"; "ZeRO One: Sharding the Optimizer", section
  "Training Memory Requirements"; the float64 bookkeeping table of
  "Data parallelism and ZeRO stages 1 to 3", section 3).
* ``tensor_shard_bounds`` -- shards of whole tensors ("ZeRO One: Sharding the
  Optimizer", "Sharding Parameters").
* ``bucket_bounds``  -- 25 MiB gradient buckets built from the end of the flat
  gradient ("ZeRO One: Sharding the Optimizer", section "Bucketing").
* ``zero_step_sgd`` -- the same ZeRO step with momentum SGD as the wrapped
  optimizer ("Data parallelism and ZeRO stages 1 to 3", section 2, stage 1:
  SGD is elementwise like AdamW, so the chunked update equals the unsharded
  one; section 4 tests DDP with momentum-SGD steps); ``sgd_full`` is its
  unsharded reference.
* ``grad_norm`` / ``grad_multiplier`` -- the global gradient norm from squared
  chunk norms, and the clip / accumulation factor applied to the mean gradient
  ("Data parallelism and ZeRO stages 1 to 3", "Going further"; "Data
  Parallelism & ZeRO", "Two more things you'll actually hit").

Arithmetic modes:

* ``"fp64"``  -- every operation in float64 on upcast inputs: the mathematical
  reference.
* ``"fp32"``  -- fp32-mirror: each operation is one IEEE float32 operation, in
  the order written below, never fused. Host-side scalars (decay factor,
  1-beta, bias-correction step and sqrt) are formed in float64 from the float64
  hyperparameters and rounded to float32 once.

Readings taken where the pages are silent (each is listed in the design notes):

1. The Adam update itself is not printed on the pages (the problem page
   treats ``adam_update`` as supplied and never shows its body). Reading: Adam with bias correction and eps
   added outside the square root; AdamW's weight decay is decoupled and scaled
   by lr, applied before the moment update. The course page fixes the t=1
   behaviour (m = (1-b1) g, v = (1-b2) g^2, m_hat = g, sqrt(v_hat) = |g|).
2. fp32 operation order: ``p*=decay; m=b1*m+(1-b1)*g; v=b2*v+(1-b2)*(g*g);
   d=sqrt(v)/bc2s+eps; p=p-step*(m/d)`` with ``step=lr/(1-b1^t)`` and
   ``bc2s=sqrt(1-b2^t)``.
3. Mean of the gradients: summed in fp32 (fp64 in the fp64 mode) in rank order
   0..N-1, then divided by N.
4. Mixed precision: bf16 replicas and gradients, fp32 master/m/v; gradients
   are upcast exactly, the mean is kept in fp32, replicas are the
   round-to-nearest-even bf16 of the new master.
5. NaN/Inf propagate as IEEE arithmetic gives them.
6. Clipping: coefficient max_norm / (norm + 1e-6) capped at 1, applied with the
   accumulation factor as one float64 multiplier rounded to float32.
7. Momentum SGD is named, not printed. Reading: torch.optim.SGD -- coupled
   weight decay g <- g + wd*p (skipped at wd = 0); with momentum mu the buffer
   is g at t = 1 and mu*buf + (1-dampening)*g after; the direction is the
   buffer, or g + mu*buf with Nesterov; p <- p - lr*direction. Without
   momentum there is no buffer and the direction is g. fp32 constants lr, wd,
   mu and (1 - dampening) are formed in float64 and rounded once.

Parity status: every function here is pinned by a CPU test against values the
pages print, closed forms, invariants or library routines (np.array_split,
np.mean, torch.optim.Adam/AdamW/SGD, torch.nn.utils.clip_grad_norm_, torch's
bf16 cast); none is "parity unpinned".
"""

from __future__ import annotations

import math

import numpy as np

__all__ = [
    "FP32", "BF16_MIXED", "FP64_EMU",
    "shard_bounds", "init_states", "zero_step", "adam_full", "allreduce_mean",
    "zero_step_sgd", "sgd_full", "init_states_sgd",
    "grad_norm", "grad_multiplier", "tensor_shard_bounds", "gather",
    "memory_bytes", "memory_breakdown", "bucket_bounds",
    "bf16_to_f32", "f32_to_bf16_rne", "mirror_scalars",
]

# Precision of the stored training state (same meaning as the C library's enum).
FP32 = 0        # fp32 params, grads, m, v (4+4+8 bytes per parameter)
BF16_MIXED = 1  # bf16 params and grads, fp32 master, m, v (2+2+12)
FP64_EMU = 2    # the course's float64 emulation bookkeeping (memory only)


# --------------------------------------------------------------------------
# Shards
# --------------------------------------------------------------------------

def shard_bounds(n: int, N: int) -> list[int]:
    """Offsets a_0..a_N of the N shards of [0, n).

    "ZeRO-Sharded Adam Step", "The shards": shard i is the i-th piece of
    np.array_split(np.arange(n), N). array_split gives the first n mod N pieces
    one extra element, so with q = n // N and r = n mod N the i-th piece starts
    at i*q + min(i, r).
    """
    if N < 1:
        raise ValueError("number of workers must be >= 1")
    if n < 0:
        raise ValueError("number of parameters must be >= 0")
    q, r = divmod(n, N)
    return [i * q + min(i, r) for i in range(N + 1)]


def tensor_shard_bounds(numels, N: int) -> list[int]:
    """Element offsets of N shards made of whole tensors.

    "ZeRO One: Sharding the Optimizer", "Sharding Parameters": the list of
    parameter tensors (in parameters() order) is divided like the indices are
    in "The shards" -- rank i gets tensors [i*q + min(i, r), (i+1)*q + min(i+1, r))
    with q, r = divmod(len(tensors), N) -- so a shard never splits a tensor.
    Returns the flat-vector offsets of those tensor boundaries.
    """
    T = len(numels)
    if any(int(x) < 0 for x in numels):
        raise ValueError("tensor sizes must be >= 0")
    first = shard_bounds(T, N)                      # tensor indices
    offsets = [0]
    for x in numels:
        offsets.append(offsets[-1] + int(x))
    return [offsets[k] for k in first]


def _check_bounds(bounds, n, N):
    if len(bounds) != N + 1 or bounds[0] != 0 or bounds[-1] != n or any(
            b > c for b, c in zip(bounds, bounds[1:])):
        raise ValueError("shard bounds must rise from 0 to n in N steps")
    return list(bounds)


# --------------------------------------------------------------------------
# bf16 <-> fp32 (bit level, for the mixed-precision mode)
# --------------------------------------------------------------------------

def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float32."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def f32_to_bf16_rne(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); uint16 bits.

    Adds 0x7FFF plus the lowest kept bit to the 32-bit pattern and keeps the top
    16 bits: a carry into the kept half happens exactly when the dropped half is
    above one half, or equal to one half with an odd kept part. NaN inputs map
    to a quiet NaN with the same sign.
    """
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    kept_lsb = (b >> np.uint64(16)) & np.uint64(1)
    rounded = ((b + np.uint64(0x7FFF) + kept_lsb) >> np.uint64(16)) & np.uint64(0xFFFF)
    is_nan = (b & np.uint64(0x7FFFFFFF)) > np.uint64(0x7F800000)
    quiet = ((b >> np.uint64(16)) | np.uint64(0x0040)) & np.uint64(0xFFFF)
    return np.where(is_nan, quiet, rounded).astype(np.uint16)


# --------------------------------------------------------------------------
# Adam / AdamW on one array
# --------------------------------------------------------------------------

def mirror_scalars(t: int, lr: float, beta1: float, beta2: float, eps: float,
                   weight_decay: float) -> dict:
    """Per-step float32 constants of the fp32-mirror mode.

    The hyperparameters are float64 values (as the C library receives them);
    each constant is formed in float64 and rounded to float32 once.
    """
    lr, beta1, beta2, eps, weight_decay = (float(x) for x in
                                           (lr, beta1, beta2, eps, weight_decay))
    return {
        "decay": np.float32(1.0 - lr * weight_decay),
        "b1": np.float32(beta1),
        "omb1": np.float32(1.0 - beta1),
        "b2": np.float32(beta2),
        "omb2": np.float32(1.0 - beta2),
        "step": np.float32(lr / (1.0 - beta1 ** t)),
        "bc2s": np.float32(math.sqrt(1.0 - beta2 ** t)),
        "eps": np.float32(eps),
    }


def _adam(p, g, m, v, t, lr, beta1, beta2, eps, weight_decay, mode):
    """One Adam/AdamW step on arrays of equal length; returns new (p, m, v).

    AdamW (decoupled decay): p <- p*(1 - lr*wd); m <- b1*m + (1-b1)*g;
    v <- b2*v + (1-b2)*g^2; p <- p - lr * m_hat / (sqrt(v_hat) + eps) with
    m_hat = m/(1-b1^t), v_hat = v/(1-b2^t). With wd = 0 this is Adam.
    """
    if t < 1:
        raise ValueError("step number t starts at 1")
    if mode == "fp64":
        p = np.asarray(p, dtype=np.float64)
        g = np.asarray(g, dtype=np.float64)
        m = np.asarray(m, dtype=np.float64)
        v = np.asarray(v, dtype=np.float64)
        p = p * (1.0 - lr * weight_decay)
        m = beta1 * m + (1.0 - beta1) * g
        v = beta2 * v + (1.0 - beta2) * (g * g)
        m_hat = m / (1.0 - beta1 ** t)
        v_hat = v / (1.0 - beta2 ** t)
        p = p - lr * m_hat / (np.sqrt(v_hat) + eps)
        return p, m, v
    if mode == "fp32":
        c = mirror_scalars(t, lr, beta1, beta2, eps, weight_decay)
        p = np.asarray(p, dtype=np.float32)
        g = np.asarray(g, dtype=np.float32)
        m = np.asarray(m, dtype=np.float32)
        v = np.asarray(v, dtype=np.float32)
        p = p * c["decay"]
        m = c["b1"] * m + c["omb1"] * g
        v = c["b2"] * v + c["omb2"] * (g * g)
        denom = np.sqrt(v) / c["bc2s"] + c["eps"]
        p = p - c["step"] * (m / denom)
        return p, m, v
    raise ValueError(f"unknown arithmetic mode {mode!r}")


def _sgd(p, g, buf, t, lr, momentum, dampening, weight_decay, nesterov, mode):
    """One momentum-SGD step on arrays of equal length; returns new (p, buf).

    g <- g + wd*p (wd != 0); buf <- g at t = 1, else mu*buf + (1-dampening)*g
    (mu != 0); direction d = g + mu*buf (Nesterov) or buf, or d = g without
    momentum (buf stays None); p <- p - lr*d.
    """
    if t < 1:
        raise ValueError("step number t starts at 1")
    if nesterov and (momentum <= 0 or dampening != 0):
        raise ValueError("Nesterov momentum needs momentum > 0 and zero dampening")
    dt = _dtype(mode)
    lr_, wd_, mu_, omd_ = (dt(x) for x in (float(lr), float(weight_decay), float(momentum),
                                           1.0 - float(dampening)))
    p = np.asarray(p, dtype=dt)
    g = np.asarray(g, dtype=dt)
    if weight_decay != 0:
        g = g + wd_ * p
    if momentum != 0:
        if t == 1:
            buf = g.copy()
        else:
            buf = mu_ * np.asarray(buf, dtype=dt) + omd_ * g
        d = g + mu_ * buf if nesterov else buf
    else:
        buf = None
        d = g
    p = p - lr_ * d
    return p, buf


def _dtype(mode):
    return np.float64 if mode == "fp64" else np.float32


def _as_compute(x, precision, mode):
    """Gradient or parameter storage -> the arithmetic type of ``mode``."""
    if precision == BF16_MIXED:
        x = bf16_to_f32(x)
    return np.asarray(x, dtype=_dtype(mode))


def _mean_over_ranks(pieces, mode):
    """(((g_0 + g_1) + g_2) + ... + g_{N-1}) / N, accumulated in rank order."""
    acc = np.array(pieces[0], dtype=_dtype(mode), copy=True)
    for piece in pieces[1:]:
        acc = acc + piece
    return acc / _dtype(mode)(len(pieces))


def _replica_from(p, precision, mode="fp32"):
    """Value written into every rank's parameter replica by the all-gather.

    fp32 storage keeps the arithmetic type of the mode (fp64 mode: no storage
    rounding); bf16 storage is the round-to-nearest-even of the fp32 value.
    """
    if precision == BF16_MIXED:
        return f32_to_bf16_rne(np.asarray(p, dtype=np.float32))
    return np.asarray(p, dtype=_dtype(mode))


# --------------------------------------------------------------------------
# The ZeRO step
# --------------------------------------------------------------------------

def init_states(n: int, N: int, precision: int = FP32, master_init=None, mode: str = "fp32",
                bounds=None):
    """One state dict per worker, each the size of that worker's shard.

    "ZeRO-Sharded Adam Step", "What to implement": init_states gives N pairs
    (m_shard, v_shard) of zeros. In mixed precision every worker also holds the
    fp32 master copy of its shard ("Data parallelism and ZeRO optimization",
    "Memory Consumption Analysis": master weights are part of the 12 bytes of
    optimizer state); it starts as the fp32 initial weights.
    """
    bounds = shard_bounds(n, N) if bounds is None else _check_bounds(bounds, n, N)
    dt = _dtype(mode)
    states = []
    for i in range(N):
        a, b = bounds[i], bounds[i + 1]
        st = {"m": np.zeros(b - a, dtype=dt), "v": np.zeros(b - a, dtype=dt)}
        if precision == BF16_MIXED:
            if master_init is None:
                raise ValueError("mixed precision needs the fp32 initial weights")
            st["master"] = np.asarray(master_init[a:b], dtype=np.float32).astype(dt)
        states.append(st)
    return states


def init_states_sgd(n: int, N: int, precision: int = FP32, master_init=None,
                    mode: str = "fp32", bounds=None, momentum: bool = True):
    """Momentum-SGD state per worker: the momentum buffer of its shard (zeros;
    none without momentum) and, in mixed precision, the fp32 master copy."""
    bounds = shard_bounds(n, N) if bounds is None else _check_bounds(bounds, n, N)
    dt = _dtype(mode)
    states = []
    for i in range(N):
        a, b = bounds[i], bounds[i + 1]
        st = {"buf": np.zeros(b - a, dtype=dt) if momentum else None}
        if precision == BF16_MIXED:
            if master_init is None:
                raise ValueError("mixed precision needs the fp32 initial weights")
            st["master"] = np.asarray(master_init[a:b], dtype=np.float32).astype(dt)
        states.append(st)
    return states


def _reduce_scatter_mean(grads, a, b, precision, mode):
    """Step 1 for one worker: the mean over all workers of grads[.][a:b]."""
    return _mean_over_ranks([_as_compute(g[a:b], precision, mode) for g in grads], mode)


def _all_gather(new_shards, N, precision, mode):
    """Step 3: every worker's replica becomes the concatenation of all shards."""
    full = np.concatenate(new_shards) if new_shards else np.zeros(0, dtype=_dtype(mode))
    replica = _replica_from(full, precision, mode)
    return [replica.copy() for _ in range(N)]


def grad_norm(grads, precision=FP32, mode="fp32") -> float:
    """Global L2 norm of the mean gradient, assembled from the shards.

    "Data parallelism and ZeRO stages 1 to 3", "Going further" (clipping):
    sharded global-norm clipping all-reduces the squared norms of the chunks
    before the step. Each worker squares and sums its shard of the mean
    gradient (float64 sums of the mode's mean values); the N squared chunk
    norms are added in rank order and the square root taken.
    """
    N = len(grads)
    n = len(grads[0])
    bounds = shard_bounds(n, N)
    total = 0.0
    for i in range(N):
        a, b = bounds[i], bounds[i + 1]
        g_bar = _reduce_scatter_mean(grads, a, b, precision, mode).astype(np.float64)
        total += float(np.sum(g_bar * g_bar))           # squared chunk norm
    return math.sqrt(total)


def grad_multiplier(norm: float, grad_scale: float = 1.0, max_grad_norm=None) -> float:
    """The factor that multiplies the mean gradient before the update.

    ``grad_scale`` turns a sum of k accumulated micro-batch gradients into their
    mean (1/k; "Data Parallelism & ZeRO", "Two more things you'll actually
    hit": scale by 1/k so the accumulated gradient is a mean). With
    ``max_grad_norm`` the scaled gradient is clipped to that global norm; the
    pages give no formula, the reading is the usual one: coefficient
    max_norm / (norm + 1e-6), never above 1. Formed in float64.
    """
    coef = 1.0
    if max_grad_norm is not None and max_grad_norm > 0:
        coef = min(1.0, max_grad_norm / (grad_scale * norm + 1e-6))
    return grad_scale * coef


def zero_step(params, grads, states, t, lr=1e-2, beta1=0.9, beta2=0.999, eps=1e-8,
              weight_decay=0.0, precision=FP32, mode="fp32", grad_scale=1.0,
              max_grad_norm=None, bounds=None, all_gather=True):
    """One ZeRO step; returns (new_params, new_states).

    ``params``: N full-length replicas (float32, or bf16 bits as uint16).
    ``grads``:  N full-length local gradients, same storage type.
    ``states``: from ``init_states`` or a previous step.

    Follows "ZeRO-Sharded Adam Step", "The step":
      1. reduce-scatter: worker i receives the mean over all workers of the
         gradient, only for the indices of its shard;
      2. worker i runs Adam on its shard with its own m and v (its parameter
         source is its own replica's shard in fp32, its master in mixed mode);
      3. all-gather: the updated shards are concatenated and every worker's
         replica becomes the full updated vector.
    ``bounds`` (N+1 offsets, default the array_split shards) sets who owns
    what, e.g. whole tensors from ``tensor_shard_bounds``; it must match the
    bounds ``states`` were built with.
    With ``all_gather=False`` (ZeRO-3) step 3 is left out: each rank's entry
    of the result is only its own updated chunk (``gather`` assembles them).
    With ``grad_scale`` != 1 or ``max_grad_norm`` set, the mean gradient is
    first multiplied by ``grad_multiplier`` (rounded to float32 in the fp32
    mode); the global norm it needs comes from ``grad_norm`` of the same
    gradients.
    """
    N = len(grads)
    if len(params) != N or len(states) != N:
        raise ValueError("params, grads and states need one entry per worker")
    n = len(params[0])
    bounds = shard_bounds(n, N) if bounds is None else _check_bounds(bounds, n, N)
    mult = None
    if grad_scale != 1.0 or (max_grad_norm is not None and max_grad_norm > 0):
        norm = grad_norm(grads, precision, mode) if max_grad_norm else 0.0
        mult = _dtype(mode)(grad_multiplier(norm, grad_scale, max_grad_norm))
    new_shards, new_states = [], []
    for i in range(N):                                   # loop over workers only
        a, b = bounds[i], bounds[i + 1]
        g_bar = _reduce_scatter_mean(grads, a, b, precision, mode)          # 1.
        if mult is not None:
            g_bar = g_bar * mult
        st = states[i]
        if precision == BF16_MIXED:
            p_src = st["master"]
        else:
            p_src = _as_compute(params[i][a:b], precision, mode)
        p_new, m_new, v_new = _adam(p_src, g_bar, st["m"], st["v"], t, lr, beta1,  # 2.
                                    beta2, eps, weight_decay, mode)
        ns = {"m": m_new, "v": v_new}
        if precision == BF16_MIXED:
            ns["master"] = p_new
        new_states.append(ns)
        new_shards.append(p_new)
    if not all_gather:
        # ZeRO-3 ("Data parallelism and ZeRO stages 1 to 3", section 2, stage 3):
        # between steps each rank keeps only its own chunk of the parameters
        return [_replica_from(sh, precision, mode) for sh in new_shards], new_states
    return _all_gather(new_shards, N, precision, mode), new_states                # 3.


def zero_step_sgd(params, grads, states, t, lr=1e-2, momentum=0.0, dampening=0.0,
                  weight_decay=0.0, nesterov=False, precision=FP32, mode="fp32",
                  grad_scale=1.0, max_grad_norm=None, bounds=None, all_gather=True):
    """One ZeRO step with momentum SGD on each shard; returns (new_params, new_states).

    The same three steps as ``zero_step`` ("Data parallelism and ZeRO stages 1
    to 3", section 2, stage 1: the wrapped optimizer steps the rank's chunk
    with the chunk of the mean gradient, then the chunks are all-gathered),
    with ``_sgd`` in place of Adam. ``states`` come from ``init_states_sgd``.
    """
    N = len(grads)
    if len(params) != N or len(states) != N:
        raise ValueError("params, grads and states need one entry per worker")
    n = len(params[0])
    bounds = shard_bounds(n, N) if bounds is None else _check_bounds(bounds, n, N)
    mult = None
    if grad_scale != 1.0 or (max_grad_norm is not None and max_grad_norm > 0):
        norm = grad_norm(grads, precision, mode) if max_grad_norm else 0.0
        mult = _dtype(mode)(grad_multiplier(norm, grad_scale, max_grad_norm))
    new_shards, new_states = [], []
    for i in range(N):
        a, b = bounds[i], bounds[i + 1]
        g_bar = _reduce_scatter_mean(grads, a, b, precision, mode)
        if mult is not None:
            g_bar = g_bar * mult
        st = states[i]
        if precision == BF16_MIXED:
            p_src = st["master"]
        else:
            p_src = _as_compute(params[i][a:b], precision, mode)
        p_new, buf = _sgd(p_src, g_bar, st["buf"], t, lr, momentum, dampening, weight_decay,
                          nesterov, mode)
        ns = {"buf": buf}
        if precision == BF16_MIXED:
            ns["master"] = p_new
        new_states.append(ns)
        new_shards.append(p_new)
    if not all_gather:
        return [_replica_from(sh, precision, mode) for sh in new_shards], new_states
    return _all_gather(new_shards, N, precision, mode), new_states


def sgd_full(param, mean_grad, buf, t, lr=1e-2, momentum=0.0, dampening=0.0,
             weight_decay=0.0, nesterov=False, mode="fp32"):
    """Unsharded momentum SGD on the whole vector with the mean gradient."""
    return _sgd(param, mean_grad, buf, t, lr, momentum, dampening, weight_decay, nesterov, mode)


def gather(shards, precision=FP32, mode="fp32"):
    """ZeRO-3 gather(): all-gather the ranks' parameter chunks into the full
    parameters on every rank ("Data parallelism and ZeRO stages 1 to 3", section
    2, stage 3, and section 4, ``gather()`` before the forward pass). ``shards``
    are the chunks in storage form (float32, or bf16 bits)."""
    full = np.concatenate(shards) if shards else np.zeros(0, np.float32)
    return [full.copy() for _ in range(len(shards))]


def adam_full(param, mean_grad, m, v, t, lr=1e-2, beta1=0.9, beta2=0.999, eps=1e-8,
              weight_decay=0.0, mode="fp32"):
    """Unsharded Adam/AdamW on the whole vector with the mean gradient.

    The reference that the sharded step must equal entry by entry
    ("ZeRO-Sharded Adam Step", "Requirements"; "Data parallelism and ZeRO
    stages 1 to 3", section 2: the chunked update equals the single-process
    update because the optimizer is elementwise).
    """
    return _adam(param, mean_grad, m, v, t, lr, beta1, beta2, eps, weight_decay, mode)


def allreduce_mean(grads, precision=FP32, mode="fp32"):
    """DDP all_reduce(op="mean"): every rank ends with the same mean gradient.

    "Data parallelism and ZeRO stages 1 to 3", section 2 ("DDP"): one all-reduce
    with op mean gives every rank the averaged gradient with identical bits.
    Stored back in the gradients' own type (bf16: round to nearest even).
    """
    g_bar = _mean_over_ranks([_as_compute(g, precision, mode) for g in grads], mode)
    out = _replica_from(g_bar, precision, mode)
    return [out.copy() for _ in range(len(grads))]


# --------------------------------------------------------------------------
# Memory accounting
# --------------------------------------------------------------------------

# bytes per parameter for (params, grads, optimizer state):
#   fp32 training: 4, 4, 8 (m, v)        -- "ZeRO One", "Training Memory Requirements"
#   mixed bf16:    2, 2, 12 (master,m,v) -- "Data parallelism and ZeRO optimization",
#                                           "Memory Consumption Analysis"
_PER_PARAM = {FP32: (4, 4, 8), BF16_MIXED: (2, 2, 12)}


def memory_breakdown(n: int, N: int, stage: int, precision: int, rank: int = 0,
                     bounds=None) -> tuple:
    """(params, grads, optimizer) bytes held by ``rank`` after a step.

    Stage 0 is plain data parallelism (everything replicated). Stages 1, 2, 3
    shard the optimizer state, then also the gradients, then also the
    parameters ("Data Parallelism & ZeRO", "ZeRO, stage by stage"; "Data
    parallelism and ZeRO optimization", ZeRO-1/2/3 memory formulas). A rank's
    share is its np.array_split shard, so the per-rank sizes are exact when N
    does not divide n.

    FP64_EMU follows the course's float64 emulation bookkeeping ("Data
    parallelism and ZeRO stages 1 to 3", section 2 "Your emulation's
    bookkeeping" and the byte table of section 3): 8-byte values; stage 1 keeps
    the full averaged .grad plus the chunk's gradient; stages 1 and 2 hold m, v
    and a master copy of the chunk; in stage 3 the chunk is the parameter
    storage (m and v only); one process holds m and v for all n.
    ``bounds`` replaces the array_split shards (e.g. whole-tensor shards).
    """
    if N < 1 or n < 0 or stage not in (0, 1, 2, 3) or not 0 <= rank < N:
        raise ValueError("bad memory-accounting arguments")
    bounds = shard_bounds(n, N) if bounds is None else _check_bounds(bounds, n, N)
    s = bounds[rank + 1] - bounds[rank]
    if precision == FP64_EMU:
        b = 8
        params = s * b if stage == 3 else n * b
        if stage == 0:
            grads = n * b
        elif stage == 1:
            grads = n * b + s * b
        else:
            grads = s * b
        if stage == 0:
            opt = 2 * n * b
        elif stage == 3:
            opt = 2 * s * b
        else:
            opt = 3 * s * b
        return params, grads, opt
    if precision not in _PER_PARAM:
        raise ValueError("unknown precision")
    P, G, K = _PER_PARAM[precision]
    params = P * (s if stage == 3 else n)
    grads = G * (s if stage >= 2 else n)
    opt = K * (s if stage >= 1 else n)
    return params, grads, opt


def memory_bytes(n: int, N: int, stage: int, precision: int) -> int:
    """Model-state bytes on the most loaded rank (rank 0 holds the largest shard).

    With N | n this is 16n, 4n + 12n/N, 2n + 14n/N and 16n/N for mixed
    precision at stages 0..3 (16n, 8n + 8n/N, 4n + 12n/N, 16n/N for fp32).
    """
    return int(sum(memory_breakdown(n, N, stage, precision, 0)))


# --------------------------------------------------------------------------
# Gradient buckets
# --------------------------------------------------------------------------

def bucket_bounds(n: int, elem_bytes: int, bucket_bytes: int = 25 * 1024 * 1024) -> list:
    """Buckets of one rank's flat gradient, in the order they become ready.

    "ZeRO One: Sharding the Optimizer", "Bucketing": gradients are collected in
    the order backward produces them (reverse parameter order) and a bucket is
    synchronised once it holds bucket_cap_mb * 1024 * 1024 bytes. At element
    granularity over the flat gradient, bucket k covers
    [max(0, n - (k+1)*B), n - k*B) with B = bucket_bytes // elem_bytes; the last
    bucket to arrive (lowest indices) may be partial.
    """
    B = bucket_bytes // elem_bytes
    if B < 1:
        raise ValueError("bucket smaller than one element")
    out = []
    hi = n
    while hi > 0:
        lo = max(0, hi - B)
        out.append((lo, hi))
        hi = lo
    return out
