"""Seeded synthetic inputs for the ZeRO step: workloads, parameters, gradients.

This module only draws numbers. It holds none of the step's arithmetic, so the
CPU oracle and the CUDA path can both be fed from it without sharing code.

Workloads (each a flat parameter vector in ``parameters()`` order, N simulated
ranks whose buffers live in one GPU's memory):

* ``tiny_adam``   n=10,007 fp32, N=2; params U(-1,1) then per-rank grads N(0,1)
                  from ``numpy.random.default_rng(0)``; Adam lr=1e-2, (0.9, 0.999),
                  eps=1e-8, wd=0; steps t=1..5.
* ``fp32_25m``    n=25,000,000 fp32, N=4; params N(0,0.02); grads N(0,1e-3) per
                  rank with one shared mask of 1% exact zeros; AdamW 3e-4,
                  (0.9, 0.95), 1e-8, wd=0.01; 10 steps.
* ``gpt2_small``  the GPT-2-small parameter list (12 layers, d=768, 4x MLP,
                  vocab 50257, context 1024, tied head; 124,439,808 params),
                  bf16 params/grads with fp32 master/m/v, N=8; grads N(0,1e-3);
                  AdamW 6e-4, (0.9, 0.999), 1e-8, wd=0.1; 10 steps.
* ``fp32_320m``   n=320,000,000 fp32 (16 bytes/param of state), N=4; params
                  N(0,0.02); grads N(0,1e-3); AdamW 1e-4, (0.9, 0.999), 1e-8,
                  wd=0.01; 5 steps.
* ``mixed_1p3b``  n=1.3e9 mixed precision, N=8; gradients arrive as 25 MiB
                  buckets in reverse parameter order on a producer stream;
                  AdamW 1e-4, (0.9, 0.999), 1e-8, wd=0.1; 3 steps.

N(mu, s) means standard deviation s. Gradients are fresh at every step, drawn
from (seed, step, rank); the zero mask of ``fp32_25m`` is drawn once per step
from (seed, step) and applied to every rank, so the mean gradient is exactly
zero there.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

FP32 = 0
BF16_MIXED = 1


@dataclass(frozen=True)
class Workload:
    name: str
    n: int
    N: int
    precision: int
    steps: int
    lr: float
    beta1: float
    beta2: float
    eps: float
    weight_decay: float
    param_init: str          # "uniform1" = U(-1,1); "normal" = N(0, param_std)
    param_std: float
    grad_std: float
    zero_frac: float = 0.0
    bucket_bytes: int = 0    # > 0: gradients arrive in buckets of this many bytes
    notes: dict = field(default_factory=dict)


def gpt2_small_shapes() -> list[tuple[str, tuple[int, ...]]]:
    """GPT-2-small parameter tensors in ``parameters()`` order (tied LM head)."""
    d, L, V, T = 768, 12, 50257, 1024
    shapes = [("wte", (V, d)), ("wpe", (T, d))]
    for i in range(L):
        shapes += [
            (f"h{i}.ln_1.w", (d,)), (f"h{i}.ln_1.b", (d,)),
            (f"h{i}.attn.c_attn.w", (d, 3 * d)), (f"h{i}.attn.c_attn.b", (3 * d,)),
            (f"h{i}.attn.c_proj.w", (d, d)), (f"h{i}.attn.c_proj.b", (d,)),
            (f"h{i}.ln_2.w", (d,)), (f"h{i}.ln_2.b", (d,)),
            (f"h{i}.mlp.c_fc.w", (d, 4 * d)), (f"h{i}.mlp.c_fc.b", (4 * d,)),
            (f"h{i}.mlp.c_proj.w", (4 * d, d)), (f"h{i}.mlp.c_proj.b", (d,)),
        ]
    shapes += [("ln_f.w", (d,)), ("ln_f.b", (d,))]
    return shapes


def gpt2_small_numel() -> int:
    return int(sum(int(np.prod(s)) for _, s in gpt2_small_shapes()))


WORKLOADS = {
    "tiny_adam": Workload("tiny_adam", 10_007, 2, FP32, 5, 1e-2, 0.9, 0.999, 1e-8, 0.0,
                          "uniform1", 0.0, 1.0),
    "fp32_25m": Workload("fp32_25m", 25_000_000, 4, FP32, 10, 3e-4, 0.9, 0.95, 1e-8, 0.01,
                         "normal", 0.02, 1e-3, zero_frac=0.01),
    "gpt2_small": Workload("gpt2_small", gpt2_small_numel(), 8, BF16_MIXED, 10, 6e-4, 0.9,
                           0.999, 1e-8, 0.1, "normal", 0.02, 1e-3),
    "fp32_320m": Workload("fp32_320m", 320_000_000, 4, FP32, 5, 1e-4, 0.9, 0.999, 1e-8, 0.01,
                          "normal", 0.02, 1e-3),
    "mixed_1p3b": Workload("mixed_1p3b", 1_300_000_000, 8, BF16_MIXED, 3, 1e-4, 0.9, 0.999,
                           1e-8, 0.1, "normal", 0.02, 1e-3, bucket_bytes=25 * 1024 * 1024),
}


# ---------------------------------------------------------------------------
# tiny_adam: the exact numpy draw sequence
# ---------------------------------------------------------------------------

def tiny_adam_numpy(n: int = 10_007, N: int = 2, steps: int = 5, seed: int = 0):
    """params U(-1,1) (n draws), then for t=1..steps and rank 0..N-1 a N(0,1)
    gradient, all from one ``default_rng(seed)`` stream, cast to float32."""
    rng = np.random.default_rng(seed)
    params = rng.uniform(-1.0, 1.0, n).astype(np.float32)
    grads = [[rng.standard_normal(n).astype(np.float32) for _ in range(N)]
             for _ in range(steps)]
    return params, grads


# ---------------------------------------------------------------------------
# General generators (torch; on any device)
# ---------------------------------------------------------------------------

def _seed_of(*parts: int) -> int:
    """Deterministic 63-bit seed from a tuple of small integers (SplitMix64 mix)."""
    x = 0x9E3779B97F4A7C15
    mask = (1 << 64) - 1
    for p in parts:
        x = (x + (int(p) & mask) + 0x9E3779B97F4A7C15) & mask
        z = x
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & mask
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & mask
        x = z ^ (z >> 31)
    return x & ((1 << 63) - 1)


def _gen(device, *parts):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(_seed_of(*parts))
    return g


def init_params_fp32(n: int, wl: Workload, seed: int = 0, device="cpu"):
    """fp32 initial weights (also the fp32 master in mixed precision)."""
    import torch
    g = _gen(device, seed, 0xA11CE)
    out = torch.empty(n, dtype=torch.float32, device=device)
    if n == 0:
        return out
    if wl.param_init == "uniform1":
        out.uniform_(-1.0, 1.0, generator=g)
    else:
        out.normal_(0.0, wl.param_std, generator=g)
    return out


def fill_grads(grads, wl: Workload, step: int, seed: int = 0, lo: int = 0, hi: int | None = None):
    """Overwrite grads[r][lo:hi] with fresh draws for ``step`` (in place).

    Draws in fp32 then casts to the gradient storage type. With ``zero_frac``
    the same seeded mask is zeroed in every rank's gradient.
    """
    import torch
    if not grads:
        return
    device = grads[0].device
    n = grads[0].numel()
    hi = n if hi is None else hi
    if hi <= lo:
        return
    m = hi - lo
    mask = None
    if wl.zero_frac > 0:
        u = torch.empty(m, dtype=torch.float32, device=device)
        u.uniform_(0.0, 1.0, generator=_gen(device, seed, step, 0x2E80, lo))
        mask = u < wl.zero_frac
    tmp = torch.empty(m, dtype=torch.float32, device=device)
    for r, g in enumerate(grads):
        tmp.normal_(0.0, wl.grad_std, generator=_gen(device, seed, step, r, lo))
        if mask is not None:
            tmp.masked_fill_(mask, 0.0)
        g[lo:hi].copy_(tmp)


def make_replicas(init_fp32, N: int, precision: int):
    """N identical parameter replicas (fp32 copies, or RNE bf16 of the fp32 init)."""
    import torch
    dt = torch.bfloat16 if precision == BF16_MIXED else torch.float32
    base = init_fp32.to(dt)
    return [base.clone() for _ in range(N)]


def make_grads(n: int, N: int, precision: int, device="cpu"):
    import torch
    dt = torch.bfloat16 if precision == BF16_MIXED else torch.float32
    return [torch.empty(n, dtype=dt, device=device) for _ in range(N)]


def to_numpy_storage(t):
    """Host copy of a tensor in storage form: float32 array, or bf16 bits as uint16."""
    import torch
    t = t.detach().to("cpu")
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    return t.numpy().copy()
