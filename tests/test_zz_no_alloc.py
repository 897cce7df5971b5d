"""zero_grad_norm_sq_noalloc: the squared gradient norm for callers that cannot
allocate device memory (a frozen memory pool, code that must not let
cudaMalloc synchronize the device, a hook that only borrows the gradients).

It uses the library's own fixed scratch array instead of a caller-provided
one, so it is checked against zero_grad_norm_sq on the same gradients, bit for
bit as its header promises, on two calls in a row (the array keeps the
previous call's partial sums; the second call must not be affected by them),
and against the oracle's squared norm of the mean gradient. One case has more
than 100 million elements, so the array is used across thousands of partial
sums. This file is collected last on purpose.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle


def _grads(rng, n, N, mixed, device):
    """N gradients on the device and their host storage (float32, or bf16 bits)."""
    dev, host = [], []
    for _ in range(N):
        g = rng.normal(0, 1e-2, n).astype(np.float32)
        t = torch.from_numpy(g).to(device)
        if mixed:
            t = t.to(torch.bfloat16)
            host.append(t.cpu().view(torch.int16).numpy().view(np.uint16))
        else:
            host.append(g)
        dev.append(t)
    return dev, host


@pytest.mark.gpu
def test_noalloc_norm_matches_scratch_version_twice(abi, cuda):
    rng = np.random.default_rng(71)
    cases = [(3_000_017, 4, oracle.FP32), (1_000_003, 8, oracle.BF16_MIXED),
             (120_000_017, 2, oracle.FP32)]
    for n, N, prec in cases:                      # calls in a row, different inputs
        grads, host = _grads(rng, n, N, prec == oracle.BF16_MIXED, cuda)
        count = abi.zero_grad_norm_scratch_count(n, prec)
        assert n < 100_000_000 or count > 3000
        scratch = torch.empty(count, dtype=torch.float64, device=cuda)
        ref = torch.empty(1, dtype=torch.float64, device=cuda)
        got = torch.full((1,), -1.0, dtype=torch.float64, device=cuda)
        abi.zero_grad_norm_sq(grads, prec, scratch, ref, n)
        abi.zero_grad_norm_sq_noalloc(grads, prec, got, n)
        torch.cuda.synchronize()
        assert torch.equal(got, ref), (float(got.item()), float(ref.item()))
        want = oracle.grad_norm(host, precision=prec, mode="fp32") ** 2
        assert float(got.item()) == pytest.approx(want, rel=1e-9, abs=1e-300)
        del grads, host, scratch


def test_noalloc_norm_rejects_sizes_beyond_its_scratch(abi):
    # rejected before any device work: the pointers are never dereferenced
    vp = ctypes.c_void_p
    grads = (vp * 2)(4096, 1 << 40)
    code = abi.raw_call("zero_grad_norm_sq_noalloc", grads, abi.ZERO_NOALLOC_MAX_N + 1, 2,
                        abi.ZERO_FP32, 8192, None)
    assert code == abi.ZERO_EINVAL
    assert "exceeds" in abi.zero_last_error()
