"""zero_grad_norm_sq_noalloc: the squared gradient norm for callers that cannot
allocate device memory (a frozen memory pool, code that must not let
cudaMalloc synchronize the device, a hook that only borrows the gradients).

It uses the library's own fixed scratch array instead of a caller-provided
one, so it is checked against zero_grad_norm_sq on the same gradients, on two
calls in a row (the array keeps the previous call's partial sums; the second
call must not be affected by them). This file is collected last on purpose.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle


def _grads(rng, n, N, mixed, device):
    out = []
    for _ in range(N):
        g = torch.from_numpy(rng.normal(0, 1e-2, n).astype(np.float32)).to(device)
        out.append(g.to(torch.bfloat16) if mixed else g)
    return out


@pytest.mark.gpu
def test_noalloc_norm_matches_scratch_version_twice(abi, cuda):
    rng = np.random.default_rng(71)
    cases = [(3_000_017, 4, oracle.FP32), (1_000_003, 8, oracle.BF16_MIXED)]
    for n, N, prec in cases:                      # two calls in a row, different inputs
        grads = _grads(rng, n, N, prec == oracle.BF16_MIXED, cuda)
        count = abi.zero_grad_norm_scratch_count(n, prec)
        scratch = torch.empty(count, dtype=torch.float64, device=cuda)
        ref = torch.empty(1, dtype=torch.float64, device=cuda)
        got = torch.full((1,), -1.0, dtype=torch.float64, device=cuda)
        abi.zero_grad_norm_sq(grads, prec, scratch, ref, n)
        abi.zero_grad_norm_sq_noalloc(grads, prec, got, n)
        torch.cuda.synchronize()
        assert float(got.item()) == pytest.approx(float(ref.item()), rel=1e-9, abs=1e-300)


def test_noalloc_norm_rejects_sizes_beyond_its_scratch(abi):
    # rejected before any device work: the pointers are never dereferenced
    vp = ctypes.c_void_p
    grads = (vp * 2)(4096, 1 << 40)
    code = abi.raw_call("zero_grad_norm_sq_noalloc", grads, abi.ZERO_NOALLOC_MAX_N + 1, 2,
                        abi.ZERO_FP32, 8192, None)
    assert code == abi.ZERO_EINVAL
    assert "exceeds" in abi.raw_call.__globals__["_lib"].zero_last_error().decode()
