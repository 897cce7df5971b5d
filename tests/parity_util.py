"""Comparison helpers for the GPU-vs-oracle parity tests.

Tolerances (written here once, used by every parity test):
  * fp32 parameters, m, v, master: |gpu - oracle| <= 1e-6 + 1e-5 * |oracle|
    against the fp32-mirror oracle;
  * bf16 replicas: within one bf16 ulp of the round-to-nearest-even of the
    oracle's fp32 master;
  * shard bounds, memory bytes, bucket plans: bit-exact (checked elsewhere).
"""

import numpy as np

import oracle

ABS_TOL = 1e-6
REL_TOL = 1e-5


def assert_fp32_close(got, ref, what=""):
    got = np.asarray(got, np.float32).astype(np.float64)
    ref = np.asarray(ref, np.float32).astype(np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    both_nan = np.isnan(got) & np.isnan(ref)
    bad = ~both_nan & ~(np.abs(got - ref) <= ABS_TOL + REL_TOL * np.abs(ref))
    if bad.any():
        i = int(np.flatnonzero(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())} of {got.size} outside tolerance; "
                             f"first at {i}: gpu={got[i]!r} oracle={ref[i]!r}")


def bf16_ulp(x):
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    a = np.abs(np.asarray(x, np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.exp2(e - 7)


def assert_bf16_within_one_ulp(got_bits, ref_master_fp32, what=""):
    ref_bits = oracle.f32_to_bf16_rne(np.asarray(ref_master_fp32, np.float32))
    got = oracle.bf16_to_f32(got_bits).astype(np.float64)
    ref = oracle.bf16_to_f32(ref_bits).astype(np.float64)
    bad = ~(np.abs(got - ref) <= bf16_ulp(np.maximum(np.abs(got), np.abs(ref))))
    if bad.any():
        i = int(np.flatnonzero(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())} bf16 values beyond 1 ulp; first at {i}: "
                             f"gpu={got[i]!r} oracle RNE={ref[i]!r}")


def exact_fraction(got, ref):
    got = np.asarray(got)
    ref = np.asarray(ref)
    if got.size == 0:
        return 1.0
    return float(np.mean(got.view(np.uint32 if got.dtype == np.float32 else got.dtype) ==
                         ref.view(np.uint32 if ref.dtype == np.float32 else ref.dtype)))


def assert_same_bits_or_both_nan(got, ref, what=""):
    """Bitwise equal, except that a NaN matches any NaN (the GPU returns one
    canonical NaN where numpy keeps an operand's payload). float32 arrays, or
    bf16 bits as uint16."""
    got, ref = np.asarray(got), np.asarray(ref)
    assert got.shape == ref.shape, what
    if got.dtype == np.uint16:
        gn, rn = (got & 0x7FFF) > 0x7F80, (ref & 0x7FFF) > 0x7F80
        gb, rb = got, ref
    else:
        gn, rn = np.isnan(got), np.isnan(ref)
        gb, rb = got.view(np.uint32), ref.view(np.uint32)
    assert np.array_equal(gn, rn), f"{what}: NaN positions differ ({int((gn != rn).sum())})"
    bad = np.flatnonzero(gb[~gn] != rb[~rn])
    assert bad.size == 0, f"{what}: {bad.size} values differ"


def flat(states, key):
    return np.concatenate([s[key] for s in states]) if states else np.zeros(0, np.float32)


# ---------------------------------------------------------------------------
# Guard regions. compute-sanitizer is not available on the GPU pool, so every
# device buffer of the small parity tests sits inside a larger allocation whose
# other elements hold a sentinel bit pattern (a NaN in both float formats, so a
# kernel that read it as data would also show). A kernel that writes past
# either end of its range -- a vector store rounded up to 16 bytes, a unit past
# `hi`, a head written before a non-zero offset -- changes a sentinel, and
# check_guards() reports it. Buffers register themselves; the conftest checks
# and forgets them after every test.
# ---------------------------------------------------------------------------

GUARD = 4096          # sentinel elements on each side of a buffer (two full tiles)
_SENTINEL_BITS = {4: 0x7FA5A5A5, 2: 0x7FA5, 8: 0x7FF5A5A5A5A5A5A5}
_guarded = []


def _bits_dtype(elem_size):
    import torch
    return {4: torch.int32, 2: torch.int16, 8: torch.int64}[elem_size]


def guarded_empty(n, dtype, device, offset=0, what="buffer"):
    """A device view of n elements, ``GUARD + offset`` elements into an
    allocation of ``n + 2*GUARD + offset`` whose elements outside the view
    hold the sentinel. The view's own elements hold the sentinel too until
    written."""
    import torch
    es = torch.empty(0, dtype=dtype).element_size()
    buf = torch.empty(n + 2 * GUARD + offset, dtype=dtype, device=device)
    buf.view(_bits_dtype(es)).fill_(_SENTINEL_BITS[es])
    lo = GUARD + offset
    _guarded.append((buf, lo, lo + n, what))
    return buf[lo:lo + n]


def check_guards():
    """Every registered buffer's elements outside its view still hold the
    sentinel, bit for bit."""
    for buf, lo, hi, what in _guarded:
        es = buf.element_size()
        bits = buf.view(_bits_dtype(es))
        s = _SENTINEL_BITS[es]
        before = int((bits[:lo] != s).sum())
        after = int((bits[hi:] != s).sum())
        if before or after:
            raise AssertionError(f"{what}: {before} element(s) written before the buffer and "
                                 f"{after} after it (guard regions of {lo} and "
                                 f"{bits.numel() - hi} elements)")


def forget_guards():
    _guarded.clear()


def guard_count():
    return len(_guarded)
