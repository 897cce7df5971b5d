"""The C-ABI library without a GPU: it loads, exports every declared symbol, and
its host-side logic (shard plan, memory accounting, bucket plan, argument
checks) agrees exactly with the oracle. No call here launches device work."""

import ctypes
import os
import re

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    src = open(os.path.join(ROOT, "include", "zero_gb300.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_boundary():
    names = header_functions()
    for required in ["zero_shard_bounds", "zero_init_states", "zero_step", "ddp_allreduce_mean",
                     "zero_memory_bytes", "zero_step_bucketed", "zero_strerror"]:
        assert required in names


def test_library_exports_every_declared_symbol(abi):
    lib = ctypes.CDLL(abi.LIB_PATH)
    names = header_functions()
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    assert sorted(names) == abi.declared_symbols()


def test_shard_bounds_bit_exact(abi):
    for n in list(range(0, 70)) + [10_007, 25_000_000, 124_439_808, 1_300_000_000, 2**40 + 3]:
        for N in (1, 2, 3, 4, 5, 7, 8, 13, 64):
            assert abi.zero_shard_bounds(n, N) == oracle.shard_bounds(n, N), (n, N)
    for n in range(0, 120):
        for N in range(1, 12):
            sizes = np.diff(abi.zero_shard_bounds(n, N)).tolist()
            assert sizes == [len(p) for p in np.array_split(np.arange(n), N)]


def test_memory_accounting_bit_exact(abi):
    for prec in (abi.ZERO_FP32, abi.ZERO_BF16_MIXED, abi.ZERO_FP64_EMU):
        for n in (0, 1, 10, 44, 10_007, 124_439_808, 8_000_000_000, 175_000_000_000):
            for N in (1, 2, 3, 4, 8, 64):
                for stage in range(4):
                    assert abi.zero_memory_bytes(n, N, stage, prec) == \
                        oracle.memory_bytes(n, N, stage, prec)
                    for rank in {0, N - 1, N // 2}:
                        assert abi.zero_memory_breakdown(n, N, stage, prec, rank) == \
                            oracle.memory_breakdown(n, N, stage, prec, rank)


def test_bucket_plan_bit_exact(abi):
    for n, prec, bb in [(1_300_000_000, abi.ZERO_BF16_MIXED, 25 * 2**20),
                        (25_000_000, abi.ZERO_FP32, 25 * 2**20), (10, abi.ZERO_FP32, 12),
                        (0, abi.ZERO_FP32, 64), (7, abi.ZERO_BF16_MIXED, 2)]:
        es = 2 if prec == abi.ZERO_BF16_MIXED else 4
        ref = oracle.bucket_bounds(n, es, bb)
        assert abi.zero_bucket_count(n, prec, bb) == len(ref)
        assert [abi.zero_bucket_range(n, prec, bb, k) for k in range(len(ref))] == ref


def test_error_codes(abi):
    E = abi.ZeroError
    with pytest.raises(E) as e:
        abi.zero_shard_bounds(5, 0)
    assert e.value.code == abi.ZERO_EINVAL
    with pytest.raises(E):
        abi.zero_shard_bounds(-1, 2)
    for args in [(10, 0, 1, 0), (10, 4, 4, 0), (10, 4, -1, 0), (-1, 4, 1, 0), (10, 4, 1, 7)]:
        with pytest.raises(E) as e:
            abi.zero_memory_bytes(*args)
        assert e.value.code == abi.ZERO_EINVAL
    with pytest.raises(E):
        abi.zero_memory_breakdown(10, 4, 1, abi.ZERO_FP32, 4)
    with pytest.raises(E):
        abi.zero_memory_bytes(2**62, 1, 0, abi.ZERO_FP32)          # overflows 64 bits
    with pytest.raises(E):
        abi.zero_bucket_count(10, abi.ZERO_FP32, 3)               # holds no element
    with pytest.raises(E):
        abi.zero_bucket_range(10, abi.ZERO_FP32, 12, 4)
    with pytest.raises(E):
        abi.zero_bucket_count(10, abi.ZERO_FP64_EMU, 64)
    for code in (0, -1, -2, -3, -4, -5, 7):
        assert isinstance(abi.zero_strerror(code), str)
    assert "timed out" in abi.zero_strerror(abi.ZERO_ETIMEDOUT)


def test_raw_argument_checks_before_any_device_work(abi):
    """Rejections that happen on the host, before the CUDA runtime is touched."""
    vp = ctypes.c_void_p
    h = vp()
    # bad rank count, bad precision, NULL buffers, fp32 with a master buffer
    assert abi.raw_call("zero_init_states", 10, 0, 0, 16, 32, None, None, None, ctypes.byref(h)) \
        == abi.ZERO_EINVAL
    assert abi.raw_call("zero_init_states", 10, 65, 0, 16, 32, None, None, None,
                        ctypes.byref(h)) == abi.ZERO_EINVAL
    assert abi.raw_call("zero_init_states", 10, 2, 2, 16, 32, None, None, None, ctypes.byref(h)) \
        == abi.ZERO_EINVAL
    assert abi.raw_call("zero_init_states", 10, 2, 0, None, 32, None, None, None,
                        ctypes.byref(h)) == abi.ZERO_EINVAL
    assert abi.raw_call("zero_init_states", 10, 2, 0, 16, 32, 64, None, None, ctypes.byref(h)) \
        == abi.ZERO_EINVAL
    assert abi.raw_call("zero_init_states", 10, 2, 1, 16, 32, None, None, None,
                        ctypes.byref(h)) == abi.ZERO_EINVAL
    assert abi.raw_call("zero_init_states", -1, 2, 0, 16, 32, None, None, None,
                        ctypes.byref(h)) == abi.ZERO_EINVAL
    assert abi.raw_call("zero_init_states", 10, 2, 0, 18, 32, None, None, None,
                        ctypes.byref(h)) == abi.ZERO_EALIGN
    assert abi.raw_call("zero_init_states", 10, 2, 0, 16, 32, None, None, None, None) \
        == abi.ZERO_EINVAL
    # a NULL state handle
    arr = (vp * 2)(16, 32)
    assert abi.raw_call("zero_step", arr, arr, None, 1, 1e-3, 0.9, 0.999, 1e-8, 0.0, None) \
        == abi.ZERO_EINVAL
    # ddp: bad N, bad precision, overlapping buffers, misaligned bf16 pointer
    assert abi.raw_call("ddp_allreduce_mean", arr, 10, 0, 0, None) == abi.ZERO_EINVAL
    assert abi.raw_call("ddp_allreduce_mean", arr, 10, 2, 2, None) == abi.ZERO_EINVAL
    same = (vp * 2)(4096, 4096 + 8)
    assert abi.raw_call("ddp_allreduce_mean", same, 10, 2, 0, None) == abi.ZERO_EINVAL
    odd = (vp * 2)(4097, 8192)
    assert abi.raw_call("ddp_allreduce_mean", odd, 10, 2, 1, None) == abi.ZERO_EALIGN
    assert "aligned" in abi.zero_last_error()
    assert abi.raw_call("zero_free_states", None) == abi.ZERO_OK


def test_tensor_shard_bounds_bit_exact(abi):
    rng = np.random.default_rng(91)
    for T, N in [(291, 4), (148, 8), (5, 8), (1, 1), (0, 3), (37, 5)]:
        numels = rng.integers(0, 10_000, T).tolist()
        ref = oracle.tensor_shard_bounds(numels, N)
        assert abi.zero_tensor_shard_bounds(numels, N) == ref
        n = ref[-1]
        for stage in range(4):
            for prec in (abi.ZERO_FP32, abi.ZERO_BF16_MIXED, abi.ZERO_FP64_EMU):
                for rank in range(N):
                    assert abi.zero_memory_breakdown_ex(n, N, stage, prec, rank, ref) == \
                        oracle.memory_breakdown(n, N, stage, prec, rank, bounds=ref)
    with pytest.raises(abi.ZeroError):
        abi.zero_tensor_shard_bounds([3, -1], 2)
    with pytest.raises(abi.ZeroError):
        abi.zero_memory_breakdown_ex(10, 2, 1, abi.ZERO_FP32, 0, [0, 11, 10])


def test_init_states_rejects_bad_bounds_before_device_work(abi):
    vp = ctypes.c_void_p
    h = vp()
    for bad in ([1, 5, 10], [0, 5, 9], [0, 6, 5, 10]):
        arr = (ctypes.c_int64 * len(bad))(*bad)
        N = len(bad) - 1
        code = abi.raw_call("zero_init_states_ex", 10, N, 0, 4096, 8192, None, None, arr, None,
                            ctypes.byref(h))
        assert code == abi.ZERO_EINVAL
        assert "bounds" in abi.zero_last_error()


def test_option_structs_match_the_header(abi, tmp_path):
    """The ctypes mirrors of zero_step_opts_t and zero_sgd_opts_t have the C
    layout (size and every field offset), checked by compiling the header."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    structs = {"zero_step_opts_t": abi.StepOpts, "zero_sgd_opts_t": abi.SgdOpts}
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "zero_gb300.h"',
             "int main(void) {"]
    for cname, py in structs.items():
        lines.append(f'  printf("{cname} size %zu\\n", sizeof({cname}));')
        for field, _ in py._fields_:
            lines.append(f'  printf("{cname} {field} %zu\\n", offsetof({cname}, {field}));')
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    seen = {}
    for line in out.splitlines():
        cname, field, value = line.split()
        seen[(cname, field)] = int(value)
    for cname, py in structs.items():
        assert seen[(cname, "size")] == ctypes.sizeof(py), cname
        for field, _ in py._fields_:
            assert seen[(cname, field)] == getattr(py, field).offset, (cname, field)


def test_sgd_and_gather_argument_checks(abi):
    vp = ctypes.c_void_p
    arr = (vp * 2)(16, 32)
    o = abi.SgdOpts(1, 0.1, 0.9, 0.0, 0.0, 0, 1.0, 0.0, None, 0, -1, 0)
    assert abi.raw_call("zero_step_sgd", arr, arr, None, ctypes.byref(o), None) == abi.ZERO_EINVAL
    assert abi.raw_call("zero_gather", arr, None, 0, -1, None) == abi.ZERO_EINVAL
    # a host-only state (n = 0 needs no device work) to reach the option checks
    h = vp()
    assert abi.raw_call("zero_init_states", 0, 2, 0, None, None, None, None, None,
                        ctypes.byref(h)) == abi.ZERO_OK
    bad = [abi.SgdOpts(0, 0.1, 0.9, 0.0, 0.0, 0, 1.0, 0.0, None, 0, -1, 0),     # t = 0
           abi.SgdOpts(1, -0.1, 0.9, 0.0, 0.0, 0, 1.0, 0.0, None, 0, -1, 0),    # lr < 0
           abi.SgdOpts(1, 0.1, -0.9, 0.0, 0.0, 0, 1.0, 0.0, None, 0, -1, 0),    # mu < 0
           abi.SgdOpts(1, 0.1, 0.9, 0.1, 0.0, 1, 1.0, 0.0, None, 0, -1, 0),     # nesterov+damp
           abi.SgdOpts(1, 0.1, 0.0, 0.0, 0.0, 1, 1.0, 0.0, None, 0, -1, 0),     # nesterov, mu 0
           abi.SgdOpts(1, 0.1, 0.9, 0.0, 0.0, 0, 0.0, 0.0, None, 0, -1, 0),     # grad_scale 0
           abi.SgdOpts(1, 0.1, 0.9, 0.0, 0.0, 0, 1.0, 1.0, None, 0, -1, 0)]     # clip, no norm
    empty = (vp * 2)(None, None)
    for o in bad:
        assert abi.raw_call("zero_step_sgd", empty, empty, h, ctypes.byref(o), None) \
            == abi.ZERO_EINVAL
    assert abi.raw_call("zero_gather", empty, h, 0, 1, None) == abi.ZERO_EINVAL  # hi > n
    assert abi.raw_call("zero_free_states", h) == abi.ZERO_OK


def test_host_input_step_option_checks(abi):
    """zero_step_from_host_ex takes exactly one option set and the whole vector,
    and clipping only with a norm_sq output and the caller's norm scratch; each
    refusal comes before any device work."""
    vp = ctypes.c_void_p
    h = vp()
    assert abi.raw_call("zero_init_states", 0, 2, 0, None, None, None, None, None,
                        ctypes.byref(h)) == abi.ZERO_OK
    empty = (vp * 2)(None, None)
    mib = 25 << 20
    ad = abi.StepOpts(1, 1e-3, 0.9, 0.999, 1e-8, 0.01, 1.0, 0.0, None, 0, -1, 0)
    sg = abi.SgdOpts(1, 0.1, 0.9, 0.0, 0.0, 0, 1.0, 0.0, None, 0, -1, 0)

    def call(adamw, sgd, handle=h, grads=empty):
        return abi.raw_call("zero_step_from_host_ex", empty, grads, empty, handle,
                            None if adamw is None else ctypes.byref(adamw),
                            None if sgd is None else ctypes.byref(sgd), None, mib,
                            None, None, None)

    assert call(ad, sg) == abi.ZERO_EINVAL                    # both option sets
    assert call(None, None) == abi.ZERO_EINVAL                # neither
    assert call(ad, None, handle=None) == abi.ZERO_EINVAL     # no state handle
    assert call(ad, None, grads=None) == abi.ZERO_EINVAL      # no host gradients
    bad_adamw = [abi.StepOpts(1, 1e-3, 0.9, 0.999, 1e-8, 0.01, 1.0, 0.0, None, 1, -1, 0),  # lo
                 abi.StepOpts(1, 1e-3, 0.9, 0.999, 1e-8, 0.01, 1.0, 0.0, None, 0, 5, 0),   # hi
                 abi.StepOpts(1, 1e-3, 0.9, 0.999, 1e-8, 0.01, 1.0, 1.0, None, 0, -1, 0),  # no norm
                 abi.StepOpts(0, 1e-3, 0.9, 0.999, 1e-8, 0.01, 1.0, 0.0, None, 0, -1, 0),  # t = 0
                 abi.StepOpts(1, 1e-3, 1.0, 0.999, 1e-8, 0.01, 1.0, 0.0, None, 0, -1, 0),  # beta1
                 abi.StepOpts(1, 1e-3, 0.9, 0.999, 1e-8, 0.01, 0.0, 0.0, None, 0, -1, 0)]  # scale
    for o in bad_adamw:
        assert call(o, None) == abi.ZERO_EINVAL
    bad_sgd = [abi.SgdOpts(1, 0.1, 0.9, 0.0, 0.0, 0, 1.0, 0.0, None, 3, -1, 0),   # lo
               abi.SgdOpts(1, 0.1, 0.9, 0.0, 0.0, 0, 1.0, 2.0, None, 0, -1, 0),   # no norm
               abi.SgdOpts(1, 0.1, 0.9, 0.1, 0.0, 1, 1.0, 0.0, None, 0, -1, 0),   # nesterov+damp
               abi.SgdOpts(1, -0.1, 0.9, 0.0, 0.0, 0, 1.0, 0.0, None, 0, -1, 0)]  # lr < 0
    for o in bad_sgd:
        assert call(None, o) == abi.ZERO_EINVAL
    # clipping needs the caller's norm scratch as well as the norm_sq output
    no_scratch = abi.StepOpts(1, 1e-3, 0.9, 0.999, 1e-8, 0.01, 1.0, 1.0, 4096, 0, -1, 0)
    assert call(no_scratch, None) == abi.ZERO_EINVAL
    assert "norm_scratch" in abi.zero_last_error()
    # with both it is accepted (n = 0: nothing to queue)
    clip_ok = abi.StepOpts(1, 1e-3, 0.9, 0.999, 1e-8, 0.01, 1.0, 1.0, 4096, 0, -1, 0, 8192, 1)
    assert call(clip_ok, None) == abi.ZERO_OK
    # chunk size below one vector of elements is refused too
    assert abi.raw_call("zero_step_from_host_ex", empty, empty, empty, h, ctypes.byref(ad), None,
                        None, 0, None, None, None) == abi.ZERO_EINVAL
    assert abi.raw_call("zero_free_states", h) == abi.ZERO_OK


def test_ddp_mean_from_host_argument_checks(abi):
    """Every refusal of ddp_allreduce_mean_from_host comes before device work."""
    vp = ctypes.c_void_p
    host = (vp * 2)(16, 32)
    stg = (vp * 2)(64, 128)
    mib = 25 << 20

    def call(h, s, n, N, prec, chunk):
        return abi.raw_call("ddp_allreduce_mean_from_host", h, s, n, N, prec, None, chunk,
                            None, None, None)

    assert call(host, stg, -1, 2, abi.ZERO_FP32, mib) == abi.ZERO_EINVAL          # n < 0
    assert call(host, stg, 10, 0, abi.ZERO_FP32, mib) == abi.ZERO_EINVAL          # N = 0
    assert call(None, stg, 10, 2, abi.ZERO_FP32, mib) == abi.ZERO_EINVAL          # no host array
    assert call(host, None, 10, 2, abi.ZERO_FP32, mib) == abi.ZERO_EINVAL         # no staging
    assert call(host, stg, 10, 2, abi.ZERO_FP64_EMU, mib) == abi.ZERO_EINVAL      # precision
    assert call(host, stg, 10, 2, abi.ZERO_FP32, 3) == abi.ZERO_EINVAL            # chunk < 1 elem
    assert call((vp * 2)(16, None), stg, 10, 2, abi.ZERO_FP32, mib) == abi.ZERO_EINVAL
    assert call(host, (vp * 2)(64, 18), 10, 2, abi.ZERO_FP32, mib) == abi.ZERO_EALIGN
    assert call(host, (vp * 2)(64, 64), 10, 2, abi.ZERO_FP32, mib) == abi.ZERO_EINVAL  # same
    assert call(host, (vp * 2)(64, 96), 10, 2, abi.ZERO_FP32, mib) == abi.ZERO_EINVAL  # overlap


def test_ddp_host_handle_checks(abi):
    """The DDP host-input handle: create, reset and free; a NULL handle and
    the whole-vector argument checks are refused before any device work."""
    vp = ctypes.c_void_p
    h = vp()
    assert abi.raw_call("zero_ddp_host_create", ctypes.byref(h)) == abi.ZERO_OK
    assert h.value
    assert abi.raw_call("zero_ddp_host_create", None) == abi.ZERO_EINVAL
    assert abi.raw_call("zero_ddp_host_reset", h) == abi.ZERO_OK
    assert abi.raw_call("zero_ddp_host_reset", None) == abi.ZERO_EINVAL
    host = (vp * 2)(4096, 8192)
    staging = (vp * 2)(1 << 20, 1 << 21)
    same = (vp * 2)(1 << 20, 1 << 20)
    call = lambda hh, st, n=100, N=2, prec=0, chunk=1 << 20: abi.raw_call(  # noqa: E731
        "ddp_allreduce_mean_from_host_h", hh, host, st, n, N, prec, None, chunk, None, None, None)
    assert call(None, staging) == abi.ZERO_EINVAL            # no handle
    assert call(h, same) == abi.ZERO_EINVAL                  # the same staging buffer twice
    assert call(h, staging, N=0) == abi.ZERO_EINVAL          # no ranks
    assert call(h, staging, chunk=2) == abi.ZERO_EINVAL      # a chunk below one element
    assert call(h, staging, prec=2) == abi.ZERO_EINVAL       # not a gradient precision
    assert call(h, staging, n=0) == abi.ZERO_OK              # nothing to do
    assert abi.raw_call("zero_ddp_host_free", h) == abi.ZERO_OK
    assert abi.raw_call("zero_ddp_host_free", None) == abi.ZERO_OK


def test_injected_host_allocation_failures(abi):
    """A handle allocation that fails (injected, as if the host allocator
    returned NULL) reports ZERO_ENOMEM with a message, leaves the output NULL
    and queues nothing; the injection counts down, can be cleared, and stays
    in the thread that set it."""
    import threading
    vp = ctypes.c_void_p

    def init_states():
        h = vp(12345)
        rc = abi.raw_call("zero_init_states", 0, 2, abi.ZERO_FP32, None, None, None, None, None,
                          ctypes.byref(h))
        return rc, h

    def ddp_handle():
        h = vp(12345)
        return abi.raw_call("zero_ddp_host_create", ctypes.byref(h)), h

    abi.zero_debug_fail_host_allocs(2)
    rc, h = init_states()
    assert rc == abi.ZERO_ENOMEM and h.value is None
    assert "state handle" in abi.zero_last_error()
    rc, h = ddp_handle()
    assert rc == abi.ZERO_ENOMEM and h.value is None
    assert "DDP host-input handle" in abi.zero_last_error()
    rc, h = init_states()                      # the injection is used up
    assert rc == abi.ZERO_OK and h.value
    assert abi.raw_call("zero_free_states", h) == abi.ZERO_OK
    abi.zero_debug_fail_host_allocs(3)
    abi.zero_debug_fail_host_allocs(0)         # cleared
    rc, h = ddp_handle()
    assert rc == abi.ZERO_OK and h.value
    assert abi.raw_call("zero_ddp_host_free", h) == abi.ZERO_OK
    # another thread's injection leaves this thread's allocations alone
    seen = {}
    t = threading.Thread(target=lambda: (abi.zero_debug_fail_host_allocs(1),
                                         seen.update(other=init_states()[0])))
    t.start()
    t.join()
    assert seen["other"] == abi.ZERO_ENOMEM
    rc, h = init_states()
    assert rc == abi.ZERO_OK
    assert abi.raw_call("zero_free_states", h) == abi.ZERO_OK
    with pytest.raises(abi.ZeroError) as e:    # through the binding's handle class
        abi.zero_debug_fail_host_allocs(1)
        abi.DdpHost()
    assert e.value.code == abi.ZERO_ENOMEM
