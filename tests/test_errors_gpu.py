"""Failure paths of the bounded waits, made to run out on purpose.

The test-hooks build of the library (libw4a16_testhooks.so: the same sources
compiled with -DW4A16_TEST_HOOKS) lets a test set the limit of every bounded
wait and stop the TMA producers after a given number of copies (in the
cluster GEMV: hold back the sums sent to a row-block's finisher). With a 1 ms
limit and a producer that stops early, the GEMV's and the GEMM's waits give
up; each kernel must record W4A16_ERR_TIMEOUT in the device status word,
unwind (drain the copies it issued, free its TMEM) and return promptly, and
the next normal call on the same stream must be correct. Nothing faults or
hangs: every wait is bounded, and a stopped producer simply issues no more
copies. Before the follow-up GEMM runs, the test checks the GEMM's counters of
TMEM allocations and frees, so a leaked allocation is reported instead of
blocking the next kernel's allocation.
"""
import ctypes
import time

import numpy as np
import pytest

import oracle
import workloads
from helpers import assert_within_bound, to_dev

pytestmark = pytest.mark.gpu

TIMEOUT = 5
SHORT_NS = 1_000_000            # 1 ms
NORMAL_NS = 2_000_000_000       # the production limit, 2 s


@pytest.fixture(scope="module")
def hooks(cuda_device):
    import w4a16_group_quantized_linear_gb300 as w4
    from w4a16_group_quantized_linear_gb300 import build

    lib = ctypes.CDLL(build.build(variant="testhooks"))
    for name, (res, args) in w4.EXPORTS.items():
        f = getattr(lib, name)
        f.restype, f.argtypes = res, args
    lib.w4a16_test_set_hooks.restype = ctypes.c_int32
    lib.w4a16_test_set_hooks.argtypes = [ctypes.c_uint64, ctypes.c_int32]
    lib.w4a16_test_tmem_counters.restype = ctypes.c_int32
    lib.w4a16_test_tmem_counters.argtypes = [ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(ctypes.c_uint64)]
    yield lib
    lib.w4a16_test_set_hooks(NORMAL_NS, -1)


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream(dev):
    import torch

    return ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)


def _tmem(lib):
    a, f = ctypes.c_uint64(0), ctypes.c_uint64(0)
    assert lib.w4a16_test_tmem_counters(ctypes.byref(a), ctypes.byref(f)) == 0
    return a.value, f.value


def _status_after(lib, st):
    """The device status word after the stream drains, and how long that took."""
    t0 = time.perf_counter()
    status = lib.w4a16_device_status(st)
    return status, time.perf_counter() - t0


def test_gemv_wait_times_out_and_next_call_is_correct(hooks, cuda_device):
    import torch

    lib = hooks
    # group 64 takes the TMA-ring kernel, whose waits are the bounded ones (the
    # group-128 cluster kernel waits on nothing but its own cluster's barrier);
    # about 9 units per compute warp: a stop after 2 copies stalls every warp
    M, N, K, g = 1, 17408, 5120, 64
    r = workloads.rng(90)
    qw, s = workloads.raw_packed(r, N, K, g)
    x = workloads.activations(r, M, K)
    xd, qd, sd = to_dev(x, cuda_device), to_dev(qw, cuda_device), to_dev(s, cuda_device)
    y = torch.empty((M, N), dtype=torch.float16, device=cuda_device)
    nb = lib.w4a16_workspace_bytes(M, N, K, g, 1)
    ws = torch.empty(nb, dtype=torch.uint8, device=cuda_device)
    st = _stream(cuda_device)
    for issue_limit in (0, 2):
        assert lib.w4a16_workspace_init(_p(ws), nb, st) == 0
        assert lib.w4a16_test_set_hooks(SHORT_NS, issue_limit) == 0
        assert lib.w4a16_linear(_p(xd), _p(qd), _p(sd), _p(y), M, N, K, g, _p(ws), nb, st) == 0
        status, dt = _status_after(lib, st)
        assert status == TIMEOUT, f"issue limit {issue_limit}: status {status}"
        assert dt < 1.0, f"issue limit {issue_limit}: the kernel took {dt:.3f} s to give up"
        assert lib.w4a16_device_status(st) == 0   # read and cleared
    # a timed-out call leaves its arrival counters set: re-initialise, then run normally
    assert lib.w4a16_test_set_hooks(NORMAL_NS, -1) == 0
    assert lib.w4a16_workspace_init(_p(ws), nb, st) == 0
    assert lib.w4a16_linear(_p(xd), _p(qd), _p(sd), _p(y), M, N, K, g, _p(ws), nb, st) == 0
    assert lib.w4a16_device_status(st) == 0
    y_ref, a = oracle.linear(x, qw, s, g, threads=8)
    assert_within_bound(y.cpu().numpy(), y_ref, a, "GEMV after a timeout")


@pytest.mark.parametrize("kind", ["one token", "four tokens", "gated"])
def test_cluster_gemv_mailbox_wait_times_out_and_next_call_is_correct(hooks, cuda_device, kind):
    """The cluster decode kernels' only wait is a row-block finisher's wait for
    the other contributors' sums; with the sums held back it gives up after the
    limit, records the timeout, stores nothing for those rows and leaves the
    device usable."""
    import torch

    lib = hooks
    M, N, K, g = (4 if kind == "four tokens" else 1), 17408, 5120, 128  # every row-block split over 2-3 warps
    r = workloads.rng(93 + M)
    qw, s = workloads.raw_packed(r, N, K, g)
    x = workloads.activations(r, M, K)
    xd, qd, sd = to_dev(x, cuda_device), to_dev(qw, cuda_device), to_dev(s, cuda_device)
    y = torch.empty((M, N), dtype=torch.float16, device=cuda_device)
    gated = kind == "gated"
    nb = lib.w4a16_workspace_bytes(M, N, K, g, 1) if not gated else lib.w4a16_linear_gated_workspace_bytes(M, N, K, g)
    ws = torch.empty(nb, dtype=torch.uint8, device=cuda_device)
    st = _stream(cuda_device)

    def call():
        if gated:
            return lib.w4a16_linear_gated(_p(xd), _p(qd), _p(sd), _p(qd), _p(sd), _p(y), M, N, K, g, _p(ws), nb, st)
        return lib.w4a16_linear(_p(xd), _p(qd), _p(sd), _p(y), M, N, K, g, _p(ws), nb, st)

    assert lib.w4a16_workspace_init(_p(ws), nb, st) == 0
    assert lib.w4a16_test_set_hooks(SHORT_NS, 0) == 0
    assert call() == 0
    status, dt = _status_after(lib, st)
    assert status == TIMEOUT, f"status {status}"
    assert dt < 1.0, f"the kernel took {dt:.3f} s to give up"
    assert lib.w4a16_device_status(st) == 0   # read and cleared
    assert lib.w4a16_test_set_hooks(NORMAL_NS, -1) == 0
    assert call() == 0
    assert lib.w4a16_device_status(st) == 0
    if gated:
        y_ref, gg, uu, ag, au = oracle.gated_linear(x, qw, s, qw, s, g, threads=8)
        err = np.abs(y.cpu().numpy().astype(np.float64) - y_ref)
        assert np.all(err <= oracle.gated_tolerance(gg, uu, ag, au)), "gated GEMV after a timeout"
    else:
        y_ref, a = oracle.linear(x, qw, s, g, threads=8)
        assert_within_bound(y.cpu().numpy(), y_ref, a, f"cluster GEMV ({kind}) after a timeout")


@pytest.mark.parametrize("kind", ["dense", "grouped", "gated"])
def test_gemm_wait_times_out_frees_tmem_and_next_call_is_correct(hooks, cuda_device, kind):
    import torch

    lib = hooks
    grouped = kind == "grouped"
    N, K, g = 512, 2048, 128 if not grouped else 32
    r = workloads.rng(91 + ["dense", "grouped", "gated"].index(kind))
    st = _stream(cuda_device)
    if kind == "gated":   # both weight matrices; the epilogue swaps the up sums through shared memory
        M = 256
        qw, s = workloads.raw_packed(r, N, K, g)
        qu, su = workloads.raw_packed(r, N, K, g)
        qud, sud = to_dev(qu, cuda_device), to_dev(su, cuda_device)
    elif grouped:
        counts = [100, 0, 200, 37]
        E = len(counts)
        qw = r.integers(0, 256, (E, N, K // 2), dtype=np.uint8)
        s = (np.abs(r.normal(0, 0.02, (E, N, K // g))) / 7).astype(np.float16)
        off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
        M = int(off[-1])
        offd = to_dev(off, cuda_device)
    else:
        M = 256
        qw, s = workloads.raw_packed(r, N, K, g)
    x = workloads.activations(r, M, K)
    xd, qd, sd = to_dev(x, cuda_device), to_dev(qw, cuda_device), to_dev(s, cuda_device)
    y = torch.empty((M, N), dtype=torch.float16, device=cuda_device)

    def call():
        if grouped:
            return lib.w4a16_grouped_linear(_p(xd), _p(qd), _p(sd), _p(offd), _p(y), E, M, N, K, g, None, 0, st)
        if kind == "gated":
            return lib.w4a16_linear_gated(_p(xd), _p(qd), _p(sd), _p(qud), _p(sud), _p(y), M, N, K, g, None, 0, st)
        return lib.w4a16_linear(_p(xd), _p(qd), _p(sd), _p(y), M, N, K, g, None, 0, st)

    for issue_limit in (0, 3, 9):   # no copy; the first stage only; about half of K
        a0, f0 = _tmem(lib)
        assert lib.w4a16_test_set_hooks(SHORT_NS, issue_limit) == 0
        assert call() == 0
        status, dt = _status_after(lib, st)
        assert status == TIMEOUT, f"issue limit {issue_limit}: status {status}"
        assert dt < 1.0, f"issue limit {issue_limit}: the kernel took {dt:.3f} s to give up"
        a1, f1 = _tmem(lib)
        assert a1 - a0 > 0 and a1 - a0 == f1 - f0, f"TMEM allocations {a1 - a0} != frees {f1 - f0}"
    assert lib.w4a16_test_set_hooks(NORMAL_NS, -1) == 0
    assert call() == 0
    assert lib.w4a16_device_status(st) == 0
    if grouped:
        y_ref, a = oracle.grouped_linear(x, qw, s, off, g)
    elif kind == "gated":
        y_ref, gg, uu, ag, au = oracle.gated_linear(x, qw, s, qu, su, g, threads=8)
        err = np.abs(y.cpu().numpy().astype(np.float64) - y_ref)
        assert np.all(err <= oracle.gated_tolerance(gg, uu, ag, au)), "gated GEMM after a timeout"
        return
    else:
        y_ref, a = oracle.linear(x, qw, s, g, threads=8)
    assert_within_bound(y.cpu().numpy(), y_ref, a, "GEMM after a timeout")
