"""w4a16_linear_noalloc: the allocation-free decode entry point, called
through the C ABI.

It exists for callers that cannot allocate device memory (an allocator or
memory-pool callback, a plugin host that passes only input and output
buffers, a runtime that forbids allocation while it captures work): its
scratch is a fixed array inside the library instead of a workspace. The test
calls it twice in a row on different problems and checks each result: the
same bits as the regular entry point, w4a16_linear, and within the layer's
error bound |y - y_ref| <= 2^-9 |y_ref| + 1e-4 sum_k |x W^| of the oracle's
exact result. It runs alone or after the other tests (the shared array keeps
earlier calls' contents).
"""
import ctypes

import numpy as np
import pytest

import oracle
import workloads
from helpers import assert_within_bound, to_dev

pytestmark = pytest.mark.gpu


def _noalloc(w4, x, qw, s, g, out, stream):
    M, K = x.shape
    N = qw.shape[0]
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    return w4.lib().w4a16_linear_noalloc(p(x), p(qw), p(s), p(out), M, N, K, g, stream)


def test_noalloc_matches_linear_on_two_calls_in_a_row(cuda_device):
    import torch

    import w4a16_group_quantized_linear_gb300 as w4

    r = workloads.rng(77)
    problems = []
    for M, N, K, g in [(4, 5000, 2048, 128), (1, 17408, 5120, 128)]:
        qw, s = workloads.raw_packed(r, N, K, g)
        x = workloads.activations(r, M, K)
        problems.append((x, qw, s, g))
    dev = [(to_dev(x, cuda_device), to_dev(qw, cuda_device), to_dev(s, cuda_device), g) for x, qw, s, g in problems]
    stream = ctypes.c_void_p(torch.cuda.current_stream(cuda_device).cuda_stream)

    outs = [torch.full((x.shape[0], qw.shape[0]), float("nan"), dtype=torch.float16, device=cuda_device)
            for x, qw, _, _ in dev]
    for (x, qw, s, g), out in zip(dev, outs):  # two calls in a row, one synchronize
        assert _noalloc(w4, x, qw, s, g, out, stream) == 0
    torch.cuda.synchronize()
    assert w4.device_status(raise_on_error=False) == 0

    for (x, qw, s, g), (xh, qh, sh, _), out in zip(dev, problems, outs):
        y = out.cpu().numpy()
        # the same deterministic GEMV as the regular entry point: the same bits
        y_lin = w4.linear(x, qw, s, g).cpu().numpy()
        assert np.array_equal(y.view(np.uint16), y_lin.view(np.uint16))
        # and within the layer's bound of the oracle's exact result
        y_ref, absdot = oracle.linear(xh, qh, sh, g, threads=8)
        assert_within_bound(y, y_ref, absdot, f"noalloc M={xh.shape[0]} N={qh.shape[0]}")


def test_noalloc_rejects_problems_beyond_its_scratch(cuda_device):
    import w4a16_group_quantized_linear_gb300 as w4

    # arrival counters for N = 2^28 rows need 64 MiB, more than the fixed array
    lib = w4.lib()
    p = ctypes.c_void_p(1 << 20)
    assert lib.w4a16_workspace_bytes(1, 1 << 28, 128, 128, 1) > (8 << 20)
    assert lib.w4a16_linear_noalloc(p, p, p, p, 1, 1 << 28, 128, 128, None) == 7


def test_noalloc_rejects_invalid_arguments_before_touching_its_scratch(cuda_device):
    """Argument errors come back unchanged (as from w4a16_linear), with no work
    enqueued on the shared array."""
    import w4a16_group_quantized_linear_gb300 as w4

    lib = w4.lib()
    p, q = ctypes.c_void_p(1 << 20), ctypes.c_void_p((1 << 20) + 8)
    assert lib.w4a16_linear_noalloc(None, p, p, p, 1, 256, 1024, 128, None) == 1   # null x
    assert lib.w4a16_linear_noalloc(q, p, p, p, 1, 256, 1024, 128, None) == 3      # misaligned x
    assert lib.w4a16_linear_noalloc(p, p, p, p, 1, 256, 1000, 128, None) == 1      # K % group
    assert lib.w4a16_linear_noalloc(p, p, p, p, 1, 256, 1024, 48, None) == 2       # group
    # a bad stream handle never reaches the device: the argument error wins
    assert lib.w4a16_linear_noalloc(q, p, p, p, 1, 256, 1024, 128, ctypes.c_void_p(8)) == 3
