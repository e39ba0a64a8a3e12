"""GGUF block formats (Q4_K, Q5_1) on the GPU against the oracle.

The dequantizer must match the oracle's fp32 decode bit for bit (the infr
README's check: on-device decode byte-identical to the CPU dequant). The GEMV
must stay within |y - y_ref| <= 2^-9 |y_ref| + 1e-4 sum_k |x| (|a q| + |b|)
of the fp64 oracle (W^ = a q + b), element by element."""
import ctypes

import numpy as np
import pytest

import oracle
import workloads
from helpers import assert_within_bound, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w4(cuda_device):
    import w4a16_group_quantized_linear_gb300 as m

    m.lib()
    return m


def _inputs(fmt, M, N, K, seed):
    g = workloads.rng(seed)
    w = workloads.raw_blocks(g, fmt, N, K)
    x = workloads.activations(g, M, K)
    return x, w


def _check(w4, dev, fmt, M, N, K, seed, threads=1):
    x, w = _inputs(fmt, M, N, K, seed)
    y = w4.blocks_linear(fmt, to_dev(x, dev), to_dev(w, dev)).cpu().numpy()
    y_ref, a = oracle.blocks_linear(fmt, x, w, threads=threads)
    return assert_within_bound(y, y_ref, a, f"{fmt} M={M} N={N} K={K}")


@pytest.mark.parametrize("fmt,N,K", [("q4_k", 37, 1024), ("q4_k", 300, 5120), ("q5_1", 37, 1056),
                                     ("q5_1", 64, 32), ("q5_1", 300, 5120)])
def test_dequant_bit_exact(w4, cuda_device, fmt, N, K):
    w = workloads.raw_blocks(workloads.rng(7), fmt, N, K)
    got = w4.blocks_dequant(fmt, to_dev(w, cuda_device), K).cpu().numpy()
    ref = oracle.blocks_decode_f32(fmt, w, K)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("fmt", ["q4_k", "q5_1"])
@pytest.mark.parametrize("M", [1, 2, 3, 8, 9, 17])
def test_small_shapes_all_M(w4, cuda_device, fmt, M):
    # 203 rows: full row-blocks and a ragged last one; 11 units of 256 k a row,
    # so the warps' runs of units cross row-block boundaries
    print(fmt, M, "max err/bound", _check(w4, cuda_device, fmt, M, 203, 2816, 10 + M))


@pytest.mark.parametrize("fmt,K", [("q4_k", 256), ("q5_1", 32), ("q5_1", 96), ("q5_1", 1056), ("q5_1", 2080)])
def test_short_and_ragged_k(w4, cuda_device, fmt, K):
    # one unit, or a last unit with fewer than eight Q5_1 blocks
    for M in (1, 5):
        print(fmt, K, M, "max err/bound", _check(w4, cuda_device, fmt, M, 77, K, K + M))


@pytest.mark.parametrize("fmt", ["q4_k", "q5_1"])
def test_cluster_split(w4, cuda_device, fmt):
    # few row-blocks of 32 units each: every row-block is shared by several warps
    # and blocks of a cluster
    for M in (1, 4):
        print(fmt, M, "max err/bound", _check(w4, cuda_device, fmt, M, 1000, 8192, 40 + M, threads=8))


@pytest.mark.parametrize("fmt", ["q4_k", "q5_1"])
@pytest.mark.parametrize("M", [1, 4])
@pytest.mark.parametrize("K,N", [(5120, 17408), (17408, 5120)])
def test_decode_full_size(w4, cuda_device, fmt, M, K, N):
    print(fmt, M, K, N, "max err/bound", _check(w4, cuda_device, fmt, M, N, K, 50 + M, threads=8))


@pytest.mark.parametrize("fmt", ["q4_k", "q5_1"])
def test_deterministic_and_pinned_host_output(w4, cuda_device, fmt):
    import torch

    x, w = _inputs(fmt, 3, 5120, 17408, 60)
    xd, wd = to_dev(x, cuda_device), to_dev(w, cuda_device)
    y1 = w4.blocks_linear(fmt, xd, wd)
    y2 = w4.blocks_linear(fmt, xd, wd)
    host = torch.empty((3, 5120), dtype=torch.float16).pin_memory()
    w4.blocks_linear(fmt, xd, wd, out=host)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)
    assert torch.equal(y1.cpu(), host)


def test_edge_cases_and_errors(w4, cuda_device):
    import torch

    lib = w4.lib()
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    st = ctypes.c_void_p(torch.cuda.current_stream(cuda_device).cuda_stream)
    x = torch.zeros((2, 512), dtype=torch.float16, device=cuda_device)
    w = torch.zeros((8, 288), dtype=torch.uint8, device=cuda_device)
    y = torch.full((2, 8), 7.0, dtype=torch.float16, device=cuda_device)
    Q4K, Q51 = w4.BLOCK_FORMATS["q4_k"], w4.BLOCK_FORMATS["q5_1"]
    # nothing to do
    assert lib.w4a16_blocks_linear(Q4K, P(x), P(w), P(y), 0, 8, 512, st) == 0
    assert lib.w4a16_blocks_linear(Q4K, P(x), P(w), P(y), 2, 0, 512, st) == 0
    torch.cuda.synchronize()
    assert bool((y == 7.0).all())
    # K = 0 writes zeros
    assert lib.w4a16_blocks_linear(Q4K, P(x), P(w), P(y), 2, 8, 0, st) == 0
    torch.cuda.synchronize()
    assert bool((y == 0.0).all())
    # all-zero blocks give zeros
    y.fill_(7.0)
    assert lib.w4a16_blocks_linear(Q4K, P(x), P(w), P(y), 2, 8, 512, st) == 0
    torch.cuda.synchronize()
    assert bool((y == 0.0).all())
    # unknown format, K not whole blocks, negative sizes, misaligned pointers
    assert lib.w4a16_blocks_linear(3, P(x), P(w), P(y), 2, 8, 512, st) == 2
    assert lib.w4a16_blocks_linear(Q4K, P(x), P(w), P(y), 2, 8, 300, st) == 1
    assert lib.w4a16_blocks_linear(Q51, P(x), P(w), P(y), 2, 8, 48, st) == 1
    assert lib.w4a16_blocks_linear(Q4K, P(x), P(w), P(y), -1, 8, 512, st) == 1
    assert lib.w4a16_blocks_linear(Q4K, ctypes.c_void_p(x.data_ptr() + 2), P(w), P(y), 1, 8, 256, st) == 3
    assert lib.w4a16_blocks_linear(Q4K, P(x), ctypes.c_void_p(w.data_ptr() + 8), P(y), 1, 4, 256, st) == 3
    out = torch.empty((8, 512), dtype=torch.float32, device=cuda_device)
    assert lib.w4a16_blocks_dequant(3, P(w), 8, 512, P(out), st) == 2
    assert lib.w4a16_blocks_dequant(Q4K, P(w), 8, 500, P(out), st) == 1
    assert lib.w4a16_blocks_dequant(Q4K, P(w), 0, 512, P(out), st) == 0
    assert lib.w4a16_blocks_row_bytes(Q4K, 512) == 288 and lib.w4a16_blocks_row_bytes(Q51, 64) == 48
    assert lib.w4a16_blocks_row_bytes(Q4K, 100) == -1 and lib.w4a16_blocks_row_bytes(9, 256) == -1
    assert w4.device_status() == 0


def test_many_rows_take_several_launches(w4, cuda_device):
    # 2500 row-blocks at 8 tokens: more than one launch's clusters may hold, so the
    # rows go in two launches
    print("q4_k M=8 N=40000 max err/bound", _check(w4, cuda_device, "q4_k", 8, 40000, 5120, 70, threads=8))
