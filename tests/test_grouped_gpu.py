"""Routed-expert grouped GEMM on the GPU against the oracle."""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

import oracle
import workloads
from helpers import assert_within_bound, to_dev

pytestmark = pytest.mark.gpu

THREADS = max(1, os.cpu_count() or 1)


@pytest.fixture(scope="module")
def w4(cuda_device):
    import w4a16_group_quantized_linear_gb300 as m

    m.lib()
    return m


def _run(w4, dev, x, qw, s, off, g):
    out = w4.grouped_linear(to_dev(x, dev), to_dev(qw, dev), to_dev(s.view(np.float16), dev), to_dev(off, dev), g)
    w4.device_status()
    return out.cpu().numpy()


def _experts(r, E, N, K, g):
    qw = r.integers(0, 256, (E, N, K // 2), dtype=np.uint8)
    s = (np.abs(r.normal(0, 0.02, (E, N, K // g))) / 7).astype(np.float16)
    return qw, s


@pytest.mark.parametrize("counts,N,K,g", [
    ([3, 0, 130, 1, 0, 260, 128], 256, 256, 32),  # empty experts, tails of 1..127
    ([0, 0, 0, 5], 128, 128, 64),
    ([700], 300, 512, 128),                         # E = 1
    ([1] * 40, 200, 96, 32),                        # many single-row experts, K % 64 = 32
])
def test_grouped_segments(w4, cuda_device, counts, N, K, g):
    r = workloads.rng(sum(counts) + N + K)
    E = len(counts)
    qw, s = _experts(r, E, N, K, g)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    x = workloads.activations(r, int(off[-1]), K)
    y = _run(w4, cuda_device, x, qw, s, off, g)
    y_ref, a = oracle.grouped_linear(x, qw, s, off, g)
    assert_within_bound(y, y_ref, a, f"grouped {counts}")


def test_grouped_E1_equals_dense(w4, cuda_device):
    r = workloads.rng(50)
    qw, s = _experts(r, 1, 256, 512, 32)
    x = workloads.activations(r, 300, 512)
    off = np.array([0, 300], np.int32)
    yg = _run(w4, cuda_device, x, qw, s, off, 32)
    yd = w4.linear(to_dev(x, cuda_device), to_dev(qw[0], cuda_device), to_dev(s[0], cuda_device), 32).cpu().numpy()
    assert np.array_equal(yg.view(np.uint16), yd.view(np.uint16))


@pytest.mark.parametrize("K,N", [(2048, 512), (512, 2048)])
def test_moe_full_size_every_row(w4, cuda_device, K, N):
    """E=128 experts, 4096 tokens, top-8 uniform routing (R = 32768 rows),
    group 32; weights quantized by the oracle; every row and column checked
    (the experts run in parallel on the host, each through the dense oracle)."""
    W, x, rt = workloads.moe(K, N)
    E = W.shape[0]
    qw = np.empty((E, N, K // 2), np.uint8)
    s = np.empty((E, N, K // 32), np.uint16)
    for e in range(E):
        qw[e], s[e] = oracle.quantize(W[e], 32)
    y = _run(w4, cuda_device, x, qw, s, rt.offsets, 32)

    def one(e):
        r0, r1 = int(rt.offsets[e]), int(rt.offsets[e + 1])
        if r1 == r0:
            return 0.0
        y_ref, a = oracle.linear(x[r0:r1], qw[e], s[e], 32)
        return assert_within_bound(y[r0:r1], y_ref, a, f"expert {e}")

    with ThreadPoolExecutor(THREADS) as ex:
        worst = max(ex.map(one, range(E)))
    print(f"moe K={K} N={N} max err/bound (all {x.shape[0]} rows) {worst:.3f}")


def test_bad_offsets_reported_not_faulted(w4, cuda_device):
    r = workloads.rng(52)
    qw, s = _experts(r, 3, 128, 128, 32)
    x = workloads.activations(r, 64, 128)
    import w4a16_group_quantized_linear_gb300 as m
    for off in ([0, 40, 20, 64], [0, 10, 20, 63], [5, 10, 20, 64]):
        m.grouped_linear(to_dev(x, cuda_device), to_dev(qw, cuda_device), to_dev(s, cuda_device),
                         to_dev(np.array(off, np.int32), cuda_device), 32)
        assert m.device_status(raise_on_error=False) == 6
    assert m.device_status(raise_on_error=False) == 0
