"""Prefill GEMM (M >= 17, tcgen05) on the GPU against the oracle, within
|y - y_ref| <= 2^-9 |y_ref| + 1e-4 sum_k |x W^| per element."""
import os

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


def _run(w4, dev, x, qw, s, g):
    out = w4.linear(to_dev(x, dev), to_dev(qw, dev), to_dev(s.view(np.float16), dev), g)
    w4.device_status()
    return out.cpu().numpy()


@pytest.mark.parametrize("M,N,K,g", [
    (17, 128, 128, 128),      # smallest GEMM M, one tile (32-token tiles up to M=32)
    (32, 384, 2048, 128),     # 32-token tile, full
    (33, 200, 512, 64),       # 64-token tiles from M=33, ragged N
    (64, 300, 1024, 32),      # 64-token tile, full, group 32
    (65, 130, 768, 128),      # first M on 128-token tiles, K % 256 != 0
    (128, 128, 64, 64),       # one chunk
    (200, 384, 512, 128),     # several tiles, ragged M
    (300, 257, 1024, 32),     # ragged N (one row past a tile), g32
    (129, 130, 96, 32),       # K % 64 == 32, ragged everything
    (256, 512, 2048, 64),
    (511, 200, 160, 32),      # K = 5 groups of 32
    (100, 200, 544, 32),      # 128-k stages from K = 512: a last stage of 32 k
    (300, 130, 800, 32),      # ... of 32 k, ragged N
    (97, 264, 576, 64),       # ... of 64 k, group 64
])
def test_gemm_raw_nibbles(w4, cuda_device, M, N, K, g):
    r = workloads.rng(M * 31 + N + K + g)
    qw, s = workloads.raw_packed(r, N, K, g)
    x = workloads.activations(r, M, K)
    y = _run(w4, cuda_device, x, qw, s, g)
    y_ref, a = oracle.linear(x, qw, s, g, threads=4)
    print(f"M={M} N={N} K={K} g={g} max err/bound", assert_within_bound(y, y_ref, a, "gemm"))


@pytest.mark.parametrize("g", [32, 128])
def test_gemm_minimum_K_is_one_group(w4, cuda_device, g):
    r = workloads.rng(40 + g)
    qw, s = workloads.raw_packed(r, 160, g, g)
    x = workloads.activations(r, 150, g)
    y = _run(w4, cuda_device, x, qw, s, g)
    y_ref, a = oracle.linear(x, qw, s, g)
    assert_within_bound(y, y_ref, a, "K=g")


def test_gemm_quantized_weights_with_outliers(w4, cuda_device):
    W, x, g = workloads.prefill(384, K=2048, N=640)
    qw, s = oracle.quantize(W, g)
    y = _run(w4, cuda_device, x, qw, s, g)
    y_ref, a = oracle.linear(x, qw, s, g, threads=4)
    print("prefill-like max err/bound", assert_within_bound(y, y_ref, a, "prefill"))


def test_gemm_zero_weights_and_one_hot(w4, cuda_device):
    r = workloads.rng(41)
    N, K, g = 256, 512, 64
    x = workloads.activations(r, 100, K)
    qw0 = np.full((N, K // 2), 0x88, np.uint8)
    _, s = workloads.raw_packed(r, N, K, g)
    assert np.all(_run(w4, cuda_device, x, qw0, s, g) == 0)
    qw, s = workloads.raw_packed(r, N, K, g)
    ks = list(range(0, K, 7))[:40]
    xo = np.zeros((len(ks), K), np.float16)
    for i, k in enumerate(ks):
        xo[i, k] = 1
    y = _run(w4, cuda_device, xo, qw, s, g)
    q = oracle.unpack(qw, K).astype(np.float64)
    sd = oracle.half_to_double(s.view(np.uint16))
    for i, k in enumerate(ks):
        assert np.array_equal(y[i], (sd[:, k // g] * q[:, k]).astype(np.float16))


def test_gemm_deterministic(w4, cuda_device):
    r = workloads.rng(42)
    qw, s = workloads.raw_packed(r, 640, 1024, 128)
    x = workloads.activations(r, 333, 1024)
    y1 = _run(w4, cuda_device, x, qw, s, 128)
    y2 = _run(w4, cuda_device, x, qw, s, 128)
    assert np.array_equal(y1.view(np.uint16), y2.view(np.uint16))


def test_prefill_m512_full_size_every_element(w4, cuda_device):
    """The full prefill workload at M = 512 (K=5120, N=17408, group 128, 1%
    outlier channels): every element against the oracle."""
    W, x, g = workloads.prefill(512)
    qw, s = oracle.quantize(W, g)
    y = _run(w4, cuda_device, x, qw, s, g)
    y_ref, a = oracle.linear(x, qw, s, g, threads=THREADS)
    print(f"prefill M=512 max err/bound (all elements) {assert_within_bound(y, y_ref, a, 'M=512'):.3f}")


def test_prefill_m4096_full_size_stratified(w4, cuda_device):
    """The full prefill workload at M = 4096: 256 random rows x all N columns,
    plus all rows x 256 random columns."""
    M = 4096
    W, x, g = workloads.prefill(M)
    qw, s = oracle.quantize(W, g)
    y = _run(w4, cuda_device, x, qw, s, g)
    r = workloads.rng(43)
    rows = np.sort(r.choice(M, 256, replace=False))
    cols = np.sort(r.choice(W.shape[0], 256, replace=False))
    y_r, a_r = oracle.linear(x[rows], qw, s, g, threads=THREADS)
    w1 = assert_within_bound(y[rows], y_r, a_r, "rows")
    y_c, a_c = oracle.linear(x, qw[cols], s[cols], g, threads=THREADS)
    w2 = assert_within_bound(y[:, cols], y_c, a_c, "cols")
    print(f"prefill M={M} max err/bound rows {w1:.3f} cols {w2:.3f}")
