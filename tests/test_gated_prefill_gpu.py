"""Fused gate + up projections with the SiLU * up epilogue on the tensor-core
GEMM (M > 16): y = silu(x Wg^T) * (x Wu^T) against the oracle, within the
bound that follows from the linear tolerance on g and u
(oracle.gated_tolerance). Each tile holds 64 rows of Wg and the same 64 rows
of Wu, so ragged N (not a multiple of 64) and every token-tile width (32, 64
and 128 tokens) appear below."""
import os

import numpy as np
import pytest

import oracle
import workloads
from helpers import to_dev

pytestmark = pytest.mark.gpu

THREADS = max(1, os.cpu_count() or 1)


@pytest.fixture(scope="module")
def w4(cuda_device):
    import w4a16_group_quantized_linear_gb300 as m

    m.lib()
    return m


def _run(w4, dev, x, qg, sg, qu, su, g):
    y = w4.linear_gated(to_dev(x, dev), to_dev(qg, dev), to_dev(sg.view(np.float16), dev), to_dev(qu, dev),
                        to_dev(su.view(np.float16), dev), g)
    w4.device_status()
    return y.cpu().numpy()


def _check(y, x, qg, sg, qu, su, g, what):
    y_ref, gg, uu, ag, au = oracle.gated_linear(x, qg, sg, qu, su, g, threads=THREADS)
    bound = oracle.gated_tolerance(gg, uu, ag, au)
    err = np.abs(y.astype(np.float64) - y_ref)
    assert np.all(np.isfinite(y)), what
    bad = err > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements out of bound, "
                           f"worst err/bound {np.max(err / np.maximum(bound, 1e-300))}")
    return float(np.max(err / np.maximum(bound, 1e-300)))


def _scaled(r, N, K, g, gain):
    qw, s = workloads.raw_packed(r, N, K, g)
    s = oracle.float_to_half_bits(np.float32(gain) * oracle.half_to_double(s).astype(np.float32))
    return qw, s


@pytest.mark.parametrize("M,N,K,g", [
    (17, 128, 128, 128),     # smallest GEMM M; 32-token tiles
    (17, 300, 512, 64),      # ragged N: the last tile has 44 of 64 outputs
    (32, 1000, 2080, 32),    # K % 256 != 0: a partial stage
    (33, 200, 512, 32),      # 64-token tiles from M = 33
    (64, 130, 768, 128),     # 64-token tile, full; two outputs past a tile
    (65, 129, 1536, 64),     # first M on 128-token tiles
    (129, 65, 96, 32),       # K = 3 groups; ragged everything
    (200, 257, 1024, 32),
    (300, 64, 2048, 128),    # exactly one tile of outputs
])
def test_gated_gemm_raw(w4, cuda_device, M, N, K, g):
    r = workloads.rng(M * 17 + N + K + g)
    qg, sg = _scaled(r, N, K, g, 8.0)  # gate values of order 1, where silu is far from linear
    qu, su = workloads.raw_packed(r, N, K, g)
    x = workloads.activations(r, M, K)
    y = _run(w4, cuda_device, x, qg, sg, qu, su, g)
    print(f"gated GEMM M={M} N={N} K={K} g={g} max err/bound "
          f"{_check(y, x, qg, sg, qu, su, g, f'M={M} N={N} K={K} g={g}'):.3f}")


def test_gated_gemm_zero_up_gives_exact_zero(w4, cuda_device):
    r = workloads.rng(81)
    qg, sg = workloads.raw_packed(r, 300, 1024, 128)
    qu = np.full_like(qg, 0x88)  # every q = 0
    x = workloads.activations(r, 100, 1024)
    assert np.all(_run(w4, cuda_device, x, qg, sg, qu, sg, 128) == 0)


def test_gated_gemm_gate_and_up_are_not_swapped(w4, cuda_device):
    """silu(g) * u is not symmetric in g and u: one-hot x reads single weights
    of both matrices, and swapping the matrices must change the result (a
    kernel that loaded Wu's rows into the gate half of the tile would not)."""
    r = workloads.rng(82)
    N, K, g = 96, 256, 64
    qg, sg = _scaled(r, N, K, g, 8.0)
    qu, su = workloads.raw_packed(r, N, K, g)
    ks = list(range(0, K, 5))[:40]
    x = np.zeros((len(ks), K), np.float16)
    for i, k in enumerate(ks):
        x[i, k] = 1
    y = _run(w4, cuda_device, x, qg, sg, qu, su, g)
    _check(y, x, qg, sg, qu, su, g, "one-hot x")
    ys = _run(w4, cuda_device, x, qu, su, qg, sg, g)   # swapped roles give a different result
    assert not np.array_equal(y.view(np.uint16), ys.view(np.uint16))


def test_gated_gemm_deterministic(w4, cuda_device):
    r = workloads.rng(83)
    qg, sg = _scaled(r, 640, 1024, 128, 8.0)
    qu, su = workloads.raw_packed(r, 640, 1024, 128)
    x = workloads.activations(r, 333, 1024)
    y1 = _run(w4, cuda_device, x, qg, sg, qu, su, 128)
    y2 = _run(w4, cuda_device, x, qg, sg, qu, su, 128)
    assert np.array_equal(y1.view(np.uint16), y2.view(np.uint16))


def _full_pair():
    """The 27B-class gate/up pair (K=5120 -> N=17408, group 128) quantized by
    the oracle from N(0, 0.02) weights."""
    K, N, g = 5120, 17408, 128
    qg, sg = oracle.quantize(workloads.weights(workloads.rng(0), N, K), g)
    qu, su = oracle.quantize(workloads.weights(workloads.rng(1), N, K), g)
    return qg, sg, qu, su, K, N, g


@pytest.mark.parametrize("M", [17, 512])
def test_gated_prefill_full_size_every_element(w4, cuda_device, M):
    qg, sg, qu, su, K, N, g = _full_pair()
    x = workloads.activations(workloads.rng(2 + M), M, K, outlier_frac=0.01)  # prefill x: 1% outlier channels
    y = _run(w4, cuda_device, x, qg, sg, qu, su, g)
    print(f"gated prefill M={M} max err/bound (all elements) {_check(y, x, qg, sg, qu, su, g, f'M={M}'):.3f}")


def test_gated_prefill_m4096_full_size_stratified(w4, cuda_device):
    """M = 4096: 256 random rows x all N outputs, plus all rows x 256 random
    outputs (each output n needs row n of both Wg and Wu)."""
    M = 4096
    qg, sg, qu, su, K, N, g = _full_pair()
    x = workloads.activations(workloads.rng(2 + M), M, K, outlier_frac=0.01)  # prefill x: 1% outlier channels
    y = _run(w4, cuda_device, x, qg, sg, qu, su, g)
    r = workloads.rng(84)
    rows = np.sort(r.choice(M, 256, replace=False))
    cols = np.sort(r.choice(N, 256, replace=False))
    w1 = _check(y[rows], x[rows], qg, sg, qu, su, g, "rows")
    w2 = _check(y[:, cols], x, qg[cols], sg[cols], qu[cols], su[cols], g, "cols")
    print(f"gated prefill M={M} max err/bound rows {w1:.3f} cols {w2:.3f}")
