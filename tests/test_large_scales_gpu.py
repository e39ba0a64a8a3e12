"""Rows whose fp16 scales exceed 8188: the split-scale kernel (dense M > 64,
routed experts, the gated pair) computes such a row with its scales divided by
a power of two and multiplies the result back, which is exact. These rows must
match the oracle like any other, at every group size, next to ordinary rows."""
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


def _big_scales(r, N, K, g):
    """Packed bytes with every third row's scales in [8192, 60000) (two to three
    halvings needed) and the other rows ordinary."""
    qw, s = workloads.raw_packed(r, N, K, g)
    sd = oracle.half_to_double(s.view(np.uint16))
    big = r.uniform(8192.0, 60000.0, sd.shape)
    rows = np.arange(N) % 3 == 0
    sd[rows] = big[rows]
    return qw, oracle.float_to_half_bits(sd.astype(np.float32))


@pytest.mark.parametrize("g", [32, 64, 128])
@pytest.mark.parametrize("M,N,K", [(100, 130, 512), (300, 257, 1024)])
def test_dense_rows_with_large_scales(w4, cuda_device, M, N, K, g):
    r = workloads.rng(M + N + K + g + 7)
    qw, s = _big_scales(r, N, K, g)
    x = (workloads.activations(r, M, K).astype(np.float32) * np.float32(1e-4)).astype(np.float16)
    y = w4.linear(to_dev(x, cuda_device), to_dev(qw, cuda_device), to_dev(s.view(np.float16), cuda_device),
                  g).cpu().numpy()
    w4.device_status()
    assert np.all(np.isfinite(y))
    y_ref, a = oracle.linear(x, qw, s, g)
    print(f"large scales M={M} N={N} K={K} g={g} max err/bound "
          f"{assert_within_bound(y, y_ref, a, 'large scales'):.3f}")


@pytest.mark.parametrize("g", [32, 128])
def test_grouped_rows_with_large_scales(w4, cuda_device, g):
    r = workloads.rng(500 + g)
    counts = [70, 0, 190, 33]
    E, N, K = len(counts), 200, 512
    qw = np.empty((E, N, K // 2), np.uint8)
    s = np.empty((E, N, K // g), np.uint16)
    for e in range(E):
        qw[e], s[e] = _big_scales(r, N, K, g)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    x = (workloads.activations(r, int(off[-1]), K).astype(np.float32) * np.float32(1e-4)).astype(np.float16)
    y = w4.grouped_linear(to_dev(x, cuda_device), to_dev(qw, cuda_device), to_dev(s.view(np.float16), cuda_device),
                          to_dev(off, cuda_device), g).cpu().numpy()
    w4.device_status()
    y_ref, a = oracle.grouped_linear(x, qw, s, off, g)
    assert_within_bound(y, y_ref, a, "grouped, large scales")


def test_gated_rows_with_large_scales(w4, cuda_device):
    r = workloads.rng(601)
    M, N, K, g = 150, 192, 1024, 64
    qg, sg = workloads.raw_packed(r, N, K, g)
    qu, su = _big_scales(r, N, K, g)
    x = (workloads.activations(r, M, K).astype(np.float32) * np.float32(1e-2)).astype(np.float16)
    y = w4.linear_gated(to_dev(x, cuda_device), to_dev(qg, cuda_device), to_dev(sg.view(np.float16), cuda_device),
                        to_dev(qu, cuda_device), to_dev(su.view(np.float16), cuda_device), g).cpu().numpy()
    w4.device_status()
    y_ref, gg, uu, ag, au = oracle.gated_linear(x, qg, sg, qu, su, g)
    err = np.abs(y.astype(np.float64) - y_ref)
    assert np.all(np.isfinite(y))
    assert np.all(err <= oracle.gated_tolerance(gg, uu, ag, au))
