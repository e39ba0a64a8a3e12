"""Fused gate + up projections with the SiLU * up epilogue (decode GEMV,
M <= 16) on the GPU against the oracle: y = silu(x Wg^T) * (x Wu^T), within
the bound that follows from the linear tolerance on g and u (see
oracle.gated_tolerance)."""
import numpy as np
import pytest

import oracle
import workloads
from helpers import to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w4(cuda_device):
    import w4a16_group_quantized_linear_gb300 as m

    m.lib()
    return m


def _run(w4, dev, x, qg, sg, qu, su, g):
    return w4.linear_gated(to_dev(x, dev), to_dev(qg, dev), to_dev(sg.view(np.float16), dev), to_dev(qu, dev),
                           to_dev(su.view(np.float16), dev), g).cpu().numpy()


def _check(y, x, qg, sg, qu, su, g, what, threads=1):
    y_ref, gg, uu, ag, au = oracle.gated_linear(x, qg, sg, qu, su, g, threads=threads)
    bound = oracle.gated_tolerance(gg, uu, ag, au)
    err = np.abs(y.astype(np.float64) - y_ref)
    assert np.all(np.isfinite(y)), what
    bad = err > bound
    assert not bad.any(), f"{what}: {int(bad.sum())} elements out of bound, worst err/bound {np.max(err / np.maximum(bound, 1e-300))}"
    ratio = float(np.max(err / np.maximum(bound, 1e-300)))
    print(f"{what} max err/bound {ratio:.3f}")
    return ratio


def _scaled(r, N, K, g, gain):
    qw, s = workloads.raw_packed(r, N, K, g)
    s = oracle.float_to_half_bits(np.float32(gain) * oracle.half_to_double(s).astype(np.float32))
    return qw, s


# Scale rows of K/g halves travel by TMA when they are a multiple of 16 bytes
# and are read from global memory otherwise; both kinds appear below, with
# partial units (K % 512 != 0), ragged N and the two-tile path (M > 8).
@pytest.mark.parametrize("M,N,K,g", [(1, 256, 1024, 128), (4, 1000, 2080, 32), (16, 300, 512, 64),
                                     (3, 17, 192, 64), (9, 129, 1536, 64), (1, 4099, 384, 128)])
def test_gated_raw(w4, cuda_device, M, N, K, g):
    r = workloads.rng(M * 13 + N + K)
    qg, sg = _scaled(r, N, K, g, 8.0)  # gate values of order 1, where silu is far from linear
    qu, su = workloads.raw_packed(r, N, K, g)
    x = workloads.activations(r, M, K)
    y = _run(w4, cuda_device, x, qg, sg, qu, su, g)
    _check(y, x, qg, sg, qu, su, g, f"gated M={M} N={N} K={K} g={g}")


def test_gated_zero_up_gives_exact_zero(w4, cuda_device):
    r = workloads.rng(71)
    qg, sg = workloads.raw_packed(r, 300, 1024, 128)
    qu = np.full_like(qg, 0x88)  # every q = 0
    x = workloads.activations(r, 2, 1024)
    y = _run(w4, cuda_device, x, qg, sg, qu, sg, 128)
    assert np.all(y == 0)


def test_gated_two_calls_and_plain_calls_share_a_workspace(w4, cuda_device):
    """Gated and plain calls alternate on one stream (one cached workspace):
    each call leaves its counters at zero for the next."""
    r = workloads.rng(72)
    K, N, g = 2048, 777, 64
    qg, sg = _scaled(r, N, K, g, 8.0)
    qu, su = workloads.raw_packed(r, N, K, g)
    for i in range(3):
        x = workloads.activations(workloads.rng(100 + i), 1 + 2 * i, K)
        y = _run(w4, cuda_device, x, qg, sg, qu, su, g)
        _check(y, x, qg, sg, qu, su, g, f"gated round {i}")
        yl = w4.linear(to_dev(x, cuda_device), to_dev(qu, cuda_device), to_dev(su.view(np.float16), cuda_device),
                       g).cpu().numpy()
        y_ref, a = oracle.linear(x, qu, su, g)
        assert np.all(np.abs(yl - y_ref) <= oracle.tolerance(y_ref, a))


@pytest.mark.parametrize("M", [1, 4])
def test_gated_decode_full_size(w4, cuda_device, M):
    """The 27B-class gate/up pair (K=5120 -> N=17408, group 128) with weights
    quantized by the oracle from N(0, 0.02)."""
    K, N, g = 5120, 17408, 128
    qg, sg = oracle.quantize(workloads.weights(workloads.rng(0), N, K), g)
    qu, su = oracle.quantize(workloads.weights(workloads.rng(1), N, K), g)
    x = workloads.activations(workloads.rng(2), M, K)
    y = _run(w4, cuda_device, x, qg, sg, qu, su, g)
    _check(y, x, qg, sg, qu, su, g, f"gated decode M={M}", threads=8)


@pytest.mark.parametrize("N,K", [(8192, 4096), (4096, 16384)])
def test_gated_cluster_decode(w4, cuda_device, N, K):
    """M = 1, group 128, aligned N and K: the cluster kernel for the pair (units
    of 16 Wg rows and the same 16 Wu rows, both sums sent to a row-block's
    finisher). Checked against the oracle, rerun bit for bit, and with
    W4A16_STATIC_WEIGHTS."""
    r = workloads.rng(N + K + 5)
    qg, sg = _scaled(r, N, K, 128, 8.0)
    qu, su = workloads.raw_packed(r, N, K, 128)
    x = workloads.activations(r, 1, K)
    args = [to_dev(x, cuda_device), to_dev(qg, cuda_device), to_dev(sg.view(np.float16), cuda_device),
            to_dev(qu, cuda_device), to_dev(su.view(np.float16), cuda_device)]
    y0 = w4.linear_gated(*args, 128).cpu().numpy()
    _check(y0, x, qg, sg, qu, su, 128, f"gated cluster N={N} K={K}", threads=8)
    assert np.array_equal(y0.view(np.uint16), w4.linear_gated(*args, 128).cpu().numpy().view(np.uint16))
    y1 = w4.linear_gated(*args, 128, static_weights=True).cpu().numpy()
    assert np.array_equal(y0.view(np.uint16), y1.view(np.uint16))


def test_gated_static_weights_same_bits(w4, cuda_device):
    """W4A16_STATIC_WEIGHTS changes no result bit of the fused pair."""
    r = workloads.rng(61)
    M, N, K, g = 2, 1000, 2048, 128
    qg, sg = _scaled(r, N, K, g, 8.0)
    qu, su = workloads.raw_packed(r, N, K, g)
    x = workloads.activations(r, M, K)
    args = [to_dev(x, cuda_device), to_dev(qg, cuda_device), to_dev(sg.view(np.float16), cuda_device),
            to_dev(qu, cuda_device), to_dev(su.view(np.float16), cuda_device)]
    y0 = w4.linear_gated(*args, g).cpu().numpy()
    y1 = w4.linear_gated(*args, g, static_weights=True).cpu().numpy()
    assert np.array_equal(y0.view(np.uint16), y1.view(np.uint16))
    _check(y1, x, qg, sg, qu, su, g, "gated static weights")


def test_gated_then_plain_share_one_workspace(w4, cuda_device):
    """A fused gate+up call and a plain GEMV may share one workspace: every
    call leaves it ready for the next, including the fp32 gate/up parking
    area, whose bytes lie where a wide plain GEMV keeps its arrival counters."""
    import torch

    lib = w4.lib()
    r = workloads.rng(62)
    M, N, K, g = 2, 4096, 1024, 128
    qg, sg = _scaled(r, N, K, g, 8.0)
    qu, su = workloads.raw_packed(r, N, K, g)
    x = workloads.activations(r, M, K)
    Np, Kp = 17408, 1024                      # 1088 row-blocks of counters
    qp, sp = workloads.raw_packed(r, Np, Kp, g)
    xp = workloads.activations(r, 1, Kp)
    nb = max(lib.w4a16_linear_gated_workspace_bytes(M, N, K, g), lib.w4a16_workspace_bytes(1, Np, Kp, g, 1))
    ws = torch.empty(nb, dtype=torch.uint8, device=cuda_device)
    st = w4._stream(cuda_device)
    assert lib.w4a16_workspace_init(w4._ptr(ws), nb, st) == 0
    d = [to_dev(t, cuda_device) for t in (x, qg, sg.view(np.float16), qu, su.view(np.float16))]
    y = torch.empty((M, N), dtype=torch.float16, device=cuda_device)
    assert lib.w4a16_linear_gated(*(w4._ptr(t) for t in d), w4._ptr(y), M, N, K, g, w4._ptr(ws), nb, st) == 0
    dp = [to_dev(t, cuda_device) for t in (xp, qp, sp)]
    yp = torch.empty((1, Np), dtype=torch.float16, device=cuda_device)
    assert lib.w4a16_linear(*(w4._ptr(t) for t in dp), w4._ptr(yp), 1, Np, Kp, g, w4._ptr(ws), nb, st) == 0
    w4.device_status()
    _check(y.cpu().numpy(), x, qg, sg, qu, su, g, "gated on a shared workspace")
    y_ref, a = oracle.linear(xp, qp, sp, g, threads=8)
    from helpers import assert_within_bound
    assert_within_bound(yp.cpu().numpy(), y_ref, a, "plain GEMV after the gated call")
