"""Outputs stored straight into pinned host memory (unified addressing): every
path (decode GEMV, narrow tiles, split-scale GEMM, both fused gate+up paths)
gives the same bits as with a device output, and they match the oracle."""
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


@pytest.mark.parametrize("M,N,K,g", [(1, 4099, 1024, 128), (4, 1000, 2080, 32), (32, 300, 512, 64),
                                     (200, 257, 1024, 32), (512, 640, 2048, 128),
                                     (1, 8192, 4096, 128), (4, 8192, 4096, 128)])  # the cluster decode kernels
def test_linear_into_pinned_host_memory(w4, cuda_device, M, N, K, g):
    import torch

    r = workloads.rng(M + N + K + g)
    qw, s = workloads.raw_packed(r, N, K, g)
    x = workloads.activations(r, M, K)
    xd, qd, sd = to_dev(x, cuda_device), to_dev(qw, cuda_device), to_dev(s, cuda_device)
    y_dev = w4.linear(xd, qd, sd, g).cpu().numpy()
    y_host = torch.full((M, N), 7.0, dtype=torch.float16).pin_memory()
    w4.linear(xd, qd, sd, g, out=y_host)
    torch.cuda.synchronize()
    w4.device_status()
    assert np.array_equal(y_host.numpy().view(np.uint16), y_dev.view(np.uint16))
    y_ref, a = oracle.linear(x, qw, s, g)
    assert_within_bound(y_host.numpy(), y_ref, a, f"M={M} into host memory")


@pytest.mark.parametrize("M,N,K,g", [(2, 384, 1024, 64), (100, 384, 1024, 64), (1, 8192, 4096, 128)])
def test_gated_into_pinned_host_memory(w4, cuda_device, M, N, K, g):
    import torch

    r = workloads.rng(300 + M)
    qg, sg = workloads.raw_packed(r, N, K, g)
    qu, su = workloads.raw_packed(r, N, K, g)
    x = workloads.activations(r, M, K)
    d = [to_dev(t, cuda_device) for t in (x, qg, sg, qu, su)]
    y_dev = w4.linear_gated(*d, g).cpu().numpy()
    y_host = torch.zeros((M, N), dtype=torch.float16).pin_memory()
    w4.linear_gated(*d, g, out=y_host)
    torch.cuda.synchronize()
    w4.device_status()
    assert np.array_equal(y_host.numpy().view(np.uint16), y_dev.view(np.uint16))


def test_unpinned_host_output_is_refused(w4, cuda_device):
    import torch

    x = torch.zeros((1, 256), dtype=torch.float16, device=cuda_device)
    qw = torch.full((64, 128), 0x88, dtype=torch.uint8, device=cuda_device)
    s = torch.ones((64, 2), dtype=torch.float16, device=cuda_device)
    with pytest.raises(ValueError):
        w4.linear(x, qw, s, 128, out=torch.empty((1, 64), dtype=torch.float16))
