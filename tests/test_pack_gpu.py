"""w4a16_pack / w4a16_unpack on the GPU: bit-exact against the oracle."""
import numpy as np
import pytest

import oracle
import workloads
from helpers import to_dev
from test_oracle import _quantize_cases

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w4(cuda_device):
    import w4a16_group_quantized_linear_gb300 as m

    m.lib()
    return m


def _pack_both(w4, W, g, dev):
    qw, s = oracle.quantize(W, g)
    qd, sd = w4.pack(to_dev(W, dev), g)
    return qw, s, qd.cpu().numpy(), sd.cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("N,K,g", [(256, 1024, 128), (17408, 5120, 128), (5120, 17408, 128),
                                   (512, 2048, 32), (2048, 512, 32), (33, 192, 64), (1, 32, 32)])
def test_pack_bit_exact(w4, cuda_device, N, K, g):
    W = workloads.weights(workloads.rng(N + K + g), N, K)
    qw, s, qd, sd = _pack_both(w4, W, g, cuda_device)
    assert np.array_equal(qd, qw)
    assert np.array_equal(sd, s)


def test_pack_golden_cases(w4, cuda_device):
    for case in _quantize_cases():
        g = case["g"]
        K = g * len(case["s"])
        W = np.zeros((1, K), np.float32)
        W[0, :len(case["w"])] = case["w"]
        qw, s, qd, sd = _pack_both(w4, W, g, cuda_device)
        assert sd[0].tolist() == case["s"], case["name"]
        assert np.array_equal(qd, qw), case["name"]


def test_pack_edge_values(w4, cuda_device):
    r = workloads.rng(9)
    W = workloads.weights(r, 64, 256)
    W[0] = 0                                             # all-zero groups
    W[1] *= 1e-6                                         # scales round to zero
    W[5] *= 1e-3                                         # subnormal scales
    W[2, :32] = np.float32(7.0) * np.arange(-16, 16) / 16  # exact ties
    W[3] = np.float32(1e4) * np.sign(W[3])               # equal magnitudes
    W[4, ::2] = -W[4, 1::2]                              # odd symmetry
    for g in (32, 64, 128):
        qw, s, qd, sd = _pack_both(w4, W, g, cuda_device)
        assert np.array_equal(qd, qw) and np.array_equal(sd, s)


def test_unpack_bit_exact(w4, cuda_device):
    b = np.arange(256, dtype=np.uint8).reshape(4, 64)
    b = np.concatenate([b, workloads.rng(3).integers(0, 256, (60, 64), dtype=np.uint8)])
    q = w4.unpack(to_dev(b, cuda_device), 128).cpu().numpy()
    assert np.array_equal(q, oracle.unpack(b, 128))


def test_pack_unpack_round_trip(w4, cuda_device):
    W = workloads.weights(workloads.rng(4), 100, 384)
    qd, sd = w4.pack(to_dev(W, cuda_device), 128)
    q = w4.unpack(qd, 384).cpu().numpy()
    assert np.array_equal(oracle.pack_q(q), qd.cpu().numpy())
