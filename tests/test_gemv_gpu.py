"""Decode GEMV (M <= 16) on the GPU against the oracle, within
|y - y_ref| <= 2^-9 |y_ref| + 1e-4 sum_k |x W^| per element."""
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


def _run(w4, dev, x, qw, s, g):
    return w4.linear(to_dev(x, dev), to_dev(qw, dev), to_dev(s.view(np.float16), dev), g).cpu().numpy()


def test_config0(w4, cuda_device):
    W, x, g = workloads.config0()
    qw, s = oracle.quantize(W, g)
    y = _run(w4, cuda_device, x, qw, s, g)
    y_ref, a = oracle.linear(x, qw, s, g)
    print("config0 max err/bound", assert_within_bound(y, y_ref, a, "config0"))


@pytest.mark.parametrize("M", [1, 4])
@pytest.mark.parametrize("K,N", [(5120, 17408), (17408, 5120)])
def test_decode_full_size(w4, cuda_device, M, K, N):
    W, x, g = workloads.decode(M, K, N)
    qw, s = oracle.quantize(W, g)
    y = _run(w4, cuda_device, x, qw, s, g)
    y_ref, a = oracle.linear(x, qw, s, g, threads=8)
    print(f"decode M={M} K={K} N={N} max err/bound", assert_within_bound(y, y_ref, a, "decode"))


@pytest.mark.parametrize("M", [1, 2, 3, 5, 8, 9, 13, 16])
@pytest.mark.parametrize("g", [32, 64, 128])
def test_raw_nibbles_all_M(w4, cuda_device, M, g):
    r = workloads.rng(100 * M + g)
    N, K = 203, 1536
    qw, s = workloads.raw_packed(r, N, K, g)
    x = workloads.activations(r, M, K)
    y = _run(w4, cuda_device, x, qw, s, g)
    y_ref, a = oracle.linear(x, qw, s, g)
    assert_within_bound(y, y_ref, a, f"M={M} g={g}")


@pytest.mark.parametrize("M,N,K", [(1, 32, 65536), (2, 48, 30720), (1, 2500, 4096), (3, 16, 40960), (2, 1, 512)])
def test_row_blocks_split_across_many_warps(w4, cuda_device, M, N, K):
    """Group 128: row-blocks whose units are split over up to about 24 warps of
    a cluster (their partials summed in batches), clusters left without work,
    the two x paths (per warp for M <= 2, per block above)."""
    r = workloads.rng(M * 31 + N + K)
    qw, s = workloads.raw_packed(r, N, K, 128)
    x = workloads.activations(r, M, K)
    y = _run(w4, cuda_device, x, qw, s, 128)
    y_ref, a = oracle.linear(x, qw, s, 128)
    assert_within_bound(y, y_ref, a, f"M={M} N={N} K={K}")
    assert np.array_equal(y.view(np.uint16), _run(w4, cuda_device, x, qw, s, 128).view(np.uint16))


@pytest.mark.parametrize("M", [2, 5, 8, 9, 12, 16])
def test_decode_kernel_several_tokens(w4, cuda_device, M):
    """Group 128, aligned N and K, 2 to 16 tokens: the written-out decode kernel
    with x staged once per block (one or two 8-token MMA tiles) and each
    contributor's 16 x M sums sent to the row-block's finisher."""
    r = workloads.rng(700 + M)
    N, K = 8192, 4096
    qw, s = workloads.raw_packed(r, N, K, 128)
    x = workloads.activations(r, M, K)
    y = _run(w4, cuda_device, x, qw, s, 128)
    y_ref, a = oracle.linear(x, qw, s, 128, threads=8)
    assert_within_bound(y, y_ref, a, f"M={M}")
    assert np.array_equal(y.view(np.uint16), _run(w4, cuda_device, x, qw, s, 128).view(np.uint16))
    ys = w4.linear(to_dev(x, cuda_device), to_dev(qw, cuda_device), to_dev(s.view(np.float16), cuda_device), 128,
                   static_weights=True).cpu().numpy()
    assert np.array_equal(y.view(np.uint16), ys.view(np.uint16))


@pytest.mark.parametrize("N,K,g", [(1, 32, 32), (7, 96, 32), (17, 192, 64), (100, 640, 128), (1000, 2080, 32),
                                   (4099, 384, 128), (16, 128, 128), (31, 8192, 64)])
def test_ragged_shapes(w4, cuda_device, N, K, g):
    r = workloads.rng(N * 7 + K)
    qw, s = workloads.raw_packed(r, N, K, g)
    for M in (1, 4, 11):
        x = workloads.activations(r, M, K)
        y = _run(w4, cuda_device, x, qw, s, g)
        y_ref, a = oracle.linear(x, qw, s, g)
        assert_within_bound(y, y_ref, a, f"N={N} K={K} g={g} M={M}")


def test_zero_weights_give_exact_zero(w4, cuda_device):
    r = workloads.rng(21)
    x = workloads.activations(r, 3, 1024)
    qw = np.full((300, 512), 0x88, np.uint8)
    s = (np.abs(r.normal(0, 0.02, (300, 8))) / 7).astype(np.float16)
    y = _run(w4, cuda_device, x, qw, s, 128)
    assert np.all(y == 0)


def test_one_hot_x_reads_one_weight_exactly(w4, cuda_device):
    r = workloads.rng(22)
    N, K, g = 300, 1024, 64
    qw, s = workloads.raw_packed(r, N, K, g)
    ks = [0, 1, 63, 64, 500, 1023]
    x = np.zeros((len(ks), K), np.float16)
    for i, k in enumerate(ks):
        x[i, k] = 1
    y = _run(w4, cuda_device, x, qw, s, g)
    q = oracle.unpack(qw, K).astype(np.float64)
    sd = oracle.half_to_double(s.view(np.uint16))
    for i, k in enumerate(ks):
        want = (sd[:, k // g] * q[:, k]).astype(np.float16)   # one exact product, rounded once
        assert np.array_equal(y[i], want)


def test_deterministic_and_workspace_reuse(w4, cuda_device):
    r = workloads.rng(23)
    qw, s = workloads.raw_packed(r, 5000, 4096, 128)
    x = workloads.activations(r, 4, 4096)
    y1 = _run(w4, cuda_device, x, qw, s, 128)
    # a different shape in between reuses (and must leave clean) the workspace counters
    qw2, s2 = workloads.raw_packed(r, 77, 1024, 32)
    _run(w4, cuda_device, x[:, :1024], qw2, s2, 32)
    y2 = _run(w4, cuda_device, x, qw, s, 128)
    assert np.array_equal(y1.view(np.uint16), y2.view(np.uint16))


def test_output_canary_untouched(w4, cuda_device):
    import torch

    r = workloads.rng(24)
    N, K = 100, 512
    qw, s = workloads.raw_packed(r, N, K, 128)
    x = workloads.activations(r, 3, K)
    buf = torch.full((3 * N + 64,), 12345, dtype=torch.int16, device=cuda_device)
    out = buf[: 3 * N].view(torch.float16).view(3, N)
    w4.linear(to_dev(x, cuda_device), to_dev(qw, cuda_device), to_dev(s, cuda_device), 128, out=out)
    tail = buf[3 * N:].cpu().numpy()
    assert np.all(tail == 12345)
    y_ref, a = oracle.linear(x, qw, s, 128)
    assert_within_bound(out.cpu().numpy(), y_ref, a, "canary")


def test_workspace_shared_across_shapes(w4, cuda_device):
    """Calls of different M and N share one workspace; each must see clean counters."""
    r = workloads.rng(25)
    cases = [(16, 64, 2048), (1, 20000, 1024), (9, 333, 4096), (4, 7000, 640), (1, 64, 128)]
    data = []
    for M, N, K in cases:
        qw, s = workloads.raw_packed(r, N, K, 128)
        data.append((workloads.activations(r, M, K), qw, s))
    for _ in range(2):
        for x, qw, s in data:
            y = _run(w4, cuda_device, x, qw, s, 128)
            y_ref, a = oracle.linear(x, qw, s, 128)
            assert_within_bound(y, y_ref, a, f"M={x.shape[0]} N={qw.shape[0]}")


def test_weights_written_by_previous_kernel(w4, cuda_device):
    """The GEMV may start before the kernel ahead of it on the stream ends; it
    must still read the weights that kernel wrote. The quantizer writes the
    packed weights and the GEMV follows at once on the same stream, several
    times over; the allocator hands back the same memory with the previous
    round's contents, so reading too early would give the old weights."""
    import torch

    K, N, g = 2048, 1536, 128
    x = workloads.activations(workloads.rng(77), 1, K)
    xd = to_dev(x, cuda_device)
    for i in range(6):
        W = workloads.weights(workloads.rng(100 + i), N, K)
        Wd = torch.from_numpy(W).to(cuda_device)
        torch.cuda.synchronize()
        qw, s = w4.pack(Wd, g)
        y = w4.linear(xd, qw, s, g).cpu().numpy()
        del qw, s
        qh, sh = oracle.quantize(W, g)
        y_ref, a = oracle.linear(x, qh, sh, g)
        assert_within_bound(y, y_ref, a, f"pack then GEMV, round {i}")


@pytest.mark.parametrize("M,N,K,g", [(1, 4099, 384, 128), (4, 1000, 2080, 32), (9, 203, 1536, 64),
                                     (16, 300, 4096, 128), (1, 17408, 5120, 128), (2, 31, 8192, 64)])
def test_static_weights_same_bits(w4, cuda_device, M, N, K, g):
    """W4A16_STATIC_WEIGHTS only lets the weights stream before the previous
    kernel completes: the result bits are those of the default mode."""
    r = workloads.rng(M + N + K + g)
    qw, s = workloads.raw_packed(r, N, K, g)
    x = workloads.activations(r, M, K)
    xd, qd, sd = to_dev(x, cuda_device), to_dev(qw, cuda_device), to_dev(s, cuda_device)
    y0 = w4.linear(xd, qd, sd, g).cpu().numpy()
    y1 = w4.linear(xd, qd, sd, g, static_weights=True).cpu().numpy()
    assert np.array_equal(y0.view(np.uint16), y1.view(np.uint16))
    y_ref, a = oracle.linear(x, qw, s, g)
    assert_within_bound(y1, y_ref, a, "static weights")


def test_static_weights_chain_reads_x_after_the_previous_kernel(w4, cuda_device):
    """A decode-like chain queued back to back: x_i -> layer 1 -> h -> layer 2
    -> o_i, with one h buffer for every step. Layer 2 streams its weights
    early but must read h only after layer 1 of the same step has written it;
    reading early would give the previous step's h."""
    import torch

    g, K1, N1 = 128, 1024, 1536
    r = workloads.rng(26)
    q1, s1 = workloads.raw_packed(r, N1, K1, g)
    q2, s2 = workloads.raw_packed(r, K1, N1, g)
    xs = [workloads.activations(r, 1, K1) * np.float16(1 + i) for i in range(8)]
    dq1, ds1, dq2, ds2 = (to_dev(t, cuda_device) for t in (q1, s1, q2, s2))
    dxs = [to_dev(x, cuda_device) for x in xs]
    torch.cuda.synchronize()
    h = torch.empty((1, N1), dtype=torch.float16, device=cuda_device)
    outs = [torch.empty((1, K1), dtype=torch.float16, device=cuda_device) for _ in xs]
    for x, o in zip(dxs, outs):
        w4.linear(x, dq1, ds1, g, out=h, static_weights=True)
        w4.linear(h, dq2, ds2, g, out=o, static_weights=True)
    got = [o.cpu().numpy() for o in outs]
    w4.device_status()
    for i, (x, y) in enumerate(zip(xs, got)):
        hh = w4.linear(dxs[i], dq1, ds1, g)
        want = w4.linear(hh, dq2, ds2, g).cpu().numpy()
        assert np.array_equal(y.view(np.uint16), want.view(np.uint16)), f"step {i}"
        y1_ref, a1 = oracle.linear(x, q1, s1, g)
        hh_h = hh.cpu().numpy()
        assert_within_bound(hh_h, y1_ref, a1, f"step {i} layer 1")
        y2_ref, a2 = oracle.linear(hh_h, q2, s2, g)
        assert_within_bound(y, y2_ref, a2, f"step {i} layer 2")
