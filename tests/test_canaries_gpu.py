"""Guard canaries: every GPU entry point writes exactly its output and nothing
past it (the output sits at the front of a larger buffer whose tail holds a
fixed pattern), and the output itself still matches the oracle."""
import numpy as np
import pytest

import oracle
import workloads
from helpers import assert_within_bound, to_dev

pytestmark = pytest.mark.gpu

PATTERN = 12345


@pytest.fixture(scope="module")
def w4(cuda_device):
    import w4a16_group_quantized_linear_gb300 as m

    m.lib()
    return m


def _guarded(rows, cols, dev, tail=4096):
    """An fp16 [rows, cols] view at the front of a buffer with `tail` guard elements."""
    import torch

    buf = torch.full((rows * cols + tail,), PATTERN, dtype=torch.int16, device=dev)
    return buf, buf[: rows * cols].view(torch.float16).view(rows, cols)


def _tail_intact(buf, n):
    return bool(np.all(buf[n:].cpu().numpy() == PATTERN))


@pytest.mark.parametrize("M,N,K,g", [(200, 100, 512, 128), (40, 130, 256, 64), (17, 8, 32, 32)])
def test_gemm_writes_only_its_output(w4, cuda_device, M, N, K, g):
    r = workloads.rng(M + N + K)
    qw, s = workloads.raw_packed(r, N, K, g)
    x = workloads.activations(r, M, K)
    buf, out = _guarded(M, N, cuda_device)
    w4.linear(to_dev(x, cuda_device), to_dev(qw, cuda_device), to_dev(s, cuda_device), g, out=out)
    w4.device_status()
    assert _tail_intact(buf, M * N)
    y_ref, a = oracle.linear(x, qw, s, g)
    assert_within_bound(out.cpu().numpy(), y_ref, a, "gemm canary")


def test_grouped_writes_only_its_output(w4, cuda_device):
    r = workloads.rng(31)
    counts = [5, 0, 140, 3]
    E, N, K, g = len(counts), 72, 256, 32
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    R = int(off[-1])
    qw = r.integers(0, 256, (E, N, K // 2), dtype=np.uint8)
    s = (np.abs(r.normal(0, 0.02, (E, N, K // g))) / 7).astype(np.float16)
    x = workloads.activations(r, R, K)
    buf, out = _guarded(R, N, cuda_device)
    w4.grouped_linear(to_dev(x, cuda_device), to_dev(qw, cuda_device), to_dev(s, cuda_device),
                      to_dev(off, cuda_device), g, out=out)
    w4.device_status()
    assert _tail_intact(buf, R * N)
    y_ref, a = oracle.grouped_linear(x, qw, s, off, g)
    assert_within_bound(out.cpu().numpy(), y_ref, a, "grouped canary")


def test_gated_writes_only_its_output(w4, cuda_device):
    r = workloads.rng(32)
    M, N, K, g = 3, 100, 512, 128
    qg, sg = workloads.raw_packed(r, N, K, g)
    qu, su = workloads.raw_packed(r, N, K, g)
    x = workloads.activations(r, M, K)
    buf, out = _guarded(M, N, cuda_device)
    d = cuda_device
    w4.linear_gated(to_dev(x, d), to_dev(qg, d), to_dev(sg, d), to_dev(qu, d), to_dev(su, d), g, out=out)
    w4.device_status()
    assert _tail_intact(buf, M * N)
    y_ref, g_ref, u_ref, ag, au = oracle.gated_linear(x, qg, sg, qu, su, g)
    got = out.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - y_ref) <= oracle.gated_tolerance(g_ref, u_ref, ag, au))


def test_moe_dispatch_and_combine_write_only_their_outputs(w4, cuda_device):
    import torch

    r = workloads.rng(33)
    T, E, k, K = 300, 12, 3, 64
    logits = workloads.router_logits(r, T, E)
    x = workloads.activations(r, T, K)
    d = cuda_device
    xd = to_dev(x, d)
    ids, wts = w4.moe_route(to_dev(logits, d), k)
    off, row_of, tok, xs = w4.moe_dispatch(ids, E, xd)
    # dispatch again into guarded buffers through the C ABI
    P = T * k
    xs_buf, xs_view = _guarded(P, K, d)
    tok_buf = torch.full((P + 1024,), -777, dtype=torch.int32, device=d)
    row_buf = torch.full((P + 1024,), -777, dtype=torch.int32, device=d)
    off_buf = torch.full((E + 1 + 1024,), -777, dtype=torch.int32, device=d)
    nb = int(w4.lib().w4a16_moe_dispatch_workspace_bytes(T, k, E))
    ws = torch.empty(max(nb, 1), dtype=torch.uint8, device=d)
    st = w4._stream(d)
    assert w4.lib().w4a16_moe_dispatch(w4._ptr(ids), T, k, E, w4._ptr(xd), K, w4._ptr(off_buf),
                                       w4._ptr(row_buf), w4._ptr(tok_buf), w4._ptr(xs_view), w4._ptr(ws), nb,
                                       st) == 0
    w4.device_status()
    assert np.all(tok_buf[P:].cpu().numpy() == -777) and np.all(row_buf[P:].cpu().numpy() == -777)
    assert np.all(off_buf[E + 1:].cpu().numpy() == -777)
    assert _tail_intact(xs_buf, P * K)
    assert np.array_equal(xs_view.cpu().numpy().view(np.uint16), xs.cpu().numpy().view(np.uint16))
    assert np.array_equal(off_buf[: E + 1].cpu().numpy(), off.cpu().numpy())
    # combine into a guarded output
    y_buf, y_view = _guarded(T, K, d)
    w4.moe_combine(xs, row_of, wts, out=y_view)
    w4.device_status()
    assert _tail_intact(y_buf, T * K)
    y_ref, a = oracle.moe_combine(xs.cpu().numpy(), row_of.cpu().numpy(), wts.cpu().numpy())
    assert np.all(np.abs(y_view.cpu().numpy().astype(np.float64) - y_ref) <= oracle.combine_tolerance(y_ref, a, k))


@pytest.mark.parametrize("fmt,M,N,K", [("q4_k", 3, 203, 2816), ("q5_1", 9, 77, 1056), ("q4_k", 1, 1000, 8192)])
def test_blocks_gemv_writes_only_its_output(w4, cuda_device, fmt, M, N, K):
    r = workloads.rng(M + N + K)
    wb = workloads.raw_blocks(r, fmt, N, K)
    x = workloads.activations(r, M, K)
    buf, out = _guarded(M, N, cuda_device)
    w4.blocks_linear(fmt, to_dev(x, cuda_device), to_dev(wb, cuda_device), out=out)
    w4.device_status()
    assert _tail_intact(buf, M * N)
    y_ref, a = oracle.blocks_linear(fmt, x, wb)
    assert_within_bound(out.cpu().numpy(), y_ref, a, f"{fmt} canary")
