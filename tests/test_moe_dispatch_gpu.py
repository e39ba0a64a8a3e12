"""Routed-MoE router, dispatch and combine on the GPU against the oracle: ids,
offsets and permutations bit-exact, weights and combined outputs within the
oracle's fp32 bounds, and the whole route -> dispatch -> grouped layer ->
combine chain."""
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


def _route(w4, dev, logits, k, renorm):
    ids, w = w4.moe_route(to_dev(logits, dev), k, renorm)
    w4.device_status()
    return ids.cpu().numpy(), w.cpu().numpy()


@pytest.mark.parametrize("T,E,k,ties", [
    (4096, 128, 8, False),   # the routed-expert workload: 4096 tokens, 8 of 128
    (333, 40, 5, False),     # E not a multiple of 32, ragged token blocks
    (257, 128, 8, True),     # integer logits: many equal values
    (64, 1024, 32, False),   # largest E and top_k
    (9, 1, 1, False),        # one expert
    (5, 32, 32, True),       # top_k = E: the whole ordering
])
@pytest.mark.parametrize("renorm", [True, False])
def test_route_matches_oracle(w4, cuda_device, T, E, k, ties, renorm):
    r = workloads.rng(T + E + k)
    logits = workloads.router_logits(r, T, E, 3.0)
    if ties:
        logits = np.round(logits).astype(np.float32)
    ids, w = _route(w4, cuda_device, logits, k, renorm)
    ids_ref, w_ref, ms = oracle.moe_route(logits, k, renorm)
    assert np.array_equal(ids, ids_ref)
    err = np.abs(w.astype(np.float64) - w_ref)
    assert np.all(err <= oracle.route_tolerance(w_ref, ms, E, k)), float((err / np.abs(w_ref)).max())


def test_route_empty_and_limits(w4, cuda_device):
    import torch

    ids, w = w4.moe_route(torch.empty((0, 16), dtype=torch.float32, device=cuda_device), 4)
    assert ids.shape == (0, 4)
    for E, k, code in ((16, 17, 1), (16, 0, 1), (1025, 8, 2), (64, 33, 2)):
        with pytest.raises(w4.W4A16Error) as e:
            w4.moe_route(torch.zeros((2, E), dtype=torch.float32, device=cuda_device), k)
        assert e.value.status == code


def _dispatch(w4, dev, ids, E, x=None):
    off, row_of, tok, xs = w4.moe_dispatch(to_dev(ids.astype(np.int32), dev), E,
                                           None if x is None else to_dev(x, dev))
    status = w4.device_status(raise_on_error=False)
    return off.cpu().numpy(), row_of.cpu().numpy(), tok.cpu().numpy(), None if xs is None else xs.cpu().numpy(), status


@pytest.mark.parametrize("T,k,E,K,dup", [
    (4096, 8, 128, 2048, False),  # the routed-expert workload (R = 32768 rows)
    (1000, 3, 7, 64, True),       # 3 chunks, the last one partial; repeated experts per token
    (300, 4, 4096, 8, False),     # largest E: most experts empty
    (1, 1, 1, 16, False),
    (2047, 2, 33, 0, True),       # permutation only, no gather
])
def test_dispatch_matches_oracle(w4, cuda_device, T, k, E, K, dup):
    r = workloads.rng(T * k + E)
    if dup:
        ids = r.integers(0, E, size=(T, k))
    else:
        ids, _, _ = oracle.moe_route(workloads.router_logits(r, T, E), k)
    x = workloads.activations(r, T, K) if K else None
    off, row_of, tok, xs, status = _dispatch(w4, cuda_device, ids, E, x)
    assert status == 0
    off_ref, row_ref, tok_ref = oracle.moe_dispatch(ids, E)
    assert np.array_equal(off, off_ref)
    assert np.array_equal(row_of, row_ref)
    assert np.array_equal(tok, tok_ref)
    if K:
        assert np.array_equal(xs.view(np.uint16), oracle.moe_gather(x, tok_ref).view(np.uint16))


def test_dispatch_no_tokens_writes_zero_offsets(w4, cuda_device):
    import torch

    off, row_of, tok, xs = w4.moe_dispatch(torch.empty((0, 4), dtype=torch.int32, device=cuda_device), 9)
    w4.device_status()
    assert off.cpu().tolist() == [0] * 10 and row_of.shape == (0, 4) and xs is None


def test_dispatch_reports_out_of_range_ids(w4, cuda_device):
    """An id of E (or negative) is caught by the kernel's own range check: the pair
    gets row -1, no row, and the device word reports BAD_ROUTING."""
    E, T, k = 6, 50, 2
    r = workloads.rng(3)
    ids = r.integers(0, E, size=(T, k))
    ids[7, 1] = E
    ids[20, 0] = -3
    off, row_of, tok, _, status = _dispatch(w4, cuda_device, ids, E)
    assert status == 8
    assert row_of[7, 1] == -1 and row_of[20, 0] == -1
    assert off[-1] == T * k - 2
    keep = np.ones((T, k), bool)
    keep[7, 1] = keep[20, 0] = False
    good = ids.copy()
    good[~keep] = 0
    # the valid pairs are ordered as the oracle orders them with the bad pairs left out
    order = [(int(ids[t, j]), t, j) for t in range(T) for j in range(k) if keep[t, j]]
    order.sort()
    for rr, (_, t, j) in enumerate(order):
        assert row_of[t, j] == rr and tok[rr] == t


@pytest.mark.parametrize("T,k,N,drop", [
    (4096, 8, 2048, False),  # the routed-expert workload (down projection output)
    (100, 3, 100, False),    # N % 8 != 0: one element per thread
    (37, 4, 264, True),      # some pairs dropped (row -1)
    (1, 1, 8, False),
])
def test_combine_matches_oracle(w4, cuda_device, T, k, N, drop):
    r = workloads.rng(T + k + N)
    R = T * k
    ys = r.normal(0, 2, size=(R, N)).astype(np.float16)
    row_of = r.permutation(R).reshape(T, k).astype(np.int32)
    if drop:
        row_of[::5, 0] = -1
    w = r.random((T, k)).astype(np.float32)
    y = w4.moe_combine(to_dev(ys, cuda_device), to_dev(row_of, cuda_device), to_dev(w, cuda_device))
    w4.device_status()
    keep = row_of >= 0
    y_ref, a = oracle.moe_combine(ys, np.where(keep, row_of, 0), np.where(keep, w, 0.0))
    got = y.cpu().numpy().astype(np.float64)
    err = np.abs(got - y_ref)
    assert np.all(err <= oracle.combine_tolerance(y_ref, a, k))


def test_combine_reports_rows_out_of_range(w4, cuda_device):
    T, k, N = 4, 2, 16
    ys = np.ones((T * k, N), np.float16)
    row_of = np.arange(T * k, dtype=np.int32).reshape(T, k)
    row_of[2, 1] = T * k  # one past the end: reported, adds nothing
    w = np.ones((T, k), np.float32)
    y = w4.moe_combine(to_dev(ys, cuda_device), to_dev(row_of, cuda_device), to_dev(w, cuda_device))
    assert w4.device_status(raise_on_error=False) == 8
    got = y.cpu().numpy().astype(np.float64)
    assert np.all(got[2] == 1.0) and np.all(got[[0, 1, 3]] == 2.0)


def test_moe_chain_matches_oracle(w4, cuda_device):
    """route -> dispatch (with gather) -> grouped layer (group 32) -> combine, each step
    against the oracle on the GPU's own inputs to that step."""
    T, E, k, K, N, g = 200, 16, 4, 256, 96, 32
    r = workloads.rng(99)
    logits = workloads.router_logits(r, T, E)
    x = workloads.activations(r, T, K)
    qw = r.integers(0, 256, (E, N, K // 2), dtype=np.uint8)
    s = (np.abs(r.normal(0, 0.02, (E, N, K // g))) / 7).astype(np.float16)
    dev = cuda_device
    ids_d, w_d = w4.moe_route(to_dev(logits, dev), k)
    off_d, row_d, tok_d, xs_d = w4.moe_dispatch(ids_d, E, to_dev(x, dev))
    ys_d = w4.grouped_linear(xs_d, to_dev(qw, dev), to_dev(s, dev), off_d, g)
    y_d = w4.moe_combine(ys_d, row_d, w_d)
    w4.device_status()
    ids_ref, w_ref, ms = oracle.moe_route(logits, k)
    assert np.array_equal(ids_d.cpu().numpy(), ids_ref)
    off_ref, row_ref, tok_ref = oracle.moe_dispatch(ids_ref, E)
    assert np.array_equal(off_d.cpu().numpy(), off_ref) and np.array_equal(row_d.cpu().numpy(), row_ref)
    xs_ref = oracle.moe_gather(x, tok_ref)
    assert np.array_equal(xs_d.cpu().numpy().view(np.uint16), xs_ref.view(np.uint16))
    ys = ys_d.cpu().numpy()
    ys_ref, a = oracle.grouped_linear(xs_ref, qw, s, off_ref, g)
    assert_within_bound(ys, ys_ref, a, "experts")
    wg = w_d.cpu().numpy()
    y_ref, a = oracle.moe_combine(ys, row_ref, wg)
    err = np.abs(y_d.cpu().numpy().astype(np.float64) - y_ref)
    assert np.all(err <= oracle.combine_tolerance(y_ref, a, k))
