"""Routed experts with the token gather fused into the activation loads
(w4a16_grouped_linear_gather): bit-identical to the unfused path (dispatch
writes the expert-sorted x, then w4a16_grouped_linear), within the oracle's
bound of the exact routed layer, and reporting bad token ids without faulting."""
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


def _experts(r, E, N, K, g=32):
    qw = r.integers(0, 256, (E, N, K // 2), dtype=np.uint8)
    s = (np.abs(r.normal(0, 0.02, (E, N, K // g))) / 7).astype(np.float16)
    return qw, s


@pytest.mark.parametrize("T,E,k,N,K", [
    (4096, 128, 8, 512, 2048),   # the routed-expert workload's gate/up projection
    (300, 16, 4, 200, 512),      # ragged tiles, few experts
    (37, 8, 2, 130, 96),         # K % 128 != 0: a partial stage; tiny expert tiles
    (1000, 64, 8, 256, 256),
])
def test_gather_equals_unfused_and_oracle(w4, cuda_device, T, E, k, N, K):
    r = workloads.rng(T + E + N + K)
    logits = workloads.router_logits(r, T, E)
    x = workloads.activations(r, T, K)
    qw, s = _experts(r, E, N, K)
    dev = cuda_device
    xd, qd, sd = to_dev(x, dev), to_dev(qw, dev), to_dev(s, dev)
    ids, _ = w4.moe_route(to_dev(logits, dev), k)
    off, row_of, tok, xs = w4.moe_dispatch(ids, E, xd)
    y_unfused = w4.grouped_linear(xs, qd, sd, off, 32).cpu().numpy()
    y_fused = w4.grouped_linear_gather(xd, tok, qd, sd, off, 32).cpu().numpy()
    w4.device_status()
    assert np.array_equal(y_fused.view(np.uint16), y_unfused.view(np.uint16))
    # the oracle on the gathered rows (checked on a sample of rows at the full workload)
    off_h, tok_h = off.cpu().numpy(), tok.cpu().numpy()
    rows = np.arange(len(tok_h)) if len(tok_h) <= 4096 else np.sort(workloads.rng(9).choice(len(tok_h), 2048, False))
    exp_of_row = np.searchsorted(off_h, rows, side="right") - 1
    worst = 0.0
    for e in np.unique(exp_of_row):
        rs = rows[exp_of_row == e]
        y_ref, a = oracle.linear(x[tok_h[rs]], qw[e], s[e], 32)
        worst = max(worst, assert_within_bound(y_fused[rs], y_ref, a, f"expert {e}"))
    print(f"gather T={T} E={E} k={k} N={N} K={K} max err/bound {worst:.3f}")


def test_gather_chain_matches_oracle(w4, cuda_device):
    """route -> dispatch (no copy of x) -> fused gather GEMM -> combine, against
    the oracle's route -> dispatch -> gather -> grouped linear -> combine."""
    r = workloads.rng(71)
    T, E, k, N, K = 200, 16, 4, 96, 256
    logits = workloads.router_logits(r, T, E)
    x = workloads.activations(r, T, K)
    qw, s = _experts(r, E, N, K)
    dev = cuda_device
    ids, wts = w4.moe_route(to_dev(logits, dev), k)
    off, row_of, tok, xs = w4.moe_dispatch(ids, E)   # offsets and permutation only
    assert xs is None
    ys = w4.grouped_linear_gather(to_dev(x, dev), tok, to_dev(qw, dev), to_dev(s, dev), off, 32)
    y = w4.moe_combine(ys, row_of, wts).cpu().numpy()
    w4.device_status()
    ids_ref, _, _ = oracle.moe_route(logits, k)
    off_ref, row_ref, tok_ref = oracle.moe_dispatch(ids_ref, E)
    assert np.array_equal(tok.cpu().numpy(), tok_ref)
    ys_ref, a_ref = oracle.grouped_linear(oracle.moe_gather(x, tok_ref), qw, s, off_ref, 32)
    assert_within_bound(ys.cpu().numpy(), ys_ref, a_ref, "expert rows")
    y_ref, a = oracle.moe_combine(ys.cpu().numpy(), row_ref, wts.cpu().numpy())
    assert np.all(np.abs(y.astype(np.float64) - y_ref) <= oracle.combine_tolerance(y_ref, a, k))


def test_gather_reports_bad_tokens(w4, cuda_device):
    """A token id outside [0, T) is reported as W4A16_ERR_BAD_ROUTING and its
    row reads zeros; the other rows are unaffected."""
    import torch

    r = workloads.rng(72)
    T, E, N, K = 50, 2, 128, 128
    x = workloads.activations(r, T, K)
    qw, s = _experts(r, E, N, K)
    tok = np.arange(40, dtype=np.int32) % T
    tok[5], tok[33] = T + 7, -3
    off = np.array([0, 20, 40], np.int32)
    dev = cuda_device
    y = w4.grouped_linear_gather(to_dev(x, dev), to_dev(tok, dev), to_dev(qw, dev), to_dev(s, dev),
                                 to_dev(off, dev), 32).cpu().numpy()
    assert w4.device_status(raise_on_error=False) == 8
    assert np.all(y[5] == 0) and np.all(y[33] == 0)
    good = np.array([i for i in range(40) if i not in (5, 33)])
    for e, rows in ((0, good[good < 20]), (1, good[good >= 20])):
        y_ref, a = oracle.linear(x[tok[rows]], qw[e], s[e], 32)
        assert_within_bound(y[rows], y_ref, a, f"expert {e}")
    del torch
