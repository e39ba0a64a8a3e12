"""The C ABI: the library builds, loads and exports every declared symbol, and
host-side validation returns the documented status codes (no GPU needed)."""
import ctypes
import os
import re

import pytest

from conftest import ROOT


@pytest.fixture(scope="module")
def lib():
    from w4a16_group_quantized_linear_gb300 import build

    build.build()
    import w4a16_group_quantized_linear_gb300 as w4

    return w4.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "w4a16.h")).read()
    return re.findall(r"W4A16_API\s+[\w\s\*]+?\b(w4a16_\w+)\s*\(", src)


def test_header_declares_the_api():
    names = set(_declared())
    assert {"w4a16_pack", "w4a16_unpack", "w4a16_linear", "w4a16_grouped_linear",
            "w4a16_workspace_bytes", "w4a16_device_status", "w4a16_status_string"} <= names


def test_library_exports_every_declared_symbol(lib):
    import w4a16_group_quantized_linear_gb300 as w4

    for name in _declared():
        assert hasattr(lib, name), name
        assert name in w4.EXPORTS, f"binding misses {name}"
    assert lib.w4a16_version() >= 100


def test_status_strings(lib):
    import w4a16_group_quantized_linear_gb300 as w4

    for code, name in w4.STATUS.items():
        assert lib.w4a16_status_string(code).decode().startswith(name)


def _fake(addr):
    return ctypes.c_void_p(addr)


@pytest.mark.parametrize("group,K,want", [(16, 256, 2), (96, 288, 2), (128, 200, 1), (32, 48, 1), (64, -64, 1)])
def test_linear_rejects_bad_group_or_K(lib, group, K, want):
    p = _fake(1 << 20)
    assert lib.w4a16_linear(p, p, p, p, 4, 8, K, group, None, 0, None) == want


def test_linear_rejects_negative_sizes_and_nulls(lib):
    p = _fake(1 << 20)
    assert lib.w4a16_linear(p, p, p, p, -1, 8, 128, 128, None, 0, None) == 1
    assert lib.w4a16_linear(p, p, p, p, 4, -8, 128, 128, None, 0, None) == 1
    assert lib.w4a16_linear(None, p, p, p, 4, 8, 128, 128, None, 0, None) == 1
    assert lib.w4a16_linear(p, p, p, None, 4, 8, 128, 128, None, 0, None) == 1


def test_linear_rejects_misaligned(lib):
    p, q = _fake(1 << 20), _fake((1 << 20) + 8)
    assert lib.w4a16_linear(q, p, p, p, 4, 8, 128, 128, None, 0, None) == 3
    assert lib.w4a16_linear(p, q, p, p, 4, 8, 128, 128, None, 0, None) == 3
    assert lib.w4a16_linear(p, p, q, p, 4, 8, 128, 128, None, 0, None) == 3


def test_empty_problems_are_no_ops(lib):
    p = _fake(1 << 20)
    assert lib.w4a16_linear(p, p, p, p, 0, 8, 128, 128, None, 0, None) == 0
    assert lib.w4a16_linear(p, p, p, p, 4, 0, 128, 128, None, 0, None) == 0
    assert lib.w4a16_pack(p, 0, 128, 128, p, p, None) == 0
    assert lib.w4a16_unpack(p, 0, 128, p, None) == 0


def test_grouped_and_pack_validation(lib):
    p = _fake(1 << 20)
    assert lib.w4a16_grouped_linear(p, p, p, p, p, 0, 16, 8, 128, 32, None, 0, None) == 1   # E < 1
    assert lib.w4a16_grouped_linear(p, p, p, None, p, 4, 16, 8, 128, 32, None, 0, None) == 1
    assert lib.w4a16_grouped_linear(p, p, p, p, p, 4, 16, 8, 100, 32, None, 0, None) == 1
    assert lib.w4a16_pack(p, 4, 100, 32, p, p, None) == 1
    assert lib.w4a16_pack(p, 4, 128, 48, p, p, None) == 2
    assert lib.w4a16_unpack(p, 4, 7, p, None) == 1


def test_moe_validation(lib):
    p, q = _fake(1 << 20), _fake((1 << 20) + 8)
    # router: 1 <= top_k <= E, E <= 1024, top_k <= 32
    assert lib.w4a16_moe_route(p, 4, 16, 17, 1, p, p, None) == 1
    assert lib.w4a16_moe_route(p, 4, 0, 1, 1, p, p, None) == 1
    assert lib.w4a16_moe_route(p, 4, 2048, 8, 1, p, p, None) == 2
    assert lib.w4a16_moe_route(p, 4, 64, 33, 1, p, p, None) == 2
    assert lib.w4a16_moe_route(None, 4, 64, 8, 1, p, p, None) == 1
    assert lib.w4a16_moe_route(None, 0, 64, 8, 1, None, None, None) == 0
    # dispatch: one int per (chunk of 1024 pairs, expert) of workspace
    assert lib.w4a16_moe_dispatch_workspace_bytes(4096, 8, 128) == 32 * 128 * 4
    assert lib.w4a16_moe_dispatch_workspace_bytes(4, 8, 5000) == 0
    big = 1 << 20
    assert lib.w4a16_moe_dispatch(p, 4, 2, 0, p, 64, p, p, p, p, p, big, None) == 1
    assert lib.w4a16_moe_dispatch(p, 4, 2, 5000, p, 64, p, p, p, p, p, big, None) == 2
    assert lib.w4a16_moe_dispatch(p, 4, 2, 8, p, 60, p, p, p, p, p, big, None) == 2
    assert lib.w4a16_moe_dispatch(p, 4, 2, 8, q, 64, p, p, p, p, p, big, None) == 3
    assert lib.w4a16_moe_dispatch(p, 4, 2, 8, p, 64, p, p, p, p, None, 0, None) == 7
    assert lib.w4a16_moe_dispatch(p, 4, 2, 8, p, 64, None, p, p, p, p, big, None) == 1
    assert lib.w4a16_moe_dispatch(p, 4, 2, 8, None, 64, p, p, p, p, p, big, None) == 1
    # combine
    assert lib.w4a16_moe_combine(p, 8, p, p, 4, 0, 16, p, None) == 1
    assert lib.w4a16_moe_combine(p, 8, p, p, 0, 2, 16, p, None) == 0
    assert lib.w4a16_moe_combine(p, 8, None, p, 4, 2, 16, p, None) == 1
    assert lib.w4a16_moe_combine(p, -1, p, p, 4, 2, 16, p, None) == 1


def test_grouped_gather_validation(lib):
    p, q = _fake(1 << 20), _fake((1 << 20) + 8)
    # E < 1, no offsets, negative T
    assert lib.w4a16_grouped_linear_gather(p, 64, p, p, p, p, p, 0, 16, 8, 128, 32, None) == 1
    assert lib.w4a16_grouped_linear_gather(p, 64, p, p, p, None, p, 4, 16, 8, 128, 32, None) == 1
    assert lib.w4a16_grouped_linear_gather(p, -1, p, p, p, p, p, 4, 16, 8, 128, 32, None) == 1
    # misaligned x; K not a multiple of the group
    assert lib.w4a16_grouped_linear_gather(q, 64, p, p, p, p, p, 4, 16, 8, 128, 32, None) == 3
    assert lib.w4a16_grouped_linear_gather(p, 64, p, p, p, p, p, 4, 16, 8, 100, 32, None) == 1
    # nothing to do
    assert lib.w4a16_grouped_linear_gather(p, 64, p, p, p, p, p, 4, 0, 8, 128, 32, None) == 0


def test_blocks_validation(lib):
    """GGUF block formats: row sizes and the host checks, all before any device work."""
    import oracle

    p, q = _fake(1 << 20), _fake((1 << 20) + 8)
    Q4K, Q51 = 1, 2
    for fmt, name in ((Q4K, "q4_k"), (Q51, "q5_1")):
        for K in (0, 32, 96, 256, 288, 5120, 17408, 100, -256):
            assert lib.w4a16_blocks_row_bytes(fmt, K) == oracle.blocks_row_bytes(name, K), (name, K)
    assert lib.w4a16_blocks_row_bytes(Q4K, 5120) == 20 * 144 and lib.w4a16_blocks_row_bytes(Q51, 5120) == 160 * 24
    assert lib.w4a16_blocks_row_bytes(3, 256) == -1
    # unknown format; K not whole blocks; negative sizes; null pointers; misaligned pointers
    assert lib.w4a16_blocks_linear(3, p, p, p, 1, 8, 256, None) == 2
    assert lib.w4a16_blocks_linear(Q4K, p, p, p, 1, 8, 288, None) == 1
    assert lib.w4a16_blocks_linear(Q51, p, p, p, 1, 8, 48, None) == 1
    assert lib.w4a16_blocks_linear(Q4K, p, p, p, -1, 8, 256, None) == 1
    assert lib.w4a16_blocks_linear(Q4K, None, p, p, 1, 8, 256, None) == 1
    assert lib.w4a16_blocks_linear(Q4K, p, p, None, 1, 8, 256, None) == 1
    assert lib.w4a16_blocks_linear(Q4K, q, p, p, 1, 8, 256, None) == 3
    assert lib.w4a16_blocks_linear(Q51, p, q, p, 1, 8, 64, None) == 3
    # nothing to do
    assert lib.w4a16_blocks_linear(Q4K, p, p, p, 0, 8, 256, None) == 0
    assert lib.w4a16_blocks_linear(Q4K, p, p, p, 1, 0, 256, None) == 0
    # the dequantizer
    assert lib.w4a16_blocks_dequant(3, p, 8, 256, p, None) == 2
    assert lib.w4a16_blocks_dequant(Q4K, p, 8, 300, p, None) == 1
    assert lib.w4a16_blocks_dequant(Q4K, p, -1, 256, p, None) == 1
    assert lib.w4a16_blocks_dequant(Q4K, None, 8, 256, p, None) == 1
    assert lib.w4a16_blocks_dequant(Q4K, p, 8, 256, q, None) == 3
    assert lib.w4a16_blocks_dequant(Q4K, p, 0, 256, p, None) == 0
    assert lib.w4a16_blocks_dequant(Q51, p, 8, 0, p, None) == 0
