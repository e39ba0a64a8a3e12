"""W4A16 group-quantized linear layer for GB300 (sm_103a).

y = x W^T with int4-symmetric weights (nibble q+8, even k in the low nibble),
one fp16 scale per group of 32/64/128 input features and fp16 activations
(LLM170 page, introduction: "W4A16 (int4 sym g128, f16 activations)").

This module is a thin ctypes binding over the C ABI of ``libw4a16.so``
(declared in ``include/w4a16.h``): it checks tensor dtypes and shapes,
allocates outputs with PyTorch and passes raw device pointers and the current
CUDA stream. Every step of the computation runs in the library's CUDA
kernels; there is no fallback. If the library is missing, every call raises.
Build it with ``python -m w4a16_group_quantized_linear_gb300.build`` (or
``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = ["pack", "unpack", "linear", "linear_gated", "grouped_linear", "grouped_linear_gather", "moe_route",
           "moe_dispatch", "moe_combine", "blocks_row_bytes", "blocks_linear", "blocks_dequant", "BLOCK_FORMATS",
           "workspace_bytes", "device_status", "STATIC_WEIGHTS",
           "W4A16Error", "lib", "LIB_PATH", "EXPORTS", "STATUS"]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libw4a16.so")

STATUS = {0: "W4A16_OK", 1: "W4A16_ERR_INVALID_ARG", 2: "W4A16_ERR_UNSUPPORTED", 3: "W4A16_ERR_MISALIGNED",
          4: "W4A16_ERR_CUDA", 5: "W4A16_ERR_TIMEOUT", 6: "W4A16_ERR_BAD_OFFSETS", 7: "W4A16_ERR_WORKSPACE",
          8: "W4A16_ERR_BAD_ROUTING"}

_P, _I64, _I32, _SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
# name -> (restype, argtypes); mirrors include/w4a16.h
EXPORTS = {
    "w4a16_pack": (_I32, [_P, _I64, _I64, _I32, _P, _P, _P]),
    "w4a16_unpack": (_I32, [_P, _I64, _I64, _P, _P]),
    "w4a16_linear": (_I32, [_P, _P, _P, _P, _I64, _I64, _I64, _I32, _P, _SZ, _P]),
    "w4a16_linear_ex": (_I32, [_P, _P, _P, _P, _I64, _I64, _I64, _I32, ctypes.c_uint32, _P, _SZ, _P]),
    "w4a16_linear_noalloc": (_I32, [_P, _P, _P, _P, _I64, _I64, _I64, _I32, _P]),
    "w4a16_linear_gated": (_I32, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I32, _P, _SZ, _P]),
    "w4a16_linear_gated_ex": (_I32, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I32, ctypes.c_uint32, _P, _SZ,
                                     _P]),
    "w4a16_linear_gated_workspace_bytes": (_SZ, [_I64, _I64, _I64, _I32]),
    "w4a16_grouped_linear": (_I32, [_P, _P, _P, _P, _P, _I32, _I64, _I64, _I64, _I32, _P, _SZ, _P]),
    "w4a16_grouped_linear_gather": (_I32, [_P, _I64, _P, _P, _P, _P, _P, _I32, _I64, _I64, _I64, _I32, _P]),
    "w4a16_moe_route": (_I32, [_P, _I64, _I32, _I32, _I32, _P, _P, _P]),
    "w4a16_moe_dispatch_workspace_bytes": (_SZ, [_I64, _I32, _I32]),
    "w4a16_moe_dispatch": (_I32, [_P, _I64, _I32, _I32, _P, _I64, _P, _P, _P, _P, _P, _SZ, _P]),
    "w4a16_moe_combine": (_I32, [_P, _I64, _P, _P, _I64, _I32, _I64, _P, _P]),
    "w4a16_blocks_row_bytes": (_I64, [_I32, _I64]),
    "w4a16_blocks_linear": (_I32, [_I32, _P, _P, _P, _I64, _I64, _I64, _P]),
    "w4a16_blocks_dequant": (_I32, [_I32, _P, _I64, _I64, _P, _P]),
    "w4a16_workspace_bytes": (_SZ, [_I64, _I64, _I64, _I32, _I32]),
    "w4a16_workspace_init": (_I32, [_P, _SZ, _P]),
    "w4a16_device_status": (_I32, [_P]),
    "w4a16_status_string": (ctypes.c_char_p, [_I32]),
    "w4a16_version": (_I32, []),
    "w4a16_last_cuda_error": (ctypes.c_char_p, []),
}


# flags of w4a16_linear_ex / w4a16_linear_gated_ex (include/w4a16.h)
STATIC_WEIGHTS = 1

# GGUF block formats (W4A16_FORMAT_* in include/w4a16.h)
BLOCK_FORMATS = {"q4_k": 1, "q5_1": 2}


class W4A16Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        detail = ""
        if status == 4 and _lib is not None:
            detail = " (" + _lib.w4a16_last_cuda_error().decode(errors="replace") + ")"
        super().__init__(f"{where}: {STATUS.get(status, status)}{detail}")


_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """The loaded C library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libw4a16.so not built ({LIB_PATH}); run "
                                   "python -m w4a16_group_quantized_linear_gb300.build")
            h = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in EXPORTS.items():
                f = getattr(h, name)
                f.restype, f.argtypes = res, args
            _lib = h
    return _lib


def _check(status: int, where: str):
    if status != 0:
        raise W4A16Error(status, where)


def _stream(dev: torch.device):
    return ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)


def _ptr(t: torch.Tensor):
    return ctypes.c_void_p(t.data_ptr())


def _need(t: torch.Tensor, name: str, dtype, dim: int):
    if not isinstance(t, torch.Tensor) or t.dtype != dtype or t.dim() != dim or not t.is_cuda:
        raise ValueError(f"{name}: expected a {dim}-d {dtype} CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")


def _out(out, shape, device: torch.device, K: int):
    """The output of a dense layer: new on x's device, or the caller's tensor,
    which may be on x's device or in pinned host memory (the kernels then store
    to it directly through unified addressing: no separate copy)."""
    if out is None:
        return torch.empty(shape, dtype=torch.float16, device=device)
    if not isinstance(out, torch.Tensor) or out.dtype != torch.float16 or out.dim() != 2:
        raise ValueError("out: expected a 2-d torch.float16 tensor")
    if not out.is_contiguous():
        raise ValueError("out: must be contiguous")
    if tuple(out.shape) != tuple(shape):
        raise ValueError("out must be [M, N]")
    if out.is_cuda:
        if out.device != device:
            raise ValueError("out must be on x's device")
    elif not out.is_pinned() or K == 0:
        raise ValueError("out must be a CUDA tensor, or pinned host memory (K > 0)")
    return out


# one zero-initialised workspace per (device, stream), grown on demand
_ws: dict = {}


def _workspace(dev: torch.device, stream, nbytes: int):
    if nbytes == 0:
        return None
    key = (dev.index, stream.value)
    buf = _ws.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = torch.empty(max(nbytes, 1 << 20), dtype=torch.uint8, device=dev)
        _check(lib().w4a16_workspace_init(_ptr(buf), buf.numel(), stream), "w4a16_workspace_init")
        _ws[key] = buf
    return buf


def workspace_bytes(M: int, N: int, K: int, group: int, E: int = 1) -> int:
    return int(lib().w4a16_workspace_bytes(M, N, K, group, E))


def pack(w: torch.Tensor, group: int = 128):
    """fp32 [N, K] -> (qweight uint8 [N, K/2], scales fp16 [N, K/group])."""
    _need(w, "w", torch.float32, 2)
    N, K = w.shape
    qw = torch.empty((N, K // 2), dtype=torch.uint8, device=w.device)
    s = torch.empty((N, K // group if group else 0), dtype=torch.float16, device=w.device)
    _check(lib().w4a16_pack(_ptr(w), N, K, group, _ptr(qw), _ptr(s), _stream(w.device)), "w4a16_pack")
    return qw, s


def unpack(qw: torch.Tensor, K: int) -> torch.Tensor:
    """uint8 [N, K/2] -> int8 q [N, K] in [-8, 7]."""
    _need(qw, "qweight", torch.uint8, 2)
    N = qw.shape[0]
    if qw.shape[1] * 2 != K:
        raise ValueError("qweight must be [N, K/2]")
    q = torch.empty((N, K), dtype=torch.int8, device=qw.device)
    _check(lib().w4a16_unpack(_ptr(qw), N, K, _ptr(q), _stream(qw.device)), "w4a16_unpack")
    return q


def linear(x: torch.Tensor, qweight: torch.Tensor, scales: torch.Tensor, group: int = 128,
           out: torch.Tensor | None = None, static_weights: bool = False) -> torch.Tensor:
    """y = x W^T for x fp16 [M, K], qweight uint8 [N, K/2], scales fp16 [N, K/group].
    ``out`` may be a CUDA tensor on x's device or pinned host memory (K > 0).

    ``static_weights=True`` passes W4A16_STATIC_WEIGHTS: the caller promises
    that no work still pending on the stream writes qweight or scales (the
    weights of a decode loop), so the decode GEMV may stream them before the
    previous kernel on the stream completes. Results are identical."""
    _need(x, "x", torch.float16, 2)
    _need(qweight, "qweight", torch.uint8, 2)
    _need(scales, "scales", torch.float16, 2)
    M, K = x.shape
    N = qweight.shape[0]
    if qweight.shape[1] * 2 != K or (group and tuple(scales.shape) != (N, K // group)):
        raise ValueError("shape mismatch between x, qweight and scales")
    out = _out(out, (M, N), x.device, K)
    st = _stream(x.device)
    nb = workspace_bytes(M, N, K, group, 1)
    ws = _workspace(x.device, st, nb)
    _check(lib().w4a16_linear_ex(_ptr(x), _ptr(qweight), _ptr(scales), _ptr(out), M, N, K, group,
                                 STATIC_WEIGHTS if static_weights else 0,
                                 _ptr(ws) if ws is not None else None, ws.numel() if ws is not None else 0, st),
           "w4a16_linear")
    return out


def _format(fmt) -> int:
    if isinstance(fmt, str):
        if fmt not in BLOCK_FORMATS:
            raise ValueError(f"unknown block format {fmt!r}")
        return BLOCK_FORMATS[fmt]
    return int(fmt)


def blocks_row_bytes(fmt, K: int) -> int:
    """Bytes of one row of K weights in a GGUF block format (-1: not whole blocks)."""
    return int(lib().w4a16_blocks_row_bytes(_format(fmt), K))


def blocks_linear(fmt, x: torch.Tensor, blocks: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
    """y = x W^T for x fp16 [M, K] and GGUF block-format weights ("q4_k" or
    "q5_1"), blocks uint8 [N, blocks_row_bytes(fmt, K)]."""
    _need(x, "x", torch.float16, 2)
    _need(blocks, "blocks", torch.uint8, 2)
    M, K = x.shape
    N = blocks.shape[0]
    f = _format(fmt)
    if blocks.shape[1] != blocks_row_bytes(f, K):
        raise ValueError("blocks: expected [N, blocks_row_bytes(fmt, K)] bytes")
    out = _out(out, (M, N), x.device, K)
    _check(lib().w4a16_blocks_linear(f, _ptr(x), _ptr(blocks), _ptr(out), M, N, K, _stream(x.device)),
           "w4a16_blocks_linear")
    return out


def blocks_dequant(fmt, blocks: torch.Tensor, K: int) -> torch.Tensor:
    """W^ fp32 [N, K] from GGUF block-format weights uint8 [N, row_bytes]."""
    _need(blocks, "blocks", torch.uint8, 2)
    f = _format(fmt)
    N = blocks.shape[0]
    if blocks.shape[1] != blocks_row_bytes(f, K):
        raise ValueError("blocks: expected [N, blocks_row_bytes(fmt, K)] bytes")
    w = torch.empty((N, K), dtype=torch.float32, device=blocks.device)
    _check(lib().w4a16_blocks_dequant(f, _ptr(blocks), N, K, _ptr(w), _stream(blocks.device)),
           "w4a16_blocks_dequant")
    return w


def linear_gated(x: torch.Tensor, qweight_gate: torch.Tensor, scales_gate: torch.Tensor,
                 qweight_up: torch.Tensor, scales_up: torch.Tensor, group: int = 128,
                 out: torch.Tensor | None = None, static_weights: bool = False) -> torch.Tensor:
    """y = silu(x Wg^T) * (x Wu^T) in one launch (the decode GEMV for M <= 16,
    the tensor-core GEMM above); both weight matrices uint8 [N, K/2] with fp16
    scales [N, K/group]. ``static_weights`` as in :func:`linear`."""
    _need(x, "x", torch.float16, 2)
    for t, name in ((qweight_gate, "qweight_gate"), (qweight_up, "qweight_up")):
        _need(t, name, torch.uint8, 2)
    for t, name in ((scales_gate, "scales_gate"), (scales_up, "scales_up")):
        _need(t, name, torch.float16, 2)
    M, K = x.shape
    N = qweight_gate.shape[0]
    if (qweight_gate.shape[1] * 2 != K or tuple(qweight_up.shape) != tuple(qweight_gate.shape)
            or tuple(scales_gate.shape) != (N, K // group) or tuple(scales_up.shape) != (N, K // group)):
        raise ValueError("shape mismatch between x, the weights and the scales")
    out = _out(out, (M, N), x.device, K)
    st = _stream(x.device)
    nb = int(lib().w4a16_linear_gated_workspace_bytes(M, N, K, group))
    ws = _workspace(x.device, st, nb)
    _check(lib().w4a16_linear_gated_ex(_ptr(x), _ptr(qweight_gate), _ptr(scales_gate), _ptr(qweight_up),
                                       _ptr(scales_up), _ptr(out), M, N, K, group,
                                       STATIC_WEIGHTS if static_weights else 0,
                                       _ptr(ws) if ws is not None else None, ws.numel() if ws is not None else 0,
                                       st), "w4a16_linear_gated")
    return out


def grouped_linear(x_sorted: torch.Tensor, qweight: torch.Tensor, scales: torch.Tensor,
                   expert_offsets: torch.Tensor, group: int = 32,
                   out: torch.Tensor | None = None) -> torch.Tensor:
    """Routed experts: x_sorted fp16 [R, K] (rows sorted by expert), qweight uint8
    [E, N, K/2], scales fp16 [E, N, K/group], expert_offsets int32 [E+1] on the device."""
    _need(x_sorted, "x_sorted", torch.float16, 2)
    _need(qweight, "qweight", torch.uint8, 3)
    _need(scales, "scales", torch.float16, 3)
    _need(expert_offsets, "expert_offsets", torch.int32, 1)
    R, K = x_sorted.shape
    E, N = qweight.shape[0], qweight.shape[1]
    if qweight.shape[2] * 2 != K or tuple(scales.shape) != (E, N, K // group) or expert_offsets.numel() != E + 1:
        raise ValueError("shape mismatch between x_sorted, qweight, scales and expert_offsets")
    if out is None:
        out = torch.empty((R, N), dtype=torch.float16, device=x_sorted.device)
    else:
        _need(out, "out", torch.float16, 2)
    st = _stream(x_sorted.device)
    nb = workspace_bytes(R, N, K, group, E)
    ws = _workspace(x_sorted.device, st, nb)
    _check(lib().w4a16_grouped_linear(_ptr(x_sorted), _ptr(qweight), _ptr(scales), _ptr(expert_offsets),
                                      _ptr(out), E, R, N, K, group,
                                      _ptr(ws) if ws is not None else None, ws.numel() if ws is not None else 0,
                                      st), "w4a16_grouped_linear")
    return out


def grouped_linear_gather(x: torch.Tensor, token_of_row: torch.Tensor, qweight: torch.Tensor, scales: torch.Tensor,
                          expert_offsets: torch.Tensor, group: int = 32,
                          out: torch.Tensor | None = None) -> torch.Tensor:
    """Routed experts reading their rows straight from the token-major x:
    y_sorted[r] = x[token_of_row[r]] W_e^T for the expert e of row r. x fp16
    [T, K]; token_of_row int32 [R] (from moe_dispatch); qweight uint8
    [E, N, K/2]; scales fp16 [E, N, K/group] (group 32); expert_offsets int32
    [E+1]. The same bits as grouped_linear on the gathered rows."""
    _need(x, "x", torch.float16, 2)
    _need(token_of_row, "token_of_row", torch.int32, 1)
    _need(qweight, "qweight", torch.uint8, 3)
    _need(scales, "scales", torch.float16, 3)
    _need(expert_offsets, "expert_offsets", torch.int32, 1)
    T, K = x.shape
    R = token_of_row.shape[0]
    E, N = qweight.shape[0], qweight.shape[1]
    if qweight.shape[2] * 2 != K or tuple(scales.shape) != (E, N, K // group) or expert_offsets.numel() != E + 1:
        raise ValueError("shape mismatch between x, qweight, scales and expert_offsets")
    if out is None:
        out = torch.empty((R, N), dtype=torch.float16, device=x.device)
    else:
        _need(out, "out", torch.float16, 2)
        if tuple(out.shape) != (R, N):
            raise ValueError("out must be [R, N]")
    _check(lib().w4a16_grouped_linear_gather(_ptr(x), T, _ptr(token_of_row), _ptr(qweight), _ptr(scales),
                                             _ptr(expert_offsets), _ptr(out), E, R, N, K, group,
                                             _stream(x.device)), "w4a16_grouped_linear_gather")
    return out


def moe_route(logits: torch.Tensor, top_k: int, renormalize: bool = True):
    """Softmax top-k router: logits fp32 [T, E] -> (topk_ids int32 [T, top_k],
    topk_weights fp32 [T, top_k])."""
    _need(logits, "logits", torch.float32, 2)
    T, E = logits.shape
    ids = torch.empty((T, top_k), dtype=torch.int32, device=logits.device)
    w = torch.empty((T, top_k), dtype=torch.float32, device=logits.device)
    _check(lib().w4a16_moe_route(_ptr(logits), T, E, top_k, 1 if renormalize else 0, _ptr(ids), _ptr(w),
                                 _stream(logits.device)), "w4a16_moe_route")
    return ids, w


def moe_dispatch(topk_ids: torch.Tensor, E: int, x: torch.Tensor | None = None):
    """Expert-major order of the (token, slot) pairs: returns (expert_offsets int32
    [E+1], row_of int32 [T, top_k], token_of_row int32 [T*top_k], x_sorted fp16
    [T*top_k, K] or None when x is None)."""
    _need(topk_ids, "topk_ids", torch.int32, 2)
    T, k = topk_ids.shape
    dev = topk_ids.device
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    row_of = torch.empty((T, k), dtype=torch.int32, device=dev)
    token_of_row = torch.empty(T * k, dtype=torch.int32, device=dev)
    x_sorted, K = None, 0
    if x is not None:
        _need(x, "x", torch.float16, 2)
        if x.shape[0] != T:
            raise ValueError("x must have one row per token")
        K = x.shape[1]
        x_sorted = torch.empty((T * k, K), dtype=torch.float16, device=dev)
    nb = int(lib().w4a16_moe_dispatch_workspace_bytes(T, k, E))
    ws = torch.empty(nb, dtype=torch.uint8, device=dev) if nb else None
    _check(lib().w4a16_moe_dispatch(_ptr(topk_ids), T, k, E, _ptr(x) if x is not None else None, K,
                                    _ptr(offsets), _ptr(row_of), _ptr(token_of_row),
                                    _ptr(x_sorted) if x_sorted is not None else None,
                                    _ptr(ws) if ws is not None else None, nb, _stream(dev)), "w4a16_moe_dispatch")
    return offsets, row_of, token_of_row, x_sorted


def moe_combine(y_sorted: torch.Tensor, row_of: torch.Tensor, topk_weights: torch.Tensor,
                out: torch.Tensor | None = None) -> torch.Tensor:
    """y[t] = sum_j topk_weights[t, j] * y_sorted[row_of[t, j]] (fp32 sum, fp16 result)."""
    _need(y_sorted, "y_sorted", torch.float16, 2)
    _need(row_of, "row_of", torch.int32, 2)
    _need(topk_weights, "topk_weights", torch.float32, 2)
    if tuple(topk_weights.shape) != tuple(row_of.shape):
        raise ValueError("row_of and topk_weights must both be [T, top_k]")
    T, k = row_of.shape
    R, N = y_sorted.shape
    if out is None:
        out = torch.empty((T, N), dtype=torch.float16, device=y_sorted.device)
    else:
        _need(out, "out", torch.float16, 2)
        if tuple(out.shape) != (T, N):
            raise ValueError("out must be [T, N]")
    _check(lib().w4a16_moe_combine(_ptr(y_sorted), R, _ptr(row_of), _ptr(topk_weights), T, k, N, _ptr(out),
                                   _stream(y_sorted.device)), "w4a16_moe_combine")
    return out


def device_status(raise_on_error: bool = True) -> int:
    """Synchronizes the current stream and reads/clears the device error word."""
    st = _stream(torch.device("cuda", torch.cuda.current_device()))
    status = int(lib().w4a16_device_status(st))
    if raise_on_error:
        _check(status, "device")
    return status
