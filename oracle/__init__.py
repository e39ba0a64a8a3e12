"""CPU oracle for the W4A16 group-quantized linear layer (fp64, plain C).

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg may import this package; the product path never does. The C
source (``oracle.c``) shares no code with the CUDA library.

What it follows: the LLM170 page, introduction ("W4A16 (int4 sym g128, f16
activations)", group 32 for the MoE models) and its Repository layout section
(GPU kernel outputs must match the CPU reference quant lane). The quantizer
(s = fp16(max|w|/7), q = clamp(rint(w/s), -8, 7), nibble q+8, even k in the
low nibble) is the workload specification's reading of "int4 sym".

The block-format functions (``blocks_*``) decode the GGUF block types Q4_K
and Q5_1 that the infr README lists among its validated formats ("Also
validated for correctness"; footnote 3 for Q5_1 expert banks), in the ggml
layouts the C source describes, and form y = x W^T from them in fp64.

The routed-MoE functions (``moe_route``, ``moe_dispatch``, ``moe_gather``,
``moe_combine``) are numpy fp64: the softmax top-k router the infr README's
model table names, the expert-major permutation, and the router-weighted sum
of the selected experts' outputs.

Every function here is pinned by ``tests/test_oracle.py`` against closed
forms, exact rational arithmetic, numpy's own binary16 conversion and the
hand-worked fixtures in ``tests/golden/``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

_CFLAGS = ["-std=c99", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc into oracle/_build/liboracle.so."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".{os.getpid()}.tmp"
        subprocess.run(["gcc", *_CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _SO)
    return _SO


def _bind(path: str):
    """Load a compiled oracle library and declare its C signatures."""
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    I32 = ctypes.c_int32
    lib.oracle_half_to_double_n.argtypes = [P, I64, P]
    lib.oracle_float_to_half_rn_n.argtypes = [P, I64, P]
    lib.oracle_quantize.argtypes = [P, I64, I64, I32, P, P]
    lib.oracle_unpack.argtypes = [P, I64, I64, P]
    lib.oracle_pack_q.argtypes = [P, I64, I64, P]
    lib.oracle_dequantize.argtypes = [P, I64, I64, I64, I32, P]
    lib.oracle_linear.argtypes = [P, P, P, I64, I64, I64, I32, P, P]
    lib.oracle_grouped_linear.argtypes = [P, P, P, P, I32, I64, I64, I64, I32, P, P]
    lib.oracle_blocks_row_bytes.argtypes = [I32, I64]
    lib.oracle_blocks_row_bytes.restype = I64
    lib.oracle_blocks_decode.argtypes = [I32, P, I64, I64, P]
    lib.oracle_blocks_decode_f32.argtypes = [I32, P, I64, I64, P]
    lib.oracle_blocks_linear.argtypes = [I32, P, P, I64, I64, I64, P, P]
    for f in (lib.oracle_half_to_double_n, lib.oracle_float_to_half_rn_n,
              lib.oracle_quantize, lib.oracle_unpack, lib.oracle_pack_q,
              lib.oracle_dequantize, lib.oracle_linear, lib.oracle_grouped_linear,
              lib.oracle_blocks_decode, lib.oracle_blocks_decode_f32, lib.oracle_blocks_linear):
        f.restype = None
    return lib


def compile_variant(src_text: str, out_dir: str) -> str:
    """Compile C source text with the oracle's flags (used by the mutation tests)."""
    src = os.path.join(out_dir, "variant.c")
    so = os.path.join(out_dir, "libvariant.so")
    with open(src, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", *_CFLAGS, "-o", so, src, "-lm"], check=True)
    return so


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(build())
    return _lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def half_bits(x) -> np.ndarray:
    """fp16 array (or uint16 bits) -> uint16 bit patterns, no arithmetic."""
    a = np.asarray(x)
    if a.dtype == np.float16:
        return np.ascontiguousarray(a).view(np.uint16)
    return _c(a, np.uint16)


def half_to_double(bits) -> np.ndarray:
    b = half_bits(bits)
    out = np.empty(b.shape, np.float64)
    _load().oracle_half_to_double_n(_p(b), b.size, _p(out))
    return out


def float_to_half_bits(f) -> np.ndarray:
    a = _c(f, np.float32)
    out = np.empty(a.shape, np.uint16)
    _load().oracle_float_to_half_rn_n(_p(a), a.size, _p(out))
    return out


def quantize(w: np.ndarray, group: int):
    """fp32 [N, K] -> (qw uint8 [N, K/2], s fp16-bits uint16 [N, K/group])."""
    w = _c(w, np.float32)
    N, K = w.shape
    assert K % group == 0 and K % 2 == 0
    qw = np.empty((N, K // 2), np.uint8)
    s = np.empty((N, K // group), np.uint16)
    _load().oracle_quantize(_p(w), N, K, group, _p(qw), _p(s))
    return qw, s


def unpack(qw: np.ndarray, K: int) -> np.ndarray:
    qw = _c(qw, np.uint8)
    N = qw.shape[0]
    q = np.empty((N, K), np.int8)
    _load().oracle_unpack(_p(qw), N, K, _p(q))
    return q


def pack_q(q: np.ndarray) -> np.ndarray:
    q = _c(q, np.int8)
    N, K = q.shape
    qw = np.empty((N, K // 2), np.uint8)
    _load().oracle_pack_q(_p(q), N, K, _p(qw))
    return qw


def dequantize(qw: np.ndarray, s: np.ndarray, K: int, group: int) -> np.ndarray:
    qw = _c(qw, np.uint8)
    s = half_bits(s)
    N = qw.shape[0]
    out = np.empty((N, K), np.float64)
    _load().oracle_dequantize(_p(qw), _p(s), N, K, group, _p(out))
    return out


def linear(x, qw, s, group: int, threads: int = 1):
    """y = x @ W^T in fp64 and sum_k |x W^| ; x fp16 [M, K]. Returns (y, absdot).

    ``threads > 1`` splits the output columns n over threads (each element's
    sum is computed exactly as in the single-threaded case)."""
    xb = half_bits(x)
    M, K = xb.shape
    qw = _c(qw, np.uint8)
    s = half_bits(s)
    N = qw.shape[0]
    assert qw.shape == (N, K // 2) and s.shape == (N, K // group)
    if threads <= 1 or N < 2 * threads:
        y = np.empty((M, N), np.float64)
        a = np.empty((M, N), np.float64)
        _load().oracle_linear(_p(xb), _p(qw), _p(s), M, N, K, group, _p(y), _p(a))
        return y, a
    lib = _load()
    bounds = np.linspace(0, N, threads + 1).astype(np.int64)

    def part(i):
        n0, n1 = int(bounds[i]), int(bounds[i + 1])
        qs, ss = np.ascontiguousarray(qw[n0:n1]), np.ascontiguousarray(s[n0:n1])
        yp = np.empty((M, n1 - n0), np.float64)
        ap = np.empty((M, n1 - n0), np.float64)
        lib.oracle_linear(_p(xb), _p(qs), _p(ss), M, n1 - n0, K, group, _p(yp), _p(ap))
        return yp, ap

    with ThreadPoolExecutor(threads) as ex:
        parts = list(ex.map(part, range(threads)))
    return np.concatenate([p[0] for p in parts], 1), np.concatenate([p[1] for p in parts], 1)


def grouped_linear(x, qw, s, offsets, group: int):
    """Routed-expert linear over expert-sorted rows. x fp16 [R, K], qw [E, N, K/2],
    s [E, N, K/g], offsets int32 [E+1]. Returns (y, absdot) fp64 [R, N]."""
    xb = half_bits(x)
    R, K = xb.shape
    qw = _c(qw, np.uint8)
    s = half_bits(s)
    off = _c(offsets, np.int32)
    E, N = qw.shape[0], qw.shape[1]
    assert off.shape == (E + 1,) and off[0] == 0 and off[-1] == R
    y = np.zeros((R, N), np.float64)
    a = np.zeros((R, N), np.float64)
    _load().oracle_grouped_linear(_p(xb), _p(qw), _p(s), _p(off), E, R, N, K, group, _p(y), _p(a))
    return y, a


# ----------------------------------------------------------------------------
# GGUF block formats (format codes as in oracle.c)

BLOCK_FORMATS = {"q4_k": 1, "q5_1": 2}


def _fmt(fmt) -> int:
    return BLOCK_FORMATS[fmt] if isinstance(fmt, str) else int(fmt)


def blocks_row_bytes(fmt, K: int) -> int:
    """Bytes of one row of K weights in a block format (-1: not whole blocks)."""
    return int(_load().oracle_blocks_row_bytes(_fmt(fmt), K))


def _blocks(fmt, w, K: int) -> np.ndarray:
    w = _c(w, np.uint8)
    rb = blocks_row_bytes(fmt, K)
    if rb < 0 or w.ndim != 2 or w.shape[1] != rb:
        raise ValueError(f"blocks: expected uint8 [N, {rb}] for K={K}")
    return w


def blocks_decode(fmt, w, K: int) -> np.ndarray:
    """W^ fp64 [N, K] from the block bytes uint8 [N, row_bytes]."""
    w = _blocks(fmt, w, K)
    out = np.empty((w.shape[0], K), np.float64)
    _load().oracle_blocks_decode(_fmt(fmt), _p(w), w.shape[0], K, _p(out))
    return out


def blocks_decode_f32(fmt, w, K: int) -> np.ndarray:
    """W^ fp32 [N, K] as a CPU dequantizer forms it: a * q + b with the step a
    and offset b in fp32, rounded once."""
    w = _blocks(fmt, w, K)
    out = np.empty((w.shape[0], K), np.float32)
    _load().oracle_blocks_decode_f32(_fmt(fmt), _p(w), w.shape[0], K, _p(out))
    return out


def blocks_linear(fmt, x, w, threads: int = 1):
    """y = x W^T in fp64 for block-format weights; x fp16 [M, K], w uint8
    [N, row_bytes]. Returns (y, absterm), absterm = sum_k |x| (|a q| + |b|)
    for W^ = a q + b: the size of what a kernel adds up, which takes the place
    of sum_k |x W^| in tolerance(). ``threads > 1`` splits the rows n."""
    xb = half_bits(x)
    M, K = xb.shape
    w = _blocks(fmt, w, K)
    N = w.shape[0]
    lib, f = _load(), _fmt(fmt)
    if threads <= 1 or N < 2 * threads:
        y = np.empty((M, N), np.float64)
        a = np.empty((M, N), np.float64)
        lib.oracle_blocks_linear(f, _p(xb), _p(w), M, N, K, _p(y), _p(a))
        return y, a
    bounds = np.linspace(0, N, threads + 1).astype(np.int64)

    def part(i):
        n0, n1 = int(bounds[i]), int(bounds[i + 1])
        wp = np.ascontiguousarray(w[n0:n1])
        yp = np.empty((M, n1 - n0), np.float64)
        ap = np.empty((M, n1 - n0), np.float64)
        lib.oracle_blocks_linear(f, _p(xb), _p(wp), M, n1 - n0, K, _p(yp), _p(ap))
        return yp, ap

    with ThreadPoolExecutor(threads) as ex:
        parts = list(ex.map(part, range(threads)))
    return np.concatenate([p[0] for p in parts], 1), np.concatenate([p[1] for p in parts], 1)


def tolerance(y_ref: np.ndarray, absdot: np.ndarray) -> np.ndarray:
    """Per-element bound |y - y_ref| <= 2^-9 |y_ref| + 1e-4 sum_k |x_k W^_nk| + 2^-25.

    The first two terms are the workload's bound. The last is the final
    rounding of y to fp16 where the first term cannot cover it: below 2^-14
    binary16 values are spaced a fixed 2^-24 apart, so even the correctly
    rounded exact result can be 2^-25 away (relative to such a y that is far
    more than 2^-9). It matters only when sum_k |x W^| is tiny too."""
    return np.ldexp(np.abs(y_ref), -9) + 1e-4 * absdot + np.ldexp(1.0, -25)


def silu(v):
    """SiLU(v) = v / (1 + e^(-v)) in fp64: the activation of the gated MLP
    (rust-inference page, list of accuracy fixes, item 5: the SiLU-activated
    gate projection multiplies the up projection)."""
    v = np.asarray(v, dtype=np.float64)
    with np.errstate(over="ignore"):
        return v / (1.0 + np.exp(-v))


def gated_linear(x, qw_gate, s_gate, qw_up, s_up, group: int, threads: int = 1):
    """y = silu(x Wg^T) * (x Wu^T) in fp64, the two projections as linear()
    forms them. Returns (y, g, u, absdot_g, absdot_u)."""
    g, ag = linear(x, qw_gate, s_gate, group, threads)
    u, au = linear(x, qw_up, s_up, group, threads)
    return silu(g) * u, g, u, ag, au


def gated_tolerance(g, u, absdot_g, absdot_u):
    """Per-element bound on |y - y_ref| for a kernel whose g and u each meet
    the linear bound (tolerance()) and which evaluates silu(g) * u in fp32 and
    rounds once to fp16. First-order propagation with |silu'| <= 1.1 on the
    real line, the cross term of the two errors, and 2^-9 |y| + 2^-25 for the
    fp32 evaluation and the final rounding: rounding to fp16 errs by at most
    half a unit in the last place, 2^-11 |y| for normal values and the
    absolute 2^-25 (half the subnormal spacing 2^-24) below 2^-14, where
    silu(g) * u lands when g and u are both small."""
    eg = tolerance(g, absdot_g)
    eu = tolerance(u, absdot_u)
    y = silu(g) * u
    return (1.1 * eg * np.abs(u) + np.abs(silu(g)) * eu + 1.1 * eg * eu + np.ldexp(np.abs(y), -9)
            + np.ldexp(1.0, -25))



# ----------------------------------------------------------------------------
# Routed-MoE dispatch around the grouped layer. The pages name the router
# ("softmax router, top-k experts" for Qwen3 MoE and "8-of-128 routed" for the
# Gemma 4 MoE in the infr README's model table) and run the experts "MoE
# resident" at group 32 (LLM170 page, benchmark table). The permutation and the
# weighted combine are the plain reading of a routed layer: each token's output
# is the router-weighted sum of its selected experts' outputs.


def moe_route(logits, top_k: int, renormalize: bool = True):
    """Softmax router: for each token the top_k experts by logit (ties go to the
    lower expert index) and their softmax probabilities as weights, divided by
    their sum when ``renormalize``. The selection compares the fp32 logits
    themselves; the probabilities are fp64. Returns (ids int32 [T, top_k],
    weights fp64 [T, top_k], max_shift fp64 [T]) where max_shift is the largest
    |l - max l| over the row (it enters the error bound of an fp32 softmax)."""
    lf = np.asarray(logits, dtype=np.float32)
    T, E = lf.shape
    if not 1 <= top_k <= E:
        raise ValueError("need 1 <= top_k <= E")
    l64 = lf.astype(np.float64)
    ids = np.argsort(-l64, axis=1, kind="stable")[:, :top_k].astype(np.int32)
    shifted = l64 - l64.max(axis=1, keepdims=True)
    p = np.exp(shifted)
    p /= p.sum(axis=1, keepdims=True)
    w = np.take_along_axis(p, ids.astype(np.int64), axis=1)
    if renormalize:
        w = w / w.sum(axis=1, keepdims=True)
    return ids, w, np.abs(shifted).max(axis=1)


def moe_dispatch(ids, E: int):
    """Expert-major order of the (token t, slot j) pairs: rows sorted by
    (expert, t, j). Returns (expert_offsets int32 [E+1], row_of int32 [T, k]
    (the row of pair (t, j)), token_of_row int32 [R]) with R = T k."""
    ids = np.asarray(ids)
    T, k = ids.shape
    flat = ids.reshape(-1).astype(np.int64)
    if flat.size and (flat.min() < 0 or flat.max() >= E):
        raise ValueError("expert id out of range")
    order = np.argsort(flat, kind="stable")          # pair index t*k + j, stable within an expert
    offsets = np.zeros(E + 1, np.int64)
    offsets[1:] = np.cumsum(np.bincount(flat, minlength=E))
    row_of = np.empty(T * k, np.int64)
    row_of[order] = np.arange(T * k)
    return offsets.astype(np.int32), row_of.reshape(T, k).astype(np.int32), (order // k).astype(np.int32)


def moe_gather(x, token_of_row):
    """x_sorted[r] = x[token_of_row[r]] (a row copy)."""
    return np.asarray(x)[np.asarray(token_of_row, dtype=np.int64)]


def moe_combine(y_sorted, row_of, weights):
    """y[t] = sum_j weights[t, j] * y_sorted[row_of[t, j]] in fp64, y_sorted fp16.
    Returns (y, absdot) with absdot = sum_j |weights[t, j] * y_sorted[row_of[t, j]]|."""
    ys = half_to_double(half_bits(y_sorted))
    row_of = np.asarray(row_of, dtype=np.int64)
    w = np.asarray(weights, dtype=np.float64)
    T, k = row_of.shape
    y = np.zeros((T, ys.shape[1]), np.float64)
    a = np.zeros_like(y)
    for j in range(k):
        term = w[:, j:j + 1] * ys[row_of[:, j]]
        y += term
        a += np.abs(term)
    return y, a


def route_tolerance(w_ref, max_shift, E: int, top_k: int):
    """Bound on |w - w_ref| for weights computed in fp32: each exp(l - max) with
    its argument rounded (relative error <= 2^-24 |l - max|) and a few ulp of
    exp, an E-term fp32 sum, and up to three fp32 divisions."""
    eps = 2.0 ** -24
    return np.abs(w_ref) * eps * (np.asarray(max_shift)[:, None] + 2 * E + 2 * top_k + 16)


def combine_tolerance(y_ref, absdot, top_k: int):
    """Bound on |y - y_ref| for an fp32 weighted sum of top_k fp16 rows rounded
    once to fp16: the fp16 rounding (2^-11 relative, 2^-25 absolute below the
    normal range, doubled) and (top_k + 1) fp32 roundings of the running sum."""
    return np.ldexp(np.abs(y_ref), -10) + (top_k + 1) * 2.0 ** -23 * absdot + 2.0 ** -24
