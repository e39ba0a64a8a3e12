"""Seeded synthetic inputs for the W4A16 linear layer (tests and benchmark).

This module draws random numbers and arranges them; it holds none of the
layer's arithmetic (no quantization, no dequantization, no dot products), so
both the CPU oracle and the CUDA path can take their inputs from it.

Recipes (one numpy PCG64 generator per call, seed 0 unless given; draws in
the fixed order W, then x, then routing):

* dense weights: fp32 ~ N(0, 0.02), shape [N, K] (quantized afterwards by
  whichever side is under test);
* activations: fp16 ~ N(0, 1), shape [M, K];
* prefill activations additionally get round(0.01 K) distinct "outlier"
  channels (columns of x) multiplied by 20 before the fp16 cast;
* routed MoE: each token picks ``top_k`` distinct experts uniformly at
  random; rows are the (expert, token) pairs sorted by expert, then token;
  ``offsets`` is the exclusive prefix sum of the per-expert row counts
  (empty experts allowed);
* raw packed weights: uniform random bytes (all 16 nibble values, including
  nibble 0, i.e. q = -8, which the quantizer never emits) with fp16 scales
  drawn as |N(0, 0.02)| / 7;
* GGUF block formats (Q4_K: 144-byte blocks of 256 weights; Q5_1: 24-byte
  blocks of 32): uniform random bytes for every block, then the two fp16
  fields at the start of each block replaced: Q4_K d ~ U(0.5, 2) 2^-12 and
  dmin ~ U(0.5, 2) 2^-13 (weights within about [-0.015, 0.46], spread 0.07,
  with the random 6-bit scales and minimums); Q5_1 d ~ U(0.5, 2) 2^-9 and m ~ -U(0.5, 2) 2^-5.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

# Workload shapes (M tokens, K input features, N output features, group).
CONFIG0 = dict(M=1, K=1024, N=256, group=128)
DECODE_SHAPES = [dict(K=5120, N=17408), dict(K=17408, N=5120)]  # gate/up, down
PREFILL_SHAPE = dict(K=5120, N=17408, group=128)
PREFILL_M = (512, 4096)
MOE = dict(E=128, tokens=4096, top_k=8, hidden=2048, inter=512, group=32)


def rng(seed: int = 0) -> np.random.Generator:
    return np.random.default_rng(np.random.PCG64(seed))


def weights(g: np.random.Generator, N: int, K: int, std: float = 0.02) -> np.ndarray:
    return g.normal(0.0, std, size=(N, K)).astype(np.float32)


def activations(g: np.random.Generator, M: int, K: int, outlier_frac: float = 0.0,
                outlier_gain: float = 20.0) -> np.ndarray:
    x = g.normal(0.0, 1.0, size=(M, K))
    if outlier_frac > 0.0:
        n_out = int(round(outlier_frac * K))
        cols = g.choice(K, size=n_out, replace=False)
        x[:, cols] *= outlier_gain
    return x.astype(np.float16)


def raw_packed(g: np.random.Generator, N: int, K: int, group: int):
    """Uniform random packed bytes and random positive fp16 scales."""
    qw = g.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    s = (np.abs(g.normal(0.0, 0.02, size=(N, K // group))) / 7.0).astype(np.float16)
    return qw, s


# GGUF block formats: (weights per block, bytes per block), and where the two
# fp16 fields of a block sit (bytes 0-1 and 2-3 in both formats).
BLOCK_FORMATS = {"q4_k": (256, 144), "q5_1": (32, 24)}


def raw_blocks(g: np.random.Generator, fmt: str, N: int, K: int) -> np.ndarray:
    """Random block bytes uint8 [N, K / weights_per_block * bytes_per_block]."""
    bw, bb = BLOCK_FORMATS[fmt]
    assert K % bw == 0
    nb = N * (K // bw)
    raw = g.integers(0, 256, size=(nb, bb), dtype=np.uint8)
    if fmt == "q4_k":
        f0 = g.uniform(0.5, 2.0, nb) * 2.0 ** -12
        f1 = g.uniform(0.5, 2.0, nb) * 2.0 ** -13
    else:
        f0 = g.uniform(0.5, 2.0, nb) * 2.0 ** -9
        f1 = -g.uniform(0.5, 2.0, nb) * 2.0 ** -5
    raw[:, 0:2] = f0.astype("<f2").view(np.uint8).reshape(nb, 2)
    raw[:, 2:4] = f1.astype("<f2").view(np.uint8).reshape(nb, 2)
    return raw.reshape(N, (K // bw) * bb)


@dataclass
class Routing:
    offsets: np.ndarray      # int32 [E+1]
    token_of_row: np.ndarray  # int64 [R], token index of each expert-sorted row
    expert_of_row: np.ndarray  # int64 [R]


def routing(g: np.random.Generator, tokens: int, E: int, top_k: int) -> Routing:
    keys = g.random((tokens, E))
    experts = np.argsort(keys, axis=1)[:, :top_k]          # distinct, uniform
    tok = np.repeat(np.arange(tokens), top_k)
    exp = experts.reshape(-1)
    order = np.lexsort((tok, exp))                          # by expert, then token
    counts = np.bincount(exp, minlength=E)
    offsets = np.zeros(E + 1, np.int64)
    offsets[1:] = np.cumsum(counts)
    return Routing(offsets.astype(np.int32), tok[order], exp[order])


def router_logits(g: np.random.Generator, tokens: int, E: int, std: float = 1.0) -> np.ndarray:
    """Router logits fp32 [tokens, E] ~ N(0, std); the pages give no distribution."""
    return g.normal(0.0, std, size=(tokens, E)).astype(np.float32)


def config0(seed: int = 0):
    """M=1, K=1024, N=256, group 128: W ~ N(0, 0.02) fp32, x ~ N(0, 1) fp16."""
    g = rng(seed)
    W = weights(g, CONFIG0["N"], CONFIG0["K"])
    x = activations(g, CONFIG0["M"], CONFIG0["K"])
    return W, x, CONFIG0["group"]


def decode(M: int, K: int, N: int, seed: int = 0):
    """Decode GEMV inputs (M = 1 or 4 independent rows), group 128."""
    g = rng(seed)
    W = weights(g, N, K)
    x = activations(g, M, K)
    return W, x, 128


def prefill(M: int, K: int = 5120, N: int = 17408, seed: int = 0):
    """Prefill GEMM inputs with 1% outlier channels scaled by 20, group 128."""
    g = rng(seed)
    W = weights(g, N, K)
    x = activations(g, M, K, outlier_frac=0.01)
    return W, x, 128


def moe(K: int, N: int, E: int = 128, tokens: int = 4096, top_k: int = 8, seed: int = 0):
    """Routed-expert inputs for one projection (K -> N per expert), group 32.

    Returns (W [E, N, K] fp32, x_sorted [R, K] fp16, Routing)."""
    g = rng(seed)
    W = g.normal(0.0, 0.02, size=(E, N, K)).astype(np.float32)
    x_tok = activations(g, tokens, K)
    r = routing(g, tokens, E, top_k)
    return W, np.ascontiguousarray(x_tok[r.token_of_row]), r
