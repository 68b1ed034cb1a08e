"""Seeded synthetic inputs: canonical weight blocks and fp32 activations.

This module draws random numbers and lays them out as canonical block bytes.
It holds none of the product's arithmetic (no dequantisation, no dot
products), so both the CUDA path and the CPU oracle may use it.

Canonical block layouts (little-endian), per format:
    Q4_0      18 B / 32 weights : [d fp16][qs 16 B]        two 4-bit q per byte
    Q8_0      34 B / 32 weights : [d fp16][32 x int8]
    I8_B64    66 B / 64 weights : [d fp16][64 x int8]
    Q6_K     210 B / 256 weights: [ql 128 B][qh 64 B][sc 16 x int8][d fp16]

Value distributions (draw order per matrix: q, then d, then x):
    Q4_0   q ~ U{0..15}; d = fp16(|N(0,1)| * 0.02)
    Q8_0,
    I8_B64 q = clip(rint(N(0, 40)), -127, 127); d = fp16(|N(0,1)| * 0.002)
    Q6_K   6-bit q ~ U{0..63}; sc ~ U{-32..31}; d = fp16(|N(0,1)| * 0.001)
    x      fp32 ~ N(0, 1)
Uniform 4-bit q are drawn as uniform bytes (each byte holds two independent
U{0..15} values); Q6_K's ql and qh planes are uniform bytes, which makes every
6-bit q uniform on 0..63 whatever the bit assignment.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

Q4_0, Q8_0, I8_B64, Q6_K = 0, 1, 2, 3
FORMAT_NAMES = {Q4_0: "q4_0", Q8_0: "q8_0", I8_B64: "i8_b64", Q6_K: "q6_k"}
BLOCK_ELEMS = {Q4_0: 32, Q8_0: 32, I8_B64: 64, Q6_K: 256}
BLOCK_BYTES = {Q4_0: 18, Q8_0: 34, I8_B64: 66, Q6_K: 210}


def canonical_bytes(fmt: int, N: int, K: int) -> int:
    """Size of an N x K matrix in canonical blocks."""
    return N * (K // BLOCK_ELEMS[fmt]) * BLOCK_BYTES[fmt]


def _fp16_bytes(d: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(d.astype("<f2")).view(np.uint8).reshape(d.shape + (2,))


def gen_weights(fmt: int, N: int, K: int, rng: np.random.Generator) -> np.ndarray:
    """Canonical block bytes for an N x K weight matrix, shape [N, row_bytes]."""
    be, bb = BLOCK_ELEMS[fmt], BLOCK_BYTES[fmt]
    if K % be:
        raise ValueError("K=%d is not a multiple of the block size %d" % (K, be))
    nb = K // be
    out = np.empty((N, nb, bb), dtype=np.uint8)
    if fmt == Q4_0:
        qs = rng.integers(0, 256, size=(N, nb, 16), dtype=np.uint8)
        d = (np.abs(rng.standard_normal((N, nb))) * 0.02).astype(np.float16)
        out[..., 0:2] = _fp16_bytes(d)
        out[..., 2:] = qs
    elif fmt in (Q8_0, I8_B64):
        q = np.clip(np.rint(rng.normal(0.0, 40.0, size=(N, nb, be))), -127, 127).astype(np.int8)
        d = (np.abs(rng.standard_normal((N, nb))) * 0.002).astype(np.float16)
        out[..., 0:2] = _fp16_bytes(d)
        out[..., 2:] = q.view(np.uint8)
    elif fmt == Q6_K:
        ql = rng.integers(0, 256, size=(N, nb, 128), dtype=np.uint8)
        qh = rng.integers(0, 256, size=(N, nb, 64), dtype=np.uint8)
        sc = rng.integers(-32, 32, size=(N, nb, 16)).astype(np.int8)
        d = (np.abs(rng.standard_normal((N, nb))) * 0.001).astype(np.float16)
        out[..., 0:128] = ql
        out[..., 128:192] = qh
        out[..., 192:208] = sc.view(np.uint8)
        out[..., 208:210] = _fp16_bytes(d)
    else:
        raise ValueError("unknown format %r" % fmt)
    return out.reshape(N, nb * bb)


def gen_x(M: int, K: int, rng: np.random.Generator) -> np.ndarray:
    """fp32 activations x[M][K] ~ N(0, 1)."""
    return rng.standard_normal((M, K), dtype=np.float32)


def make_problem(fmt: int, N: int, K: int, M: int, seed):
    """(W canonical bytes [N, row_bytes], x [M, K] fp32) from one seed."""
    rng = np.random.default_rng(seed)
    W = gen_weights(fmt, N, K, rng)
    x = gen_x(M, K, rng)
    return W, x


# ---- the workloads: shapes of the models the engines serve ------------------

@dataclass(frozen=True)
class Linear:
    name: str
    fmt: int
    N: int
    K: int
    M: int
    seed: tuple

    @property
    def weight_bytes(self) -> int:
        return canonical_bytes(self.fmt, self.N, self.K)

    @property
    def algorithmic_bytes(self) -> int:
        """Packed weights + fp32 x + fp32 y: what the product must move."""
        return self.weight_bytes + 4 * self.M * (self.K + self.N)

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    def make(self):
        return make_problem(self.fmt, self.N, self.K, self.M, self.seed)


@dataclass(frozen=True)
class Workload:
    name: str
    linears: tuple = field(default_factory=tuple)

    @property
    def algorithmic_bytes(self) -> int:
        return sum(l.algorithmic_bytes for l in self.linears)

    @property
    def weight_bytes(self) -> int:
        return sum(l.weight_bytes for l in self.linears)


# SmolLM2-360M: hidden 960, 15 query heads / 5 KV heads of 64, MLP 2560, 32 layers.
SMOLLM2_360M_LAYER = (("q_proj", 960, 960), ("k_proj", 320, 960), ("v_proj", 320, 960),
                      ("o_proj", 960, 960), ("gate_proj", 2560, 960),
                      ("up_proj", 2560, 960), ("down_proj", 960, 2560))
TINYLLAMA_SHAPES = ((2048, 2048), (256, 2048), (5632, 2048), (2048, 5632))
QWEN25_3B_FFN_SHAPES = ((11008, 2048), (2048, 11008))
QWEN25_3B_FFN_BATCHES = (1, 4, 16, 64, 256)


def q4_0_gemv_960() -> Workload:
    """Q4_0 GEMV, M=1, N=960, K=960, seed 0."""
    return Workload("q4_0_gemv_960x960", (Linear("gemv", Q4_0, 960, 960, 1, (0,)),))


def smollm2_360m_decode_stack(layers: int = 32) -> Workload:
    """All Q4_0 linears of one SmolLM2-360M decode step (M=1), fresh x per linear."""
    lins = []
    for l in range(layers):
        for j, (nm, N, K) in enumerate(SMOLLM2_360M_LAYER):
            lins.append(Linear("layer%d.%s" % (l, nm), Q4_0, N, K, 1, (0, 2, l, j)))
    return Workload("smollm2_360m_q4_0_decode_stack_%dL" % layers, tuple(lins))


def tinyllama_gemv(fmt: int) -> Workload:
    """Q8_0 or I8_B64 GEMVs at TinyLlama-1.1B shapes, M=1."""
    lins = tuple(Linear("%dx%d" % (N, K), fmt, N, K, 1, (0, 3, i, fmt))
                 for i, (N, K) in enumerate(TINYLLAMA_SHAPES))
    return Workload("tinyllama_1.1b_%s_gemv" % FORMAT_NAMES[fmt], lins)


def qwen25_3b_ffn(M: int) -> Workload:
    """Q4_0 FFN GEMM at Qwen2.5-3B shapes with M activation rows."""
    lins = tuple(Linear("%dx%d_M%d" % (N, K, M), Q4_0, N, K, M, (0, 4, i, M))
                 for i, (N, K) in enumerate(QWEN25_3B_FFN_SHAPES))
    return Workload("qwen2.5_3b_ffn_q4_0_M%d" % M, lins)


def qwen25_3b_lm_head() -> Workload:
    """Q6_K lm_head GEMV, vocab 151936 x hidden 2048, M=1."""
    return Workload("qwen2.5_3b_lm_head_q6_k",
                    (Linear("lm_head", Q6_K, 151936, 2048, 1, (0, 5, 0, Q6_K)),))
