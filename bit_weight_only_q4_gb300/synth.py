"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle.

This module only draws random numbers and stores them in the two weight layouts;
it holds none of the arithmetic of the dequantise-and-multiply path.  The random
source is numpy's PCG64 bit generator (O'Neill, "PCG: A Family of Simple Fast
Space-Efficient Statistically Good Algorithms for Random Number Generation",
2014) seeded through ``numpy.random.SeedSequence``; normals come from numpy's
``standard_normal``.  Both are platform independent, so x86 and Arm hosts draw
identical inputs.  Conversions to bf16 / fp16 / float8_e4m3fn are library
round-to-nearest-even casts (torch / numpy).

Value distributions follow the workloads the pages describe for a speech-token
LLM's decode projections:
  * int4-g128-minmax ("rumik-oss-1-int4", "Format"): codes uniform 0..15 (a
    uniform random byte holds two independent uniform nibbles), fp16 scale
    U[1e-3, 2e-2], fp16 min = -7.5 * scale * U[0.8, 1.2].
  * NVFP4 weight-only ("VoxCPM2 NVFP4 (GPTQ)", "NVFP4 settings"): codes uniform
    over the 16 E2M1 bit patterns, e4m3 group-16 scales from U[0.25, 4], fp32
    global scale 1e-2.
  * activations bf16 ~ N(0, 1); the restricted audio head bf16 ~ N(0, 0.02)
    (0.02 read as the standard deviation).

Every array is returned on the CPU: uint8 for packed codes and e4m3 scales, uint16
for the bit patterns of fp16 / bf16 values, float32 for the global scale.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


def rng_for(*key: int) -> np.random.Generator:
    """A PCG64 generator keyed by a tuple of non-negative ints (seed, layer, ...)."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(list(key))))


def _to_bf16_bits(a: np.ndarray) -> np.ndarray:
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def _to_e4m3_bits(a: np.ndarray) -> np.ndarray:
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy().copy()


def activations(rng: np.random.Generator, M: int, K: int, std: float = 1.0) -> np.ndarray:
    """bf16 bits [M, K] drawn from N(0, std^2)."""
    return _to_bf16_bits(rng.standard_normal((M, K), dtype=np.float32) * np.float32(std))


@dataclass
class Int4Matrix:
    qweight: np.ndarray          # uint8 [N, K/2], low nibble = even column
    scale: np.ndarray            # uint16 fp16 bits [N, K/128]
    minv: np.ndarray             # uint16 fp16 bits [N, K/128]

    @property
    def N(self) -> int:
        return self.qweight.shape[0]

    @property
    def K(self) -> int:
        return 2 * self.qweight.shape[1]


@dataclass
class Nvfp4Matrix:
    codes: np.ndarray            # uint8 [N, K/2], low nibble = even column
    scale: np.ndarray            # uint8 e4m3 bits [N, K/16]
    global_scale: np.float32 = field(default_factory=lambda: np.float32(1e-2))

    @property
    def N(self) -> int:
        return self.codes.shape[0]

    @property
    def K(self) -> int:
        return 2 * self.codes.shape[1]


def int4_matrix(rng: np.random.Generator, N: int, K: int) -> Int4Matrix:
    if K % 128:
        raise ValueError("int4-g128 needs K % 128 == 0")
    q = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    s = rng.uniform(1e-3, 2e-2, size=(N, K // 128)).astype(np.float16)
    mn = (-7.5 * s.astype(np.float64) * rng.uniform(0.8, 1.2, size=s.shape)).astype(np.float16)
    return Int4Matrix(q, s.view(np.uint16).copy(), mn.view(np.uint16).copy())


def nvfp4_matrix(rng: np.random.Generator, N: int, K: int,
                 global_scale: float = 1e-2) -> Nvfp4Matrix:
    if K % 16:
        raise ValueError("NVFP4 needs K % 16 == 0")
    q = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    s = _to_e4m3_bits(rng.uniform(0.25, 4.0, size=(N, K // 16)))
    return Nvfp4Matrix(q, s, np.float32(global_scale))


@dataclass
class Int8Matrix:
    qweight: np.ndarray          # int8 [N, K]
    scale: np.ndarray            # uint16 fp16 bits [N]

    @property
    def N(self) -> int:
        return self.qweight.shape[0]

    @property
    def K(self) -> int:
        return self.qweight.shape[1]


def int8_matrix(rng: np.random.Generator, N: int, K: int) -> Int8Matrix:
    """INT8 weight-only matrix: codes uniform over -128..127, fp16 row scales
    U[2e-4, 1e-3] (a weight's absolute maximum over 127 for weights ~ N(0, 0.02))."""
    q = rng.integers(-128, 128, size=(N, K), dtype=np.int8)
    s = rng.uniform(2e-4, 1e-3, size=N).astype(np.float16)
    return Int8Matrix(q, s.view(np.uint16).copy())


def head_matrix(rng: np.random.Generator, rows: int = 2049, hidden: int = 2048,
                std: float = 0.02) -> np.ndarray:
    """bf16 bits [rows, hidden] of the restricted audio head."""
    return activations(rng, rows, hidden, std)


# ------------------------------------------------------------------ workloads
# Each workload is named by what it is and its sizes; the seed is part of it.

INT4_GEMV_2048 = dict(name="int4-g128 GEMV M=1 N=2048 K=2048", seed=0, M=1, N=2048, K=2048)
INT8_GEMV_16384 = dict(name="int8 weight-only GEMV M=1 N=16384 K=2048", seed=5, M=1,
                       N=16384, K=2048)
NVFP4_GEMV_16384 = dict(name="nvfp4 GEMV M=1 N=16384 K=2048", seed=1, M=1, N=16384, K=2048)
DECODE_STACK_28 = dict(name="int4-g128 decode step, 28 layers, hidden 2048, ffn 8192, "
                            "restricted head 2049x2048", seed=2, layers=28, hidden=2048,
                       ffn=8192, head_rows=2049)
NVFP4_BATCHED_48 = dict(name="nvfp4 batched decode M=48, 2048->8192 and 8192->2048",
                        seed=3, M=48, shapes=((8192, 2048), (2048, 8192)),
                        m_sweep=(1, 3, 8, 16, 32, 48))
PREFILL_2048 = dict(name="prefill M=2048, 2048->8192 and 8192->2048, int4-g128 and nvfp4",
                    seed=4, M=2048, shapes=((8192, 2048), (2048, 8192)))

# Projections of one synthetic decode layer: (name, N, K).  q/k/v/o are
# hidden x hidden, gate/up expand to the FFN width, down contracts back.
DECODE_LAYER_PROJS = (("q", 2048, 2048), ("k", 2048, 2048), ("v", 2048, 2048),
                      ("o", 2048, 2048), ("gate", 8192, 2048), ("up", 8192, 2048),
                      ("down", 2048, 8192))


def int4_gemv_2048():
    c = INT4_GEMV_2048
    rng = rng_for(c["seed"])
    w = int4_matrix(rng, c["N"], c["K"])
    x = activations(rng, c["M"], c["K"])
    return x, w


def int8_gemv_16384():
    c = INT8_GEMV_16384
    rng = rng_for(c["seed"])
    w = int8_matrix(rng, c["N"], c["K"])
    x = activations(rng, c["M"], c["K"])
    return x, w


def nvfp4_gemv_16384():
    c = NVFP4_GEMV_16384
    rng = rng_for(c["seed"])
    w = nvfp4_matrix(rng, c["N"], c["K"])
    x = activations(rng, c["M"], c["K"])
    return x, w


def decode_stack_layer(layer: int):
    """The seven int4 matrices of one layer of the synthetic decode stack."""
    seed = DECODE_STACK_28["seed"]
    return {name: int4_matrix(rng_for(seed, 1, layer, i), N, K)
            for i, (name, N, K) in enumerate(DECODE_LAYER_PROJS)}


def decode_stack_head():
    seed = DECODE_STACK_28["seed"]
    return head_matrix(rng_for(seed, 2), DECODE_STACK_28["head_rows"],
                       DECODE_STACK_28["hidden"])


def decode_stack_input():
    seed = DECODE_STACK_28["seed"]
    return activations(rng_for(seed, 3), 1, DECODE_STACK_28["hidden"])


def nvfp4_batched(shape_index: int, M: int):
    c = NVFP4_BATCHED_48
    N, K = c["shapes"][shape_index]
    w = nvfp4_matrix(rng_for(c["seed"], shape_index), N, K)
    x = activations(rng_for(c["seed"], shape_index, M), M, K)
    return x, w


def prefill(layout: str, shape_index: int, M: int | None = None):
    c = PREFILL_2048
    N, K = c["shapes"][shape_index]
    M = c["M"] if M is None else M
    lay = 0 if layout == "int4" else 1
    wrng = rng_for(c["seed"], lay, shape_index)
    w = int4_matrix(wrng, N, K) if layout == "int4" else nvfp4_matrix(wrng, N, K)
    x = activations(rng_for(c["seed"], lay, shape_index, 1), M, K)
    return x, w
