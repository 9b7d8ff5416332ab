"""Byte accounting of the two 4-bit weight layouts (host-side, no GPU).

int4-g128-minmax ("rumik-oss-1-int4", "Format"): 4-bit codes plus an fp16 scale
and an fp16 min per 128 columns of a row.  NVFP4 weight-only ("VoxCPM2 NVFP4
(GPTQ)", "NVFP4 settings"): 4-bit E2M1 codes plus one e4m3 scale per 16 columns
and one fp32 global scale per matrix.  INT8 weight-only (the reading of "Rumik
TTS Fast Inference", "What Made It Faster"): int8 codes plus one fp16 scale per
row.  These are the algorithmic bytes a
weight-streaming kernel must move; the benchmark divides them by time.
"""
from __future__ import annotations

INT4_GROUP = 128
NVFP4_GROUP = 16


def int4_bytes_per_weight() -> float:
    return 0.5 + 2 * 2 / INT4_GROUP


def nvfp4_bytes_per_weight() -> float:
    return 0.5 + 1 / NVFP4_GROUP


def weight_bytes(layout: str, N: int, K: int) -> int:
    """Bytes of one packed weight matrix [N, K] in the given layout."""
    if layout == "int4":
        return N * K // 2 + 2 * 2 * N * (K // INT4_GROUP)
    if layout == "nvfp4":
        return N * K // 2 + N * (K // NVFP4_GROUP) + 4
    if layout == "int8":                  # int8 codes + one fp16 scale per row
        return N * K + 2 * N
    raise ValueError(layout)


def linear_bytes(layout: str, M: int, N: int, K: int) -> int:
    """Algorithmic bytes of one call y[M,N] = x[M,K] W^T: packed weights once,
    bf16 activations in, bf16 outputs out."""
    return weight_bytes(layout, N, K) + 2 * M * K + 2 * M * N


def head_bytes(M: int, rows: int, hidden: int) -> int:
    """Bytes of the restricted head: bf16 rows read once, bf16 h in, bf16 out."""
    return 2 * rows * hidden + 2 * M * hidden + 2 * M * rows
