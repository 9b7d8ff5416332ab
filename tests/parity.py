"""Helpers for GPU-vs-oracle parity tests: moving seeded inputs to the device and
checking outputs against the fp64 oracle with the stated tolerances.

Tolerance (per output element y[m,n], and over the whole output):
    |y_gpu - y_oracle| <= 1e-2 * sum_k |x[m,k] w[n,k]| + 1e-3
    ||y_gpu - y_oracle||_F / ||y_oracle||_F <= 2e-3
The oracle is the unrounded fp64 result; the GPU output is bf16.
"""
from __future__ import annotations

import numpy as np
import torch

REL_FRO = 2e-3
ABS_REL = 1e-2
ABS_ADD = 1e-3
FRO_MIN_ELEMS = 1024


# device upload helpers live in the package (bench.py uses them too)
from bit_weight_only_q4_gb300.upload import (bf16_bits_host, bf16_dev, f16_dev, int4_dev,  # noqa: F401
                                             int8_dev, nvfp4_dev, u8_dev)


def check(y_gpu: torch.Tensor, y_ref: np.ndarray, abs_ref: np.ndarray, what: str = "",
          rel_fro: float = REL_FRO) -> dict:
    yg = y_gpu.detach().float().cpu().numpy().astype(np.float64)
    assert yg.shape == y_ref.shape, (yg.shape, y_ref.shape)
    assert np.isfinite(yg).all(), f"{what}: non-finite output"
    err = np.abs(yg - y_ref)
    bound = ABS_REL * abs_ref + ABS_ADD
    worst = float((err / bound).max()) if err.size else 0.0
    nref = float(np.linalg.norm(y_ref))
    rf = float(np.linalg.norm(yg - y_ref) / nref) if nref > 0 else float(np.linalg.norm(yg))
    assert worst <= 1.0, f"{what}: max |err| / bound = {worst:.3g}"
    # The Frobenius bound is a statistical property of many outputs: bf16 output
    # rounding alone is up to 2^-8 relative per element, so it is applied to
    # outputs of at least FRO_MIN_ELEMS elements (the element-wise bound always is).
    if y_ref.size >= FRO_MIN_ELEMS:
        assert rf <= rel_fro, f"{what}: relative Frobenius error {rf:.3g} > {rel_fro}"
    return {"worst_ratio": worst, "rel_fro": rf}
