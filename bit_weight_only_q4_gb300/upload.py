"""Host -> device marshalling of the seeded synthetic inputs (numpy bit patterns
from :mod:`bit_weight_only_q4_gb300.synth`) into torch CUDA tensors of the dtypes
the C ABI expects.  Pure data movement: no arithmetic of the method happens here.
"""
from __future__ import annotations

import numpy as np
import torch


def bf16_dev(bits: np.ndarray, device="cuda") -> torch.Tensor:
    """bf16 tensor from uint16 bit patterns."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def u8_dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def f16_dev(bits: np.ndarray, device="cuda") -> torch.Tensor:
    """fp16 tensor from uint16 bit patterns."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.float16).to(device)


def bf16_bits_host(t: torch.Tensor) -> np.ndarray:
    """uint16 bit patterns of a bf16 tensor, on the host."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16).copy()


def int4_dev(w, device="cuda"):
    """(qweight, scale, min) of an int4-g128 matrix on the device."""
    return u8_dev(w.qweight, device), f16_dev(w.scale, device), f16_dev(w.minv, device)


def nvfp4_dev(w, device="cuda"):
    """(codes, e4m3 scales, global scale as a one-element fp32 tensor) on the device."""
    g = torch.tensor([float(w.global_scale)], dtype=torch.float32, device=device)
    return u8_dev(w.codes, device), u8_dev(w.scale, device), g


def int8_dev(w, device="cuda"):
    """(qweight int8, scale fp16) of an INT8 weight-only matrix on the device."""
    return (torch.from_numpy(np.ascontiguousarray(w.qweight)).to(device),
            torch.from_numpy(np.ascontiguousarray(w.scale).view(np.int16)).view(torch.float16).to(device))
