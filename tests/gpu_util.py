"""Helpers for the GPU parity tests (CUDA path through the C ABI)."""
import numpy as np


def torch_bf16_bits(x_bf16: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x_bf16).view(np.int16)).cuda()


def rel_err(got: np.ndarray, ref: np.ndarray) -> float:
    return float(np.abs(got.astype(np.float64) - ref.astype(np.float64)).max() / np.abs(ref).max())


def ulp_diff_f32(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in fp32 units in the last place (same-sign finite values)."""
    ia = np.ascontiguousarray(a, np.float32).view(np.int32).astype(np.int64)
    ib = np.ascontiguousarray(b, np.float32).view(np.int32).astype(np.int64)
    ia = np.where(ia < 0, -(ia & 0x7FFFFFFF), ia)
    ib = np.where(ib < 0, -(ib & 0x7FFFFFFF), ib)
    return np.abs(ia - ib)
