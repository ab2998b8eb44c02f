"""Helpers shared by the GPU tests: moving seeded bf16 bit patterns to the
device and back.  No method arithmetic."""
import numpy as np
import torch


def to_dev(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)
