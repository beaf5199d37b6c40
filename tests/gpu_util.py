"""Host<->device marshalling for the GPU tests (no arithmetic of the layer)."""

import numpy as np
import torch


def x_to_device(x: np.ndarray, act_dtype: str) -> torch.Tensor:
    if act_dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def empty_out(T: int, H: int, act_dtype: str) -> torch.Tensor:
    dt = torch.bfloat16 if act_dtype == "bf16" else torch.float32
    return torch.empty((T, H), dtype=dt, device="cuda")


def out_to_host(out: torch.Tensor) -> np.ndarray:
    return out.float().cpu().numpy().astype(np.float64)
