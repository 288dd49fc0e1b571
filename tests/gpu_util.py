"""Host <-> device helpers for the GPU tests (plumbing only)."""
import numpy as np


def dev_bf16(a, device="cuda"):
    """uint16 bf16 bit patterns (numpy) -> torch.bfloat16 device tensor."""
    import torch
    a = np.ascontiguousarray(a, dtype=np.uint16)
    return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)


def dev(a, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def host_bf16(t) -> np.ndarray:
    """torch.bfloat16 tensor -> uint16 bit patterns (numpy)."""
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host(t) -> np.ndarray:
    return t.detach().contiguous().cpu().numpy()
