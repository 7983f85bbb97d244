"""Shared test helpers: moving bf16 bit patterns and e4m3 bytes between numpy
(the oracle's side) and torch device tensors (the CUDA path's side)."""
import numpy as np
import torch


def dev_bf16(h: np.ndarray, device="cuda") -> torch.Tensor:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    return torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).to(device)


def host_bf16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host_u8(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.uint8).cpu().numpy()


def f32(*shape, device="cuda"):
    return torch.empty(shape if shape else (1,), dtype=torch.float32, device=device)


def u8(*shape, device="cuda"):
    return torch.empty(shape, dtype=torch.uint8, device=device)


def bf16_out(*shape, device="cuda"):
    return torch.empty(shape, dtype=torch.bfloat16, device=device)


def first_diff(a: np.ndarray, b: np.ndarray) -> str:
    bad = np.argwhere(a != b)
    if bad.size == 0:
        return "equal"
    i = tuple(bad[0])
    return f"{len(bad)} differences, first at {i}: got {a[i]!r} expected {b[i]!r}"
