"""Helpers for the GPU parity tests: host <-> device copies of seeded inputs."""
import numpy as np
import torch


def dev():
    return torch.device("cuda:0")


def to_dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev()).view(torch.bfloat16)


def to_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev())


def bf16_to_np_f32(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy()


def status() -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=dev())
