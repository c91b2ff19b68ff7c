"""Helpers shared by the GPU tests: moving seeded numpy inputs to the device."""
import numpy as np


def torch_bf16(bits: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def torch_u8(a: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, np.uint8)).cuda()


def torch_of(a: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def np_of(t) -> np.ndarray:
    return t.cpu().numpy()


def wd_bits(t) -> np.ndarray:
    """fp16 scale tensor (stored as int16) -> uint16 bit patterns."""
    return t.cpu().numpy().view(np.uint16)
