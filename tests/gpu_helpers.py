"""Helpers for the GPU tests: move uint32 / float32 numpy arrays to and from
the device bit for bit (torch has no full uint32 dtype, so int32 views)."""
import numpy as np


def to_dev_u32(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint32).view(np.int32)).cuda()


def to_dev_f32(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def from_dev_u32(t):
    return t.cpu().numpy().view(np.uint32)
