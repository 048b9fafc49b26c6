"""Small helpers shared by the GPU tests (device transfer, oracle operands)."""
import numpy as np
import torch

import oracle.dsa_oracle as O


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def bf16_dev(bits):
    """uint16 BF16 bit patterns -> CUDA bfloat16 tensor."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def host(t):
    return t.cpu().numpy()


def bf16_values(bits):
    return O.bf16_bits_to_float(bits)
