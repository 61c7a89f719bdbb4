"""Helpers for the GPU parity tests: moving synthetic host arrays to the device and
reading results back.  No verification arithmetic lives here."""
import numpy as np
import torch

import synth


def dev():
    return torch.device("cuda", 0)


def to_dev(x: np.ndarray, bf16: bool):
    """fp32 numpy array (bf16-exact values when bf16) -> CUDA tensor of the right dtype."""
    if bf16:
        bits = synth.bf16_bits(np.ascontiguousarray(x, dtype=np.float32))
        t = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16)
        return t.to(dev())
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(dev())


def i32(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.int32)).to(dev())


def host(t):
    if t.dtype == torch.bfloat16:
        return t.float().cpu().numpy()
    return t.cpu().numpy()
