"""Torch tensors -> the oracle's numpy form (test infrastructure).

bf16 travels as raw uint16 bits; pools keep their strides so that the oracle
writes through the same [slot, channel, column] view the kernel sees. No
arithmetic happens here.
"""
import numpy as np
import torch


def to_np(t):
    """CPU numpy array (float32 or uint16 bf16 bits) sharing memory with a CPU copy."""
    if t is None:
        return None
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype in (torch.int32, torch.uint8, torch.float32):
        return t.numpy()
    raise TypeError(t.dtype)


def pool_np(pool):
    """Numpy view of a pool that keeps its [slot, channel, column] strides."""
    t = pool.detach().cpu()
    if t.dtype == torch.bfloat16:
        a = t.view(torch.int16).numpy().view(np.uint16)
    else:
        a = t.numpy()
    assert a.strides == tuple(s * a.itemsize for s in t.stride())
    return a


def np_to_f64(a):
    """Numpy storage array (float32 or uint16 bf16 bits) -> float64 values."""
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)
