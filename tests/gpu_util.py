"""Shared setup for GPU tests: the device, the library, host<->device copies."""
import numpy as np
import pytest


def cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from lattice_vq_weight_gb300 import build
    build.build()
    import lattice_vq_weight_gb300 as L
    return torch, L


def to_dev_bf16(torch, a):
    """float32 numpy values representable in bf16 -> device bf16 tensor (exact)."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to("cuda").to(torch.bfloat16)


def to_dev(torch, a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.to("cuda")
