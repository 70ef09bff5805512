"""Helpers for the GPU parity tests: host<->device views of uint64 records."""

import numpy as np
import pytest

try:
    import torch
except ImportError:  # pragma: no cover
    torch = None


def need_gpu():
    if torch is None or not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def lib():
    """The CUDA library's binding (built on demand, fails loudly if it cannot load)."""
    import importlib.util
    import os
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    spec = importlib.util.spec_from_file_location(
        "_descbuild_build", os.path.join(root, "descriptor_build_gb300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build()
    import descriptor_build_gb300 as db
    return db


def dev64(a: np.ndarray) -> "torch.Tensor":
    """uint64 (or any 8-byte) numpy array -> int64 CUDA tensor with the same bits."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int64)).cuda()


def dev32(a: np.ndarray) -> "torch.Tensor":
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int32)).cuda()


def host64(t: "torch.Tensor") -> np.ndarray:
    return t.cpu().numpy().view(np.uint64)


def host32(t: "torch.Tensor") -> np.ndarray:
    return t.cpu().numpy().view(np.uint32)
