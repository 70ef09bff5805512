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


def assert_arena_equal(got: np.ndarray, want: np.ndarray, fill: int, where: str = ""):
    """List pages from the GPU against the oracle's, word for word.

    Both arenas started filled with ``fill``; no list word can equal it (list
    words are 4 KiB-aligned bus addresses, ``fill`` is not). Slots the oracle
    wrote must match. Slots it left as they were must still hold ``fill``,
    except that the library may write 0 into the slots that share a list's
    last entry's 32-byte sector (the header allows it: the kernel ends every
    list on a whole sector)."""
    got = np.ascontiguousarray(got).view(np.uint64).reshape(-1, 4)
    want = np.ascontiguousarray(want).view(np.uint64).reshape(-1, 4)
    assert got.shape == want.shape, where
    f = np.uint64(fill & (2**64 - 1))
    defined = want != f
    ok = np.where(defined, got == want, got == f)
    # a sector holding a list's last entry: its undefined slots may be 0
    tail = defined.any(axis=1, keepdims=True) & ~defined & (got == 0)
    bad = ~(ok | tail)
    if bad.any():
        r, c = np.argwhere(bad)[0]
        raise AssertionError(f"{where}: arena word {4 * r + c}: got {int(got[r, c]):#x}, "
                             f"want {int(want[r, c]):#x} ({int(bad.sum())} words differ)")
