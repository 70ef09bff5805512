"""Host-side parts of the registration-cache batches, without a GPU."""

import ctypes

import pytest

from conftest import ROOT  # noqa: F401  (puts the repository on sys.path)


@pytest.fixture(scope="module")
def db():
    import descriptor_build_gb300 as d
    return d


def test_capacity_grows_as_the_ib_mr_cache_does(db):
    """'IB Backend MR Cache': capacity 0, first grown to 32, then 32 -> 64 -> 128."""
    assert [db.mr_capacity_for(n) for n in (0, 1, 31, 32, 33, 64, 65, 128, 129)] == \
        [0, 32, 32, 32, 64, 64, 128, 128, 256]
    assert db.mr_capacity_for(1 << 40) == 1 << 40 and db.mr_capacity_for((1 << 40) + 1) == 1 << 41


def test_workspace_sizes(db):
    a = db.mr_register_workspace_size(1000, 100)
    b = db.mr_register_workspace_size(100000, 100)
    assert 0 < a < b and b >= 100000 * (8 + 8 + 4 + 4)      # sort buffers at least
    assert db.mr_deregister_workspace_size(0, 0) > 0
    lib = ctypes.CDLL(db.lib_path)
    out = ctypes.c_size_t()
    lib.db_mr_register_workspace_size.argtypes = [ctypes.c_uint64, ctypes.c_uint64,
                                                  ctypes.POINTER(ctypes.c_size_t)]
    assert lib.db_mr_register_workspace_size(1 << 31, 1, ctypes.byref(out)) == -22
    assert lib.db_mr_register_workspace_size(1, 1 << 31, ctypes.byref(out)) == -22
