"""The C ABI library builds, loads and exports what include/*.h declares.

No compute calls: only the host-side entry points (workspace sizes, error
strings, argument checks that return before touching a GPU).
"""

import ctypes
import glob
import os
import re

import pytest

from conftest import ROOT


@pytest.fixture(scope="module")
def libpath():
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "_descbuild_build", os.path.join(ROOT, "descriptor_build_gb300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    try:
        mod.nvcc()
    except RuntimeError:
        pytest.skip("no nvcc")
    return mod.build()


def declared_functions():
    names = []
    for hdr in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(hdr).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(db_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_three_calls():
    names = declared_functions()
    for n in ("db_prp_build", "db_mr_lookup", "db_wqe_bucket", "db_prp_workspace_size",
              "db_mr_workspace_size", "db_wqe_workspace_size", "db_strerror"):
        assert n in names


def test_library_exports_every_declared_symbol(libpath):
    lib = ctypes.CDLL(libpath)
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_workspace_sizes(libpath):
    lib = ctypes.CDLL(libpath)
    out = ctypes.c_size_t()
    assert lib.db_prp_workspace_size(ctypes.c_uint64(4_194_304), ctypes.byref(out)) == 0
    assert out.value >= 256 + 8 * (4_194_304 // 2048)   # a status word per tile
    assert lib.db_mr_workspace_size(ctypes.c_uint64(1 << 20), ctypes.byref(out)) == 0
    assert out.value >= 32 * (1 << 20)
    assert lib.db_wqe_workspace_size(ctypes.c_uint64(8 << 20), ctypes.c_uint32(32),
                                     ctypes.byref(out)) == 0
    assert out.value >= 4 * 33 * ((8 << 20) // 1024)   # a count per (ring + invalid, tile)
    # out of range
    assert lib.db_wqe_workspace_size(ctypes.c_uint64(10), ctypes.c_uint32(0),
                                     ctypes.byref(out)) == -22
    assert lib.db_wqe_workspace_size(ctypes.c_uint64(10), ctypes.c_uint32(1025),
                                     ctypes.byref(out)) == -22
    assert lib.db_prp_workspace_size(ctypes.c_uint64((1 << 28) + 1), ctypes.byref(out)) == -22
    assert lib.db_prp_workspace_size(ctypes.c_uint64(1), None) == -22


def test_argument_checks_need_no_gpu(libpath):
    lib = ctypes.CDLL(libpath)
    vp = ctypes.c_void_p
    lib.db_prp_build.argtypes = [vp, ctypes.c_uint64, vp, ctypes.c_uint64, ctypes.c_uint64,
                                 ctypes.c_uint64, vp, vp, vp, vp, vp, ctypes.c_uint32, vp,
                                 ctypes.c_size_t, vp]
    fake = 1 << 20  # never dereferenced: the checks fail first
    # heap size not a multiple of 64 KiB
    assert lib.db_prp_build(fake, 10, fake, 1000, 0, 1, fake, fake, None, None, None, 0, fake,
                            1 << 20, None) == -22
    # arena base not page aligned
    assert lib.db_prp_build(fake, 10, fake, 1 << 20, 5, 1, fake, fake, None, None, None, 0, fake,
                            1 << 20, None) == -22
    # misaligned request array
    assert lib.db_prp_build(fake + 8, 10, fake, 1 << 20, 0, 1, fake, fake, None, None, None, 0,
                            fake, 1 << 20, None) == -22
    # workspace too small
    assert lib.db_prp_build(fake, 10, fake, 1 << 20, 0, 1, fake, fake, None, None, None, 0,
                            fake, 16, None) == -28
    lib.db_strerror.restype = ctypes.c_char_p
    assert b"workspace" in lib.db_strerror(-28)
    lib.db_wqe_bucket.argtypes = [vp, ctypes.c_uint64, vp, vp, ctypes.c_uint32, ctypes.c_uint32,
                                  ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint64, vp,
                                  ctypes.c_uint64, vp, vp, vp, vp, ctypes.c_size_t, vp]
    # depth not a power of two
    assert lib.db_wqe_bucket(fake, 5, fake, fake, 8, 4, 0, 0, 1 << 20, fake, 6, fake, fake, None,
                             fake, 1 << 20, None) == -22
    # more than 1024 rings
    assert lib.db_wqe_bucket(fake, 5, fake, fake, 64, 32, 0, 0, 1 << 20, fake, 8, fake, fake,
                             None, fake, 1 << 20, None) == -22


def test_transport_argument_checks_need_no_gpu(libpath):
    lib = ctypes.CDLL(libpath)
    vp, u32, u64 = ctypes.c_void_p, ctypes.c_uint32, ctypes.c_uint64
    lib.db_wqe_bucket_transport.argtypes = [vp, u64, vp, vp, vp, u32, u32, u64, u32, u64, vp,
                                            u64, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
    fake = 1 << 20  # never dereferenced: the checks fail first
    call = lambda direct, n_direct, transport=fake: lib.db_wqe_bucket_transport(
        fake, 5, fake, fake, transport, 8, 4, 0, 0, 1 << 20, fake, 8, fake, fake, direct,
        n_direct, None, fake, 1 << 20, None)
    assert call(fake, None) == -22           # no n_direct
    assert call(fake + 16, fake) == -22      # direct records not 32-byte aligned
    assert call(fake, fake, transport=None) == -22
