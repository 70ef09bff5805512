"""Python binding of libdescbuild.so: batched GPU-range -> DMA-descriptor translation.

The functions here have the names of the C ABI in ``include/descbuild.h``
(without the ``db_`` prefix) and only marshal arguments: torch CUDA tensors
become device pointers, the stream becomes a ``cudaStream_t``, and a negative
return code becomes a ``DescBuildError``. Every step of the computation runs
in the library's CUDA kernels; there is no fallback. Importing this package
fails loudly when the library has not been built.

Record layouts (all tensors contiguous, on the GPU):
  PRP request  16 B  {u64 off; u32 len; u32 rsvd}     -> int64 [n, 2]
  PRP output   16 B  {u64 prp1; u64 prp2}             -> int64 [n, 2]
  range        16 B  {u64 addr; u64 size}             -> int64 [n, 2]
  put          16 B  {u64 off; u32 bytes; u16 pe; u16 qp} -> int64 [n, 2]
  WQE          64 B                                    -> uint8 [rings, depth, 64]
  counters     32 B  {total, n_invalid, n_overflow, err} -> int64 [4]
"""

from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

from . import build as _build

__all__ = [
    "DescBuildError", "lib_path", "workspace", "prp_workspace_size", "prp_build",
    "prp_build_static", "PRP_STATIC_MAX_REQUESTS",
    "mr_workspace_size", "mr_lookup", "mr_lookup_overlap", "wqe_workspace_size",
    "wqe_vmm_workspace_size", "wqe_bucket", "wqe_bucket_vmm", "wqe_bucket_transport",
    "XPORT_RDMA", "XPORT_P2P", "XPORT_SDMA",
    "strerror", "CQ_SLOT_DTYPE", "CQ_MAX_SLOTS", "CQ_MAX_DEPTH", "CQ_TIMED", "cq_slots",
    "cq_slot_fields",
    "mr_capacity_for", "mr_register_workspace_size", "mr_register",
    "mr_deregister_workspace_size", "mr_deregister", "MR_NEW", "MR_NEW_DUP", "DEREG_OK",
    "DEREG_RELEASED", "DEREG_STALE",
    "cq_mirror", "cq_attach", "cq_detach", "cq_wait_ack", "cq_host_reap", "cq_request_stop",
    "PRP_OK", "PRP_INVALID", "PRP_OVERFLOW", "MR_MISS", "MR_EXACT", "MR_CONTAINED",
    "MR_INVALID", "ERR_TIMEOUT", "ERR_RING_OVERFLOW", "ERR_TABLE_ORDER", "PRP_ZERO_TAIL",
    "PRP_SCHED_SINGLE", "PRP_SCHED_SPLIT",
]

PRP_OK, PRP_INVALID, PRP_OVERFLOW = 0, 1, 2
MR_MISS, MR_EXACT, MR_CONTAINED, MR_INVALID = 0, 1, 2, 3
ERR_TIMEOUT, ERR_RING_OVERFLOW, ERR_TABLE_ORDER = 1, 2, 4
PRP_ZERO_TAIL = 1
PRP_SCHED_SINGLE, PRP_SCHED_SPLIT = 2, 4
XPORT_RDMA, XPORT_P2P, XPORT_SDMA = 0, 1, 2

lib_path = _build.LIB


class DescBuildError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        msg = _lib.db_strerror(code).decode()
        if code == -5:
            msg += f" (cudaError {_lib.db_last_cuda_error()})"
        super().__init__(f"{fn}: {msg} [{code}]")


def _load():
    if not os.path.exists(lib_path):
        raise ImportError(
            f"{lib_path} is missing: build it with `python -c 'import __graft_entry__ as g; "
            f"g.build()'` (needs nvcc)")
    lib = ctypes.CDLL(lib_path)
    vp, u64, u32, i32, sz = (ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int,
                             ctypes.c_size_t)
    psz = ctypes.POINTER(ctypes.c_size_t)
    lib.db_prp_workspace_size.argtypes = [u64, psz]
    lib.db_prp_build.argtypes = [vp, u64, vp, u64, u64, u64, vp, vp, vp, vp, vp, u32, vp, sz, vp]
    lib.db_prp_build_static.argtypes = [vp, u64, vp, u64, u64, u64, vp, vp, vp, vp, vp, u32, vp]
    lib.db_mr_workspace_size.argtypes = [u64, psz]
    lib.db_mr_lookup.argtypes = [vp, u64, vp, vp, vp, u64, vp, vp, vp, vp, vp, sz, vp]
    lib.db_mr_lookup_overlap.argtypes = lib.db_mr_lookup.argtypes
    lib.db_wqe_workspace_size.argtypes = [u64, u32, psz]
    lib.db_wqe_vmm_workspace_size.argtypes = [u64, u32, u32, u64, u32, psz]
    lib.db_wqe_vmm_workspace_size.restype = i32
    lib.db_wqe_bucket.argtypes = [vp, u64, vp, vp, u32, u32, u64, u32, u64, vp, u64, vp, vp, vp,
                                  vp, sz, vp]
    lib.db_wqe_bucket_vmm.argtypes = [vp, u64, vp, vp, vp, u32, u32, u32, u64, u64, vp, u64, vp,
                                      vp, u32, vp, vp, vp, sz, vp]
    lib.db_wqe_bucket_transport.argtypes = [vp, u64, vp, vp, vp, u32, u32, u64, u32, u64, vp,
                                            u64, vp, vp, vp, vp, vp, vp, sz, vp]
    for name in ("db_prp_workspace_size", "db_prp_build", "db_prp_build_static",
                 "db_mr_workspace_size",
                 "db_mr_lookup", "db_mr_lookup_overlap", "db_wqe_workspace_size", "db_wqe_bucket",
                 "db_wqe_bucket_vmm", "db_wqe_bucket_transport",
                 "db_last_cuda_error"):
        getattr(lib, name).restype = i32
    lib.db_mr_capacity_for.argtypes = [u64]
    lib.db_mr_capacity_for.restype = u64
    lib.db_mr_register_workspace_size.argtypes = [u64, u64, psz]
    lib.db_mr_register.argtypes = [vp, u64, vp, u32, vp, vp, vp, vp, u64, vp, vp, vp, vp, u64,
                                   vp, vp, vp, vp, vp, sz, vp]
    lib.db_mr_deregister_workspace_size.argtypes = [u64, u64, psz]
    lib.db_mr_deregister.argtypes = [vp, u64, vp, vp, vp, vp, u64, vp, vp, vp, vp, vp, vp, vp,
                                     vp, sz, vp]
    for name in ("db_mr_register_workspace_size", "db_mr_register",
                 "db_mr_deregister_workspace_size", "db_mr_deregister"):
        getattr(lib, name).restype = i32
    lib.db_cq_mirror.argtypes = [vp, u32, vp, u64, vp, vp]
    lib.db_cq_attach.argtypes = [vp, u64, u64, u32, ctypes.POINTER(ctypes.c_uint32)]
    lib.db_cq_detach.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
    lib.db_cq_wait_ack.argtypes = [vp, u32, u64]
    lib.db_cq_host_reap.argtypes = [vp, u32, ctypes.POINTER(ctypes.c_uint32),
                                    ctypes.POINTER(ctypes.c_uint32), vp, u32]
    lib.db_cq_request_stop.argtypes = [vp]
    lib.db_cq_request_stop.restype = None
    for name in ("db_cq_mirror", "db_cq_attach", "db_cq_detach", "db_cq_wait_ack",
                 "db_cq_host_reap"):
        getattr(lib, name).restype = i32
    lib.db_strerror.argtypes = [i32]
    lib.db_strerror.restype = ctypes.c_char_p
    lib.db_last_cuda_error.argtypes = []
    return lib


_lib = _load()


def _check(fn: str, rc: int) -> None:
    if rc != 0:
        raise DescBuildError(fn, rc)


def _ptr(t: torch.Tensor | None) -> int | None:
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to libdescbuild must be contiguous")
    return t.data_ptr()


def _records(t: torch.Tensor, size: int) -> int:
    nbytes = t.numel() * t.element_size()
    if nbytes % size:
        raise ValueError(f"buffer of {nbytes} bytes is not a whole number of {size}-byte records")
    return nbytes // size


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _size(fn, *args) -> int:
    out = ctypes.c_size_t(0)
    _check(fn.__name__, fn(*args, ctypes.byref(out)))
    return out.value


def workspace(nbytes: int, device=None) -> torch.Tensor:
    """A zero-filled device workspace of ``nbytes`` (256-byte aligned by torch)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device or "cuda")


def strerror(code: int) -> str:
    return _lib.db_strerror(code).decode()


# ------------------------------------------------------------------ PRP build
def prp_workspace_size(n: int) -> int:
    return _size(_lib.db_prp_workspace_size, n)


def prp_build(req: torch.Tensor, lut: torch.Tensor, heap_size: int, arena_base: int,
              arena_cap_pages: int, arena: torch.Tensor | None, prp: torch.Tensor,
              ws: torch.Tensor, page_base: torch.Tensor | None = None,
              status: torch.Tensor | None = None, ctr: torch.Tensor | None = None,
              flags: int = 0, stream=None) -> None:
    """db_prp_build: PRP1/PRP2 per request and the chained list pages in ``arena``."""
    n = _records(req, 16)
    _check("db_prp_build", _lib.db_prp_build(
        _ptr(req), n, _ptr(lut), heap_size, arena_base, arena_cap_pages, _ptr(arena), _ptr(prp),
        _ptr(page_base), _ptr(status), _ptr(ctr), flags, _ptr(ws),
        ws.numel() * ws.element_size(), _stream(stream)))


PRP_STATIC_MAX_REQUESTS = 1 << 24


def prp_build_static(req: torch.Tensor, lut: torch.Tensor, heap_size: int, arena_base: int,
                     arena_cap_pages: int, arena: torch.Tensor | None, prp: torch.Tensor,
                     page_base: torch.Tensor | None = None, status: torch.Tensor | None = None,
                     ctr: torch.Tensor | None = None, flags: int = 0, stream=None) -> None:
    """db_prp_build_static: prp_build with the library's own static scratch
    array, for callers that must not allocate device memory while submitting
    (cudaMalloc may wait on queued device work and takes driver locks).
    At most PRP_STATIC_MAX_REQUESTS requests per call; calls that may overlap
    on the GPU share the array and must be ordered by the caller. The first
    call on a device looks the array up, so make it before any stream capture."""
    n = _records(req, 16)
    _check("db_prp_build_static", _lib.db_prp_build_static(
        _ptr(req), n, _ptr(lut), heap_size, arena_base, arena_cap_pages, _ptr(arena), _ptr(prp),
        _ptr(page_base), _ptr(status), _ptr(ctr), flags, _stream(stream)))


# ------------------------------------------------------------------ MR lookup
def mr_workspace_size(n_mr: int) -> int:
    return _size(_lib.db_mr_workspace_size, n_mr)


def mr_lookup(q: torch.Tensor, mr_start: torch.Tensor, mr_end: torch.Tensor,
              mr_lkey: torch.Tensor, idx: torch.Tensor, lkey: torch.Tensor, kind: torch.Tensor,
              ws: torch.Tensor, ctr: torch.Tensor | None = None, stream=None) -> None:
    """db_mr_lookup: classify each range against a sorted registration table."""
    n_q = _records(q, 16)
    n_mr = _records(mr_start, 8)
    _check("db_mr_lookup", _lib.db_mr_lookup(
        _ptr(q), n_q, _ptr(mr_start), _ptr(mr_end), _ptr(mr_lkey), n_mr, _ptr(idx), _ptr(lkey),
        _ptr(kind), _ptr(ctr), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def mr_lookup_overlap(q: torch.Tensor, mr_start: torch.Tensor, mr_end: torch.Tensor,
                      mr_lkey: torch.Tensor, idx: torch.Tensor, lkey: torch.Tensor,
                      kind: torch.Tensor, ws: torch.Tensor, ctr: torch.Tensor | None = None,
                      stream=None) -> None:
    """db_mr_lookup_overlap: the same on a start-sorted table whose ranges may overlap."""
    n_q = _records(q, 16)
    n_mr = _records(mr_start, 8)
    _check("db_mr_lookup_overlap", _lib.db_mr_lookup_overlap(
        _ptr(q), n_q, _ptr(mr_start), _ptr(mr_end), _ptr(mr_lkey), n_mr, _ptr(idx), _ptr(lkey),
        _ptr(kind), _ptr(ctr), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


# ------------------------------------------------------- MR cache mutation
MR_NEW, MR_NEW_DUP = 4, 5
DEREG_OK, DEREG_RELEASED, DEREG_STALE = 0, 1, 2


def mr_capacity_for(n: int) -> int:
    """Table capacity after growth to n records: 0, 32, then doubling."""
    return int(_lib.db_mr_capacity_for(n))


def mr_register_workspace_size(n_q: int, n_mr: int) -> int:
    return _size(_lib.db_mr_register_workspace_size, n_q, n_mr)


def mr_register(q: torch.Tensor, new_lkey: torch.Tensor, start: torch.Tensor, end: torch.Tensor,
                lkey: torch.Tensor, refs: torch.Tensor, out_start: torch.Tensor,
                out_end: torch.Tensor, out_lkey: torch.Tensor, out_refs: torch.Tensor,
                handle: torch.Tensor, kind: torch.Tensor, remap: torch.Tensor, ws: torch.Tensor,
                granule_shift: int = 12, ctr: torch.Tensor | None = None, stream=None) -> None:
    """db_mr_register: a batch of registrations; the table after it goes to out_*."""
    n_q = _records(q, 16)
    n_mr = _records(start, 8)
    out_cap = _records(out_start, 8)
    _check("db_mr_register", _lib.db_mr_register(
        _ptr(q), n_q, _ptr(new_lkey), granule_shift, _ptr(start), _ptr(end), _ptr(lkey),
        _ptr(refs), n_mr, _ptr(out_start), _ptr(out_end), _ptr(out_lkey), _ptr(out_refs),
        out_cap, _ptr(handle), _ptr(kind), _ptr(remap), _ptr(ctr), _ptr(ws),
        ws.numel() * ws.element_size(), _stream(stream)))


def mr_deregister_workspace_size(n_h: int, n_mr: int) -> int:
    return _size(_lib.db_mr_deregister_workspace_size, n_h, n_mr)


def mr_deregister(handle: torch.Tensor, start: torch.Tensor, end: torch.Tensor,
                  lkey: torch.Tensor, refs: torch.Tensor, out_start: torch.Tensor,
                  out_end: torch.Tensor, out_lkey: torch.Tensor, out_refs: torch.Tensor,
                  remap: torch.Tensor, status: torch.Tensor, ws: torch.Tensor,
                  ctr: torch.Tensor | None = None, stream=None) -> None:
    """db_mr_deregister: a batch of deregistrations, in batch order."""
    n_h = _records(handle, 8)
    n_mr = _records(start, 8)
    _check("db_mr_deregister", _lib.db_mr_deregister(
        _ptr(handle), n_h, _ptr(start), _ptr(end), _ptr(lkey), _ptr(refs), n_mr,
        _ptr(out_start), _ptr(out_end), _ptr(out_lkey), _ptr(out_refs), _ptr(remap),
        _ptr(status), _ptr(ctr), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


# --------------------------------------------------------------- WQE bucketing
def wqe_workspace_size(n: int, n_rings: int) -> int:
    return _size(_lib.db_wqe_workspace_size, n, n_rings)


def wqe_vmm_workspace_size(n: int, world: int, n_qp: int, heap_size: int,
                           chunk_shift: int) -> int:
    """Workspace bytes of db_wqe_bucket_vmm (columns plus the packed chunk tables)."""
    return _size(_lib.db_wqe_vmm_workspace_size, n, world, n_qp, heap_size, chunk_shift)


def wqe_bucket(req: torch.Tensor, peer_ptrs: torch.Tensor, rkeys: torch.Tensor, world: int,
               n_qp: int, local_base: int, lkey: int, heap_size: int, rings: torch.Tensor,
               depth: int, head: torch.Tensor, count: torch.Tensor, ws: torch.Tensor,
               ctr: torch.Tensor | None = None, stream=None) -> None:
    """db_wqe_bucket: translate puts and stable-partition them into WQE rings."""
    n = _records(req, 16)
    _check("db_wqe_bucket", _lib.db_wqe_bucket(
        _ptr(req), n, _ptr(peer_ptrs), _ptr(rkeys), world, n_qp, local_base, lkey, heap_size,
        _ptr(rings), depth, _ptr(head), _ptr(count), _ptr(ctr), _ptr(ws),
        ws.numel() * ws.element_size(), _stream(stream)))


def wqe_bucket_transport(req: torch.Tensor, peer_ptrs: torch.Tensor, rkeys: torch.Tensor,
                         transport: torch.Tensor, world: int, n_qp: int, local_base: int,
                         lkey: int, heap_size: int, rings: torch.Tensor, depth: int,
                         head: torch.Tensor, count: torch.Tensor, direct: torch.Tensor,
                         n_direct: torch.Tensor, ws: torch.Tensor,
                         ctr: torch.Tensor | None = None, stream=None) -> None:
    """db_wqe_bucket_transport: puts dispatched on their PE's transport (uint8
    [world] of XPORT_*): RDMA puts into WQE rings as wqe_bucket, P2P and SDMA
    puts as 32-byte direct records (uint8 [n, 32]) in batch order; n_direct
    (int64 [1]) gets their number."""
    n = _records(req, 16)
    _check("db_wqe_bucket_transport", _lib.db_wqe_bucket_transport(
        _ptr(req), n, _ptr(peer_ptrs), _ptr(rkeys), _ptr(transport), world, n_qp, local_base,
        lkey, heap_size, _ptr(rings), depth, _ptr(head), _ptr(count), _ptr(direct),
        _ptr(n_direct), _ptr(ctr), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def wqe_bucket_vmm(req: torch.Tensor, chunk_raddr: torch.Tensor, chunk_rkey: torch.Tensor,
                   chunk_lkey: torch.Tensor, chunk_shift: int, world: int, n_qp: int,
                   local_base: int, heap_size: int, rings: torch.Tensor, depth: int,
                   head: torch.Tensor, count: torch.Tensor, ws: torch.Tensor,
                   ctr: torch.Tensor | None = None, stream=None, mtu: int = 0,
                   psn_head: torch.Tensor | None = None) -> None:
    """db_wqe_bucket_vmm: puts on a chunked (VMM) heap, one WQE per chunk
    touched; with an mtu, each WQE also gets its first PSN."""
    n = _records(req, 16)
    _check("db_wqe_bucket_vmm", _lib.db_wqe_bucket_vmm(
        _ptr(req), n, _ptr(chunk_raddr), _ptr(chunk_rkey), _ptr(chunk_lkey), chunk_shift, world,
        n_qp, local_base, heap_size, _ptr(rings), depth, _ptr(head), _ptr(count), mtu,
        _ptr(psn_head), _ptr(ctr), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


# ------------------------------------------------------------------ CQ mirror
CQ_MAX_SLOTS, CQ_MAX_DEPTH = 64, 65536
CQ_TIMED = 1  # slot flag: record each batch's latency in lat_ns / lat_seq
# db_cq_slot, 64 bytes
CQ_SLOT_DTYPE = np.dtype([("dev_cq", "<u8"), ("host_cq", "<u8"), ("depth", "<u4"),
                          ("generation", "<u4"), ("ack", "<u4"), ("seen", "<u4"),
                          ("head", "<u4"), ("phase", "<u4"), ("copied", "<u8"),
                          ("flags", "<u4"), ("lat_ns", "<u4"), ("lat_seq", "<u8")])
assert CQ_SLOT_DTYPE.itemsize == 64


def _host(t: torch.Tensor) -> int:
    if t.device.type != "cpu" or not t.is_contiguous():
        raise ValueError("expected a contiguous host tensor")
    return t.data_ptr()


def cq_slots(n: int) -> torch.Tensor:
    """A zero-filled slot table of n slots in pinned host memory."""
    return torch.zeros((n, 64), dtype=torch.uint8).pin_memory()


def cq_slot_fields(slots: torch.Tensor) -> np.ndarray:
    """A live structured view of a slot table (reads see the kernel's writes)."""
    return slots.numpy().view(CQ_SLOT_DTYPE).reshape(-1)


def cq_mirror(slots: torch.Tensor, stop: torch.Tensor, limit_s: float,
              ctr: torch.Tensor | None = None, stream=None, n_slots: int | None = None) -> None:
    """db_cq_mirror: launch the bounded resident mirror over the slots."""
    n = slots.shape[0] if n_slots is None else n_slots
    _check("db_cq_mirror", _lib.db_cq_mirror(_host(slots), n, _host(stop),
                                             int(limit_s * 1e9), _ptr(ctr), _stream(stream)))


def cq_attach(slots: torch.Tensor, i: int, dev_cq: torch.Tensor, host_cq: torch.Tensor) -> int:
    """db_cq_attach: serve the device CQ dev_cq ([depth, 4] int32, device)
    into host_cq ([depth, 4] int32, pinned); returns the odd generation."""
    depth = _records(dev_cq, 16)
    if _records(host_cq, 16) != depth:
        raise ValueError("device and host CQ differ in depth")
    g = ctypes.c_uint32(0)
    _check("db_cq_attach", _lib.db_cq_attach(_host(slots) + 64 * i, _ptr(dev_cq),
                                             _host(host_cq), depth, ctypes.byref(g)))
    return g.value


def cq_detach(slots: torch.Tensor, i: int) -> int:
    """db_cq_detach: returns the odd generation whose acknowledgement to wait for."""
    g = ctypes.c_uint32(0)
    _check("db_cq_detach", _lib.db_cq_detach(_host(slots) + 64 * i, ctypes.byref(g)))
    return g.value


def cq_wait_ack(slots: torch.Tensor, i: int, generation: int, timeout_s: float) -> bool:
    rc = _lib.db_cq_wait_ack(_host(slots) + 64 * i, generation, int(timeout_s * 1e9))
    if rc not in (0, -110):
        _check("db_cq_wait_ack", rc)
    return rc == 0


def cq_host_reap(host_cq: torch.Tensor, head: int, phase: int, max_entries: int | None = None):
    """db_cq_host_reap: returns (entries [n, 4] uint32, head, phase)."""
    depth = _records(host_cq, 16)
    m = depth if max_entries is None else max_entries
    out = np.zeros((max(m, 1), 4), dtype=np.uint32)
    h, ph = ctypes.c_uint32(head), ctypes.c_uint32(phase)
    n = _lib.db_cq_host_reap(_host(host_cq), depth, ctypes.byref(h), ctypes.byref(ph),
                             out.ctypes.data, m)
    if n < 0:
        _check("db_cq_host_reap", n)
    return out[:n], h.value, ph.value


def cq_request_stop(stop: torch.Tensor) -> None:
    _lib.db_cq_request_stop(_host(stop))
