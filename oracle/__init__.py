"""CPU oracle for batched descriptor building -- test infrastructure only.

A ctypes front end over ``oracle.cpp``: plain single-threaded C++ written
from the source pages' definitions. Only the tests, ``__graft_entry__``'s
smoke check and the benchmark's CPU-baseline leg may import this package;
the CUDA library never does, and this package never imports the library.

All functions take and return numpy arrays (host memory).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

PRP_OK, PRP_INVALID, PRP_OVERFLOW = 0, 1, 2
MR_MISS, MR_EXACT, MR_CONTAINED, MR_INVALID = 0, 1, 2, 3
ERR_RING_OVERFLOW = 2


def build(force: bool = False) -> str:
    """Compile liboracle.so beside its source (plain g++, no GPU needed)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-o", tmp, _SRC],
                       check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # A test may point this at a deliberately broken build of the
            # oracle to check that the pins notice (tests/test_oracle_mutations.py).
            path = os.environ.get("DB_ORACLE_LIB") or build()
            lib = ctypes.CDLL(path)
            u64, u32, i32, vp = ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int, ctypes.c_void_p
            lib.oracle_prp_list_pages.restype = u64
            lib.oracle_prp_list_pages.argtypes = [u64, u64, u64]
            lib.oracle_prp_one.restype = u64
            lib.oracle_prp_one.argtypes = [u64, u64, vp, u64, u64, u64, u64, vp, vp, i32]
            lib.oracle_prp_build.restype = None
            lib.oracle_prp_build.argtypes = [vp, u64, vp, u64, u64, u64, u64, vp, vp, vp, vp,
                                             vp, i32]
            lib.oracle_mr_round.restype = None
            lib.oracle_mr_round.argtypes = [u64, u64, vp]
            for name in ("oracle_mr_linear", "oracle_mr_bsearch", "oracle_mr_prefix_max"):
                fn = getattr(lib, name)
                fn.restype = None
                fn.argtypes = [vp, u64, vp, vp, vp, u64, vp, vp, vp]
            lib.oracle_wqe_bucket.restype = None
            lib.oracle_wqe_bucket.argtypes = [vp, u64, vp, vp, u32, u32, u64, u32, u64, vp, u64,
                                              vp, vp, vp]
            lib.oracle_wqe_bucket_transport.restype = None
            lib.oracle_wqe_bucket_transport.argtypes = [vp, u64, vp, vp, vp, u32, u32, u64, u32,
                                                        u64, vp, u64, vp, vp, vp, vp, vp]
            lib.oracle_wqe_bucket_vmm.restype = None
            lib.oracle_wqe_bucket_vmm.argtypes = [vp, u64, vp, vp, vp, u32, u32, u32, u64, u64,
                                                  vp, u64, vp, u32, vp, vp, vp]
            lib.oracle_mr_register.restype = None
            lib.oracle_mr_register.argtypes = [vp, u64, vp, u32, vp, vp, vp, vp, u64, vp, vp, vp,
                                               vp, u64, vp, vp, vp, vp]
            for name in ("oracle_mr_register_seq", "oracle_mr_register_seq_indexed"):
                fn = getattr(lib, name)
                fn.restype = None
                fn.argtypes = lib.oracle_mr_register.argtypes
            lib.oracle_mr_deregister.restype = None
            lib.oracle_mr_deregister.argtypes = [vp, u64, vp, vp, vp, vp, u64, vp, vp, vp, vp, vp,
                                                 vp, vp]
            lib.oracle_cq_mirror_pass.restype = u32
            lib.oracle_cq_mirror_pass.argtypes = [vp, u32, vp, vp, vp, u32]
            lib.oracle_cq_ack.restype = u32
            lib.oracle_cq_ack.argtypes = [u32, u32, u32]
            _lib = lib
    return _lib


def _p(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _u64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.uint64)


# ----------------------------------------------------------------------- PRP
def prp_list_pages(off: int, length: int, heap_size: int) -> int:
    """List pages one request needs (0 for no list or an invalid request)."""
    return int(_load().oracle_prp_list_pages(off, length, heap_size))


def prp_one(off: int, length: int, lut: np.ndarray, heap_size: int, arena_base: int,
            page_base: int, zero_tail: bool = False, fill: int = 0):
    """Descriptors of one request placed at list page ``page_base``.

    Returns (prp1, prp2, list) where ``list`` is [list_pages, 512] uint64
    (slots the request leaves unwritten hold ``fill``).
    """
    lut = _u64(lut)
    pages = prp_list_pages(off, length, heap_size)
    lst = np.full((max(pages, 1), 512), fill, dtype=np.uint64)
    prp = np.zeros(2, dtype=np.uint64)
    got = _load().oracle_prp_one(off, length, _p(lut), lut.shape[0], heap_size, arena_base,
                                 page_base, _p(prp), _p(lst), int(zero_tail))
    assert got == pages
    return int(prp[0]), int(prp[1]), lst[:pages]


def prp_build(req: np.ndarray, lut: np.ndarray, heap_size: int, arena_base: int,
              arena_cap_pages: int, zero_tail: bool = False, fill: int = 0,
              lists: bool = True, arena: np.ndarray | None = None) -> dict:
    """Whole batch; returns prp [n,2], page_base [n], status [n], ctr [4], arena.

    With ``lists=False`` no arena is allocated or written (everything else is
    computed as if the lists had been written). ``arena`` may be given as a
    preallocated uint64 [>= arena_cap_pages, 512] array."""
    req = _u64(req).reshape(-1, 2)
    lut = _u64(lut)
    n = req.shape[0]
    if not lists:
        arena = None
    elif arena is None:
        arena = np.full((max(arena_cap_pages, 1), 512), fill, dtype=np.uint64)
    else:
        assert arena.dtype == np.uint64 and arena.shape[0] >= arena_cap_pages
    prp = np.zeros((n, 2), dtype=np.uint64)
    page_base = np.zeros(n, dtype=np.uint64)
    status = np.zeros(n, dtype=np.uint8)
    ctr = np.zeros(4, dtype=np.uint64)
    _load().oracle_prp_build(_p(req), n, _p(lut), lut.shape[0], heap_size, arena_base,
                             arena_cap_pages, _p(arena), _p(prp), _p(page_base), _p(status),
                             _p(ctr), int(zero_tail))
    return dict(prp=prp, page_base=page_base, status=status, ctr=ctr,
                arena=arena[:arena_cap_pages] if lists else None)


# ------------------------------------------------------------------------ MR
def mr_round(addr: int, size: int):
    """(valid, base, aend) of one range rounded to whole 4 KiB pages."""
    out = np.zeros(3, dtype=np.uint64)
    _load().oracle_mr_round(addr, size, _p(out))
    return bool(out[0]), int(out[1]), int(out[2])


def _mr(fn_name, queries, start, end, lkey):
    q = _u64(queries).reshape(-1, 2)
    start, end = _u64(start), _u64(end)
    lkey = np.ascontiguousarray(lkey, dtype=np.uint32)
    n = q.shape[0]
    idx = np.zeros(n, dtype=np.int32)
    lk = np.zeros(n, dtype=np.uint32)
    kind = np.zeros(n, dtype=np.uint8)
    getattr(_load(), fn_name)(_p(q), n, _p(start), _p(end), _p(lkey), start.shape[0],
                              _p(idx), _p(lk), _p(kind))
    return dict(idx=idx, lkey=lk, kind=kind)


def mr_linear(queries, start, end, lkey) -> dict:
    """The definition: first containing range by index, for every query."""
    return _mr("oracle_mr_linear", queries, start, end, lkey)


def mr_prefix_max(queries, start, end, lkey) -> dict:
    """Same result for tables sorted by start whose ranges may overlap."""
    return _mr("oracle_mr_prefix_max", queries, start, end, lkey)


def mr_bsearch(queries, start, end, lkey) -> dict:
    """Same result for sorted non-overlapping tables, by binary search."""
    return _mr("oracle_mr_bsearch", queries, start, end, lkey)


MR_HIT_EXACT, MR_HIT_CONTAINED, MR_NEW, MR_NEW_DUP = 1, 2, 4, 5
DEREG_OK, DEREG_RELEASED, DEREG_STALE = 0, 1, 2


def _table(start, end, lkey, refs):
    return (_u64(start), _u64(end), np.ascontiguousarray(lkey, dtype=np.uint32),
            np.ascontiguousarray(refs, dtype=np.uint32))


def mr_register(queries, new_lkey, start, end, lkey, refs, granule_shift: int = 12,
                out_cap: int | None = None, one_at_a_time: bool = False,
                indexed: bool = False) -> dict:
    """A batch of registrations against a table sorted by start (records may
    overlap). Returns the table after the batch (start, end, lkey, refs,
    trimmed to its size), handle / kind per request, remap per old record and
    ctr [records after, invalid, overflow, error bits]. With one_at_a_time,
    the pages' per-call definition (each request looked up in the table as
    the requests before it left it) instead of the batch reading; with
    indexed as well, the same definition computed with an index (for large
    batches; pinned equal to the scan)."""
    q = _u64(queries).reshape(-1, 2)
    start, end, lkey, refs = _table(start, end, lkey, refs)
    new_lkey = np.ascontiguousarray(new_lkey, dtype=np.uint32)
    n_q, n = q.shape[0], start.shape[0]
    cap = n + n_q if out_cap is None else out_cap
    o = dict(start=np.zeros(max(cap, 1), np.uint64), end=np.zeros(max(cap, 1), np.uint64),
             lkey=np.zeros(max(cap, 1), np.uint32), refs=np.zeros(max(cap, 1), np.uint32))
    handle = np.full(max(n_q, 1), -1, dtype=np.int64)
    kind = np.zeros(max(n_q, 1), dtype=np.uint8)
    remap = np.full(max(n, 1), -1, dtype=np.int64)
    ctr = np.zeros(4, dtype=np.uint64)
    if one_at_a_time:
        fn = "oracle_mr_register_seq_indexed" if indexed else "oracle_mr_register_seq"
        getattr(_load(), fn)(_p(q), n_q, _p(new_lkey), granule_shift, _p(start), _p(end),
                             _p(lkey), _p(refs), n, _p(o["start"]), _p(o["end"]), _p(o["lkey"]),
                             _p(o["refs"]), cap, _p(handle), _p(kind), _p(remap), _p(ctr))
    else:
        _load().oracle_mr_register(_p(q), n_q, _p(new_lkey), granule_shift, _p(start), _p(end),
                                   _p(lkey), _p(refs), n, _p(o["start"]), _p(o["end"]),
                                   _p(o["lkey"]), _p(o["refs"]), cap, _p(handle), _p(kind),
                                   _p(remap), _p(ctr))
    m = int(ctr[0]) if int(ctr[2]) == 0 else 0
    return dict(start=o["start"][:m], end=o["end"][:m], lkey=o["lkey"][:m], refs=o["refs"][:m],
                handle=handle[:n_q], kind=kind[:n_q], remap=remap[:n], ctr=ctr)


def mr_deregister(handles, start, end, lkey, refs) -> dict:
    """A batch of deregistrations (record indices), applied in batch order."""
    h = np.ascontiguousarray(handles, dtype=np.int64)
    start, end, lkey, refs = _table(start, end, lkey, refs)
    n = start.shape[0]
    o = dict(start=np.zeros(max(n, 1), np.uint64), end=np.zeros(max(n, 1), np.uint64),
             lkey=np.zeros(max(n, 1), np.uint32), refs=np.zeros(max(n, 1), np.uint32))
    remap = np.full(max(n, 1), -1, dtype=np.int64)
    status = np.zeros(max(h.shape[0], 1), dtype=np.uint8)
    ctr = np.zeros(4, dtype=np.uint64)
    _load().oracle_mr_deregister(_p(h), h.shape[0], _p(start), _p(end), _p(lkey), _p(refs), n,
                                 _p(o["start"]), _p(o["end"]), _p(o["lkey"]), _p(o["refs"]),
                                 _p(remap), _p(status), _p(ctr))
    m = int(ctr[0])
    return dict(start=o["start"][:m], end=o["end"][:m], lkey=o["lkey"][:m], refs=o["refs"][:m],
                remap=remap[:n], status=status[:h.shape[0]], ctr=ctr)


# ----------------------------------------------------------------------- WQE
def wqe_bucket(req, peer_ptrs, rkeys, world: int, n_qp: int, local_base: int, lkey: int,
               heap_size: int, depth: int, head, fill: int = 0,
               rings: np.ndarray | None = None) -> dict:
    """Whole batch; returns rings [R, depth, 64] u8, head, count, ctr.
    ``rings`` may be given preallocated."""
    req = _u64(req).reshape(-1, 2)
    peer_ptrs = _u64(peer_ptrs)
    rkeys = np.ascontiguousarray(rkeys, dtype=np.uint32)
    n_rings = world * n_qp
    if rings is None:
        rings = np.full((n_rings, depth, 64), fill, dtype=np.uint8)
    else:
        assert rings.dtype == np.uint8 and rings.shape == (n_rings, depth, 64)
    head = _u64(head).copy()
    count = np.zeros(n_rings, dtype=np.uint32)
    ctr = np.zeros(4, dtype=np.uint64)
    _load().oracle_wqe_bucket(_p(req), req.shape[0], _p(peer_ptrs), _p(rkeys), world, n_qp,
                              local_base, lkey, heap_size, _p(rings), depth, _p(head),
                              _p(count), _p(ctr))
    return dict(rings=rings, head=head, count=count, ctr=ctr)


DIRECT_DTYPE = np.dtype([("dst", "<u8"), ("src", "<u8"), ("len", "<u4"), ("req_index", "<u4"),
                         ("pe", "<u2"), ("transport", "u1"), ("rsvd0", "u1"), ("rsvd1", "<u4")])
XPORT_RDMA, XPORT_P2P, XPORT_SDMA = 0, 1, 2


def wqe_bucket_transport(req, peer_ptrs, rkeys, transport, world: int, n_qp: int,
                         local_base: int, lkey: int, heap_size: int, depth: int, head,
                         fill: int = 0, rings: np.ndarray | None = None) -> dict:
    """Puts dispatched on their target PE's transport: RDMA puts become WQEs
    in their rings (as wqe_bucket), P2P and SDMA puts direct descriptors in
    request order. Returns rings, head, count, ctr, direct [n_direct, 32] u8
    and n_direct."""
    req = _u64(req).reshape(-1, 2)
    peer_ptrs = _u64(peer_ptrs)
    rkeys = np.ascontiguousarray(rkeys, dtype=np.uint32)
    transport = np.ascontiguousarray(transport, dtype=np.uint8)
    assert transport.shape[0] >= world
    n_rings = world * n_qp
    if rings is None:
        rings = np.full((n_rings, depth, 64), fill, dtype=np.uint8)
    else:
        assert rings.dtype == np.uint8 and rings.shape == (n_rings, depth, 64)
    head = _u64(head).copy()
    count = np.zeros(n_rings, dtype=np.uint32)
    ctr = np.zeros(4, dtype=np.uint64)
    n = req.shape[0]
    direct = np.full((max(n, 1), 32), fill, dtype=np.uint8)
    nd = np.zeros(1, dtype=np.uint64)
    _load().oracle_wqe_bucket_transport(_p(req), n, _p(peer_ptrs), _p(rkeys), _p(transport),
                                        world, n_qp, local_base, lkey, heap_size, _p(rings),
                                        depth, _p(head), _p(count), _p(ctr), _p(direct), _p(nd))
    k = int(nd[0])
    return dict(rings=rings, head=head, count=count, ctr=ctr, direct=direct[:k], n_direct=k)


def wqe_bucket_vmm(req, chunk_raddr, chunk_rkey, chunk_lkey, chunk_shift: int, world: int,
                   n_qp: int, local_base: int, heap_size: int, depth: int, head,
                   fill: int = 0, rings: np.ndarray | None = None, mtu: int = 0,
                   psn_head=None) -> dict:
    """Put translation on a VMM heap: one WQE per chunk a put touches.
    chunk_raddr / chunk_rkey are [world, n_chunks], chunk_lkey [n_chunks].
    With an mtu, each WQE gets its first PSN; psn_head is updated."""
    req = _u64(req).reshape(-1, 2)
    n_chunks = -(-heap_size // (1 << chunk_shift))
    chunk_raddr = _u64(chunk_raddr).reshape(-1)
    chunk_rkey = np.ascontiguousarray(chunk_rkey, dtype=np.uint32).reshape(-1)
    chunk_lkey = np.ascontiguousarray(chunk_lkey, dtype=np.uint32).reshape(-1)
    assert chunk_raddr.shape[0] == world * n_chunks and chunk_rkey.shape[0] == world * n_chunks
    assert chunk_lkey.shape[0] == n_chunks
    n_rings = world * n_qp
    if rings is None:
        rings = np.full((n_rings, depth, 64), fill, dtype=np.uint8)
    else:
        assert rings.dtype == np.uint8 and rings.shape == (n_rings, depth, 64)
    head = _u64(head).copy()
    psn = _u64(psn_head if psn_head is not None else np.zeros(n_rings)).copy()
    count = np.zeros(n_rings, dtype=np.uint32)
    ctr = np.zeros(4, dtype=np.uint64)
    _load().oracle_wqe_bucket_vmm(_p(req), req.shape[0], _p(chunk_raddr), _p(chunk_rkey),
                                  _p(chunk_lkey), chunk_shift, world, n_qp, local_base,
                                  heap_size, _p(rings), depth, _p(head), mtu, _p(psn),
                                  _p(count), _p(ctr))
    out = dict(rings=rings, head=head, count=count, ctr=ctr)
    if mtu:
        out["psn_head"] = psn
    return out


# ------------------------------------------------------------------ CQ mirror
def cq_mirror_pass(dev_cq: np.ndarray, head: int, phase: int, host_cq: np.ndarray,
                   max_entries: int | None = None):
    """One mirror pass over a completion queue ([depth, 4] uint32 entries):
    copies the entries whose phase tag is the expected one into ``host_cq``
    (in place). Returns (copied, head, phase)."""
    assert dev_cq.dtype == np.uint32 and dev_cq.shape[1] == 4 and dev_cq.flags["C_CONTIGUOUS"]
    assert host_cq.dtype == np.uint32 and host_cq.shape == dev_cq.shape
    assert host_cq.flags["C_CONTIGUOUS"]
    depth = dev_cq.shape[0]
    h = np.array([head], dtype=np.uint32)
    ph = np.array([phase], dtype=np.uint32)
    n = _load().oracle_cq_mirror_pass(_p(dev_cq), depth, _p(h), _p(ph), _p(host_cq),
                                      depth if max_entries is None else max_entries)
    return int(n), int(h[0]), int(ph[0])


def cq_ack(cur: int, now: int, keep: int) -> int:
    """Acknowledgement after working under generation ``cur`` and finding ``now``."""
    return int(_load().oracle_cq_ack(cur, now, keep))
