"""Seeded synthetic inputs for the descriptor-building workloads.

This module only draws inputs. It holds none of the arithmetic of the
methods themselves (no page counting, no rounding, no address translation,
no bucketing): the same arrays feed the CUDA library, the CPU oracle, the
tests and the benchmark.

Every generator takes an integer seed and uses numpy's PCG64 bit generator,
so a seed fixes the inputs on one machine. Shapes and value distributions
follow the five workloads of the descriptor-building study:

* ``prp_tiny``    1 GiB heap, 4,096 requests of 512 B .. 128 KiB, plus a
                  64-range registration table over the heap.
* ``prp_small``   1 GiB heap, 1,048,576 requests of 512 B .. 4 KiB.
* ``prp_large``   16 GiB heap, 4,194,304 requests, log-uniform 4 KiB .. 4 MiB.
* ``mr_lookup``   1,048,576 registered ranges over a 48-bit space and
                  16,777,216 query ranges (40 % exact, 40 % contained,
                  20 % miss).
* ``put_bucket``  8 PEs x 4 queues, 8,388,608 puts of 16 B .. 64 KiB.

Request records are returned as ``uint64`` arrays of shape ``[n, 2]``:

* PRP request:  word 0 = heap offset, word 1 = length (low 32 bits).
* MR query:     word 0 = address, word 1 = size.
* put request:  word 0 = heap offset, word 1 = bytes | pe << 32 | qp << 48.
"""

from __future__ import annotations

import numpy as np

KiB = 1024
MiB = 1024 * KiB
GiB = 1024 * MiB

SEED_BASE = 0xDB5EED00

# Workload names in the order of the study's configuration list.
WORKLOADS = ("prp_tiny", "prp_small", "prp_large", "mr_lookup", "put_bucket", "put_bucket_vmm",
             "mr_lookup_overlap", "mr_register", "mr_deregister", "put_bucket_transport")


def seed_of(name: str) -> int:
    """Default seed of a named workload."""
    return SEED_BASE + WORKLOADS.index(name)


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def pack_prp_requests(off: np.ndarray, length: np.ndarray) -> np.ndarray:
    """AoS PRP requests {u64 off; u32 len; u32 rsvd=0} as uint64 [n, 2]."""
    off = np.asarray(off, dtype=np.uint64)
    length = np.asarray(length, dtype=np.uint64)
    out = np.empty((off.shape[0], 2), dtype=np.uint64)
    out[:, 0] = off
    out[:, 1] = length & np.uint64(0xFFFFFFFF)
    return out


def pack_ranges(addr: np.ndarray, size: np.ndarray) -> np.ndarray:
    """AoS ranges {u64 addr; u64 size} as uint64 [n, 2]."""
    out = np.empty((np.asarray(addr).shape[0], 2), dtype=np.uint64)
    out[:, 0] = np.asarray(addr, dtype=np.uint64)
    out[:, 1] = np.asarray(size, dtype=np.uint64)
    return out


def pack_put_requests(off, nbytes, pe, qp) -> np.ndarray:
    """AoS puts {u64 off; u32 bytes; u16 pe; u16 qp} as uint64 [n, 2]."""
    off = np.asarray(off, dtype=np.uint64)
    out = np.empty((off.shape[0], 2), dtype=np.uint64)
    out[:, 0] = off
    out[:, 1] = (np.asarray(nbytes, dtype=np.uint64) & np.uint64(0xFFFFFFFF)) \
        | ((np.asarray(pe, dtype=np.uint64) & np.uint64(0xFFFF)) << np.uint64(32)) \
        | ((np.asarray(qp, dtype=np.uint64) & np.uint64(0xFFFF)) << np.uint64(48))
    return out


def physical_lut(rng: np.random.Generator, n_entries: int) -> np.ndarray:
    """Distinct, non-zero, 64 KiB-aligned bus addresses, one per 64 KiB chunk.

    Frame numbers are drawn uniformly from [1, 2^32) and redrawn on
    duplicates, so addresses lie in [64 KiB, 2^48).
    """
    frames = rng.integers(1, 1 << 32, size=n_entries, dtype=np.uint64)
    while True:
        _, first = np.unique(frames, return_index=True)
        if first.shape[0] == n_entries:
            break
        dup = np.ones(n_entries, dtype=bool)
        dup[first] = False
        frames[dup] = rng.integers(1, 1 << 32, size=int(dup.sum()), dtype=np.uint64)
    return frames << np.uint64(16)


def prp_tiny(seed: int | None = None) -> dict:
    """4,096 requests on a 1 GiB heap, plus a 64-range registration table.

    Offsets are uniform 4-byte-aligned in the heap, lengths uniform multiples
    of 512 B in [512 B, 128 KiB], clipped at the heap end. The table holds 64
    non-overlapping 4 KiB-aligned ranges covering about 70 % of the heap; the
    same (offset, length) pairs serve as its query ranges.
    """
    rng = _rng(seed_of("prp_tiny") if seed is None else seed)
    heap = 1 * GiB
    n = 4096
    lut = physical_lut(rng, heap // (64 * KiB))
    off = np.uint64(4) * rng.integers(0, heap // 4, size=n, dtype=np.uint64)
    length = np.uint64(512) * rng.integers(1, 257, size=n, dtype=np.uint64)
    length = np.minimum(length, np.uint64(heap) - off)
    # 64 slots cut at sorted distinct page boundaries; each registered range
    # takes the first ~70 % of its slot (at least one page).
    pages = heap // 4096
    cuts = np.sort(rng.choice(np.arange(1, pages, dtype=np.int64), size=63, replace=False))
    lo = np.concatenate(([0], cuts)).astype(np.int64)
    hi = np.concatenate((cuts, [pages])).astype(np.int64)
    span = np.maximum(1, (0.7 * (hi - lo)).astype(np.int64))
    mr_start = (lo * 4096).astype(np.uint64)
    mr_end = ((lo + span) * 4096).astype(np.uint64)
    mr_lkey = rng.integers(0, 1 << 32, size=64, dtype=np.uint64).astype(np.uint32)
    return dict(name="prp_tiny", heap_size=heap, lut=lut,
                req=pack_prp_requests(off, length),
                arena_base=0x1_0000_0000,
                mr_start=mr_start, mr_end=mr_end, mr_lkey=mr_lkey,
                queries=pack_ranges(off, length))


def prp_small(seed: int | None = None, n: int = 1_048_576) -> dict:
    """Small-I/O regime: 60 % 4 KiB-aligned, 40 % 512 B-aligned offsets.

    Lengths are uniform over {512, 1024, 2048, 4096} B and every request lies
    inside the 1 GiB heap. The 512 B-aligned offsets are never 4 KiB-aligned.
    """
    rng = _rng(seed_of("prp_small") if seed is None else seed)
    heap = 1 * GiB
    lut = physical_lut(rng, heap // (64 * KiB))
    length = np.uint64(512) << rng.integers(0, 4, size=n, dtype=np.uint64)
    aligned = rng.random(n) < 0.6
    # Pick the 4 KiB page first, then a sub-page offset; keep the end in the heap.
    last_page = (np.uint64(heap) - length) // np.uint64(4096)
    page = (rng.random(n) * (last_page.astype(np.float64) + 1)).astype(np.uint64)
    page = np.minimum(page, last_page)
    sub = np.uint64(512) * rng.integers(1, 8, size=n, dtype=np.uint64)
    off = page * np.uint64(4096) + np.where(aligned, np.uint64(0), sub)
    over = off + length > np.uint64(heap)
    off[over] -= np.uint64(4096)
    return dict(name="prp_small", heap_size=heap, lut=lut,
                req=pack_prp_requests(off, length), arena_base=0x1_0000_0000)


def prp_large(seed: int | None = None, n: int = 4_194_304) -> dict:
    """Large/chained regime on a 16 GiB heap.

    Lengths are 512 * round(8 * exp(U * ln 1024)) bytes, a log-uniform spread
    over 4 KiB .. 4 MiB in 512 B multiples. 90 % of offsets are 4 KiB-aligned;
    10 % are 4-byte-aligned with a non-zero in-page offset.
    """
    rng = _rng(seed_of("prp_large") if seed is None else seed)
    heap = 16 * GiB
    lut = physical_lut(rng, heap // (64 * KiB))
    units = np.rint(8.0 * np.exp(rng.random(n) * np.log(1024.0))).astype(np.uint64)
    length = np.uint64(512) * units
    unaligned = rng.random(n) < 0.1
    last_page = (np.uint64(heap) - length) // np.uint64(4096) - np.uint64(1)
    page = (rng.random(n) * (last_page.astype(np.float64) + 1)).astype(np.uint64)
    page = np.minimum(page, last_page)
    sub = np.uint64(4) * rng.integers(1, 1024, size=n, dtype=np.uint64)
    off = page * np.uint64(4096) + np.where(unaligned, sub, np.uint64(0))
    return dict(name="prp_large", heap_size=heap, lut=lut,
                req=pack_prp_requests(off, length), arena_base=0x1_0000_0000)


def mr_table(rng: np.random.Generator, n_mr: int, va_bits: int = 48):
    """Sorted, non-overlapping registered ranges over a ``va_bits`` space.

    Sizes are 4096 * round(exp(U * ln 16384)) bytes (4 KiB .. 64 MiB).
    One gap in eight is zero (adjacent ranges); the others are
    4096 * U[1, 2g] bytes with g chosen so the last range ends below 2^va_bits.
    Returns (start, end, lkey, gap_pages_before).
    """
    pages = np.rint(np.exp(rng.random(n_mr) * np.log(16384.0))).astype(np.uint64)
    pages = np.maximum(pages, np.uint64(1))
    total_pages = int(pages.sum())
    space_pages = (1 << (va_bits - 12)) - 1
    free_pages = space_pages - total_pages
    n_gap = max(1, int(n_mr * 7 / 8))
    g = max(1, int(0.9 * free_pages / n_gap))
    gaps = rng.integers(1, 2 * g + 1, size=n_mr, dtype=np.uint64)
    gaps[rng.random(n_mr) < 0.125] = 0
    gaps[0] = max(int(gaps[0]), 1)
    # Scale down if the draw overshoots the space (rare).
    while int(gaps.sum()) + total_pages >= space_pages:
        gaps //= np.uint64(2)
    start_pages = np.cumsum(gaps + pages) - pages
    start = start_pages * np.uint64(4096)
    end = start + pages * np.uint64(4096)
    lkey = rng.integers(0, 1 << 32, size=n_mr, dtype=np.uint64).astype(np.uint32)
    return start, end, lkey, gaps


def mr_lookup(seed: int | None = None, n_mr: int = 1_048_576,
              n_q: int = 16_777_216) -> dict:
    """Registration table plus query ranges with a fixed kind mix.

    Queries pick a registered range uniformly by index, then:
    40 % the same range (half exactly aligned, half with in-page slack on
    both ends), 40 % a strictly smaller page run inside a range of at least
    two pages (with in-page slack), 20 % a miss (half inside a non-empty gap,
    half straddling a range's end by at least one page on each side).
    """
    rng = _rng(seed_of("mr_lookup") if seed is None else seed)
    start, end, lkey, gaps = mr_table(rng, n_mr)
    pages = (end - start) // np.uint64(4096)
    u = rng.random(n_q)
    kind = np.where(u < 0.4, 0, np.where(u < 0.8, 1, 2))
    addr = np.empty(n_q, dtype=np.uint64)
    stop = np.empty(n_q, dtype=np.uint64)  # exclusive end of the query
    P = np.uint64(4096)

    # Same range: half aligned, half with slack a (front) and b (back), a + b < 4096.
    e = np.flatnonzero(kind == 0)
    m = rng.integers(0, n_mr, size=e.shape[0])
    slack = rng.random(e.shape[0]) < 0.5
    a = rng.integers(0, 4096, size=e.shape[0], dtype=np.uint64)
    b = rng.integers(0, 4096, size=e.shape[0], dtype=np.uint64)
    b = np.where(a + b >= P, P - np.uint64(1) - a, b)
    a = np.where(slack, a, np.uint64(0))
    b = np.where(slack, b, np.uint64(0))
    addr[e] = start[m] + a
    stop[e] = end[m] - b

    # Strictly contained: a page run [p0, p1) of a >= 2-page range, not the whole.
    c = np.flatnonzero(kind == 1)
    multi = np.flatnonzero(pages >= 2)
    m = multi[rng.integers(0, multi.shape[0], size=c.shape[0])]
    npg = pages[m].astype(np.int64)
    p0 = (rng.random(c.shape[0]) * npg).astype(np.int64)
    p0 = np.minimum(p0, npg - 1)
    p1 = p0 + 1 + (rng.random(c.shape[0]) * (npg - p0)).astype(np.int64)
    p1 = np.minimum(p1, npg)
    whole = (p0 == 0) & (p1 == npg)
    # Shrink the whole-range draws by one page at a random end.
    front = rng.random(c.shape[0]) < 0.5
    p0 = np.where(whole & front, 1, p0)
    p1 = np.where(whole & ~front, npg - 1, p1)
    a = rng.integers(0, 4096, size=c.shape[0], dtype=np.uint64)
    b = rng.integers(0, 4096, size=c.shape[0], dtype=np.uint64)
    b = np.where((p1 - p0 == 1) & (a + b >= P), P - np.uint64(1) - a, b)
    addr[c] = start[m] + p0.astype(np.uint64) * P + a
    stop[c] = start[m] + p1.astype(np.uint64) * P - b

    # Miss: inside a non-empty gap, or straddling a range end.
    x = np.flatnonzero(kind == 2)
    in_gap = rng.random(x.shape[0]) < 0.5
    gi = np.flatnonzero(gaps > 0)
    g = gi[rng.integers(0, gi.shape[0], size=x.shape[0])]
    gap_lo = np.where(g == 0, np.uint64(0), end[np.maximum(g - 1, 0)])
    gpg = gaps[g].astype(np.int64)
    q0 = (rng.random(x.shape[0]) * gpg).astype(np.int64)
    q0 = np.minimum(q0, gpg - 1)
    q1 = q0 + 1 + (rng.random(x.shape[0]) * (gpg - q0)).astype(np.int64)
    q1 = np.minimum(q1, gpg)
    gap_addr = gap_lo + q0.astype(np.uint64) * P
    gap_stop = gap_lo + q1.astype(np.uint64) * P
    m = rng.integers(0, n_mr - 1, size=x.shape[0])
    back = 1 + (rng.random(x.shape[0]) * pages[m].astype(np.float64)).astype(np.uint64)
    back = np.minimum(back, pages[m])
    ahead = 1 + rng.integers(0, 16, size=x.shape[0], dtype=np.uint64)
    st_addr = end[m] - back * P
    st_stop = end[m] + ahead * P
    addr[x] = np.where(in_gap, gap_addr, st_addr)
    stop[x] = np.where(in_gap, gap_stop, st_stop)

    return dict(name="mr_lookup", mr_start=start, mr_end=end, mr_lkey=lkey,
                queries=pack_ranges(addr, stop - addr), query_mix=kind)


def mr_lookup_overlap(seed: int | None = None, n_mr: int = 1_048_576,
                      n_q: int = 16_777_216, extra: float = 0.25) -> dict:
    """A registration table whose records overlap, plus query ranges.

    The disjoint table of ``mr_table`` gets ``extra * n_mr`` more records,
    each for a range that straddles an existing record's end (from 1 page
    up to the whole record before it, 1 .. 64 pages after): the ranges a
    cache registers anew after a partial-overlap miss. The merged table is
    sorted by start (stably, so an original record precedes an extra one
    with the same start). Queries pick a merged record uniformly: 40 % the
    record itself (half with in-page slack), 40 % a page run inside it,
    20 % a range straddling its end by 1 .. 128 pages. Which record answers
    a query depends on the overlaps, so no kind is fixed by the mix.
    """
    rng = _rng(seed_of("mr_lookup_overlap") if seed is None else seed)
    start, end, lkey, _ = mr_table(rng, n_mr)
    P = np.uint64(4096)
    pages = (end - start) // P
    n_x = int(n_mr * extra)
    m = rng.integers(0, n_mr, size=n_x)
    back = 1 + (rng.random(n_x) * pages[m].astype(np.float64)).astype(np.uint64)
    back = np.minimum(back, pages[m])
    ahead = 1 + rng.integers(0, 64, size=n_x, dtype=np.uint64)
    xs = end[m] - back * P
    xe = end[m] + ahead * P
    xk = rng.integers(0, 1 << 32, size=n_x, dtype=np.uint64).astype(np.uint32)
    all_s = np.concatenate([start, xs])
    order = np.argsort(all_s, kind="stable")
    start = all_s[order]
    end = np.concatenate([end, xe])[order]
    lkey = np.concatenate([lkey, xk])[order]
    n = start.shape[0]
    pages = (end - start) // P

    u = rng.random(n_q)
    kind = np.where(u < 0.4, 0, np.where(u < 0.8, 1, 2))
    r = rng.integers(0, n, size=n_q)
    npg = pages[r]
    a = rng.integers(0, 4096, size=n_q, dtype=np.uint64)
    b = rng.integers(0, 4096, size=n_q, dtype=np.uint64)
    b = np.where(a + b >= P, P - np.uint64(1) - a, b)
    slack = rng.random(n_q) < 0.5
    # 0: the record, with or without slack
    addr0 = start[r] + np.where(slack, a, np.uint64(0))
    stop0 = end[r] - np.where(slack, b, np.uint64(0))
    # 1: a page run [p0, p1) inside the record
    p0 = np.minimum((rng.random(n_q) * npg.astype(np.float64)).astype(np.uint64), npg - np.uint64(1))
    p1 = p0 + np.uint64(1) + (rng.random(n_q) * (npg - p0).astype(np.float64)).astype(np.uint64)
    p1 = np.minimum(p1, npg)
    addr1 = start[r] + p0 * P + a
    stop1 = start[r] + p1 * P - np.where(p1 - p0 == np.uint64(1), np.minimum(b, P - np.uint64(1) - a), b)
    # 2: straddling the record's end
    bk = np.minimum(np.uint64(1) + (rng.random(n_q) * npg.astype(np.float64)).astype(np.uint64), npg)
    addr2 = end[r] - bk * P
    stop2 = end[r] + (np.uint64(1) + rng.integers(0, 128, size=n_q, dtype=np.uint64)) * P
    addr = np.where(kind == 0, addr0, np.where(kind == 1, addr1, addr2))
    stop = np.where(kind == 0, stop0, np.where(kind == 1, stop1, stop2))
    return dict(name="mr_lookup_overlap", mr_start=start, mr_end=end, mr_lkey=lkey,
                queries=pack_ranges(addr, stop - addr), query_mix=kind)


def mr_register(seed: int | None = None, n_mr: int = 1_048_576,
                n_q: int = 16_777_216) -> dict:
    """A registration batch: the ``mr_lookup`` table and queries as requests
    (40 % the same range as a record, 40 % inside one, 20 % missing), each
    record holding 1..4 references, and the lkey a new registration for each
    request would get (uniform u32)."""
    d = mr_lookup(seed_of("mr_register") if seed is None else seed, n_mr, n_q)
    rng = _rng((seed_of("mr_register") if seed is None else seed) + 1)
    d["name"] = "mr_register"
    d["mr_refs"] = rng.integers(1, 5, size=n_mr).astype(np.uint32)
    d["new_lkey"] = rng.integers(0, 1 << 32, size=n_q, dtype=np.uint64).astype(np.uint32)
    return d


def mr_deregister(seed: int | None = None, n_mr: int = 1_048_576,
                  n_h: int = 2_097_152) -> dict:
    """A deregistration batch over the ``mr_lookup`` table with 1..4
    references per record: 94 % of the handles name a record (uniform), 3 %
    are -1 and 3 % lie past the table, so some records lose every reference
    and some handles arrive after their record was released."""
    s0 = seed_of("mr_deregister") if seed is None else seed
    rng = _rng(s0)
    start, end, lkey, _ = mr_table(rng, n_mr)
    refs = rng.integers(1, 5, size=n_mr).astype(np.uint32)
    h = rng.integers(0, n_mr, size=n_h).astype(np.int64)
    u = rng.random(n_h)
    h = np.where(u < 0.03, -1, np.where(u < 0.06, n_mr + rng.integers(0, n_mr, size=n_h), h))
    return dict(name="mr_deregister", mr_start=start, mr_end=end, mr_lkey=lkey, mr_refs=refs,
                handles=h.astype(np.int64))


def put_bucket(seed: int | None = None, n: int = 8_388_608, world: int = 8,
               n_qp: int = 4, depth: int = 1 << 19) -> dict:
    """Symmetric-heap puts over ``world`` PEs x ``n_qp`` queues.

    peerPtrs are random 2 MiB-aligned bases in [2^40, 2^47), rkeys random
    u32, the local base 2 MiB-aligned, the lkey random. Each put has pe and
    qp uniform, bytes = 16 * U[1, 4096] and a 16 B-aligned offset uniform in
    a 4 GiB heap with offset + bytes inside the heap.
    """
    rng = _rng(seed_of("put_bucket") if seed is None else seed)
    heap = 4 * GiB
    two_mib = 2 * MiB
    peer_ptrs = rng.integers((1 << 40) // two_mib, (1 << 47) // two_mib,
                             size=world, dtype=np.uint64) * np.uint64(two_mib)
    rkeys = rng.integers(0, 1 << 32, size=world, dtype=np.uint64).astype(np.uint32)
    local_base = int(rng.integers((1 << 40) // two_mib, (1 << 47) // two_mib)) * two_mib
    lkey = int(rng.integers(0, 1 << 32))
    pe = rng.integers(0, world, size=n, dtype=np.uint64)
    qp = rng.integers(0, n_qp, size=n, dtype=np.uint64)
    nbytes = np.uint64(16) * rng.integers(1, 4097, size=n, dtype=np.uint64)
    slots = (np.uint64(heap) - nbytes) // np.uint64(16)
    off = np.uint64(16) * np.minimum(
        (rng.random(n) * (slots.astype(np.float64) + 1)).astype(np.uint64), slots)
    return dict(name="put_bucket", heap_size=heap, world=world, n_qp=n_qp,
                depth=depth, peer_ptrs=peer_ptrs, rkeys=rkeys,
                local_base=local_base, lkey=lkey,
                req=pack_put_requests(off, nbytes, pe, qp),
                head=np.zeros(world * n_qp, dtype=np.uint64))


def put_bucket_vmm(seed: int | None = None, n: int = 8_388_608, world: int = 8,
                   n_qp: int = 4, depth: int = 1 << 19, chunk_shift: int = 21) -> dict:
    """The put_bucket batch on a heap of 2^chunk_shift-byte chunks.

    The puts are those of put_bucket (same seed rule). Each chunk c of each PE
    sits at a random 2^chunk_shift-aligned remote address in [2^40, 2^47)
    with a random rkey; each local chunk has a random lkey.
    """
    p = put_bucket(seed, n, world, n_qp, depth)
    rng = _rng((seed_of("put_bucket_vmm") if seed is None else seed) ^ 0x5A5A)
    C = 1 << chunk_shift
    n_chunks = -(-p["heap_size"] // C)
    lo, hi = (1 << 40) // C, (1 << 47) // C
    chunk_raddr = rng.integers(lo, hi, size=(world, n_chunks), dtype=np.uint64) * np.uint64(C)
    chunk_rkey = rng.integers(0, 1 << 32, size=(world, n_chunks), dtype=np.uint64).astype(np.uint32)
    chunk_lkey = rng.integers(0, 1 << 32, size=n_chunks, dtype=np.uint64).astype(np.uint32)
    p.update(name="put_bucket_vmm", chunk_shift=chunk_shift, chunk_raddr=chunk_raddr,
             chunk_rkey=chunk_rkey, chunk_lkey=chunk_lkey)
    return p


def put_bucket_transport(seed: int | None = None, n: int = 8_388_608, world: int = 8,
                         n_qp: int = 4, depth: int = 1 << 19, p2p=(1, 2), sdma=()) -> dict:
    """The put_bucket batch with a transport per PE.

    The puts are those of put_bucket (same seed rule). transport[pe] is 0
    (RDMA) except for the PEs in ``p2p`` (1) and ``sdma`` (2): the PEs on
    this node. Their peer pointers are replaced by the addresses at which
    this process maps their heaps: random 2 MiB-aligned bases in [2^40, 2^47).
    """
    p = put_bucket(seed, n, world, n_qp, depth)
    rng = _rng((seed_of("put_bucket_transport") if seed is None else seed) ^ 0x3C3C)
    transport = np.zeros(world, dtype=np.uint8)
    transport[list(p2p)] = 1
    transport[list(sdma)] = 2
    two_mib = 2 * MiB
    mapped = rng.integers((1 << 40) // two_mib, (1 << 47) // two_mib,
                          size=world, dtype=np.uint64) * np.uint64(two_mib)
    peer = p["peer_ptrs"].copy()
    peer[transport != 0] = mapped[transport != 0]
    p.update(name="put_bucket_transport", transport=transport, peer_ptrs=peer)
    return p


GENERATORS = {
    "prp_tiny": prp_tiny,
    "prp_small": prp_small,
    "prp_large": prp_large,
    "mr_lookup": mr_lookup,
    "put_bucket": put_bucket,
    "put_bucket_vmm": put_bucket_vmm,
    "put_bucket_transport": put_bucket_transport,
}
