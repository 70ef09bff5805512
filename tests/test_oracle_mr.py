"""Pins for the MR-lookup oracle.

Follows "NCCL expert course 26" ("IB Backend MR Cache": page rounding worked
table, containment reuse, partial overlap is no hit; "Communicator User
Registration Cache": page_floor/page_cover on sorted records; the
ncclCommRegister semantics experiment).
"""

import numpy as np
import pytest

from conftest import h, load_golden

PAGE = 4096


def test_rounding_worked_table(oracle):
    fx = load_golden("mr_hand_cases.json")["rounding"]
    for c in fx["cases"]:
        ok, base, aend = oracle.mr_round(h(c["addr"]), c["size"])
        assert ok
        assert base == h(c["base"])
        assert (aend - base) // PAGE == c["pages"]


@pytest.mark.parametrize("section", ["registration_experiment", "partial_overlap"])
def test_hand_cases(oracle, section):
    fx = load_golden("mr_hand_cases.json")[section]
    base = h(fx.get("alloc_base", "0x0"))
    start = np.array([base + h(r["start"]) for r in fx["table"]], dtype=np.uint64)
    end = np.array([base + h(r["end"]) for r in fx["table"]], dtype=np.uint64)
    lkey = np.array([r["lkey"] for r in fx["table"]], dtype=np.uint32)
    q = np.array([[(base + h(x["off"])) & (2**64 - 1), x["size"]] for x in fx["queries"]],
                 dtype=np.uint64)
    for fn in (oracle.mr_linear, oracle.mr_bsearch):
        out = fn(q, start, end, lkey)
        assert out["kind"].tolist() == [x["kind"] for x in fx["queries"]]
        assert out["idx"].tolist() == [x["idx"] for x in fx["queries"]]
        assert out["lkey"].tolist() == [x["lkey"] for x in fx["queries"]]


def brute_force_kind(addr, size, table):
    """Page sets: a query hits record i when every 4 KiB page the query touches
    lies in the record's page set; exact when the page sets are equal."""
    if size == 0 or addr + size > 2**64 - PAGE:
        return 3, -1
    qp = set(range(addr // PAGE, (addr + size - 1) // PAGE + 1))
    for i, (s, e) in enumerate(table):
        rp = set(range(s // PAGE, e // PAGE))
        if qp <= rp:
            return (1 if qp == rp else 2), i
    return 0, -1


def random_sorted_table(rng, n, span_pages=400):
    cuts = np.sort(rng.choice(np.arange(1, span_pages), size=2 * n, replace=False))
    start = cuts[0::2].astype(np.uint64) * PAGE
    end = cuts[1::2].astype(np.uint64) * PAGE
    return start, end


def test_brute_force_tiny_tables(oracle):
    rng = np.random.default_rng(7)
    for trial in range(40):
        n = int(rng.integers(1, 12))
        start, end = random_sorted_table(rng, n)
        lkey = rng.integers(0, 2**32, size=n, dtype=np.uint64).astype(np.uint32)
        nq = 200
        addr = rng.integers(0, 420 * PAGE, size=nq).astype(np.uint64)
        size = rng.integers(0, 40 * PAGE, size=nq).astype(np.uint64)
        q = np.stack([addr, size], axis=1)
        lin = oracle.mr_linear(q, start, end, lkey)
        bs = oracle.mr_bsearch(q, start, end, lkey)
        table = list(zip(start.tolist(), end.tolist()))
        for k in range(nq):
            kind, idx = brute_force_kind(int(addr[k]), int(size[k]), table)
            assert lin["kind"][k] == kind and lin["idx"][k] == idx
            assert lin["lkey"][k] == (lkey[idx] if idx >= 0 else 0)
        for key in ("kind", "idx", "lkey"):
            assert (lin[key] == bs[key]).all()


def test_overlapping_table_lowest_index_wins(oracle):
    # The definition scans by index; with overlapping records the first
    # containing one is returned even when a later one matches exactly.
    start = np.array([0x0, 0x1000], dtype=np.uint64)
    end = np.array([0x10000, 0x2000], dtype=np.uint64)
    lkey = np.array([1, 2], dtype=np.uint32)
    q = np.array([[0x1000, 0x1000]], dtype=np.uint64)
    out = oracle.mr_linear(q, start, end, lkey)
    assert out["idx"][0] == 0 and out["kind"][0] == 2 and out["lkey"][0] == 1


def test_overlap_hand_cases(oracle):
    """Hand-worked values on a table of overlapping records (a partial
    overlap is registered anew), checked against page sets as well."""
    fx = load_golden("mr_hand_cases.json")["overlap_after_partial_miss"]
    table = [(h(r["start"]), h(r["end"])) for r in fx["table"]]
    start = np.array([t[0] for t in table], dtype=np.uint64)
    end = np.array([t[1] for t in table], dtype=np.uint64)
    lkey = np.array([r["lkey"] for r in fx["table"]], dtype=np.uint32)
    q = np.array([[h(x["off"]), x["size"]] for x in fx["queries"]], dtype=np.uint64)
    for x in fx["queries"]:
        assert brute_force_kind(h(x["off"]), x["size"], table) == (x["kind"], x["idx"])
    for fn in (oracle.mr_linear, oracle.mr_prefix_max):
        out = fn(q, start, end, lkey)
        assert out["kind"].tolist() == [x["kind"] for x in fx["queries"]]
        assert out["idx"].tolist() == [x["idx"] for x in fx["queries"]]
        assert out["lkey"].tolist() == [x["lkey"] for x in fx["queries"]]


def test_linear_equals_bsearch_medium(oracle):
    import synth
    rng = np.random.default_rng(11)
    start, end, lkey, _ = synth.mr_table(rng, 3000, va_bits=40)
    d = synth.mr_lookup(seed=5, n_mr=3000, n_q=4000)
    lin = oracle.mr_linear(d["queries"], d["mr_start"], d["mr_end"], d["mr_lkey"])
    bs = oracle.mr_bsearch(d["queries"], d["mr_start"], d["mr_end"], d["mr_lkey"])
    for key in ("kind", "idx", "lkey"):
        assert (lin[key] == bs[key]).all()
    # The generated mix: 40 % exact, 40 % contained, 20 % miss.
    assert (lin["kind"][d["query_mix"] == 0] == 1).all()
    assert (lin["kind"][d["query_mix"] == 1] == 2).all()
    assert (lin["kind"][d["query_mix"] == 2] == 0).all()


def test_edges(oracle):
    start = np.array([0x10000, 0x20000], dtype=np.uint64)
    end = np.array([0x20000, 0x21000], dtype=np.uint64)    # adjacent records
    lkey = np.array([5, 6], dtype=np.uint32)
    q = np.array([
        [0x1FFFF, 1],        # last byte of record 0 -> contained
        [0x20000, 1],        # first byte of the 1-page record 1 -> exact
        [0x1F000, 0x2000],   # spans two adjacent records -> miss
        [0xF000, 0x1000],    # just before record 0 -> miss
        [0x10000, 0x10000],  # the whole of record 0 -> exact
    ], dtype=np.uint64)
    for fn in (oracle.mr_linear, oracle.mr_bsearch):
        out = fn(q, start, end, lkey)
        assert out["kind"].tolist() == [2, 1, 0, 0, 1]
        assert out["idx"].tolist() == [0, 1, -1, -1, 0]
    empty = oracle.mr_linear(q, start[:0], end[:0], lkey[:0])
    assert (empty["kind"] == 0).all() and (empty["idx"] == -1).all()


def overlapping_table(rng, n, span_pages, max_pages):
    """Sorted-by-start ranges that may overlap (page-granular, non-empty)."""
    start = np.sort(rng.integers(0, span_pages, size=n)).astype(np.uint64) * np.uint64(4096)
    pages = rng.integers(1, max_pages + 1, size=n).astype(np.uint64)
    end = start + pages * np.uint64(4096)
    lkey = rng.integers(0, 2**32, size=n, dtype=np.uint64).astype(np.uint32)
    return start, end, lkey


@pytest.mark.parametrize("n,span,maxp", [(1, 10, 3), (7, 20, 8), (50, 200, 40), (300, 2000, 400),
                                          (2000, 100000, 30)])
def test_prefix_max_equals_the_definition_on_overlapping_tables(oracle, n, span, maxp):
    """The O(log N) search for sorted overlapping tables gives the lowest
    containing index, as the linear definition does."""
    rng = np.random.default_rng(n * 7 + span)
    start, end, lkey = overlapping_table(rng, n, span, maxp)
    m = 20000
    a = rng.integers(0, (span + maxp) * 4096, size=m).astype(np.uint64)
    sz = rng.integers(0, 8 * 4096, size=m).astype(np.uint64)
    pick = rng.integers(0, n, size=m)
    a = np.where(rng.random(m) < 0.4, start[pick], a)
    sz = np.where(rng.random(m) < 0.3, end[pick] - start[pick], sz)
    q = np.stack([a, sz], axis=1).astype(np.uint64)
    lin = oracle.mr_linear(q, start, end, lkey)
    pm = oracle.mr_prefix_max(q, start, end, lkey)
    for key in ("idx", "lkey", "kind"):
        assert (lin[key] == pm[key]).all(), key
    assert (lin["kind"] == 1).any() and (lin["kind"] == 2).any() and (lin["kind"] == 0).any()
