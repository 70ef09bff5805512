"""Pins for the MR-cache mutation oracle (registration and deregistration
batches).

Follows "NCCL expert course 26" ("IB Backend MR Cache": a hit takes a
reference, a miss is registered anew, deregistration drops a reference and
removes the MR at zero, an unknown handle is an error; "Communicator User
Registration Cache": records in address order; the ncclCommRegister
experiment) and the xNVMe "uPCIe CUDA" page (xnvme_buf_register refcounts
whole 64 KiB device pages).
"""

import numpy as np
import pytest

from conftest import h, load_golden

G4K, G64K = 12, 16
EMPTY = (np.zeros(0, np.uint64), np.zeros(0, np.uint64), np.zeros(0, np.uint32),
         np.zeros(0, np.uint32))


def table_of(rows):
    return (np.array([h(r["start"]) for r in rows], np.uint64),
            np.array([h(r["end"]) for r in rows], np.uint64),
            np.array([r["lkey"] for r in rows], np.uint32),
            np.array([r["refs"] for r in rows], np.uint32))


def rows_of(out, base=0):
    return [(int(s) - base, int(e) - base, int(k), int(r))
            for s, e, k, r in zip(out["start"], out["end"], out["lkey"], out["refs"])]


def test_page_experiment_one_call_at_a_time(oracle):
    """Each registration its own call: both the batch form and the
    one-at-a-time definition give the page's outcome."""
    fx = load_golden("mr_hand_cases.json")["mutation_experiment"]
    base = h(fx["alloc_base"])
    for one in (False, True):
        t = EMPTY
        for c in fx["register_calls"]:
            q = np.array([[base + h(c["off"]), c["size"]]], np.uint64)
            r = oracle.mr_register(q, [c["new_lkey"]], *t, one_at_a_time=one)
            assert r["kind"].tolist() == [c["kind"]] and r["handle"].tolist() == [c["handle"]]
            assert r["refs"].tolist() == c["refs_after"]
            t = (r["start"], r["end"], r["lkey"], r["refs"])
        want = [(h(x["start"]), h(x["end"]), x["lkey"], x["refs"]) for x in fx["table_after"]]
        assert rows_of(r, base) == want
    dr = fx["deregister_batch"]
    d = oracle.mr_deregister(dr["handles"], *t)
    assert d["status"].tolist() == dr["status"] and d["remap"].tolist() == dr["remap"]
    assert rows_of(d, base) == [(h(x["start"]), h(x["end"]), x["lkey"], x["refs"])
                                for x in dr["table_after"]]
    assert d["ctr"].tolist() == [1, 1, 0, 0]


def test_page_experiment_as_one_batch(oracle):
    fx = load_golden("mr_hand_cases.json")["mutation_experiment"]
    base = h(fx["alloc_base"])
    calls = fx["register_calls"]
    q = np.array([[base + h(c["off"]), c["size"]] for c in calls], np.uint64)
    lk = [c["new_lkey"] for c in calls]
    one = fx["one_batch_reading"]
    r = oracle.mr_register(q, lk, *EMPTY)
    assert r["kind"].tolist() == one["kind"] and r["handle"].tolist() == one["handle"]
    assert rows_of(r, base) == [(h(x["start"]), h(x["end"]), x["lkey"], x["refs"])
                                for x in one["table_after"]]
    want = fx["one_batch"]
    for indexed in (False, True):
        s = oracle.mr_register(q, lk, *EMPTY, one_at_a_time=True, indexed=indexed)
        assert s["kind"].tolist() == want["kind"] and s["handle"].tolist() == want["handle"]
        assert rows_of(s, base) == [(h(x["start"]), h(x["end"]), x["lkey"], x["refs"])
                                    for x in want["table_after"]]


@pytest.mark.parametrize("addr,size,base,end", [
    (0x12345, 10, 0x10000, 0x20000),
    (0x1FFFF, 2, 0x10000, 0x30000),
    (0x20000, 0x10000, 0x20000, 0x30000),
    (0x20000, 0x10001, 0x20000, 0x40000),
])
def test_granule_64k_hand_cases(oracle, addr, size, base, end):
    """xnvme_buf_register covers whole 64 KiB device pages."""
    r = oracle.mr_register(np.array([[addr, size]], np.uint64), [7], *EMPTY, granule_shift=G64K)
    assert r["kind"].tolist() == [4]
    assert (int(r["start"][0]), int(r["end"][0])) == (base, end)


def test_granule_4k_rounds_as_the_lookup_does(oracle):
    rng = np.random.default_rng(4)
    top = 2**64 - 1
    a = rng.integers(0, 2**63, size=300, dtype=np.uint64) * np.uint64(2)
    a[:20] = np.uint64(top - 5000)
    sz = rng.integers(0, 1 << 22, size=300, dtype=np.uint64)
    for x, s in zip(a, sz):
        r = oracle.mr_register(np.array([[x, s]], np.uint64), [1], *EMPTY)
        ok, b, e = oracle.mr_round(int(x), int(s))
        if not ok:
            assert r["kind"].tolist() == [3] and r["handle"].tolist() == [-1]
        else:
            assert (int(r["start"][0]), int(r["end"][0])) == (b, e)
    # the top granule: a range ending inside the last 64 KiB of the space is invalid at 64 KiB
    r = oracle.mr_register(np.array([[2**64 - 0x10000, 1]], np.uint64), [1], *EMPTY,
                           granule_shift=G64K)
    assert r["kind"].tolist() == [3]
    r = oracle.mr_register(np.array([[2**64 - 0x20000, 0x10000]], np.uint64), [1], *EMPTY,
                           granule_shift=G64K)
    assert r["kind"].tolist() == [4]


def disjoint_table(rng, n, span_pages):
    cuts = np.sort(rng.choice(np.arange(1, span_pages), size=2 * n, replace=False))
    s = cuts[0::2].astype(np.uint64) * np.uint64(4096)
    e = cuts[1::2].astype(np.uint64) * np.uint64(4096)
    lk = rng.integers(0, 2**32, size=n, dtype=np.uint64).astype(np.uint32)
    refs = rng.integers(1, 5, size=n).astype(np.uint32)
    return s, e, lk, refs


@pytest.mark.parametrize("seed", range(6))
def test_batch_equals_one_at_a_time_without_nesting(oracle, seed):
    """Hits on old records, new ranges inside the gaps (disjoint from each
    other and from every record), repeats of those new ranges and invalid
    requests: the batch reading gives exactly the per-call result."""
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 60))
    s, e, lk, refs = disjoint_table(rng, n, 3000)
    gaps = [(0 if i == 0 else int(e[i - 1]), int(s[i])) for i in range(n)] + [(int(e[-1]), 3100 * 4096)]
    fresh = []
    for lo, hi in gaps:        # at most one new range per gap, strictly inside it
        if hi - lo >= 3 * 4096 and rng.random() < 0.7:
            a = lo + 4096 * int(rng.integers(1, (hi - lo) // 4096 - 1))
            b = a + 4096 * int(rng.integers(1, (hi - a) // 4096))
            fresh.append((a, b - a))
    reqs = []
    for _ in range(400):
        u = rng.random()
        if u < 0.4:
            i = int(rng.integers(0, n))
            off = 4096 * int(rng.integers(0, (int(e[i]) - int(s[i])) // 4096))
            reqs.append((int(s[i]) + off + int(rng.integers(0, 100)), int(rng.integers(1, 4096))))
        elif u < 0.9 and fresh:
            a, ln = fresh[int(rng.integers(0, len(fresh)))]
            reqs.append((a + int(rng.integers(0, 64)), ln - 64))
        else:
            reqs.append((int(rng.integers(0, 1 << 30)), 0))
    q = np.array(reqs, np.uint64)
    nl = rng.integers(0, 2**32, size=q.shape[0], dtype=np.uint64).astype(np.uint32)
    b = oracle.mr_register(q, nl, s, e, lk, refs)
    o = oracle.mr_register(q, nl, s, e, lk, refs, one_at_a_time=True)
    for key in ("start", "end", "lkey", "refs", "handle", "kind", "remap", "ctr"):
        assert (b[key] == o[key]).all(), key
    assert set(b["kind"].tolist()) >= {1, 2, 3, 4, 5}


def holders(s, e, b, a):
    return [i for i in range(len(s)) if int(s[i]) <= b and a <= int(e[i])]


@pytest.mark.parametrize("seed", range(8))
def test_batch_reading_invariants(oracle, seed):
    """Arbitrary ranges (nested, overlapping, repeated) on a table whose
    records overlap: the batch result obeys the reading, checked by brute
    force."""
    rng = np.random.default_rng(100 + seed)
    n = int(rng.integers(0, 40))
    s = np.sort(rng.integers(0, 400, size=n)).astype(np.uint64) * np.uint64(4096)
    e = s + rng.integers(1, 40, size=n).astype(np.uint64) * np.uint64(4096)
    lk = rng.integers(0, 2**32, size=n, dtype=np.uint64).astype(np.uint32)
    refs = rng.integers(1, 4, size=n).astype(np.uint32)
    m = 300
    a = rng.integers(0, 450 * 4096, size=m).astype(np.uint64)
    sz = rng.integers(0, 30 * 4096, size=m).astype(np.uint64)
    pick = rng.integers(0, max(m // 4, 1), size=m)
    rep = rng.random(m) < 0.3                     # repeat an earlier request
    a = np.where(rep, a[pick], a)
    sz = np.where(rep, sz[pick], sz)
    q = np.stack([a, sz], axis=1).astype(np.uint64)
    nl = rng.integers(0, 2**32, size=m, dtype=np.uint64).astype(np.uint32)
    r = oracle.mr_register(q, nl, s, e, lk, refs)
    os_, oe = r["start"], r["end"]
    assert (np.diff(os_.astype(np.int64)) >= 0).all()                 # sorted by start
    valid = r["kind"] != 3
    assert int(r["refs"].astype(np.int64).sum()) == int(refs.astype(np.int64).sum()) + int(valid.sum())
    for i in range(n):                                                 # old records kept, in order
        j = int(r["remap"][i])
        assert (int(os_[j]), int(oe[j]), int(r["lkey"][j])) == (int(s[i]), int(e[i]), int(lk[i]))
    assert (np.diff(r["remap"]) > 0).all()
    firsts = {}
    for k in range(m):
        if r["kind"][k] == 3:
            assert (int(q[k, 1]) == 0) and r["handle"][k] == -1
            continue
        b = int(q[k, 0]) // 4096 * 4096
        ae = -(-(int(q[k, 0]) + int(q[k, 1])) // 4096) * 4096
        old = holders(s, e, b, ae)
        j = int(r["handle"][k])
        assert int(os_[j]) <= b and ae <= int(oe[j])                    # it holds the request
        if old:                                                         # lowest old holder
            assert r["kind"][k] == (1 if (int(s[old[0]]), int(e[old[0]])) == (b, ae) else 2)
            assert j == r["remap"][old[0]]
        else:                                                           # a new record of its own range
            assert (int(os_[j]), int(oe[j])) == (b, ae)
            if (b, ae) in firsts:
                assert r["kind"][k] == 5 and firsts[(b, ae)] == j
            else:
                assert r["kind"][k] == 4 and int(r["lkey"][j]) == int(nl[k])
                firsts[(b, ae)] = j
    new_idx = sorted(set(range(len(os_))) - set(r["remap"].tolist()))
    assert sorted(new_idx) == sorted(firsts.values())
    news = [(int(os_[j]), int(oe[j])) for j in new_idx]
    assert news == sorted(news)                                        # (start, end) order
    for j in new_idx:       # after every old record with the same start
        olds_same = [int(r["remap"][i]) for i in range(n) if int(s[i]) == int(os_[j])]
        assert all(x < j for x in olds_same)


def test_capacity_overflow_writes_nothing(oracle):
    s, e, lk, refs = disjoint_table(np.random.default_rng(1), 10, 500)
    q = np.array([[600 * 4096, 4096], [700 * 4096, 4096]], np.uint64)
    r = oracle.mr_register(q, [1, 2], s, e, lk, refs, out_cap=11)
    assert r["ctr"].tolist() == [12, 0, 1, 0] and r["start"].shape[0] == 0
    r = oracle.mr_register(q, [1, 2], s, e, lk, refs, out_cap=12)
    assert r["ctr"].tolist() == [12, 0, 0, 0] and r["start"].shape[0] == 12


def test_deregister_by_brute_force(oracle):
    rng = np.random.default_rng(7)
    for _ in range(30):
        n = int(rng.integers(0, 20))
        s, e, lk, refs = disjoint_table(rng, max(n, 1), 400)
        if n == 0:
            s, e, lk, refs = (x[:0] for x in (s, e, lk, refs))
        hs = rng.integers(-2, n + 2, size=int(rng.integers(0, 60)))
        d = oracle.mr_deregister(hs, s, e, lk, refs)
        left = [int(x) for x in refs]
        want = []
        for x in hs:
            if x < 0 or x >= n or left[x] == 0:
                want.append(2)
            else:
                left[x] -= 1
                want.append(1 if left[x] == 0 else 0)
        assert d["status"].tolist() == want
        keep = [i for i in range(n) if left[i] > 0]
        assert d["remap"].tolist() == [keep.index(i) if i in keep else -1 for i in range(n)]
        assert d["refs"].tolist() == [left[i] for i in keep]
        assert d["start"].tolist() == [int(s[i]) for i in keep]
        assert d["ctr"].tolist() == [len(keep), want.count(2), 0, 0]


def test_deregister_releases_once(oracle):
    """refs r and d handles naming the record: min(d, r) references drop, the
    r-th releases it, the rest are stale."""
    s, e, lk, _ = disjoint_table(np.random.default_rng(2), 3, 100)
    for r0 in (1, 2, 5):
        for d in (1, r0, r0 + 3):
            refs = np.array([r0, 1, 1], np.uint32)
            out = oracle.mr_deregister([0] * d, s, e, lk, refs)
            st = out["status"].tolist()
            assert st.count(1) == (1 if d >= r0 else 0)
            assert st.count(2) == max(0, d - r0)
            assert st[:min(d, r0)] == [0] * (min(d, r0) - (1 if d >= r0 else 0)) + ([1] if d >= r0 else [])


def test_partial_overlap_miss_with_the_same_start(oracle):
    """[0x1000, 0x3000) only partly overlaps the record [0x1000, 0x2000): a
    miss, registered anew and placed after the record with the same start."""
    s = np.array([0x1000, 0x8000], np.uint64)
    e = np.array([0x2000, 0x9000], np.uint64)
    lk = np.array([1, 2], np.uint32)
    refs = np.array([1, 1], np.uint32)
    q = np.array([[0x1000, 0x2000], [0x1000, 0x1000], [0x1800, 0x1000]], np.uint64)
    for one in (False, True):
        r = oracle.mr_register(q, [7, 8, 9], s, e, lk, refs, one_at_a_time=one)
        assert r["start"].tolist() == [0x1000, 0x1000, 0x8000]
        assert r["end"].tolist() == [0x2000, 0x3000, 0x9000]
        assert r["remap"].tolist() == [0, 2]
        assert r["kind"].tolist()[:2] == [4, 1] and r["handle"].tolist()[:2] == [1, 0]
        # the third request is [0x1000, 0x3000) after rounding: the new range again
        assert r["kind"].tolist()[2] == 5 and r["handle"].tolist()[2] == 1
        assert r["refs"].tolist() == [2, 2, 1]


def nested_batch(rng, n_old, n_q, pages, overlap):
    """A table over a few pages (overlapping records when `overlap`) and
    requests that nest in each other and in the records, in random order,
    with repeats and invalid ones."""
    if n_old:
        s = np.sort(rng.integers(0, pages - 1, size=n_old)).astype(np.uint64)
        if not overlap:
            s = np.unique(s)
        ln = rng.integers(1, 8 if overlap else 2, size=s.shape[0]).astype(np.uint64)
        if not overlap:  # disjoint: each record ends before the next starts
            nxt = np.append(s[1:], np.uint64(pages))
            ln = np.minimum(ln, nxt - s)
        e = s + ln
        s, e = s * np.uint64(4096), e * np.uint64(4096)
    else:
        s = e = np.zeros(0, np.uint64)
    lk = rng.integers(0, 2**32, size=s.shape[0], dtype=np.uint64).astype(np.uint32)
    refs = rng.integers(1, 4, size=s.shape[0]).astype(np.uint32)
    a = rng.integers(0, pages, size=n_q).astype(np.uint64) * np.uint64(4096)
    a += rng.integers(0, 4096, size=n_q).astype(np.uint64) * (rng.random(n_q) < 0.3)
    sz = rng.integers(1, 6 * 4096, size=n_q).astype(np.uint64)
    rep = rng.random(n_q) < 0.15
    for k in np.flatnonzero(rep):
        if k:
            j = int(rng.integers(0, k))
            a[k], sz[k] = a[j], sz[j]
    sz[rng.random(n_q) < 0.03] = 0  # invalid
    q = np.stack([a, sz], axis=1).astype(np.uint64)
    nl = rng.integers(0, 2**32, size=n_q, dtype=np.uint64).astype(np.uint32)
    return q, nl, (s, e, lk, refs)


@pytest.mark.parametrize("seed", range(40))
def test_indexed_one_at_a_time_equals_the_scan(oracle, seed):
    """The indexed one-at-a-time registration gives exactly the scan's
    result (table, handles, kinds, remap, counters) on batches whose new
    ranges nest in each other and in old records, on disjoint and
    overlapping tables, at 4 KiB and 64 KiB granules, and with too small an
    output capacity."""
    rng = np.random.default_rng(900 + seed)
    q, nl, t = nested_batch(rng, int(rng.integers(0, 12)), int(rng.integers(1, 300)),
                            int(rng.integers(4, 80)), overlap=seed % 2 == 1)
    g = G64K if seed % 5 == 4 else G4K
    if g == G64K:
        q[:, 0] *= np.uint64(16)
        q[:, 1] *= np.uint64(16)
        t = (t[0] * np.uint64(16), t[1] * np.uint64(16), t[2], t[3])
    for cap in (None, len(t[0]) + 1):
        a = oracle.mr_register(q, nl, *t, granule_shift=g, out_cap=cap, one_at_a_time=True)
        b = oracle.mr_register(q, nl, *t, granule_shift=g, out_cap=cap, one_at_a_time=True,
                               indexed=True)
        assert a["ctr"].tolist() == b["ctr"].tolist()
        assert a["kind"].tolist() == b["kind"].tolist()
        if int(a["ctr"][2]) == 0:
            for key in ("start", "end", "lkey", "refs", "handle", "remap"):
                assert a[key].tolist() == b[key].tolist(), key


def test_one_at_a_time_nesting_hand_case(oracle):
    """Worked by hand from the per-call definition (lowest-index holder in
    the table as it stands; a new record after every record starting at or
    before it), on the old table {[8K, 16K)}:
      0: [4K, 8K)   misses           -> new record A
      1: [4K, 6K)   inside A         -> hit on A (kind 5)
      2: [0, 16K)   misses           -> new record B, before A (lower start)
      3: [4K, 8K)   A and B hold it  -> B, the lower start (kind 5)
      4: [8K, 12K)  old record and B -> B starts lower (kind 5)
      5: [12K, 16K) inside B and old -> B
      6: [8K, 16K)  same as the old  -> B still comes first (kind 5)
    Final table: B [0, 16K) refs 5, A [4K, 8K) refs 2, old [8K, 16K) refs 1."""
    K = 1024
    t = (np.array([8 * K], np.uint64), np.array([16 * K], np.uint64), np.array([77], np.uint32),
         np.array([1], np.uint32))
    q = np.array([[4 * K, 4 * K], [4 * K, 2 * K], [0, 16 * K], [4 * K, 4 * K], [8 * K, 4 * K],
                  [12 * K, 4 * K], [8 * K, 8 * K]], np.uint64)
    for indexed in (False, True):
        r = oracle.mr_register(q, [10, 11, 12, 13, 14, 15, 16], *t, one_at_a_time=True,
                               indexed=indexed)
        assert r["kind"].tolist() == [4, 5, 4, 5, 5, 5, 5]
        assert rows_of(r) == [(0, 16 * K, 12, 5), (4 * K, 8 * K, 10, 2), (8 * K, 16 * K, 77, 1)]
        assert r["handle"].tolist() == [1, 1, 0, 0, 0, 0, 0]
        assert r["remap"].tolist() == [2]
        assert r["ctr"].tolist() == [3, 0, 0, 0]


@pytest.mark.parametrize("g", [G4K, G64K])
def test_one_at_a_time_first_range_holds_the_rest(oracle, g):
    """A closed form from the per-call definition: the first request asks for
    a range holding every later request and both old records, so it makes
    the only new record, first in the table (lowest start), and every later
    request -- a miss, a repeat, or a range inside an old record, which the
    new record precedes -- is a hit on it. Its references are the batch's
    size; the old records keep theirs and move up by one."""
    rng = np.random.default_rng(70 + g)
    unit = 1 << g
    m, pages = 4000, 3000
    a = rng.integers(1, pages, size=m).astype(np.uint64) * np.uint64(unit)
    a += rng.integers(0, unit, size=m).astype(np.uint64) * (rng.random(m) < 0.3)
    sz = rng.integers(1, 16 * unit, size=m).astype(np.uint64)
    a[0], sz[0] = 0, np.uint64((pages + 32) * unit)
    q = np.stack([a, sz], axis=1).astype(np.uint64)
    nl = np.arange(m, dtype=np.uint32) + np.uint32(5)
    s = np.array([40 * unit, 900 * unit], np.uint64)
    t = (s, s + np.uint64(8 * unit), np.array([3, 4], np.uint32), np.array([1, 2], np.uint32))
    for indexed in (False, True):
        r = oracle.mr_register(q, nl, *t, granule_shift=g, one_at_a_time=True, indexed=indexed)
        assert r["kind"][0] == 4 and (r["kind"][1:] == 5).all()
        assert (r["handle"] == 0).all() and r["remap"].tolist() == [1, 2]
        assert rows_of(r) == [(0, (pages + 32) * unit, 5, m), (40 * unit, 48 * unit, 3, 1),
                              (900 * unit, 908 * unit, 4, 2)]
        assert r["ctr"].tolist() == [3, 0, 0, 0]
