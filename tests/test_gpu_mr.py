"""db_mr_lookup on the GPU against the oracle, bit for bit."""

import numpy as np
import pytest

from conftest import h, load_golden
from gpu_util import dev32, dev64, host32, host64, lib, need_gpu, torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def db():
    need_gpu()
    return lib()


def run_gpu(db, q, start, end, lkey, ws=None):
    n = q.shape[0]
    idx = torch.full((max(n, 1),), 0x55, dtype=torch.int32, device="cuda")
    lk = torch.full((max(n, 1),), 0x55, dtype=torch.int32, device="cuda")
    kind = torch.full((max(n, 1),), 0x55, dtype=torch.uint8, device="cuda")
    ctr = torch.full((4,), -1, dtype=torch.int64, device="cuda")
    if ws is None:
        ws = db.workspace(db.mr_workspace_size(start.shape[0]))
    empty64 = torch.zeros(0, dtype=torch.int64, device="cuda")
    db.mr_lookup(dev64(q) if n else torch.zeros((0, 2), dtype=torch.int64, device="cuda"),
                 dev64(start) if start.shape[0] else empty64,
                 dev64(end) if start.shape[0] else empty64,
                 dev32(lkey) if start.shape[0] else torch.zeros(0, dtype=torch.int32, device="cuda"),
                 idx, lk, kind, ws, ctr=ctr)
    torch.cuda.synchronize()
    return dict(idx=idx.cpu().numpy()[:n], lkey=host32(lk)[:n], kind=kind.cpu().numpy()[:n],
                ctr=host64(ctr))


def check(got, want):
    assert (got["kind"] == want["kind"]).all()
    assert (got["idx"] == want["idx"]).all()
    assert (got["lkey"] == want["lkey"]).all()
    assert int(got["ctr"][0]) == int(((want["kind"] == 1) | (want["kind"] == 2)).sum())
    assert int(got["ctr"][1]) == int((want["kind"] == 3).sum())


@pytest.mark.parametrize("section", ["registration_experiment", "partial_overlap"])
def test_golden(db, section):
    fx = load_golden("mr_hand_cases.json")[section]
    base = h(fx.get("alloc_base", "0x0"))
    start = np.array([base + h(r["start"]) for r in fx["table"]], dtype=np.uint64)
    end = np.array([base + h(r["end"]) for r in fx["table"]], dtype=np.uint64)
    lkey = np.array([r["lkey"] for r in fx["table"]], dtype=np.uint32)
    q = np.array([[(base + h(x["off"])) & (2**64 - 1), x["size"]] for x in fx["queries"]],
                 dtype=np.uint64)
    got = run_gpu(db, q, start, end, lkey)
    assert got["kind"].tolist() == [x["kind"] for x in fx["queries"]]
    assert got["idx"].tolist() == [x["idx"] for x in fx["queries"]]
    assert got["lkey"].tolist() == [x["lkey"] for x in fx["queries"]]
    assert int(got["ctr"][3]) == 0


def test_tiny_workload(db, oracle):
    import synth
    w = synth.prp_tiny()
    got = run_gpu(db, w["queries"], w["mr_start"], w["mr_end"], w["mr_lkey"])
    check(got, oracle.mr_linear(w["queries"], w["mr_start"], w["mr_end"], w["mr_lkey"]))


@pytest.mark.parametrize("n_mr,n_q", [(1, 100), (37, 5000), (1000, 20001),
                                      (3000, 100000), (70000, 1 << 20)])
def test_generated_tables(db, oracle, n_mr, n_q):
    import synth
    d = synth.mr_lookup(seed=n_mr, n_mr=n_mr, n_q=n_q) if n_mr > 1 else None
    if d is None:
        start = np.array([0x7000_0000_0000], dtype=np.uint64)
        end = start + np.uint64(1 << 21)
        lkey = np.array([77], dtype=np.uint32)
        rng = np.random.default_rng(1)
        a = start[0] - np.uint64(1 << 22) + rng.integers(0, 1 << 24, size=n_q).astype(np.uint64)
        q = np.stack([a, rng.integers(0, 1 << 20, size=n_q).astype(np.uint64)], axis=1)
        d = dict(mr_start=start, mr_end=end, mr_lkey=lkey, queries=q)
    ref = oracle.mr_linear if n_mr * n_q <= 2e8 else oracle.mr_bsearch
    want = ref(d["queries"], d["mr_start"], d["mr_end"], d["mr_lkey"])
    got = run_gpu(db, d["queries"], d["mr_start"], d["mr_end"], d["mr_lkey"])
    check(got, want)


def test_random_uniform_queries_small_tables(db, oracle):
    """Uniform random ranges over tiny page-granular tables (many partial overlaps)."""
    rng = np.random.default_rng(9)
    for trial in range(20):
        n = int(rng.integers(1, 40))
        cuts = np.sort(rng.choice(np.arange(1, 300), size=2 * n, replace=False))
        start = cuts[0::2].astype(np.uint64) * np.uint64(4096)
        end = cuts[1::2].astype(np.uint64) * np.uint64(4096)
        lkey = rng.integers(0, 2**32, size=n, dtype=np.uint64).astype(np.uint32)
        q = np.stack([rng.integers(0, 310 * 4096, size=3000).astype(np.uint64),
                      rng.integers(0, 30 * 4096, size=3000).astype(np.uint64)], axis=1)
        check(run_gpu(db, q, start, end, lkey), oracle.mr_linear(q, start, end, lkey))


def test_extreme_addresses(db, oracle):
    start = np.array([0, 0x1000, 0xFFFF_FFFF_FFFF_D000], dtype=np.uint64)
    end = np.array([0x1000, 0x3000, 0xFFFF_FFFF_FFFF_F000], dtype=np.uint64)
    lkey = np.array([1, 2, 3], dtype=np.uint32)
    q = np.array([[0, 1], [0, 0], [0xFFF, 2], [0xFFFF_FFFF_FFFF_E000, 0x1000],
                  [0xFFFF_FFFF_FFFF_EFFF, 1], [0xFFFF_FFFF_FFFF_F000, 1],
                  [0xFFFF_FFFF_FFFF_D000, 0x2000], [5, 2**64 - 1]], dtype=np.uint64)
    check(run_gpu(db, q, start, end, lkey), oracle.mr_linear(q, start, end, lkey))


def byte_table(rng, n, span_pages, granule):
    """n disjoint records inside span_pages pages, with starts and ends on
    multiples of granule bytes (64: byte-granular records; 4096: pages)."""
    cuts = np.sort(rng.choice(np.arange(1, span_pages * 4096 // granule, dtype=np.int64),
                              size=2 * n, replace=False)).astype(np.uint64) * np.uint64(granule)
    if granule < 4096:
        cuts += rng.integers(0, granule, size=2 * n).astype(np.uint64)
    start, end = cuts[0::2], cuts[1::2]
    keep = start < end
    return start[keep], end[keep]


@pytest.mark.parametrize("case", ["unaligned", "clustered", "clustered_far", "long_queries"])
def test_directory_paths(db, oracle, case):
    """Byte-granular starts and ends (exact versus contained), many records
    in one bucket (the binary-step path), queries spanning more than 2^31
    pages and queries past the last record."""
    rng = np.random.default_rng({"unaligned": 1, "clustered": 2, "clustered_far": 3,
                                 "long_queries": 4}[case])
    if case == "unaligned":
        start, end = byte_table(rng, 3000, 200000, 64)
        # a quarter of the records page aligned at both ends, so exact hits exist
        al = rng.random(start.shape[0]) < 0.25
        start = np.where(al, (start + np.uint64(4095)) & ~np.uint64(4095), start)
        end = np.where(al, end & ~np.uint64(4095), end)
        ok = start < end
        ok[1:] &= end[:-1] <= start[1:]
        start, end = start[ok], end[ok]
    elif case == "clustered":
        # ten dense groups of 200 records, far apart: each group shares a bucket
        parts = []
        for base in np.sort(rng.choice(1 << 28, size=10, replace=False)).astype(np.uint64):
            s_, e_ = byte_table(rng, 200, 3000, 4096)
            parts.append((s_ + (base << np.uint64(12)), e_ + (base << np.uint64(12))))
        start = np.concatenate([x[0] for x in parts])
        end = np.concatenate([x[1] for x in parts])
        ok = np.ones(start.shape[0], dtype=bool)
        ok[1:] = end[:-1] <= start[1:]
        start, end = start[ok], end[ok]
    elif case == "clustered_far":
        start, end = byte_table(rng, 1500, 20000, 4096)
        start = np.append(start, np.uint64(1) << np.uint64(46))  # one record far away:
        end = np.append(end, (np.uint64(1) << np.uint64(46)) + np.uint64(1 << 20))  # every other bucket empty
    else:
        start = np.array([0x1000, 1 << 40, (1 << 60) + 0x3000], dtype=np.uint64)
        end = np.array([0x5000, 1 << 59, (1 << 61)], dtype=np.uint64)
    n = start.shape[0]
    lkey = rng.integers(0, 2**32, size=n, dtype=np.uint64).astype(np.uint32)
    hi = int(end[-1])
    m = 60000
    pick = rng.integers(0, n, size=m)
    mode = rng.integers(0, 4, size=m)
    a = np.empty(m, dtype=np.uint64)
    sz = np.empty(m, dtype=np.uint64)
    span = (end[pick] - start[pick]).astype(np.float64)
    # 0: exactly the record; 1: inside it; 2: anywhere; 3: past the last record
    a[mode == 0] = start[pick][mode == 0]
    sz[mode == 0] = (end[pick] - start[pick])[mode == 0]
    off = (rng.random(m) * span).astype(np.uint64)
    a[mode == 1] = (start[pick] + off)[mode == 1]
    sz[mode == 1] = np.maximum(np.uint64(1), ((end[pick] - start[pick] - off).astype(np.float64)
                                               * rng.random(m)).astype(np.uint64))[mode == 1]
    a[mode == 2] = (rng.random(m) * float(hi)).astype(np.uint64)[mode == 2]
    sz[mode == 2] = rng.integers(1, 1 << 16, size=m).astype(np.uint64)[mode == 2]
    a[mode == 3] = np.uint64(hi) + rng.integers(0, 1 << 30, size=m).astype(np.uint64)[mode == 3]
    sz[mode == 3] = rng.integers(1, 1 << 20, size=m).astype(np.uint64)[mode == 3]
    if case == "long_queries":
        # ranges of 2^43 .. 2^50 bytes inside the second record and across the third
        big = np.uint64(1) << rng.integers(43, 51, size=m).astype(np.uint64)
        a = np.where(mode == 1, np.uint64(1 << 41), a)
        sz = np.where(mode == 1, big, sz)
        a = np.where(mode == 0, np.uint64((1 << 60) + 0x3000), a)
        sz = np.where(mode == 0, big, sz)
    top = np.uint64(2**64 - 4096)
    sz = np.minimum(sz, top - np.minimum(a, top))
    q = np.stack([a, sz], axis=1).astype(np.uint64)
    want = oracle.mr_linear(q, start, end, lkey)
    got = run_gpu(db, q, start, end, lkey)
    check(got, want)
    kinds = np.bincount(want["kind"].astype(np.int64), minlength=4)
    assert kinds[2] > 0 and kinds[0] > 0, kinds
    if case == "unaligned":
        assert kinds[1] > 0, kinds


def test_empty_table_and_empty_batch(db, oracle):
    q = np.array([[0x1000, 10], [0, 0]], dtype=np.uint64)
    e = np.zeros(0, dtype=np.uint64)
    got = run_gpu(db, q, e, e, np.zeros(0, dtype=np.uint32))
    assert got["kind"].tolist() == [0, 3] and got["idx"].tolist() == [-1, -1]
    got = run_gpu(db, np.zeros((0, 2), dtype=np.uint64), np.array([0], dtype=np.uint64),
                  np.array([4096], dtype=np.uint64), np.array([1], dtype=np.uint32))
    assert got["ctr"].tolist() == [0, 0, 0, 0]


def test_unsorted_table_is_flagged(db):
    start = np.array([0x3000, 0x1000], dtype=np.uint64)
    end = np.array([0x4000, 0x2000], dtype=np.uint64)
    got = run_gpu(db, np.array([[0x1000, 1]], dtype=np.uint64), start, end,
                  np.array([1, 2], dtype=np.uint32))
    assert int(got["ctr"][3]) & db.ERR_TABLE_ORDER
    # overlapping records too
    start = np.array([0x1000, 0x1800 & ~0xFFF], dtype=np.uint64)
    end = np.array([0x3000, 0x4000], dtype=np.uint64)
    got = run_gpu(db, np.array([[0x1000, 1]], dtype=np.uint64), start, end,
                  np.array([1, 2], dtype=np.uint32))
    assert int(got["ctr"][3]) & db.ERR_TABLE_ORDER


def test_workspace_reuse(db, oracle):
    import synth
    ws = db.workspace(db.mr_workspace_size(5000))
    for n_mr, seed in ((5000, 1), (100, 2), (4000, 3)):
        d = synth.mr_lookup(seed=seed, n_mr=n_mr, n_q=30000)
        got = run_gpu(db, d["queries"], d["mr_start"], d["mr_end"], d["mr_lkey"], ws=ws)
        check(got, oracle.mr_bsearch(d["queries"], d["mr_start"], d["mr_end"], d["mr_lkey"]))


def test_full_size_workload(db, oracle):
    """1,048,576 registered ranges, 16,777,216 queries: every query against
    the oracle's binary search (equal to the definition on sorted disjoint
    tables, pinned in the oracle tests)."""
    import synth
    d = synth.mr_lookup()
    got = run_gpu(db, d["queries"], d["mr_start"], d["mr_end"], d["mr_lkey"])
    want = oracle.mr_bsearch(d["queries"], d["mr_start"], d["mr_end"], d["mr_lkey"])
    check(got, want)
    mix = d["query_mix"]
    assert (got["kind"][mix == 0] == 1).all()
    assert (got["kind"][mix == 1] == 2).all()
    assert (got["kind"][mix == 2] == 0).all()
    # and a sample against the linear definition itself
    s = np.random.default_rng(0).choice(d["queries"].shape[0], 200, replace=False)
    lin = oracle.mr_linear(d["queries"][s], d["mr_start"], d["mr_end"], d["mr_lkey"])
    assert (got["idx"][s] == lin["idx"]).all() and (got["kind"][s] == lin["kind"]).all()
