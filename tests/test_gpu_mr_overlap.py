"""db_mr_lookup_overlap on the GPU against the oracle, bit for bit: tables
sorted by start whose records may overlap (a partial-overlap miss is
registered anew, "NCCL expert course 26", "IB Backend MR Cache")."""

import numpy as np
import pytest

from conftest import h, load_golden
from gpu_util import dev32, dev64, host32, host64, lib, need_gpu, torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def db():
    need_gpu()
    return lib()


def run_gpu(db, q, start, end, lkey, ws=None, overlap=True):
    n = q.shape[0]
    idx = torch.full((max(n, 1),), 0x55, dtype=torch.int32, device="cuda")
    lk = torch.full((max(n, 1),), 0x55, dtype=torch.int32, device="cuda")
    kind = torch.full((max(n, 1),), 0x55, dtype=torch.uint8, device="cuda")
    ctr = torch.full((4,), -1, dtype=torch.int64, device="cuda")
    if ws is None:
        ws = db.workspace(db.mr_workspace_size(start.shape[0]))
    e64 = torch.zeros(0, dtype=torch.int64, device="cuda")
    fn = db.mr_lookup_overlap if overlap else db.mr_lookup
    fn(dev64(q) if n else torch.zeros((0, 2), dtype=torch.int64, device="cuda"),
       dev64(start) if start.shape[0] else e64, dev64(end) if start.shape[0] else e64,
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
    assert int(got["ctr"][3]) == 0


def overlapping_table(rng, n, span_pages, max_pages, granule=4096):
    start = np.sort(rng.integers(0, span_pages * (4096 // granule), size=n)).astype(np.uint64)
    start *= np.uint64(granule)
    size = rng.integers(1, max_pages * (4096 // granule) + 1, size=n).astype(np.uint64)
    end = start + size * np.uint64(granule)
    lkey = rng.integers(0, 2**32, size=n, dtype=np.uint64).astype(np.uint32)
    return start, end, lkey


def queries_near(rng, start, end, m, span):
    n = start.shape[0]
    a = rng.integers(0, span, size=m).astype(np.uint64)
    sz = rng.integers(0, 16 * 4096, size=m).astype(np.uint64)
    pick = rng.integers(0, n, size=m)
    a = np.where(rng.random(m) < 0.4, start[pick] + rng.integers(0, 3, size=m).astype(np.uint64)
                 * np.uint64(2048), a)
    sz = np.where(rng.random(m) < 0.3, end[pick] - start[pick], sz)
    return np.stack([a, sz], axis=1).astype(np.uint64)


def test_golden(db):
    fx = load_golden("mr_hand_cases.json")["overlap_after_partial_miss"]
    start = np.array([h(r["start"]) for r in fx["table"]], dtype=np.uint64)
    end = np.array([h(r["end"]) for r in fx["table"]], dtype=np.uint64)
    lkey = np.array([r["lkey"] for r in fx["table"]], dtype=np.uint32)
    q = np.array([[h(x["off"]), x["size"]] for x in fx["queries"]], dtype=np.uint64)
    got = run_gpu(db, q, start, end, lkey)
    assert got["kind"].tolist() == [x["kind"] for x in fx["queries"]]
    assert got["idx"].tolist() == [x["idx"] for x in fx["queries"]]
    assert got["lkey"].tolist() == [x["lkey"] for x in fx["queries"]]
    assert int(got["ctr"][3]) == 0


@pytest.mark.parametrize("n,span,maxp,granule", [(1, 10, 3, 4096), (7, 20, 8, 4096),
                                                  (50, 200, 40, 4096), (300, 2000, 400, 4096),
                                                  (3000, 20000, 3000, 4096),
                                                  (2000, 100000, 30, 64), (20000, 40000, 8, 4096)])
def test_small_tables_against_the_definition(db, oracle, n, span, maxp, granule):
    """Random overlapping tables (many records per directory bucket, long
    overlap chains, byte-granular ends) against the linear definition."""
    rng = np.random.default_rng(n * 31 + maxp)
    start, end, lkey = overlapping_table(rng, n, span, maxp, granule)
    q = queries_near(rng, start, end, 20000, (span + maxp) * 4096)
    want = oracle.mr_linear(q, start, end, lkey)
    check(run_gpu(db, q, start, end, lkey), want)
    kinds = np.bincount(want["kind"].astype(np.int64), minlength=4)
    assert kinds[0] > 0 and kinds[1] + kinds[2] > 0, kinds


def test_one_record_covering_all(db, oracle):
    """A first record spanning the whole table: every contained query's
    answer is record 0, reached by galloping back over the whole table."""
    rng = np.random.default_rng(5)
    start, end, lkey = overlapping_table(rng, 50000, 1 << 20, 64)
    start[0] = 0
    end[0] = np.uint64((1 << 20) * 4096 + 64 * 4096)
    q = queries_near(rng, start, end, 100000, (1 << 20) * 4096)
    want = oracle.mr_prefix_max(q, start, end, lkey)
    check(run_gpu(db, q, start, end, lkey), want)
    assert (want["idx"][want["kind"] == 2] == 0).all()


def test_disjoint_tables_agree_with_mr_lookup(db, oracle):
    """On a sorted disjoint table both entry points give the same answers."""
    import synth
    d = synth.mr_lookup(seed=3, n_mr=50000, n_q=400000)
    a = run_gpu(db, d["queries"], d["mr_start"], d["mr_end"], d["mr_lkey"])
    b = run_gpu(db, d["queries"], d["mr_start"], d["mr_end"], d["mr_lkey"], overlap=False)
    for k in ("idx", "lkey", "kind"):
        assert (a[k] == b[k]).all(), k
    check(a, oracle.mr_bsearch(d["queries"], d["mr_start"], d["mr_end"], d["mr_lkey"]))


def test_order_rule(db):
    """Overlaps are allowed; unsorted starts or an empty record are flagged."""
    q = np.array([[0x1000, 1]], dtype=np.uint64)
    k2 = np.array([1, 2], dtype=np.uint32)
    got = run_gpu(db, q, np.array([0x1000, 0x1000], dtype=np.uint64),
                  np.array([0x3000, 0x2000], dtype=np.uint64), k2)
    assert int(got["ctr"][3]) == 0 and got["idx"].tolist() == [0]
    got = run_gpu(db, q, np.array([0x3000, 0x1000], dtype=np.uint64),
                  np.array([0x4000, 0x2000], dtype=np.uint64), k2)
    assert int(got["ctr"][3]) & db.ERR_TABLE_ORDER
    got = run_gpu(db, q, np.array([0x1000, 0x2000], dtype=np.uint64),
                  np.array([0x3000, 0x2000], dtype=np.uint64), k2)
    assert int(got["ctr"][3]) & db.ERR_TABLE_ORDER


def test_empty_table_and_empty_batch(db):
    q = np.array([[0x1000, 10], [0, 0]], dtype=np.uint64)
    e = np.zeros(0, dtype=np.uint64)
    got = run_gpu(db, q, e, e, np.zeros(0, dtype=np.uint32))
    assert got["kind"].tolist() == [0, 3] and got["idx"].tolist() == [-1, -1]
    got = run_gpu(db, np.zeros((0, 2), dtype=np.uint64), np.array([0], dtype=np.uint64),
                  np.array([4096], dtype=np.uint64), np.array([1], dtype=np.uint32))
    assert got["ctr"].tolist() == [0, 0, 0, 0]


def test_workspace_reuse_across_entry_points(db, oracle):
    import synth
    ws = db.workspace(db.mr_workspace_size(6000))
    for n_mr, seed, ov in ((4000, 1, True), (100, 2, False), (4800, 3, True)):
        d = synth.mr_lookup_overlap(seed=seed, n_mr=n_mr, n_q=30000) if ov else \
            synth.mr_lookup(seed=seed, n_mr=n_mr, n_q=30000)
        got = run_gpu(db, d["queries"], d["mr_start"], d["mr_end"], d["mr_lkey"], ws=ws,
                      overlap=ov)
        check(got, oracle.mr_prefix_max(d["queries"], d["mr_start"], d["mr_end"],
                                        d["mr_lkey"]))


def test_full_size_workload(db, oracle):
    """1,310,720 records (a quarter of them straddling another's end) and
    16,777,216 queries: every query against the oracle's prefix-maximum
    search (equal to the definition, pinned in the oracle tests), and a
    sample against the linear definition itself."""
    import synth
    d = synth.mr_lookup_overlap()
    got = run_gpu(db, d["queries"], d["mr_start"], d["mr_end"], d["mr_lkey"])
    want = oracle.mr_prefix_max(d["queries"], d["mr_start"], d["mr_end"], d["mr_lkey"])
    check(got, want)
    s = np.random.default_rng(0).choice(d["queries"].shape[0], 200, replace=False)
    lin = oracle.mr_linear(d["queries"][s], d["mr_start"], d["mr_end"], d["mr_lkey"])
    assert (got["idx"][s] == lin["idx"]).all() and (got["kind"][s] == lin["kind"]).all()
    # the overlaps matter: some answers are not the last record starting at or below base
    base = d["queries"][:, 0] & ~np.uint64(4095)
    last = np.searchsorted(d["mr_start"], base, side="right") - 1
    hit = got["idx"] >= 0
    assert (got["idx"][hit] != last[hit]).mean() > 0.02


def test_five_million_overlapping_records(db, oracle):
    """5,000,000 overlapping records (4,883 blocks of the prefix maximum of
    the ends, more than one scan round of the block maxima) and 1,000,000
    queries against the oracle."""
    rng = np.random.default_rng(50)
    start, end, lkey = overlapping_table(rng, 5_000_000, 40_000_000, 64)
    q = queries_near(rng, start, end, 1_000_000, (40_000_000 + 64) * 4096)
    check(run_gpu(db, q, start, end, lkey), oracle.mr_prefix_max(q, start, end, lkey))
