"""db_mr_register / db_mr_deregister on the GPU against the oracle, bit for
bit ("NCCL expert course 26": IB Backend MR Cache, Communicator User
Registration Cache, the ncclCommRegister experiment; xNVMe "uPCIe CUDA":
xnvme_buf_register at 64 KiB)."""

import numpy as np
import pytest

from conftest import h, load_golden
from gpu_util import dev32, dev64, host32, host64, lib, need_gpu, torch

pytestmark = pytest.mark.gpu

EMPTY = (np.zeros(0, np.uint64), np.zeros(0, np.uint64), np.zeros(0, np.uint32),
         np.zeros(0, np.uint32))


@pytest.fixture(scope="module")
def db():
    need_gpu()
    return lib()


def d64(a):
    return dev64(a) if a.shape[0] else torch.zeros(0, dtype=torch.int64, device="cuda")


def d32(a):
    return dev32(a) if a.shape[0] else torch.zeros(0, dtype=torch.int32, device="cuda")


def register(db, q, new_lkey, start, end, lkey, refs, granule_shift=12, out_cap=None):
    q = np.ascontiguousarray(q, np.uint64).reshape(-1, 2)
    n_q, n = q.shape[0], start.shape[0]
    cap = n + n_q if out_cap is None else out_cap
    o = [torch.full((cap,), 0x55, dtype=torch.int64, device="cuda"),
         torch.full((cap,), 0x55, dtype=torch.int64, device="cuda"),
         torch.full((cap,), 0x55, dtype=torch.int32, device="cuda"),
         torch.full((cap,), 0x55, dtype=torch.int32, device="cuda")]
    handle = torch.full((n_q,), -7, dtype=torch.int64, device="cuda")
    kind = torch.full((n_q,), 0xEE, dtype=torch.uint8, device="cuda")
    remap = torch.full((n,), -7, dtype=torch.int64, device="cuda")
    ctr = torch.full((4,), -1, dtype=torch.int64, device="cuda")
    ws = db.workspace(db.mr_register_workspace_size(n_q, n))
    db.mr_register(d64(q.reshape(-1)).view(-1, 2) if n_q else torch.zeros((0, 2), dtype=torch.int64, device="cuda"),
                   d32(np.ascontiguousarray(new_lkey, np.uint32)), d64(start), d64(end), d32(lkey),
                   d32(refs), *o, handle, kind, remap, ws, granule_shift=granule_shift, ctr=ctr)
    torch.cuda.synchronize()
    c = host64(ctr)
    m = int(c[0]) if int(c[2]) == 0 else 0
    return dict(start=host64(o[0])[:m], end=host64(o[1])[:m], lkey=host32(o[2])[:m],
                refs=host32(o[3])[:m], handle=handle.cpu().numpy(), kind=kind.cpu().numpy(),
                remap=remap.cpu().numpy(), ctr=c)


def deregister(db, handles, start, end, lkey, refs):
    hs = np.ascontiguousarray(handles, np.int64)
    n = start.shape[0]
    o = [torch.full((max(n, 1),), 0x55, dtype=torch.int64, device="cuda"),
         torch.full((max(n, 1),), 0x55, dtype=torch.int64, device="cuda"),
         torch.full((max(n, 1),), 0x55, dtype=torch.int32, device="cuda"),
         torch.full((max(n, 1),), 0x55, dtype=torch.int32, device="cuda")]
    remap = torch.full((n,), -7, dtype=torch.int64, device="cuda")
    status = torch.full((hs.shape[0],), 0xEE, dtype=torch.uint8, device="cuda")
    ctr = torch.full((4,), -1, dtype=torch.int64, device="cuda")
    ws = db.workspace(db.mr_deregister_workspace_size(hs.shape[0], n))
    hd = torch.from_numpy(hs).cuda() if hs.shape[0] else torch.zeros(0, dtype=torch.int64,
                                                                      device="cuda")
    db.mr_deregister(hd, d64(start), d64(end), d32(lkey), d32(refs), *o, remap, status, ws,
                     ctr=ctr)
    torch.cuda.synchronize()
    c = host64(ctr)
    m = int(c[0])
    return dict(start=host64(o[0])[:m], end=host64(o[1])[:m], lkey=host32(o[2])[:m],
                refs=host32(o[3])[:m], remap=remap.cpu().numpy(), status=status.cpu().numpy(),
                ctr=c)


def same(got, want, keys):
    for k in keys:
        assert got[k].shape == want[k].shape, k
        assert (got[k].astype(np.int64) == want[k].astype(np.int64)).all(), k


REG_KEYS = ("start", "end", "lkey", "refs", "handle", "kind", "remap", "ctr")


def one_at_a_time(oracle, *args, **kw):
    """The oracle's one-at-a-time registration (the pages' definition),
    computed with its index; the tests of the oracle pin that equal to the
    plain scan."""
    return oracle.mr_register(*args, one_at_a_time=True, indexed=True, **kw)
DEREG_KEYS = ("start", "end", "lkey", "refs", "remap", "status", "ctr")


def test_page_experiment(db, oracle):
    fx = load_golden("mr_hand_cases.json")["mutation_experiment"]
    base = h(fx["alloc_base"])
    t = EMPTY
    for c in fx["register_calls"]:
        q = np.array([[base + h(c["off"]), c["size"]]], np.uint64)
        r = register(db, q, [c["new_lkey"]], *t)
        assert r["kind"].tolist() == [c["kind"]] and r["handle"].tolist() == [c["handle"]]
        assert r["refs"].tolist() == c["refs_after"]
        t = (r["start"], r["end"], r["lkey"], r["refs"])
    dr = fx["deregister_batch"]
    d = deregister(db, dr["handles"], *t)
    assert d["status"].tolist() == dr["status"] and d["remap"].tolist() == dr["remap"]
    assert d["refs"].tolist() == [1] and d["ctr"].tolist() == [1, 1, 0, 0]
    # The same registrations as one batch give the page's table: one record
    # with three references, and the disjoint one.
    one = fx["one_batch"]
    q = np.array([[base + h(c["off"]), c["size"]] for c in fx["register_calls"]], np.uint64)
    r = register(db, q, [c["new_lkey"] for c in fx["register_calls"]], *EMPTY)
    assert r["kind"].tolist() == one["kind"] and r["handle"].tolist() == one["handle"]
    assert [(int(a) - base, int(b) - base, int(k), int(n))
            for a, b, k, n in zip(r["start"], r["end"], r["lkey"], r["refs"])] == \
        [(h(x["start"]), h(x["end"]), x["lkey"], x["refs"]) for x in one["table_after"]]


def random_case(rng, n, m, span, granule_shift):
    g = 1 << granule_shift
    s = np.sort(rng.integers(0, span, size=n)).astype(np.uint64) * np.uint64(g)
    e = s + rng.integers(1, 40, size=n).astype(np.uint64) * np.uint64(g)
    lk = rng.integers(0, 2**32, size=n, dtype=np.uint64).astype(np.uint32)
    refs = rng.integers(1, 5, size=n).astype(np.uint32)
    a = rng.integers(0, (span + 50) * g, size=m).astype(np.uint64)
    sz = rng.integers(0, 30 * g, size=m).astype(np.uint64)
    if n:
        pick = rng.integers(0, n, size=m)
        inside = rng.random(m) < 0.4
        a = np.where(inside, s[pick] + rng.integers(0, g, size=m).astype(np.uint64), a)
        sz = np.where(inside, (e[pick] - s[pick]) // np.uint64(2), sz)
    rep = rng.random(m) < 0.25
    src = rng.integers(0, max(m // 3, 1), size=m)
    a = np.where(rep, a[src], a)
    sz = np.where(rep, sz[src], sz)
    sz[::17] = 0                                   # invalid requests
    q = np.stack([a, sz], axis=1).astype(np.uint64)
    nl = rng.integers(0, 2**32, size=m, dtype=np.uint64).astype(np.uint32)
    return q, nl, s, e, lk, refs


@pytest.mark.parametrize("n,m,span,granule_shift", [
    (0, 1, 10, 12), (0, 500, 100, 12), (1, 300, 10, 12), (37, 2000, 300, 12),
    (500, 20000, 5000, 12), (3000, 100000, 20000, 12), (20000, 300000, 400000, 12),
    (40, 3000, 200, 16), (5000, 200000, 60000, 16),
])
def test_register_against_the_oracle(db, oracle, n, m, span, granule_shift):
    """Overlapping tables; requests held by records, nested, partly
    overlapping, repeated and invalid; several tiles of the sort."""
    rng = np.random.default_rng(n * 7 + m + granule_shift)
    q, nl, s, e, lk, refs = random_case(rng, n, m, span, granule_shift)
    want = one_at_a_time(oracle, q, nl, s, e, lk, refs, granule_shift=granule_shift)
    got = register(db, q, nl, s, e, lk, refs, granule_shift=granule_shift)
    same(got, want, REG_KEYS)
    kinds = set(want["kind"].tolist())
    if m >= 300:
        assert {3, 4, 5} <= kinds and (n == 0 or {1, 2} & kinds)


@pytest.mark.parametrize("order", ["shrinking", "growing", "one_range", "same_start"])
def test_register_chains(db, oracle, order):
    """3,000 requests on a chain of ranges: each nested in the one before
    (every later one a hit on the first), each holding the one before (every
    one a new record), one range asked for 3,000 times, and ranges of one
    start and growing ends (a new record each, none holding the next)."""
    m, g = 3000, 4096
    i = np.arange(m, dtype=np.uint64)
    if order == "shrinking":
        a, sz = i * np.uint64(g), (np.uint64(2 * m) - i) * np.uint64(g)
    elif order == "growing":
        a, sz = (np.uint64(m) - i) * np.uint64(g), (np.uint64(1) + i * np.uint64(2)) * np.uint64(g)
    elif order == "one_range":
        a, sz = np.full(m, 5 * g, np.uint64), np.full(m, 7 * g, np.uint64)
    else:
        a, sz = np.full(m, 5 * g, np.uint64), (np.uint64(1) + i) * np.uint64(g)
    q = np.stack([a + np.uint64(1 << 30), sz], axis=1).astype(np.uint64)
    s = np.array([0x1000], np.uint64)
    e = np.array([0x3000], np.uint64)
    lk = np.array([9], np.uint32)
    refs = np.array([2], np.uint32)
    nl = np.arange(m, dtype=np.uint32) + np.uint32(100)
    want = one_at_a_time(oracle, q, nl, s, e, lk, refs)
    same(register(db, q, nl, s, e, lk, refs), want, REG_KEYS)


@pytest.mark.parametrize("m,pages,granule_shift", [(700, 40, 12), (5000, 300, 12),
                                                    (150000, 3000, 12), (400000, 100000, 12),
                                                    (60000, 2000, 16)])
def test_register_nesting_in_one_batch(db, oracle, m, pages, granule_shift):
    """Requests over a few pages, so that new ranges lie inside earlier new
    ranges of the batch, repeat them, end where they end, and wrap old
    records whose hits they then take (a new record that starts before the
    old one): the one-at-a-time result, on every output."""
    rng = np.random.default_rng(m + pages + granule_shift)
    g = 1 << granule_shift
    n = max(1, pages // 20)
    s = np.sort(rng.integers(0, pages, size=n)).astype(np.uint64) * np.uint64(g)
    e = s + rng.integers(1, 12, size=n).astype(np.uint64) * np.uint64(g)
    lk = rng.integers(0, 2**32, size=n, dtype=np.uint64).astype(np.uint32)
    refs = rng.integers(1, 4, size=n).astype(np.uint32)
    a = rng.integers(0, pages, size=m).astype(np.uint64) * np.uint64(g)
    a += rng.integers(0, g, size=m).astype(np.uint64) * (rng.random(m) < 0.3)
    sz = rng.integers(1, 16 * g, size=m).astype(np.uint64)
    wide = rng.random(m) < 0.05            # a few wide ranges that hold many others
    sz = np.where(wide, rng.integers(16 * g, 400 * g, size=m).astype(np.uint64), sz)
    rep = rng.random(m) < 0.1
    src = rng.integers(0, m, size=m)
    a = np.where(rep & (src < np.arange(m)), a[src], a)
    sz = np.where(rep & (src < np.arange(m)), sz[src], sz)
    sz[::23] = 0
    q = np.stack([a, sz], axis=1).astype(np.uint64)
    nl = rng.integers(0, 2**32, size=m, dtype=np.uint64).astype(np.uint32)
    want = one_at_a_time(oracle, q, nl, s, e, lk, refs, granule_shift=granule_shift)
    kinds = want["kind"]
    assert (kinds == 5).sum() > 0 and (kinds == 4).sum() > 0
    got = register(db, q, nl, s, e, lk, refs, granule_shift=granule_shift)
    same(got, want, REG_KEYS)


@pytest.mark.parametrize("pattern", ["all_same", "digit_2", "digits_0_3", "digits_5_6",
                                     "all_digits"])
@pytest.mark.parametrize("granule_shift", [12, 16])
def test_register_sort_digit_patterns(db, oracle, pattern, granule_shift):
    """Missed ranges whose page numbers vary only in some 8-bit digits: the
    sort skips the passes on the other digits, so an even or odd number of
    passes runs (the result then has to move into the expected buffer)."""
    rng = np.random.default_rng(sum(map(ord, pattern)) + granule_shift)
    m, g = 6000, 1 << granule_shift
    top = 64 - granule_shift  # bits of a granule number
    if pattern == "all_same":
        pages = np.full(m, 0x12345, np.uint64)
    elif pattern == "digit_2":
        pages = np.uint64(0x30000000) | (rng.integers(0, 256, size=m).astype(np.uint64) << np.uint64(16))
    elif pattern == "digits_0_3":
        pages = (rng.integers(0, 256, size=m).astype(np.uint64)
                 | (rng.integers(0, 256, size=m).astype(np.uint64) << np.uint64(24)))
    elif pattern == "digits_5_6":
        hi = rng.integers(0, 1 << (top - 48), size=m).astype(np.uint64)
        pages = (rng.integers(0, 256, size=m).astype(np.uint64) << np.uint64(40)) | (hi << np.uint64(48))
    else:
        pages = rng.integers(0, 1 << (top - 1), size=m, dtype=np.uint64)
    pages = np.minimum(pages, np.uint64((1 << top) - 4))
    a = pages * np.uint64(g) + rng.integers(0, g, size=m).astype(np.uint64)
    sz = rng.integers(1, 2 * g, size=m).astype(np.uint64)
    if pattern == "all_same":
        a[:] = a[0]
        sz[:] = sz[0]
    q = np.stack([a, sz], axis=1).astype(np.uint64)
    nl = rng.integers(0, 2**32, size=m, dtype=np.uint64).astype(np.uint32)
    # a small table away from the requests, so nearly all of them miss
    s = np.arange(1, 9, dtype=np.uint64) * np.uint64(0x100 * g)
    e = s + np.uint64(g)
    lk = np.arange(8, dtype=np.uint32)
    refs = np.ones(8, np.uint32)
    want = one_at_a_time(oracle, q, nl, s, e, lk, refs, granule_shift=granule_shift)
    got = register(db, q, nl, s, e, lk, refs, granule_shift=granule_shift)
    same(got, want, REG_KEYS)


@pytest.mark.parametrize("case", ["one_long_range", "one_high_start", "at_the_limits"])
@pytest.mark.parametrize("granule_shift", [12, 16])
def test_register_packed_sort_key_limits(db, oracle, case, granule_shift):
    """The misses are sorted once on a key that packs the start granule
    above 24 bits of the length in granules when every miss fits it, and
    else on the end and then on the start: nested ordinary misses with one
    range 2^24 granules long, or one starting at granule 2^40 (no packed
    key), or ranges of 2^24 - 1 granules up to granule 2^40 - 1 (the
    largest that fit)."""
    rng = np.random.default_rng(len(case) * 31 + granule_shift)
    m, g = 5000, 1 << granule_shift
    pages = 3000
    a = rng.integers(0, pages, size=m).astype(np.uint64) * np.uint64(g)
    a += rng.integers(0, g, size=m).astype(np.uint64) * (rng.random(m) < 0.3)
    sz = rng.integers(1, 40 * g, size=m).astype(np.uint64)
    rep = rng.random(m) < 0.1
    src = rng.integers(0, m, size=m)
    a = np.where(rep & (src < np.arange(m)), a[src], a)
    sz = np.where(rep & (src < np.arange(m)), sz[src], sz)
    top = np.uint64(1 << 40)                 # the first start granule the key cannot hold
    longest = np.uint64((1 << 24) - 1)       # the longest length it can
    if case == "one_long_range":             # holds every other request
        a[2500], sz[2500] = 0, (longest + np.uint64(1)) * np.uint64(g)
    elif case == "one_high_start":
        a[2500], sz[2500] = top * np.uint64(g), np.uint64(3 * g)
    else:
        k = np.arange(40, 80)
        a[k] = (top - np.uint64(1) - np.arange(40, dtype=np.uint64) % np.uint64(3)) * np.uint64(g)
        sz[k] = (longest - np.arange(40, dtype=np.uint64) % np.uint64(2)) * np.uint64(g)
        a[4900], sz[4900] = 0, longest * np.uint64(g)
    q = np.stack([a, sz], axis=1).astype(np.uint64)
    nl = rng.integers(0, 2**32, size=m, dtype=np.uint64).astype(np.uint32)
    s = np.array([0x40 * g, 0x900 * g], np.uint64)
    e = s + np.uint64(8 * g)
    lk = np.array([3, 4], np.uint32)
    refs = np.array([1, 2], np.uint32)
    want = one_at_a_time(oracle, q, nl, s, e, lk, refs, granule_shift=granule_shift)
    assert (want["kind"] == 4).sum() > 500 and (want["kind"] == 5).sum() > 500
    got = register(db, q, nl, s, e, lk, refs, granule_shift=granule_shift)
    same(got, want, REG_KEYS)


@pytest.mark.parametrize("pattern", ["one_handle", "two_records"])
def test_deregister_sort_digit_patterns(db, oracle, pattern):
    """Handles naming one record (no sort pass runs) or two records apart in
    one digit."""
    n = 70000
    s = np.arange(n, dtype=np.uint64) * np.uint64(0x10000)
    e = s + np.uint64(0x8000)
    lk = np.arange(n, dtype=np.uint32)
    refs = np.full(n, 3, np.uint32)
    if pattern == "one_handle":
        hs = np.full(5000, 4242, np.int64)
    else:
        hs = np.where(np.arange(5000) % 3 == 0, 0x10005, 0x00005).astype(np.int64)
    same(deregister(db, hs, s, e, lk, refs), oracle.mr_deregister(hs, s, e, lk, refs),
         DEREG_KEYS)


def test_register_new_record_takes_a_later_hit(db, oracle):
    """A new range that starts before an old record and covers part of it
    takes a later request inside both (it comes first in the table); a
    later miss inside it is a hit on it; a lone new range that nothing
    asks for again changes no other request."""
    s = np.array([0x10000, 0x40000], np.uint64)
    e = np.array([0x20000, 0x50000], np.uint64)
    lk = np.array([11, 12], np.uint32)
    refs = np.array([1, 1], np.uint32)
    q = np.array([[0x8000, 0x10000],    # misses: new record from 0x8000, over the old start
                  [0x11000, 0x1000],    # inside the old record and the new one
                  [0x30000, 0x1000],    # a lone new record
                  [0x9000, 0x1000],     # a miss inside the first new record
                  [0x41000, 0x1000],    # an ordinary hit
                  [0x30000, 0x1000]],   # the lone record asked for again
                 np.uint64)
    nl = np.arange(100, 106, dtype=np.uint32)
    want = one_at_a_time(oracle, q, nl, s, e, lk, refs)
    got = register(db, q, nl, s, e, lk, refs)
    same(got, want, REG_KEYS)
    assert want["kind"].tolist()[:5] == [db.MR_NEW, db.MR_NEW_DUP, db.MR_NEW, db.MR_NEW_DUP,
                                         db.MR_CONTAINED]


@pytest.mark.parametrize("case", ["bucket_sizes", "one_huge_bucket", "zero_refs"])
def test_deregister_bucket_sizes(db, oracle, case):
    """Records named by 1..40 handles each (either side of the bucket size a
    handle ranks itself in), references below, at and above the handle
    count; one record named by 300,000 handles; records holding no
    reference."""
    rng = np.random.default_rng({"bucket_sizes": 1, "one_huge_bucket": 2, "zero_refs": 3}[case])
    n = 2000
    s = np.arange(n, dtype=np.uint64) * np.uint64(0x10000)
    e = s + np.uint64(0x8000)
    lk = np.arange(n, dtype=np.uint32)
    c = np.arange(n) % 40 + 1
    refs = (rng.integers(0, 3, size=n) + np.maximum(c - 1, 0)).astype(np.uint32)
    hs = np.repeat(np.arange(n), c)
    if case == "one_huge_bucket":
        hs = np.concatenate([hs, np.full(300000, 7)])
        refs[7] = 123457
    if case == "zero_refs":
        refs[::3] = 0
    hs = rng.permutation(hs).astype(np.int64)
    hs[::97] = -1
    same(deregister(db, hs, s, e, lk, refs), oracle.mr_deregister(hs, s, e, lk, refs),
         DEREG_KEYS)


def test_register_empty_batch_and_capacity(db, oracle):
    rng = np.random.default_rng(3)
    q, nl, s, e, lk, refs = random_case(rng, 50, 400, 400, 12)
    got = register(db, q[:0], nl[:0], s, e, lk, refs)
    same(got, one_at_a_time(oracle, q[:0], nl[:0], s, e, lk, refs), REG_KEYS)
    want = one_at_a_time(oracle, q, nl, s, e, lk, refs)
    total = int(want["ctr"][0])
    small = register(db, q, nl, s, e, lk, refs, out_cap=total - 1)
    assert small["ctr"].tolist() == [total, int(want["ctr"][1]), 1, 0]
    assert (small["kind"] == want["kind"]).all()
    grown = register(db, q, nl, s, e, lk, refs, out_cap=db.mr_capacity_for(total))
    same(grown, want, REG_KEYS)


def test_register_unsorted_table_is_flagged(db):
    s = np.array([0x3000, 0x1000], np.uint64)
    e = np.array([0x4000, 0x2000], np.uint64)
    r = register(db, np.array([[0x1000, 1]], np.uint64), [1], s, e, np.array([1, 2], np.uint32),
                 np.array([1, 1], np.uint32))
    assert int(r["ctr"][3]) & db.ERR_TABLE_ORDER


def test_register_full_size(db, oracle):
    """16,777,216 requests against 1,048,576 records: a fifth miss the table,
    and many of those lie inside an earlier one of the batch."""
    import synth
    d = synth.mr_register()
    args = (d["queries"], d["new_lkey"], d["mr_start"], d["mr_end"], d["mr_lkey"], d["mr_refs"])
    got = register(db, *args)
    want = one_at_a_time(oracle, *args)
    same(got, want, REG_KEYS)


@pytest.mark.parametrize("n,m", [(0, 10), (1, 5), (10, 0), (30, 200), (1000, 5000),
                                 (70000, 300000)])
def test_deregister_against_the_oracle(db, oracle, n, m):
    rng = np.random.default_rng(n + 3 * m)
    s = np.arange(n, dtype=np.uint64) * np.uint64(0x10000)
    e = s + np.uint64(0x8000)
    lk = rng.integers(0, 2**32, size=n, dtype=np.uint64).astype(np.uint32)
    refs = rng.integers(1, 6, size=n).astype(np.uint32)
    hs = rng.integers(-3, n + 3, size=m).astype(np.int64)
    hs[: m // 10] = rng.integers(-(2**62), 2**62, size=m // 10)
    same(deregister(db, hs, s, e, lk, refs), oracle.mr_deregister(hs, s, e, lk, refs),
         DEREG_KEYS)


def test_deregister_past_the_fused_scan_limit(db, oracle):
    """40,000,000 records: the scan of the per-record handle counts runs over
    more blocks than a block sums the earlier blocks' totals for itself, so
    the block totals are scanned first by one CTA."""
    n, m = 40_000_000, 1_000_000
    rng = np.random.default_rng(40)
    s = np.arange(n, dtype=np.uint64) * np.uint64(0x10000)
    e = s + np.uint64(0x8000)
    lk = (np.arange(n, dtype=np.uint64) & np.uint64(0xFFFFFFFF)).astype(np.uint32)
    refs = rng.integers(1, 3, size=n).astype(np.uint32)
    hs = rng.integers(-1, n, size=m).astype(np.int64)
    same(deregister(db, hs, s, e, lk, refs), oracle.mr_deregister(hs, s, e, lk, refs),
         DEREG_KEYS)


def test_register_past_the_fused_scan_limit(db):
    """34,000,000 requests: the prefix maxima of the ends run over more blocks
    than a block takes the earlier blocks' maximum for itself, so the block
    maxima are scanned first by one CTA. The first request asks for a range
    holding every later one (and two old records), so the one-at-a-time
    result is plain: it makes the only new record, at the head of the table,
    and every later request is a hit on it. A range whose only holder lies
    blocks away in the sorted order (most of them) would make a record of
    its own if a block's carry were wrong."""
    m, g = 34_000_000, 4096
    assert m > 8192 * 4096
    rng = np.random.default_rng(34)
    pages = 10_000_000
    a = rng.integers(1, pages, size=m).astype(np.uint64) * np.uint64(g)
    a += rng.integers(0, g, size=m).astype(np.uint64) * (rng.random(m) < 0.3)
    sz = rng.integers(1, 16 * g, size=m).astype(np.uint64)
    a[0], sz[0] = 0, np.uint64((pages + 32) * g)
    q = np.stack([a, sz], axis=1).astype(np.uint64)
    nl = (np.arange(m, dtype=np.uint64) * np.uint64(7) & np.uint64(0xFFFFFFFF)).astype(np.uint32)
    s = np.array([0x4000 * g, 0x9000 * g], np.uint64)  # inside the first range
    e = s + np.uint64(8 * g)
    lk = np.array([3, 4], np.uint32)
    refs = np.array([1, 2], np.uint32)
    got = register(db, q, nl, s, e, lk, refs)
    assert got["ctr"].tolist() == [3, 0, 0, 0]
    assert got["kind"][0] == 4 and (got["kind"][1:] == 5).all()
    assert (got["handle"] == 0).all() and got["remap"].tolist() == [1, 2]
    assert got["start"].tolist() == [0, int(s[0]), int(s[1])]
    assert got["end"].tolist() == [(pages + 32) * g, int(e[0]), int(e[1])]
    assert got["lkey"].tolist() == [int(nl[0]), 3, 4]
    assert got["refs"].tolist() == [m, 1, 2]


def test_deregister_full_size(db, oracle):
    import synth
    d = synth.mr_deregister()
    args = (d["handles"], d["mr_start"], d["mr_end"], d["mr_lkey"], d["mr_refs"])
    want = oracle.mr_deregister(*args)
    same(deregister(db, *args), want, DEREG_KEYS)
    assert set(want["status"].tolist()) == {0, 1, 2}


def test_a_cache_over_several_batches(db, oracle):
    """Register, deregister and register again, each batch on the table the
    previous one left, handles carried forward through remap."""
    rng = np.random.default_rng(11)
    q, nl, s, e, lk, refs = random_case(rng, 200, 5000, 3000, 12)
    t_gpu = t_cpu = (s, e, lk, refs)
    for step in range(3):
        r = register(db, q, nl, *t_gpu)
        w = one_at_a_time(oracle, q, nl, *t_cpu)
        same(r, w, REG_KEYS)
        t_gpu = (r["start"], r["end"], r["lkey"], r["refs"])
        t_cpu = (w["start"], w["end"], w["lkey"], w["refs"])
        held = r["handle"][r["handle"] >= 0]
        hs = np.concatenate([held, held[: held.shape[0] // 2]])
        rng.shuffle(hs)
        d = deregister(db, hs, *t_gpu)
        v = oracle.mr_deregister(hs, *t_cpu)
        same(d, v, DEREG_KEYS)
        t_gpu = (d["start"], d["end"], d["lkey"], d["refs"])
        t_cpu = (v["start"], v["end"], v["lkey"], v["refs"])
        q, nl = q[::-1].copy(), nl[::-1].copy()


def test_argument_checks(db):
    z = torch.zeros(4, dtype=torch.int64, device="cuda")
    z32 = torch.zeros(4, dtype=torch.int32, device="cuda")
    q = torch.zeros((1, 2), dtype=torch.int64, device="cuda")
    ws = db.workspace(db.mr_register_workspace_size(1, 4))
    with pytest.raises(db.DescBuildError):             # granule neither 4 KiB nor 64 KiB
        db.mr_register(q, z32[:1], z, z, z32, z32, z, z, z32, z32, z[:1],
                       torch.zeros(1, dtype=torch.uint8, device="cuda"), z, ws, granule_shift=13)
    with pytest.raises(db.DescBuildError) as e:        # workspace too small
        db.mr_register(q, z32[:1], z, z, z32, z32, z, z, z32, z32, z[:1],
                       torch.zeros(1, dtype=torch.uint8, device="cuda"), z, ws[:256])
    assert e.value.code == -28
