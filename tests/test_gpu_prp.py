"""db_prp_build on the GPU against the oracle, bit for bit.

Integer work: every output word must equal the oracle's.
"""

import numpy as np
import pytest

from conftest import h, load_golden
from gpu_util import assert_arena_equal, dev64, host64, lib, need_gpu, torch

pytestmark = pytest.mark.gpu

FILL = -0x2152411021524111  # 0xDEADBEEFDEADBEEF as int64

# The library picks one of two schedules by batch size (one persistent kernel
# with a decoupled lookback, or a pair kernel followed by a list kernel);
# the tests run both on the same inputs, and the default choice on the
# full-size workloads.
SCHEDS = ["single", "split"]


@pytest.fixture(scope="module")
def db():
    need_gpu()
    return lib()


def sched_flags(db, sched):
    return {"auto": 0, "single": db.PRP_SCHED_SINGLE, "split": db.PRP_SCHED_SPLIT}[sched]


def run_gpu(db, req, lut, heap, arena_base, cap, flags=0, ws=None, with_arena=True,
            host_arena=False, per_request=True, sched="auto"):
    """One db_prp_build call. per_request=False leaves page_base and status
    out, as the benchmark's calls do (a tile with no list then skips its
    lookback, or its list kernel pass)."""
    flags |= sched_flags(db, sched)
    n = req.shape[0]
    d_req = dev64(req) if n else torch.zeros((0, 2), dtype=torch.int64, device="cuda")
    if not with_arena:
        arena = None
    elif host_arena:  # pinned host memory, written by the kernel across the link
        arena = torch.full((max(cap, 1), 512), FILL, dtype=torch.int64).pin_memory()
    else:
        arena = torch.full((max(cap, 1), 512), FILL, dtype=torch.int64, device="cuda")
    prp = torch.full((max(n, 1), 2), FILL, dtype=torch.int64, device="cuda")
    pb = torch.full((max(n, 1),), FILL, dtype=torch.int64, device="cuda")
    st = torch.full((max(n, 1),), 0xEE, dtype=torch.uint8, device="cuda")
    ctr = torch.full((4,), FILL, dtype=torch.int64, device="cuda")
    if ws is None:
        ws = db.workspace(db.prp_workspace_size(n))
    db.prp_build(d_req, dev64(lut), heap, arena_base, cap, arena, prp, ws,
                 page_base=pb if per_request else None, status=st if per_request else None,
                 ctr=ctr, flags=flags)
    torch.cuda.synchronize()
    return dict(prp=host64(prp)[:n], page_base=host64(pb)[:n] if per_request else None,
                status=st.cpu().numpy()[:n] if per_request else None,
                ctr=host64(ctr), arena=arena)


def compare(oracle, got, want, cap, zero_tail):
    assert (got["prp"] == want["prp"]).all()
    if got["page_base"] is not None:
        assert (got["page_base"] == want["page_base"]).all()
    if got["status"] is not None:
        assert (got["status"] == want["status"]).all()
    assert (got["ctr"] == want["ctr"]).all(), (got["ctr"], want["ctr"])
    if got["arena"] is not None:
        used = min(int(want["ctr"][0]), cap)
        a = host64(got["arena"][:max(used, 1)])[:used]
        # The oracle's arena was filled with the same marker: untouched slots agree too.
        if zero_tail:
            assert (a == want["arena"][:used]).all()
        else:
            assert_arena_equal(a, want["arena"][:used], FILL)
        if used < cap:
            rest = host64(got["arena"][used:used + 4])
            assert (rest == np.uint64(FILL & (2**64 - 1))).all()


@pytest.mark.parametrize("sched", SCHEDS)
def test_golden_hand_cases(db, sched):
    fx = load_golden("prp_hand_cases.json")
    n_lut = fx["heap_size"] // 65536
    lut = np.array([0x900000000 + c * 0x30000 for c in range(n_lut)], dtype=np.uint64)
    for c, v in enumerate(fx["lut_explicit"]):
        lut[c] = h(v)
    for case in fx["cases"]:
        cap = case.get("arena_cap_pages", fx["arena_cap_pages"])
        req = np.array([[h(o), int(n)] for o, n in case["req"]], dtype=np.uint64)
        got = run_gpu(db, req, lut, fx["heap_size"], h(fx["arena_base"]), cap, sched=sched)
        want = np.array([[h(a), h(b)] for a, b in case["prp"]], dtype=np.uint64)
        assert (got["prp"] == want).all(), case["name"]
        assert got["page_base"].tolist() == case["page_base"], case["name"]
        assert got["status"].tolist() == case["status"], case["name"]
        assert int(got["ctr"][0]) == case["total_pages"], case["name"]
        arena = host64(got["arena"])
        for lp in case["lists"]:
            for slot, val in lp["slots"].items():
                assert int(arena[lp["page"], int(slot)]) == h(val), (case["name"], lp, slot)


@pytest.mark.parametrize("sched", SCHEDS)
@pytest.mark.parametrize("zero_tail", [False, True])
def test_tiny_workload(db, oracle, zero_tail, sched):
    import synth
    w = synth.prp_tiny()
    cap = 4096
    want = oracle.prp_build(w["req"], w["lut"], w["heap_size"], w["arena_base"], cap,
                            zero_tail=zero_tail, fill=FILL & (2**64 - 1))
    got = run_gpu(db, w["req"], w["lut"], w["heap_size"], w["arena_base"], cap,
                  flags=db.PRP_ZERO_TAIL if zero_tail else 0, sched=sched)
    compare(oracle, got, want, cap, zero_tail)


def random_batch(rng, n, heap, max_len, invalid_frac=0.02):
    off = 4 * rng.integers(0, heap // 4, size=n).astype(np.uint64)
    length = rng.integers(1, max_len + 1, size=n).astype(np.uint64)
    length = np.minimum(length, np.uint64(heap) - off)
    bad = rng.random(n) < invalid_frac
    kind = rng.integers(0, 3, size=n)
    length = np.where(bad & (kind == 0), 0, length)
    off = np.where(bad & (kind == 1), off + np.uint64(2), off)
    length = np.where(bad & (kind == 2), np.uint64(heap), length)
    length[length == 0] = np.where(bad[length == 0], 0, 1)
    return np.stack([off, length], axis=1).astype(np.uint64)


@pytest.mark.parametrize("sched", SCHEDS)
@pytest.mark.parametrize("per_request", [True, False])
@pytest.mark.parametrize("n", [1, 2, 511, 512, 513, 2047, 2048, 2049, 4999, 70001])
def test_random_batches_ragged(db, oracle, n, per_request, sched):
    """Several tiles of 2048 and a ragged tail, lists of all lengths."""
    import synth
    rng = np.random.default_rng(1000 + n)
    heap = 64 * 1024 * 1024
    lut = synth.physical_lut(rng, heap // 65536)
    req = random_batch(rng, n, heap, 5 * 1024 * 1024 if n < 5000 else 300 * 1024)
    need = oracle.prp_build(req, lut, heap, 0x7_0000_0000, 1 << 40, lists=False)
    cap = max(1, int(need["ctr"][0]))
    want = oracle.prp_build(req, lut, heap, 0x7_0000_0000, cap, fill=FILL & (2**64 - 1))
    got = run_gpu(db, req, lut, heap, 0x7_0000_0000, cap, per_request=per_request, sched=sched)
    compare(oracle, got, want, cap, False)


@pytest.mark.parametrize("sched", SCHEDS)
@pytest.mark.parametrize("per_request", [True, False])
@pytest.mark.parametrize("spacing", [1, 3, 129, 300])
def test_sparse_lists(db, oracle, spacing, per_request, sched):
    """Lists in one tile of every `spacing`, the tiles between them holding
    only one- and two-page requests. Without page_base those tiles skip their
    lookback, so a list tile's lookback sums runs of zero aggregates (more
    than one 128-tile window when spacing > 128)."""
    import synth
    rng = np.random.default_rng(7000 + spacing)
    heap = 256 * 1024 * 1024
    lut = synth.physical_lut(rng, heap // 65536)
    tiles = 2 * spacing + 5 if spacing > 3 else 40
    n = tiles * 2048 - 777  # ragged last tile
    off = 4 * rng.integers(0, (heap - 8192) // 4, size=n).astype(np.uint64)
    length = rng.integers(1, 4097, size=n).astype(np.uint64)  # at most two pages
    list_tiles = np.arange(spacing - 1, tiles, spacing)
    for t in list_tiles:
        rows = t * 2048 + rng.choice(2048, size=5, replace=False)
        rows = rows[rows < n]
        off[rows] = 4096 * rng.integers(0, heap // 4096 - 1024, size=rows.size).astype(np.uint64)
        length[rows] = rng.integers(3 * 4096, 2 * 1024 * 1024, size=rows.size).astype(np.uint64)
    req = np.stack([off, length], axis=1).astype(np.uint64)
    need = oracle.prp_build(req, lut, heap, 0x7_0000_0000, 1 << 40, lists=False)
    cap = max(1, int(need["ctr"][0]))
    assert cap > 1
    want = oracle.prp_build(req, lut, heap, 0x7_0000_0000, cap, fill=FILL & (2**64 - 1))
    got = run_gpu(db, req, lut, heap, 0x7_0000_0000, cap, per_request=per_request, sched=sched)
    compare(oracle, got, want, cap, False)
    # Further calls on one workspace (next epochs), the schedules mixed.
    ws = db.workspace(db.prp_workspace_size(n))
    for s in (sched, "single", "split", sched):
        got = run_gpu(db, req, lut, heap, 0x7_0000_0000, cap, ws=ws, per_request=per_request,
                      sched=s)
    compare(oracle, got, want, cap, False)


@pytest.mark.parametrize("sched", SCHEDS)
@pytest.mark.parametrize("per_request", [True, False])
def test_more_tiles_than_resident_ctas(db, oracle, per_request, sched):
    """A batch of 700,001 requests (342 tiles of 2048, a ragged last one):
    more tiles than CTAs run at once, so CTAs take second tiles by ticket
    while others still write lists. One request in ten owns a list, so
    nearly every tile takes the list path."""
    import synth
    rng = np.random.default_rng(4343)
    n = 700_001
    heap = 256 * 1024 * 1024
    lut = synth.physical_lut(rng, heap // 65536)
    off = 4 * rng.integers(0, (heap - (1 << 21)) // 4, size=n).astype(np.uint64)
    length = rng.integers(1, 8193, size=n).astype(np.uint64)
    big = rng.random(n) < 0.1
    length[big] = rng.integers(3 * 4096, 1 << 21, size=int(big.sum())).astype(np.uint64)
    req = np.stack([off, length], axis=1).astype(np.uint64)
    need = oracle.prp_build(req, lut, heap, 0x7_0000_0000, 1 << 40, lists=False)
    cap = int(need["ctr"][0])
    want = oracle.prp_build(req, lut, heap, 0x7_0000_0000, cap, fill=FILL & (2**64 - 1))
    got = run_gpu(db, req, lut, heap, 0x7_0000_0000, cap, per_request=per_request, sched=sched)
    compare(oracle, got, want, cap, False)


@pytest.mark.parametrize("sched", SCHEDS)
@pytest.mark.parametrize("zero_tail", [False, True])
def test_arena_in_pinned_host_memory(db, oracle, zero_tail, sched):
    """The lists written straight into a pinned host arena equal the oracle's."""
    rng = np.random.default_rng(77)
    heap = 64 * 1024 * 1024
    lut = (rng.choice(np.arange(1, 1 << 20, dtype=np.uint64), size=heap // 65536, replace=False)
           << np.uint64(16))
    n = 20000
    off = 4 * rng.integers(0, heap // 4, size=n).astype(np.uint64)
    ln = rng.integers(1, 3 * 1024 * 1024, size=n).astype(np.uint64)
    ln = np.minimum(ln, np.uint64(heap) - off)
    req = np.stack([off, ln], axis=1).astype(np.uint64)
    cap = int(oracle.prp_build(req, lut, heap, 0x2_0000_0000, 1 << 40, lists=False)["ctr"][0])
    want = oracle.prp_build(req, lut, heap, 0x2_0000_0000, cap, zero_tail=zero_tail,
                            fill=FILL & (2**64 - 1))
    got = run_gpu(db, req, lut, heap, 0x2_0000_0000, cap,
                  flags=db.PRP_ZERO_TAIL if zero_tail else 0, host_arena=True, sched=sched)
    compare(oracle, got, want, cap, zero_tail)


@pytest.mark.parametrize("sched", SCHEDS)
def test_arena_overflow_and_capacity_edges(db, oracle, sched):
    import synth
    rng = np.random.default_rng(7)
    heap = 16 * 1024 * 1024
    lut = synth.physical_lut(rng, heap // 65536)
    req = random_batch(rng, 3000, heap, 3 * 1024 * 1024)
    full = oracle.prp_build(req, lut, heap, 0x10000000, 1 << 20, lists=False)
    total = int(full["ctr"][0])
    for cap in (0, 1, total // 3, total - 1, total, total + 5):
        want = oracle.prp_build(req, lut, heap, 0x10000000, cap, fill=FILL & (2**64 - 1))
        got = run_gpu(db, req, lut, heap, 0x10000000, cap, sched=sched)
        compare(oracle, got, want, cap, False)


@pytest.mark.parametrize("sched", SCHEDS)
def test_empty_and_all_invalid(db, oracle, sched):
    import synth
    lut = synth.physical_lut(np.random.default_rng(1), 16)
    got = run_gpu(db, np.zeros((0, 2), dtype=np.uint64), lut, 1 << 20, 0, 4, sched=sched)
    assert got["ctr"].tolist() == [0, 0, 0, 0]
    req = np.array([[0, 0], [3, 100], [1 << 20, 1], [(1 << 20) - 4, 8]] * 300, dtype=np.uint64)
    want = oracle.prp_build(req, lut, 1 << 20, 0, 4)
    got = run_gpu(db, req, lut, 1 << 20, 0, 4, sched=sched)
    compare(oracle, got, want, 4, False)
    assert int(got["ctr"][1]) == 1200


@pytest.mark.parametrize("sched", SCHEDS)
def test_largest_requests(db, oracle, sched):
    """Lengths up to 2^32 - 1 bytes (1,048,577 pages, 2053 list pages)."""
    import synth
    rng = np.random.default_rng(3)
    heap = 8 * 1024**3
    lut = synth.physical_lut(rng, heap // 65536)
    req = np.array([[0, 0xFFFFFFFF], [4092, 0xFFFFFFFF], [4 << 30, 0xFFFFF000],
                    [12, 513 * 4096]], dtype=np.uint64)
    want = oracle.prp_build(req, lut, heap, 0x1_0000_0000, 8192, fill=FILL & (2**64 - 1))
    assert int(want["ctr"][0]) > 6000
    got = run_gpu(db, req, lut, heap, 0x1_0000_0000, 8192, sched=sched)
    compare(oracle, got, want, 8192, False)


def test_workspace_reuse_across_calls(db, oracle):
    """One workspace, many calls of different sizes: results stay exact."""
    import synth
    rng = np.random.default_rng(11)
    heap = 32 * 1024 * 1024
    lut = synth.physical_lut(rng, heap // 65536)
    ws = db.workspace(db.prp_workspace_size(40000))
    for j, n in enumerate((40000, 100, 7, 40000, 513, 20000)):
        req = random_batch(rng, n, heap, 1024 * 1024)
        want = oracle.prp_build(req, lut, heap, 0x40000000, 1 << 16, fill=FILL & (2**64 - 1))
        got = run_gpu(db, req, lut, heap, 0x40000000, 1 << 16, ws=ws,
                      sched=("auto", "single", "split")[j % 3])
        compare(oracle, got, want, 1 << 16, False)


def test_bad_arguments(db):
    t = torch.zeros((4, 2), dtype=torch.int64, device="cuda")
    lut = torch.ones(16, dtype=torch.int64, device="cuda") << 16
    ws = db.workspace(db.prp_workspace_size(4))
    with pytest.raises(db.DescBuildError, match="invalid"):
        db.prp_build(t, lut, 1000, 0, 1, t, t, ws)           # heap not a multiple of 64 KiB
    with pytest.raises(db.DescBuildError, match="invalid"):
        db.prp_build(t, lut, 1 << 20, 100, 1, t, t, ws)      # arena base not page aligned
    with pytest.raises(db.DescBuildError, match="workspace"):
        db.prp_build(t, lut, 1 << 20, 0, 1, t, t, ws[:16])
    with pytest.raises(db.DescBuildError, match="invalid"):
        db.prp_build(t, lut, 1 << 20, 0, 1, t, t, ws, flags=8)
    with pytest.raises(db.DescBuildError, match="invalid"):           # both schedules at once
        db.prp_build(t, lut, 1 << 20, 0, 1, t, t, ws,
                     flags=db.PRP_SCHED_SINGLE | db.PRP_SCHED_SPLIT)


def test_lookback_timeout_is_reported(db, oracle):
    """A predecessor tile that never publishes: the bounded wait gives up,
    the call reports DB_ERR_TIMEOUT, and the workspace works again after
    (single-kernel schedule: the two-kernel one has no wait)."""
    import synth
    rng = np.random.default_rng(5)
    heap = 16 * 1024 * 1024
    lut = synth.physical_lut(rng, heap // 65536)
    req = random_batch(rng, 4 * 2048, heap, 64 * 1024)   # four tiles of 2048 requests
    ws = db.workspace(db.prp_workspace_size(req.shape[0]))
    # The first 8 bytes of the workspace hold the next tile ticket, 0 between
    # calls. Starting at 1 means no CTA ever takes tile 0.
    ws[:8].view(torch.int64).fill_(1)
    got = run_gpu(db, req, lut, heap, 0, 1 << 14, ws=ws, sched="single")
    assert int(got["ctr"][3]) & db.ERR_TIMEOUT
    want = oracle.prp_build(req, lut, heap, 0, 1 << 14, fill=FILL & (2**64 - 1))
    for s in ("single", "split"):
        got = run_gpu(db, req, lut, heap, 0, 1 << 14, ws=ws, sched=s)
        compare(oracle, got, want, 1 << 14, False)


def test_epoch_tag_wrap(db, oracle):
    """Calls across the wrap of the 22-bit tag of the status words, the
    schedules mixed, with and without lists: the words left by calls before
    the wrap are cleared when the tag comes round, so no call reads another
    call's words as its own. The header's epoch (bytes 16..19 of the
    workspace) starts two calls short of the wrap."""
    import synth
    rng = np.random.default_rng(2222)
    heap = 64 * 1024 * 1024
    lut = synth.physical_lut(rng, heap // 65536)
    n = 9 * 2048 + 5
    ws = db.workspace(db.prp_workspace_size(n))
    ws[16:20].view(torch.int32).fill_((1 << 22) - 2)
    with_lists = random_batch(rng, n, heap, 300 * 1024)
    no_lists = random_batch(rng, n, heap, 4096)
    plan = [(with_lists, "single"), (no_lists, "split"), (with_lists, "split"),
            (no_lists, "single"), (with_lists, "single"), (no_lists, "split"),
            (with_lists, "split")]
    for req, sched in plan:
        want = oracle.prp_build(req, lut, heap, 0x7_0000_0000, 1 << 14, fill=FILL & (2**64 - 1))
        for per_request in (False, True):
            got = run_gpu(db, req, lut, heap, 0x7_0000_0000, 1 << 14, ws=ws,
                          per_request=per_request, sched=sched)
            compare(oracle, got, want, 1 << 14, False)
    assert int(ws[16:20].view(torch.int32).item()) == (1 << 22) + 12  # 14 calls on


@pytest.mark.parametrize("sched", ["auto"] + SCHEDS)
@pytest.mark.parametrize("per_request", [True, False])
def test_small_io_workload_full(db, oracle, per_request, sched):
    """1,048,576 small requests: every output against the oracle (without
    page_base and status: the benchmark's call)."""
    import synth
    w = synth.prp_small()
    want = oracle.prp_build(w["req"], w["lut"], w["heap_size"], w["arena_base"], 1024)
    assert int(want["ctr"][0]) == 0  # the list path is never taken here
    got = run_gpu(db, w["req"], w["lut"], w["heap_size"], w["arena_base"], 1024,
                  per_request=per_request, sched=sched)
    compare(oracle, got, want, 1024, False)


@pytest.mark.parametrize("sched", ["auto", "split"])
@pytest.mark.parametrize("per_request", [True, False])
def test_large_workload_full_size(db, oracle, per_request, sched):
    """4,194,304 requests on a 16 GiB heap: PRPs, page bases and counters of
    every request, and every word of the ~17 GB list arena, against the oracle
    (per_request=False is the benchmark's call). The arena is compared in
    slices of requests: a slice [i0, i1) whose first list page is P0 is the
    oracle's batch of those requests with its arena base moved on by P0
    pages, which gives the same PRP2 values and chain pointers."""
    import synth
    w = synth.prp_large()
    req, lut = w["req"], w["lut"]
    n = req.shape[0]
    full = oracle.prp_build(req, lut, w["heap_size"], w["arena_base"], 1 << 40, lists=False)
    cap = int(full["ctr"][0])
    want = oracle.prp_build(req, lut, w["heap_size"], w["arena_base"], cap, lists=False)
    got = run_gpu(db, req, lut, w["heap_size"], w["arena_base"], cap, per_request=per_request,
                  sched=sched)
    assert (got["prp"] == want["prp"]).all()
    if per_request:
        assert (got["page_base"] == want["page_base"]).all()
        assert (got["status"] == want["status"]).all()
    assert (got["ctr"] == want["ctr"]).all()
    arena = got["arena"]
    fill = FILL & (2**64 - 1)
    pb = want["page_base"]
    step = 1 << 18
    for i0 in range(0, n, step):
        i1 = min(n, i0 + step)
        p0 = int(pb[i0])
        p1 = int(pb[i1]) if i1 < n else cap
        part = oracle.prp_build(req[i0:i1], lut, w["heap_size"], w["arena_base"] + 4096 * p0,
                                p1 - p0, fill=fill)
        assert (part["prp"] == want["prp"][i0:i1]).all()
        assert int(part["ctr"][0]) == p1 - p0
        assert_arena_equal(host64(arena[p0:p1]), part["arena"][:p1 - p0], FILL,
                           where=f"requests {i0}..{i1}")
    del arena
    torch.cuda.empty_cache()
