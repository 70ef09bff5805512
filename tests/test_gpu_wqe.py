"""db_wqe_bucket on the GPU against the oracle, bit for bit."""

import numpy as np
import pytest

from conftest import h, load_golden
from gpu_util import dev32, dev64, host32, host64, lib, need_gpu, torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def db():
    need_gpu()
    return lib()


def run_gpu(db, req, peer_ptrs, rkeys, world, n_qp, local_base, lkey, heap, depth, head,
            fill=0xCD, ws=None, rings=None):
    n = req.shape[0]
    R = world * n_qp
    if rings is None:
        rings = torch.full((R, depth, 64), fill, dtype=torch.uint8, device="cuda")
    d_head = dev64(np.asarray(head, dtype=np.uint64))
    count = torch.full((R,), -1, dtype=torch.int32, device="cuda")
    ctr = torch.full((4,), -1, dtype=torch.int64, device="cuda")
    if ws is None:
        ws = db.workspace(db.wqe_workspace_size(n, R))
    d_req = dev64(req) if n else torch.zeros((0, 2), dtype=torch.int64, device="cuda")
    db.wqe_bucket(d_req, dev64(np.asarray(peer_ptrs, dtype=np.uint64)),
                  dev32(np.asarray(rkeys, dtype=np.uint32)), world, n_qp, local_base, lkey, heap,
                  rings, depth, d_head, count, ws, ctr=ctr)
    torch.cuda.synchronize()
    return dict(rings=rings, head=host64(d_head), count=host32(count), ctr=host64(ctr))


def check(got, want, compare_rings=True):
    assert (got["head"] == want["head"]).all()
    assert (got["count"] == want["count"]).all()
    assert (got["ctr"] == want["ctr"]).all(), (got["ctr"], want["ctr"])
    if compare_rings:
        assert (got["rings"].cpu().numpy() == want["rings"]).all()


@pytest.mark.parametrize("variant", ["depth4", "depth1"])
def test_golden(db, variant):
    fx = load_golden("wqe_hand_cases.json")
    v = fx[variant]
    from synth import pack_put_requests
    req = pack_put_requests([h(r["off"]) for r in fx["req"]], [r["bytes"] for r in fx["req"]],
                            [r["pe"] for r in fx["req"]], [r["qp"] for r in fx["req"]])
    got = run_gpu(db, req, [h(x) for x in fx["peer_ptrs"]], fx["rkeys"], fx["world"],
                  fx["n_qp"], h(fx["local_base"]), fx["lkey"], fx["heap_size"], v["depth"],
                  fx["head"])
    assert got["head"].tolist() == v["head"]
    assert got["count"].tolist() == v["count"]
    assert got["ctr"].tolist() == v["ctr"]
    rings = got["rings"].cpu().numpy()
    u64 = rings.view(np.uint64).reshape(rings.shape[0], rings.shape[1], 8)
    u32 = rings.view(np.uint32).reshape(rings.shape[0], rings.shape[1], 16)
    for e in v["wqes"]:
        r, s = e["ring"], e["slot"]
        assert int(u64[r, s, 0]) == h(e["raddr"]) and int(u64[r, s, 1]) == h(e["laddr"])
        assert [int(x) for x in u32[r, s, 4:8]] == [e["len"], e["lkey"], e["rkey"], 0]
        assert int(u64[r, s, 4]) == e["seq"] and int(u32[r, s, 10]) == e["req_index"]


def random_puts(rng, n, world, n_qp, heap, invalid_frac=0.03):
    pe = rng.integers(0, world, size=n)
    qp = rng.integers(0, n_qp, size=n)
    nbytes = 16 * rng.integers(1, 4097, size=n)
    off = 16 * rng.integers(0, (heap - 65536) // 16, size=n)
    bad = rng.random(n) < invalid_frac
    kind = rng.integers(0, 4, size=n)
    pe = np.where(bad & (kind == 0), world + rng.integers(0, 100, size=n), pe)
    qp = np.where(bad & (kind == 1), n_qp + rng.integers(0, 7, size=n), qp)
    nbytes = np.where(bad & (kind == 2), 0, nbytes)
    off = np.where(bad & (kind == 3), heap - 8, off)
    from synth import pack_put_requests
    return pack_put_requests(off, nbytes, pe, qp)


@pytest.mark.parametrize("n,world,n_qp,depth", [
    (1, 8, 4, 64), (255, 8, 4, 64), (256, 8, 4, 64), (257, 8, 4, 64), (2049, 8, 4, 64),
    (1023, 8, 4, 64), (1024, 8, 4, 64), (1025, 8, 4, 64),
    (5000, 8, 4, 256), (5000, 8, 4, 128),       # 128: some rings overflow
    (20000, 3, 5, 2048), (20000, 1, 1, 32768), (7777, 16, 2, 512),
    (100000, 256, 4, 256), (60000, 1024, 1, 128), (300000, 8, 4, 16384)])
def test_random_batches(db, oracle, n, world, n_qp, depth):
    rng = np.random.default_rng(n * 7 + world)
    heap = 1 << 32
    req = random_puts(rng, n, world, n_qp, heap)
    peer = (rng.integers(1 << 19, 1 << 26, size=world) << 21).astype(np.uint64)
    rkeys = rng.integers(0, 2**32, size=world, dtype=np.uint64).astype(np.uint32)
    head = rng.integers(0, 2**40, size=world * n_qp).astype(np.uint64)
    lb, lk = 0x7F0000000000, 0xC0FFEE
    want = oracle.wqe_bucket(req, peer, rkeys, world, n_qp, lb, lk, heap, depth, head, fill=0xCD)
    got = run_gpu(db, req, peer, rkeys, world, n_qp, lb, lk, heap, depth, head)
    check(got, want)


def test_repeated_batches_advance_heads(db, oracle):
    """Four batches into the same rings: heads carry over, rings wrap."""
    rng = np.random.default_rng(21)
    world, n_qp, depth, heap = 4, 2, 4096, 1 << 30
    peer = (rng.integers(1 << 19, 1 << 26, size=world) << 21).astype(np.uint64)
    rkeys = rng.integers(0, 2**32, size=world, dtype=np.uint64).astype(np.uint32)
    head = np.zeros(world * n_qp, dtype=np.uint64)
    rings = torch.full((world * n_qp, depth, 64), 0xCD, dtype=torch.uint8, device="cuda")
    host_rings = np.full((world * n_qp, depth, 64), 0xCD, dtype=np.uint8)
    ws = db.workspace(db.wqe_workspace_size(30000, world * n_qp))
    for n in (30000, 11, 29999, 2048):
        req = random_puts(rng, n, world, n_qp, heap)
        want = oracle.wqe_bucket(req, peer, rkeys, world, n_qp, 0x1000, 5, heap, depth, head)
        # Merge what the oracle wrote into the previous ring contents.
        written = np.zeros(host_rings.shape[:2], dtype=bool)
        for r in range(world * n_qp):
            if want["head"][r] != head[r]:
                seqs = np.arange(int(head[r]), int(want["head"][r]))
                written[r, seqs % depth] = True
        host_rings[written] = want["rings"][written]
        got = run_gpu(db, req, peer, rkeys, world, n_qp, 0x1000, 5, heap, depth, head, ws=ws,
                      rings=rings)
        check(got, dict(want, rings=host_rings))
        head = want["head"]


def test_empty_batch(db):
    got = run_gpu(db, np.zeros((0, 2), dtype=np.uint64), [1 << 40], [1], 1, 3, 0, 0, 1 << 20,
                  8, [4, 5, 6])
    assert got["count"].tolist() == [0, 0, 0]
    assert got["head"].tolist() == [4, 5, 6]
    assert got["ctr"].tolist() == [0, 0, 0, 0]


def test_bad_arguments(db):
    t = torch.zeros((4, 2), dtype=torch.int64, device="cuda")
    p = torch.zeros(8, dtype=torch.int64, device="cuda")
    k = torch.zeros(8, dtype=torch.int32, device="cuda")
    rings = torch.zeros((32, 8, 64), dtype=torch.uint8, device="cuda")
    head = torch.zeros(32, dtype=torch.int64, device="cuda")
    cnt = torch.zeros(32, dtype=torch.int32, device="cuda")
    ws = db.workspace(db.wqe_workspace_size(4, 32))
    with pytest.raises(db.DescBuildError, match="invalid"):
        db.wqe_bucket(t, p, k, 8, 4, 0, 0, 1 << 20, rings, 6, head, cnt, ws)  # depth not pow2
    with pytest.raises(db.DescBuildError, match="invalid"):
        db.wqe_bucket(t, p, k, 0, 4, 0, 0, 1 << 20, rings, 8, head, cnt, ws)  # no PEs
    with pytest.raises(db.DescBuildError, match="invalid"):
        db.wqe_bucket(t, p, k, 2048, 1, 0, 0, 1 << 20, rings, 8, head, cnt, ws)  # > 1024 rings
    with pytest.raises(db.DescBuildError, match="workspace"):
        db.wqe_bucket(t, p, k, 8, 4, 0, 0, 1 << 20, rings, 8, head, cnt, ws[:256])


def test_full_size_workload(db, oracle):
    """8,388,608 puts into 32 rings of 2^19 entries, every byte against the oracle."""
    import synth
    p = synth.put_bucket()
    want = oracle.wqe_bucket(p["req"], p["peer_ptrs"], p["rkeys"], p["world"], p["n_qp"],
                             p["local_base"], p["lkey"], p["heap_size"], p["depth"], p["head"],
                             fill=0xCD)
    got = run_gpu(db, p["req"], p["peer_ptrs"], p["rkeys"], p["world"], p["n_qp"],
                  p["local_base"], p["lkey"], p["heap_size"], p["depth"], p["head"])
    check(got, want)


def test_columns_longer_than_one_scan_round(db, oracle):
    """33,072 tiles of 256 puts: the scan of each ring's column takes two
    rounds of 32,768 entries, the second one ragged."""
    rng = np.random.default_rng(4242)
    n = 32768 * 256 + 77777
    world, n_qp, depth, heap = 4, 2, 1 << 21, 1 << 32
    req = random_puts(rng, n, world, n_qp, heap)
    peer = (rng.integers(1 << 19, 1 << 26, size=world) << 21).astype(np.uint64)
    rkeys = rng.integers(0, 2**32, size=world, dtype=np.uint64).astype(np.uint32)
    head = rng.integers(0, 2**40, size=world * n_qp).astype(np.uint64)
    lb, lk = 0x7F0000000000, 0xC0FFEE
    want = oracle.wqe_bucket(req, peer, rkeys, world, n_qp, lb, lk, heap, depth, head, fill=0xCD)
    got = run_gpu(db, req, peer, rkeys, world, n_qp, lb, lk, heap, depth, head)
    check(got, want)


@pytest.mark.parametrize("depth", [1 << 14, 256])  # 256: every ring overflows and stays untouched
def test_rings_in_pinned_host_memory(db, oracle, depth):
    """The WQEs written straight into rings in pinned host memory equal the
    oracle's, and so do the slots the batch leaves alone."""
    rng = np.random.default_rng(515 + depth)
    n, world, n_qp, heap = 50000, 8, 4, 1 << 32
    req = random_puts(rng, n, world, n_qp, heap)
    peer = (rng.integers(1 << 19, 1 << 26, size=world) << 21).astype(np.uint64)
    rkeys = rng.integers(0, 2**32, size=world, dtype=np.uint64).astype(np.uint32)
    head = rng.integers(0, 2**40, size=world * n_qp).astype(np.uint64)
    lb, lk = 0x7F0000000000, 0xC0FFEE
    want = oracle.wqe_bucket(req, peer, rkeys, world, n_qp, lb, lk, heap, depth, head, fill=0xCD)
    rings = torch.full((world * n_qp, depth, 64), 0xCD, dtype=torch.uint8).pin_memory()
    got = run_gpu(db, req, peer, rkeys, world, n_qp, lb, lk, heap, depth, head, rings=rings)
    check(got, want)
