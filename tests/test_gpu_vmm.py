"""db_wqe_bucket_vmm on the GPU against the oracle, bit for bit."""

import numpy as np
import pytest

from conftest import h, load_golden
from gpu_util import dev32, dev64, host32, host64, lib, need_gpu, torch
from test_gpu_wqe import check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def db():
    need_gpu()
    return lib()


def run_vmm(db, req, chunk_raddr, chunk_rkey, chunk_lkey, chunk_shift, world, n_qp,
            local_base, heap, depth, head, fill=0xCD, mtu=0, psn_head=None):
    n = req.shape[0]
    R = world * n_qp
    rings = torch.full((R, depth, 64), fill, dtype=torch.uint8, device="cuda")
    d_head = dev64(np.asarray(head, dtype=np.uint64))
    count = torch.full((R,), -1, dtype=torch.int32, device="cuda")
    ctr = torch.full((4,), -1, dtype=torch.int64, device="cuda")
    ws = db.workspace(db.wqe_vmm_workspace_size(max(n, 1), world, n_qp, heap, chunk_shift))
    d_psn = dev64(np.asarray(psn_head, dtype=np.uint64)) if mtu else None
    d_req = dev64(req) if n else torch.zeros((0, 2), dtype=torch.int64, device="cuda")
    db.wqe_bucket_vmm(d_req, dev64(np.ascontiguousarray(chunk_raddr, dtype=np.uint64)),
                      dev32(np.ascontiguousarray(chunk_rkey, dtype=np.uint32)),
                      dev32(np.ascontiguousarray(chunk_lkey, dtype=np.uint32)), chunk_shift,
                      world, n_qp, local_base, heap, rings, depth, d_head, count, ws, ctr=ctr,
                      mtu=mtu, psn_head=d_psn)
    torch.cuda.synchronize()
    out = dict(rings=rings, head=host64(d_head), count=host32(count), ctr=host64(ctr))
    if mtu:
        out["psn_head"] = host64(d_psn)
    return out


def both(db, oracle, req, tables, chunk_shift, world, n_qp, local_base, heap, depth, head,
         mtu=0, psn_head=None):
    raddr, rkey, lkey = tables
    want = oracle.wqe_bucket_vmm(req, raddr, rkey, lkey, chunk_shift, world, n_qp, local_base,
                                 heap, depth, head, fill=0xCD, mtu=mtu, psn_head=psn_head)
    got = run_vmm(db, req, raddr, rkey, lkey, chunk_shift, world, n_qp, local_base, heap, depth,
                  head, mtu=mtu, psn_head=psn_head)
    check(got, want)
    if mtu:
        assert (got["psn_head"] == want["psn_head"]).all()
    return got, want


@pytest.mark.parametrize("variant", ["depth8", "depth2"])
def test_golden(db, oracle, variant):
    fx = load_golden("wqe_vmm_hand_cases.json")
    from test_oracle_wqe import pack
    raddr = np.array([[h(x) for x in row] for row in fx["chunk_raddr"]], dtype=np.uint64)
    got, _ = both(db, oracle, pack(fx["req"]), (raddr, np.array(fx["chunk_rkey"]),
                                                np.array(fx["chunk_lkey"])),
                  fx["chunk_shift"], fx["world"], fx["n_qp"], h(fx["local_base"]),
                  fx["heap_size"], fx[variant]["depth"], fx["head"])
    assert got["ctr"].tolist() == fx[variant]["ctr"]


def tables_for(rng, world, n_chunks, chunk_shift):
    C = 1 << chunk_shift
    raddr = rng.integers(1 << 10, 1 << 30, size=(world, n_chunks)).astype(np.uint64) * np.uint64(C)
    rkey = rng.integers(0, 2**32, size=(world, n_chunks), dtype=np.uint64).astype(np.uint32)
    lkey = rng.integers(0, 2**32, size=n_chunks, dtype=np.uint64).astype(np.uint32)
    return raddr, rkey, lkey


@pytest.mark.parametrize("n,world,n_qp,chunk_shift,depth,max_bytes", [
    (1, 2, 2, 12, 64, 20000), (255, 8, 4, 12, 256, 20000), (256, 8, 4, 12, 256, 20000),
    (257, 8, 4, 12, 256, 20000), (5000, 8, 4, 16, 1024, 200000), (5000, 8, 4, 12, 128, 20000),
    (20000, 1, 1, 12, 1 << 17, 100000), (20000, 3, 5, 21, 4096, 1 << 22),
    (100000, 64, 2, 14, 2048, 40000), (60000, 1024, 1, 13, 256, 30000),
    (3000, 2, 1, 12, 1 << 15, 1 << 20)])
def test_random_batches(db, oracle, n, world, n_qp, chunk_shift, depth, max_bytes):
    """Many chunk sizes, ring counts and depths (some rings overflow), one
    ring only, and puts spanning up to 257 chunks."""
    rng = np.random.default_rng(n + chunk_shift * 1000 + world)
    heap = 1 << 30
    while world * (heap >> chunk_shift) > (1 << 22):  # keep the chunk tables small
        heap >>= 1
    n_chunks = heap >> chunk_shift
    pe = rng.integers(0, world, size=n)
    qp = rng.integers(0, n_qp, size=n)
    off = 16 * rng.integers(0, heap // 16, size=n)
    nbytes = np.minimum(16 * rng.integers(1, max_bytes // 16 + 1, size=n), heap - off)
    bad = rng.random(n) < 0.03
    nbytes = np.where(bad, 0, nbytes)
    from synth import pack_put_requests
    req = pack_put_requests(off, nbytes, pe, qp)
    head = rng.integers(0, 2**40, size=world * n_qp).astype(np.uint64)
    both(db, oracle, req, tables_for(rng, world, n_chunks, chunk_shift), chunk_shift, world,
         n_qp, 0x7C0000000000, heap, depth, head)


@pytest.mark.parametrize("variant", ["depth8", "depth2"])
def test_golden_psn(db, oracle, variant):
    fx = load_golden("wqe_vmm_hand_cases.json")
    from test_oracle_wqe import pack
    ps = fx["psn"]
    raddr = np.array([[h(x) for x in row] for row in fx["chunk_raddr"]], dtype=np.uint64)
    got, _ = both(db, oracle, pack(fx["req"]), (raddr, np.array(fx["chunk_rkey"]),
                                                np.array(fx["chunk_lkey"])),
                  fx["chunk_shift"], fx["world"], fx["n_qp"], h(fx["local_base"]),
                  fx["heap_size"], fx[variant]["depth"], fx["head"], mtu=ps["mtu"],
                  psn_head=np.array(ps["psn_head"], dtype=np.uint64))
    assert got["psn_head"].tolist() == ps[f"{variant}_psn_head"]


@pytest.mark.parametrize("n,world,n_qp,chunk_shift,depth,max_bytes,mtu", [
    (257, 8, 4, 12, 256, 20000, 1024), (5000, 8, 4, 16, 1024, 200000, 4096),
    (5000, 8, 4, 12, 128, 20000, 512), (20000, 1, 1, 12, 1 << 17, 100000, 2048),
    (60000, 1024, 1, 13, 256, 30000, 1024), (3000, 2, 1, 12, 1 << 15, 1 << 20, 512),
    (100000, 8, 4, 21, 1 << 14, 65536, 4096)])
def test_random_batches_with_psns(db, oracle, n, world, n_qp, chunk_shift, depth, max_bytes,
                                  mtu):
    rng = np.random.default_rng(n + chunk_shift * 1000 + world + mtu)
    heap = 1 << 30
    while world * (heap >> chunk_shift) > (1 << 22):
        heap >>= 1
    pe = rng.integers(0, world, size=n)
    qp = rng.integers(0, n_qp, size=n)
    off = 16 * rng.integers(0, heap // 16, size=n)
    nbytes = np.minimum(16 * rng.integers(1, max_bytes // 16 + 1, size=n), heap - off)
    nbytes = np.where(rng.random(n) < 0.03, 0, nbytes)
    from synth import pack_put_requests
    req = pack_put_requests(off, nbytes, pe, qp)
    head = rng.integers(0, 2**40, size=world * n_qp).astype(np.uint64)
    psn0 = rng.integers(0, 2**40, size=world * n_qp).astype(np.uint64)
    both(db, oracle, req, tables_for(rng, world, heap >> chunk_shift, chunk_shift), chunk_shift,
         world, n_qp, 0x7C0000000000, heap, depth, head, mtu=mtu, psn_head=psn0)


@pytest.mark.parametrize("mtu", [777, 1500, 4000, 9000, (1 << 20) - 1])
def test_psns_with_mtus_that_are_not_powers_of_two(db, oracle, mtu):
    """PSN counts divide lengths by the MTU; besides random puts, a few puts
    of nearly 4 GiB (the longest a put can be) on a heap of 2 MiB chunks."""
    rng = np.random.default_rng(mtu)
    world, n_qp, chunk_shift, depth = 2, 2, 21, 1 << 14
    heap = 1 << 34
    n = 3000
    pe = rng.integers(0, world, size=n)
    qp = rng.integers(0, n_qp, size=n)
    off = 16 * rng.integers(0, (heap >> 1) // 16, size=n)
    nbytes = 16 * rng.integers(1, (8 << 20) // 16, size=n)
    big = rng.choice(n, size=3, replace=False)
    nbytes[big] = (1 << 32) - 16 * rng.integers(1, 1 << 12, size=3)
    from synth import pack_put_requests
    req = pack_put_requests(off, nbytes, pe, qp)
    head = rng.integers(0, 2**40, size=world * n_qp).astype(np.uint64)
    psn0 = rng.integers(0, 2**40, size=world * n_qp).astype(np.uint64)
    _, want = both(db, oracle, req, tables_for(rng, world, heap >> chunk_shift, chunk_shift),
                   chunk_shift, world, n_qp, 0x7C0000000000, heap, depth, head, mtu=mtu,
                   psn_head=psn0)
    assert want["ctr"][0] > n + 3 * 2047  # the long puts took their WQEs


def test_one_chunk_matches_static_heap(db, oracle):
    import synth
    from test_gpu_wqe import run_gpu
    p = synth.put_bucket(n=200_000, depth=1 << 14)
    world = p["world"]
    got_s = run_gpu(db, p["req"], p["peer_ptrs"], p["rkeys"], world, p["n_qp"],
                    p["local_base"], p["lkey"], p["heap_size"], p["depth"], p["head"])
    got_v = run_vmm(db, p["req"], p["peer_ptrs"].reshape(world, 1),
                    p["rkeys"].reshape(world, 1), np.array([p["lkey"]], dtype=np.uint32), 32,
                    world, p["n_qp"], p["local_base"], p["heap_size"], p["depth"], p["head"])
    for k in ("head", "count", "ctr"):
        assert (got_s[k] == got_v[k]).all(), k
    assert torch.equal(got_s["rings"], got_v["rings"])


def test_bad_arguments(db):
    t = torch.zeros((4, 2), dtype=torch.int64, device="cuda")
    tab = torch.zeros(64, dtype=torch.int64, device="cuda")
    t32 = torch.zeros(64, dtype=torch.int32, device="cuda")
    rings = torch.zeros((2, 8, 64), dtype=torch.uint8, device="cuda")
    head = torch.zeros(2, dtype=torch.int64, device="cuda")
    cnt = torch.zeros(2, dtype=torch.int32, device="cuda")
    ws = db.workspace(db.wqe_workspace_size(4, 2))
    for shift, depth in ((3, 8), (49, 8), (12, 6), (12, 1 << 32)):
        with pytest.raises(db.DescBuildError, match="invalid"):
            db.wqe_bucket_vmm(t, tab, t32, t32, shift, 2, 1, 0, 1 << 16, rings, depth, head, cnt, ws)
    for shift, mtu, psn in ((12, 256, head), (11, 1024, head), (12, 1024, None)):
        with pytest.raises(db.DescBuildError, match="invalid"):
            db.wqe_bucket_vmm(t, tab, t32, t32, shift, 2, 1, 0, 1 << 16, rings, 8, head, cnt, ws,
                              mtu=mtu, psn_head=psn)
    # a workspace without room for the packed chunk tables
    with pytest.raises(db.DescBuildError) as e:
        db.wqe_bucket_vmm(t, tab, t32, t32, 12, 2, 1, 0, 1 << 16, rings, 8, head, cnt, ws)
    assert e.value.code == -28
    assert db.wqe_vmm_workspace_size(4, 2, 1, 1 << 16, 12) >= db.wqe_workspace_size(4, 2) + 2 * 16 * 16


def test_full_size_workload(db, oracle):
    """The 8,388,608-put batch on a heap of 2 MiB chunks, every byte against
    the oracle."""
    import synth
    p = synth.put_bucket_vmm()
    both(db, oracle, p["req"], (p["chunk_raddr"], p["chunk_rkey"], p["chunk_lkey"]),
         p["chunk_shift"], p["world"], p["n_qp"], p["local_base"], p["heap_size"], p["depth"],
         p["head"])
