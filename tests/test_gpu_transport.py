"""db_wqe_bucket_transport on the GPU against the oracle, bit for bit.

Puts to RDMA PEs become WQEs in their rings; puts to P2P and SDMA PEs become
32-byte direct records in batch order (mori page: transport dispatch of the
put path). Every ring byte, every direct record and every counter is
compared with oracle_wqe_bucket_transport.
"""

import numpy as np
import pytest

from conftest import h, load_golden
from gpu_util import dev32, dev64, host32, host64, lib, need_gpu, torch
from test_gpu_wqe import random_puts

pytestmark = pytest.mark.gpu

FILL = 0xCD


@pytest.fixture(scope="module")
def db():
    need_gpu()
    return lib()


def run_gpu(db, req, peer_ptrs, rkeys, transport, world, n_qp, local_base, lkey, heap, depth,
            head, ws=None):
    n = req.shape[0]
    R = world * n_qp
    rings = torch.full((R, depth, 64), FILL, dtype=torch.uint8, device="cuda")
    direct = torch.full((max(n, 1), 32), FILL, dtype=torch.uint8, device="cuda")
    n_direct = torch.full((1,), -1, dtype=torch.int64, device="cuda")
    d_head = dev64(np.asarray(head, dtype=np.uint64))
    count = torch.full((R,), -1, dtype=torch.int32, device="cuda")
    ctr = torch.full((4,), -1, dtype=torch.int64, device="cuda")
    if ws is None:
        ws = db.workspace(db.wqe_workspace_size(n, R))
    d_req = dev64(req) if n else torch.zeros((0, 2), dtype=torch.int64, device="cuda")
    tr = torch.from_numpy(np.asarray(transport, dtype=np.uint8)).cuda()
    db.wqe_bucket_transport(d_req, dev64(np.asarray(peer_ptrs, dtype=np.uint64)),
                            dev32(np.asarray(rkeys, dtype=np.uint32)), tr, world, n_qp,
                            local_base, lkey, heap, rings, depth, d_head, count, direct,
                            n_direct, ws, ctr=ctr)
    torch.cuda.synchronize()
    return dict(rings=rings, head=host64(d_head), count=host32(count), ctr=host64(ctr),
                direct=direct.cpu().numpy(), n_direct=int(n_direct.item()))


def check(got, want):
    assert (got["head"] == want["head"]).all()
    assert (got["count"] == want["count"]).all()
    assert (got["ctr"] == want["ctr"]).all(), (got["ctr"], want["ctr"])
    assert got["n_direct"] == want["n_direct"]
    k = want["n_direct"]
    assert (got["direct"][:k] == want["direct"]).all()
    assert (got["direct"][k:] == FILL).all()  # nothing written past the last record
    assert (got["rings"].cpu().numpy() == want["rings"]).all()


def oracle_call(oracle, req, peer, rkeys, transport, world, n_qp, lb, lk, heap, depth, head):
    return oracle.wqe_bucket_transport(req, peer, rkeys, transport, world, n_qp, lb, lk, heap,
                                       depth, head, fill=FILL)


@pytest.mark.parametrize("variant", ["depth4", "depth1"])
def test_golden(db, oracle, variant):
    fx = load_golden("wqe_transport_hand_cases.json")
    v = fx[variant]
    from synth import pack_put_requests
    req = pack_put_requests([h(r["off"]) for r in fx["req"]], [r["bytes"] for r in fx["req"]],
                            [r["pe"] for r in fx["req"]], [r["qp"] for r in fx["req"]])
    args = (req, [h(x) for x in fx["peer_ptrs"]], fx["rkeys"], fx["transport"], fx["world"],
            fx["n_qp"], h(fx["local_base"]), fx["lkey"], fx["heap_size"], v["depth"], fx["head"])
    got = run_gpu(db, *args)
    assert got["head"].tolist() == v["head"]
    assert got["count"].tolist() == v["count"]
    assert got["ctr"].tolist() == v["ctr"]
    assert got["n_direct"] == len(fx["direct"])
    d = got["direct"]
    u64 = d.view(np.uint64).reshape(-1, 4)
    u32 = d.view(np.uint32).reshape(-1, 8)
    for k, e in enumerate(fx["direct"]):
        assert int(u64[k, 0]) == h(e["dst"]) and int(u64[k, 1]) == h(e["src"])
        assert int(u32[k, 4]) == e["len"] and int(u32[k, 5]) == e["req_index"]
        assert int(d[k, 24]) | int(d[k, 25]) << 8 == e["pe"] and int(d[k, 26]) == e["transport"]
        assert (d[k, 27:] == 0).all()
    check(got, oracle_call(oracle, *args))


@pytest.mark.parametrize("n", [1, 255, 256, 257, 5000, 70001])
@pytest.mark.parametrize("depth", [4096, 64])  # 64: some rings overflow
def test_mixed_transports_ragged(db, oracle, n, depth):
    """RDMA, P2P, SDMA and an unknown code over several tiles of 256 puts
    and a ragged tail."""
    rng = np.random.default_rng(9000 + n + depth)
    world, n_qp, heap = 8, 4, 1 << 32
    req = random_puts(rng, n, world, n_qp, heap)
    peer = (rng.integers(1 << 19, 1 << 26, size=world) << 21).astype(np.uint64)
    rkeys = rng.integers(0, 2**32, size=world, dtype=np.uint64).astype(np.uint32)
    head = rng.integers(0, 2**40, size=world * n_qp).astype(np.uint64)
    transport = np.array([0, 1, 0, 2, 0, 1, 7, 0], dtype=np.uint8)
    args = (req, peer, rkeys, transport, world, n_qp, 0x7F0000000000, 0xC0FFEE, heap, depth,
            head)
    check(run_gpu(db, *args), oracle_call(oracle, *args))


@pytest.mark.parametrize("code", [0, 1])
def test_single_transport(db, oracle, code):
    """All PEs RDMA (the result of db_wqe_bucket, no direct record) or all
    P2P (no ring touched, every valid put a direct record)."""
    rng = np.random.default_rng(77 + code)
    n, world, n_qp, depth, heap = 40000, 5, 3, 1 << 14, 1 << 32
    req = random_puts(rng, n, world, n_qp, heap)
    peer = (rng.integers(1 << 19, 1 << 26, size=world) << 21).astype(np.uint64)
    rkeys = rng.integers(0, 2**32, size=world, dtype=np.uint64).astype(np.uint32)
    head = rng.integers(0, 2**40, size=world * n_qp).astype(np.uint64)
    args = (req, peer, rkeys, np.full(world, code, np.uint8), world, n_qp, 0x7F0000000000, 9,
            heap, depth, head)
    want = oracle_call(oracle, *args)
    assert (want["n_direct"] == 0) == (code == 0)
    check(run_gpu(db, *args), want)


def test_full_size_two_p2p_peers(db, oracle):
    """8,388,608 puts over 8 PEs x 4 queues, PEs 1 and 2 on P2P: every ring
    byte and every direct record against the oracle."""
    import synth
    p = synth.put_bucket_transport()
    args = (p["req"], p["peer_ptrs"], p["rkeys"], p["transport"], p["world"], p["n_qp"],
            p["local_base"], p["lkey"], p["heap_size"], p["depth"], p["head"])
    want = oracle_call(oracle, *args)
    assert want["n_direct"] > 1_000_000
    check(run_gpu(db, *args), want)


def test_workspace_reuse_and_empty_batch(db, oracle):
    """One workspace for a batch, an empty batch (counters and n_direct
    zeroed) and a batch again."""
    rng = np.random.default_rng(5)
    world, n_qp, depth, heap = 4, 2, 1 << 12, 1 << 30
    peer = (rng.integers(1 << 19, 1 << 26, size=world) << 21).astype(np.uint64)
    rkeys = rng.integers(0, 2**32, size=world, dtype=np.uint64).astype(np.uint32)
    transport = np.array([1, 0, 2, 0], dtype=np.uint8)
    ws = db.workspace(db.wqe_workspace_size(3000, world * n_qp))
    for n in (3000, 0, 1234):
        req = random_puts(rng, n, world, n_qp, heap) if n else np.zeros((0, 2), np.uint64)
        head = rng.integers(0, 1000, size=world * n_qp).astype(np.uint64)
        args = (req, peer, rkeys, transport, world, n_qp, 0x10000, 3, heap, depth, head)
        got = run_gpu(db, *args, ws=ws)
        if n == 0:
            assert got["n_direct"] == 0 and got["ctr"].tolist() == [0, 0, 0, 0]
            assert got["count"].tolist() == [0] * (world * n_qp)
            continue
        check(got, oracle_call(oracle, *args))
