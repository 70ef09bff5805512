"""Pins for the per-PE transport oracle (oracle_wqe_bucket_transport).

Follows "mori communication library analysis (1)": the put path branches on
its target PE's transport type (RDMA, P2P or SDMA), fixed per PE at set-up;
for a PE not reached over RDMA the peer pointer is the address at which this
process maps that PE's heap, so the destination is peer_ptrs[pe] + offset
whatever the transport. RDMA puts become WQEs exactly as in the static-heap
path; P2P and SDMA puts become direct copy descriptors in request order.
"""

import numpy as np
import pytest

from conftest import h, load_golden
from test_oracle_wqe import make_batch, wqe_fields


def direct_fields(d):
    d = np.ascontiguousarray(d).reshape(-1, 32)
    u64 = d.view(np.uint64).reshape(-1, 4)
    u32 = d.view(np.uint32).reshape(-1, 8)
    u16 = d.view(np.uint16).reshape(-1, 16)
    return dict(dst=u64[:, 0], src=u64[:, 1], len=u32[:, 4], req_index=u32[:, 5],
                pe=u16[:, 12], transport=d[:, 26], tail=d[:, 27:])


def pack(reqs):
    from synth import pack_put_requests
    return pack_put_requests([h(r["off"]) for r in reqs], [r["bytes"] for r in reqs],
                             [r["pe"] for r in reqs], [r["qp"] for r in reqs])


@pytest.mark.parametrize("variant", ["depth4", "depth1"])
def test_hand_cases(oracle, variant):
    fx = load_golden("wqe_transport_hand_cases.json")
    v = fx[variant]
    FILL = 0xCD
    out = oracle.wqe_bucket_transport(pack(fx["req"]), [h(x) for x in fx["peer_ptrs"]],
                                      fx["rkeys"], fx["transport"], fx["world"], fx["n_qp"],
                                      h(fx["local_base"]), fx["lkey"], fx["heap_size"],
                                      v["depth"], fx["head"], fill=FILL)
    assert out["head"].tolist() == v["head"]
    assert out["count"].tolist() == v["count"]
    assert out["ctr"].tolist() == v["ctr"]
    f = wqe_fields(out["rings"])
    written = np.zeros(out["rings"].shape[:2], dtype=bool)
    for e in v["wqes"]:
        r, s = e["ring"], e["slot"]
        written[r, s] = True
        for key in ("raddr", "laddr", "len", "lkey", "rkey", "seq", "req_index"):
            assert int(f[key][r, s]) == h(e[key]), (key, r, s)
        assert f["flags"][r, s] == 0 and (f["tail"][r, s] == 0).all()
    assert (out["rings"][~written] == FILL).all()
    assert out["n_direct"] == len(fx["direct"])
    d = direct_fields(out["direct"])
    for k, e in enumerate(fx["direct"]):
        for key in ("dst", "src", "len", "req_index", "pe", "transport"):
            assert int(d[key][k]) == h(e[key]), (key, k)
        assert (d["tail"][k] == 0).all()


def random_case(rng, world, n_qp, n=1200, heap=1 << 30):
    req, cols = make_batch(rng, n, world, n_qp, heap)
    peer = (rng.integers(1 << 19, 1 << 26, size=world) << 21).astype(np.uint64)
    rkeys = rng.integers(0, 2**32, size=world, dtype=np.uint64).astype(np.uint32)
    head = rng.integers(0, 10**6, size=world * n_qp).astype(np.uint64)
    return req, cols, peer, rkeys, head, heap


@pytest.mark.parametrize("world,n_qp,depth", [(8, 4, 64), (3, 5, 16), (1, 1, 1024)])
def test_all_rdma_is_the_static_heap_bucketing(oracle, world, n_qp, depth):
    """Every PE on RDMA: the same rings, heads, counts and counters as the
    static-heap bucketing, and no direct descriptor."""
    rng = np.random.default_rng(31 + world)
    req, _, peer, rkeys, head, heap = random_case(rng, world, n_qp)
    lb, lk = 0x7F0000000000, 0xABCD
    a = oracle.wqe_bucket(req, peer, rkeys, world, n_qp, lb, lk, heap, depth, head, fill=7)
    b = oracle.wqe_bucket_transport(req, peer, rkeys, np.zeros(world, np.uint8), world, n_qp,
                                    lb, lk, heap, depth, head, fill=7)
    for key in ("rings", "head", "count", "ctr"):
        assert (a[key] == b[key]).all(), key
    assert b["n_direct"] == 0


@pytest.mark.parametrize("code", [1, 2])
def test_all_direct_makes_no_wqe(oracle, code):
    """Every PE on P2P (or SDMA): no ring is touched, heads stay, and the
    direct list is the valid puts in request order, each translated from its
    own request."""
    world, n_qp, depth = 6, 3, 32
    rng = np.random.default_rng(40 + code)
    req, (pe, qp, nbytes, off), peer, rkeys, head, heap = random_case(rng, world, n_qp)
    lb = 0x7F0000000000
    out = oracle.wqe_bucket_transport(req, peer, rkeys, np.full(world, code, np.uint8), world,
                                      n_qp, lb, 5, heap, depth, head, fill=7)
    assert (out["rings"] == 7).all()
    assert out["head"].tolist() == head.tolist()
    assert out["count"].tolist() == [0] * (world * n_qp)
    valid = (pe < world) & (qp < n_qp) & (nbytes >= 1) & (off + nbytes <= heap)
    ids = np.flatnonzero(valid)
    assert out["ctr"].tolist() == [0, int((~valid).sum()), 0, 0]
    assert out["n_direct"] == ids.size
    d = direct_fields(out["direct"])
    assert (d["req_index"] == ids).all()
    assert (d["dst"] == peer[pe[ids]] + off[ids].astype(np.uint64)).all()
    assert (d["src"] == np.uint64(lb) + off[ids].astype(np.uint64)).all()
    assert (d["len"] == nbytes[ids]).all()
    assert (d["pe"] == pe[ids]).all()
    assert (d["transport"] == code).all()
    assert (d["tail"] == 0).all()


@pytest.mark.parametrize("depth", [8, 40, 4096])
def test_mixed_transports_partition_the_batch(oracle, depth):
    """A mix of RDMA, P2P and SDMA PEs and one with an unknown code: each
    valid put is a WQE (or refused by an overflowing ring) or a direct
    descriptor, never both; the RDMA puts alone give the static-heap
    result; the direct list is the stable selection of the others."""
    world, n_qp = 8, 4
    rng = np.random.default_rng(50 + depth)
    req, (pe, qp, nbytes, off), peer, rkeys, head, heap = random_case(rng, world, n_qp, n=3000)
    transport = np.array([0, 1, 0, 2, 0, 1, 0, 9], dtype=np.uint8)
    lb, lk = 0x7F0000000000, 0x77
    out = oracle.wqe_bucket_transport(req, peer, rkeys, transport, world, n_qp, lb, lk, heap,
                                      depth, head, fill=7)
    known = np.zeros(pe.shape, dtype=bool)
    known[pe < world] = transport[pe[pe < world]] <= 2
    valid = (pe < world) & (qp < n_qp) & (nbytes >= 1) & (off + nbytes <= heap) & known
    tr = np.where(pe < world, transport[np.minimum(pe, world - 1)], 255)
    rdma = valid & (tr == 0)
    direct = valid & (tr != 0)
    # The RDMA puts on their own (other puts made invalid) give the rings,
    # heads and counts; their request indices are kept by giving the others
    # zero bytes.
    rdma_only = req.copy()
    rdma_only[~rdma, 1] &= ~np.uint64(0xFFFFFFFF)
    ref = oracle.wqe_bucket(rdma_only, peer, rkeys, world, n_qp, lb, lk, heap, depth, head,
                            fill=7)
    for key in ("rings", "head", "count"):
        assert (out[key] == ref[key]).all(), key
    assert out["ctr"][0] == ref["ctr"][0] and out["ctr"][2] == ref["ctr"][2]
    assert out["ctr"][3] == ref["ctr"][3]
    assert out["ctr"][1] == (~valid).sum()
    assert out["ctr"][0] + out["ctr"][2] + out["n_direct"] == valid.sum()
    d = direct_fields(out["direct"])
    ids = np.flatnonzero(direct)
    assert (d["req_index"] == ids).all()
    assert (d["transport"] == tr[ids]).all()
    assert (d["dst"] == peer[pe[ids]] + off[ids].astype(np.uint64)).all()


def test_empty_batch(oracle):
    out = oracle.wqe_bucket_transport(np.zeros((0, 2), dtype=np.uint64), [0, 0], [0, 0], [0, 1],
                                      2, 1, 0, 0, 64, 4, [5, 6])
    assert out["count"].tolist() == [0, 0]
    assert out["head"].tolist() == [5, 6]
    assert out["ctr"].tolist() == [0, 0, 0, 0]
    assert out["n_direct"] == 0
