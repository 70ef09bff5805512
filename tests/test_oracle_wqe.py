"""Pins for the put-translation / WQE-bucketing oracle.

Follows "mori communication library analysis (1)": static-heap translation
(raddr = peerPtrs[pe] + offset, rkey = peerRkeys[pe], lkey of the source
object) and the per-queue post index a WQE takes.
"""

import numpy as np
import pytest

from conftest import h, load_golden


def wqe_fields(rings):
    """Decode [R, D, 64] u8 rings into named field arrays."""
    w = rings.reshape(rings.shape[0], rings.shape[1], 64)
    u64 = w.view(np.uint64).reshape(w.shape[0], w.shape[1], 8)
    u32 = w.view(np.uint32).reshape(w.shape[0], w.shape[1], 16)
    return dict(raddr=u64[..., 0], laddr=u64[..., 1], len=u32[..., 4], lkey=u32[..., 5],
                rkey=u32[..., 6], flags=u32[..., 7], seq=u64[..., 4], req_index=u32[..., 10],
                tail=w[..., 44:])


def pack(reqs):
    from synth import pack_put_requests
    return pack_put_requests([h(r["off"]) for r in reqs], [r["bytes"] for r in reqs],
                             [r["pe"] for r in reqs], [r["qp"] for r in reqs])


@pytest.mark.parametrize("variant", ["depth4", "depth1"])
def test_hand_cases(oracle, variant):
    fx = load_golden("wqe_hand_cases.json")
    v = fx[variant]
    FILL = 0xCD
    out = oracle.wqe_bucket(pack(fx["req"]), [h(x) for x in fx["peer_ptrs"]], fx["rkeys"],
                            fx["world"], fx["n_qp"], h(fx["local_base"]), fx["lkey"],
                            fx["heap_size"], v["depth"], fx["head"], fill=FILL)
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


def make_batch(rng, n, world, n_qp, heap, invalid_frac=0.05):
    pe = rng.integers(0, world, size=n)
    qp = rng.integers(0, n_qp, size=n)
    nbytes = 16 * rng.integers(1, 64, size=n)
    off = 16 * rng.integers(0, (heap - 1024) // 16, size=n)
    bad = rng.random(n) < invalid_frac
    kind = rng.integers(0, 4, size=n)
    pe = np.where(bad & (kind == 0), world + rng.integers(0, 3, size=n), pe)
    qp = np.where(bad & (kind == 1), n_qp, qp)
    nbytes = np.where(bad & (kind == 2), 0, nbytes)
    off = np.where(bad & (kind == 3), heap - 8, off)
    from synth import pack_put_requests
    return pack_put_requests(off, nbytes, pe, qp), (pe, qp, nbytes, off)


@pytest.mark.parametrize("world,n_qp,depth", [(8, 4, 64), (3, 5, 16), (1, 1, 1024), (2, 3, 8)])
def test_stable_partition_properties(oracle, world, n_qp, depth):
    rng = np.random.default_rng(world * 100 + n_qp)
    heap = 1 << 30
    n = 900
    req, (pe, qp, nbytes, off) = make_batch(rng, n, world, n_qp, heap)
    peer = (rng.integers(1 << 19, 1 << 26, size=world) << 21).astype(np.uint64)
    rkeys = rng.integers(0, 2**32, size=world, dtype=np.uint64).astype(np.uint32)
    head = rng.integers(0, 10**6, size=world * n_qp).astype(np.uint64)
    lb, lk = 0x7F0000000000, 0xABCD
    out = oracle.wqe_bucket(req, peer, rkeys, world, n_qp, lb, lk, heap, depth, head)
    valid = (pe < world) & (qp < n_qp) & (nbytes >= 1) & (off + nbytes <= heap)
    ring = np.where(valid, pe * n_qp + qp, -1)
    demand = np.bincount(ring[valid], minlength=world * n_qp)
    assert out["count"].tolist() == demand.tolist()
    full = demand > depth
    assert out["ctr"][1] == (~valid).sum()
    assert out["ctr"][2] == demand[full].sum()
    assert out["ctr"][3] == (2 if full.any() else 0)
    assert out["head"].tolist() == (head + np.where(full, 0, demand)).tolist()
    f = wqe_fields(out["rings"])
    # Library routine: a stable sort of valid requests by ring gives, ring by
    # ring, the order in which they must appear from the old head onwards.
    order = np.argsort(np.where(valid, ring, 1 << 30), kind="stable")[: valid.sum()]
    posted = 0
    for r in range(world * n_qp):
        if full[r]:
            continue
        ids = order[ring[order] == r]
        seqs = head[r] + np.arange(ids.shape[0], dtype=np.uint64)
        slots = (seqs % np.uint64(depth)).astype(np.int64)
        assert (f["req_index"][r, slots] == ids).all()
        assert (f["seq"][r, slots] == seqs).all()
        # the translation of each entry, recomputed from its request
        p = pe[ids]
        assert (f["raddr"][r, slots] == peer[p] + off[ids].astype(np.uint64)).all()
        assert (f["laddr"][r, slots] == np.uint64(lb) + off[ids].astype(np.uint64)).all()
        assert (f["rkey"][r, slots] == rkeys[p]).all()
        assert (f["lkey"][r, slots] == lk).all()
        assert (f["len"][r, slots] == nbytes[ids]).all()
        posted += ids.shape[0]
    assert out["ctr"][0] == posted


def test_single_queue_is_order_preserving(oracle):
    rng = np.random.default_rng(2)
    req, (pe, qp, nbytes, off) = make_batch(rng, 300, 1, 1, 1 << 24, invalid_frac=0.0)
    out = oracle.wqe_bucket(req, [1 << 40], [9], 1, 1, 0, 1, 1 << 24, 512, [0])
    f = wqe_fields(out["rings"])
    assert f["req_index"][0, :300].tolist() == list(range(300))
    assert f["seq"][0, :300].tolist() == list(range(300))


def test_ring_wraps_at_depth(oracle):
    # head close to a multiple of depth: the run wraps to slot 0
    req, _ = make_batch(np.random.default_rng(4), 6, 1, 1, 1 << 20, invalid_frac=0.0)
    out = oracle.wqe_bucket(req, [0x1000000], [1], 1, 1, 0, 0, 1 << 20, 8, [13])
    f = wqe_fields(out["rings"])
    # seq 13..18 -> slots 5, 6, 7, 0, 1, 2
    assert [int(f["seq"][0, s]) for s in (5, 6, 7, 0, 1, 2)] == [13, 14, 15, 16, 17, 18]
    assert out["head"].tolist() == [19]


def test_empty_batch(oracle):
    out = oracle.wqe_bucket(np.zeros((0, 2), dtype=np.uint64), [0], [0], 1, 2, 0, 0, 64, 4,
                            [5, 6])
    assert out["count"].tolist() == [0, 0]
    assert out["head"].tolist() == [5, 6]
    assert out["ctr"].tolist() == [0, 0, 0, 0]
