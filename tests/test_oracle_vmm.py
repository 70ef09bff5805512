"""Pins for the VMM-heap put translation in the oracle.

Follows "mori communication library analysis (1)", the VMM-heap branch of the
put path: a put becomes one WQE per chunk it touches, each carrying
min(source chunk remainder, destination chunk remainder, remaining) bytes with
that chunk's keys.
"""

import numpy as np
import pytest

from conftest import h, load_golden
from test_oracle_wqe import make_batch, pack, wqe_fields


@pytest.mark.parametrize("variant", ["depth8", "depth2"])
def test_hand_cases(oracle, variant):
    fx = load_golden("wqe_vmm_hand_cases.json")
    v = fx[variant]
    FILL = 0xCD
    raddr = np.array([[h(x) for x in row] for row in fx["chunk_raddr"]], dtype=np.uint64)
    out = oracle.wqe_bucket_vmm(pack(fx["req"]), raddr, np.array(fx["chunk_rkey"]),
                                np.array(fx["chunk_lkey"]), fx["chunk_shift"], fx["world"],
                                fx["n_qp"], h(fx["local_base"]), fx["heap_size"], v["depth"],
                                fx["head"], fill=FILL)
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


def chunk_tables(rng, world, n_chunks):
    raddr = (rng.integers(1 << 10, 1 << 30, size=(world, n_chunks)) << 16).astype(np.uint64)
    rkey = rng.integers(0, 2**32, size=(world, n_chunks), dtype=np.uint64).astype(np.uint32)
    lkey = rng.integers(0, 2**32, size=n_chunks, dtype=np.uint64).astype(np.uint32)
    return raddr, rkey, lkey


def test_one_chunk_is_the_static_heap(oracle):
    """A chunk as large as the heap reduces to the static-heap translation."""
    rng = np.random.default_rng(2)
    world, n_qp, heap = 5, 3, 1 << 24
    req, _ = make_batch(rng, 3000, world, n_qp, heap)
    peer = (rng.integers(1 << 19, 1 << 26, size=world) << 21).astype(np.uint64)
    rk = rng.integers(0, 2**32, size=world, dtype=np.uint64).astype(np.uint32)
    head = rng.integers(0, 1 << 30, size=world * n_qp).astype(np.uint64)
    a = oracle.wqe_bucket(req, peer, rk, world, n_qp, 0x7E0000000000, 0xBEEF, heap, 512, head)
    v = oracle.wqe_bucket_vmm(req, peer.reshape(world, 1), rk.reshape(world, 1),
                              np.array([0xBEEF], dtype=np.uint32), 24, world, n_qp,
                              0x7E0000000000, heap, 512, head)
    for k in ("rings", "head", "count", "ctr"):
        assert (a[k] == v[k]).all(), k


@pytest.mark.parametrize("chunk_shift,depth", [(12, 4096), (16, 1024), (13, 8)])
def test_fragments_cover_each_put_chunk_by_chunk(oracle, chunk_shift, depth):
    """Every valid put's WQEs are consecutive in its ring, in address order,
    cover [off, off + bytes) exactly, stay inside one chunk each and carry
    that chunk's keys; post indices run on from the old head."""
    rng = np.random.default_rng(chunk_shift)
    world, n_qp, heap = 3, 2, 1 << 20
    C = 1 << chunk_shift
    n_chunks = heap // C
    n = 700
    pe = rng.integers(0, world, size=n)
    qp = rng.integers(0, n_qp, size=n)
    off = 16 * rng.integers(0, heap // 16, size=n)
    nbytes = np.minimum(rng.integers(1, 6 * C, size=n), heap - off)
    nbytes[::50] = 0  # some invalid puts
    from synth import pack_put_requests
    req = pack_put_requests(off, nbytes, pe, qp)
    raddr, rkey, lkey = chunk_tables(rng, world, n_chunks)
    head = rng.integers(0, 1 << 20, size=world * n_qp).astype(np.uint64)
    out = oracle.wqe_bucket_vmm(req, raddr, rkey, lkey, chunk_shift, world, n_qp,
                                0x7D0000000000, heap, depth, head, fill=0xCD)
    f = wqe_fields(out["rings"])
    posted = 0
    for r in range(world * n_qp):
        valid = [i for i in range(n) if pe[i] * n_qp + qp[i] == r and nbytes[i] > 0]
        frags = [(((int(o) + int(b) - 1) // C) - (int(o) // C) + 1) for o, b in
                 ((off[i], nbytes[i]) for i in valid)]
        total = sum(frags)
        assert int(out["count"][r]) == total
        if total > depth:
            assert int(out["head"][r]) == int(head[r])
            continue
        seq = int(head[r])
        for i, k in zip(valid, frags):
            cur = int(off[i])
            for _ in range(k):
                s = seq % depth
                end = min((cur // C + 1) * C, int(off[i]) + int(nbytes[i]))
                c = cur // C
                assert int(f["seq"][r, s]) == seq and int(f["req_index"][r, s]) == i
                assert int(f["len"][r, s]) == end - cur
                assert int(f["laddr"][r, s]) == 0x7D0000000000 + cur
                assert int(f["raddr"][r, s]) == int(raddr[pe[i], c]) + cur % C
                assert int(f["rkey"][r, s]) == int(rkey[pe[i], c])
                assert int(f["lkey"][r, s]) == int(lkey[c])
                cur = end
                seq += 1
            assert cur == int(off[i]) + int(nbytes[i])
        assert int(out["head"][r]) == seq
        posted += total
    assert int(out["ctr"][0]) == posted
    assert int(out["ctr"][1]) == int((nbytes == 0).sum())


@pytest.mark.parametrize("variant", ["depth8", "depth2"])
def test_hand_cases_with_psns(oracle, variant):
    fx = load_golden("wqe_vmm_hand_cases.json")
    ps = fx["psn"]
    raddr = np.array([[h(x) for x in row] for row in fx["chunk_raddr"]], dtype=np.uint64)
    out = oracle.wqe_bucket_vmm(pack(fx["req"]), raddr, np.array(fx["chunk_rkey"]),
                                np.array(fx["chunk_lkey"]), fx["chunk_shift"], fx["world"],
                                fx["n_qp"], h(fx["local_base"]), fx["heap_size"],
                                fx[variant]["depth"], fx["head"], fill=0xCD, mtu=ps["mtu"],
                                psn_head=np.array(ps["psn_head"], dtype=np.uint64))
    assert out["psn_head"].tolist() == ps[f"{variant}_psn_head"]
    assert out["head"].tolist() == fx[variant]["head"]
    if variant == "depth8":
        w = out["rings"].reshape(out["rings"].shape[0], out["rings"].shape[1], 64)
        psn = w.view(np.uint32).reshape(w.shape[0], w.shape[1], 16)[..., 11]
        for e in ps["depth8_psn"]:
            assert int(psn[e["ring"], e["slot"]]) == e["psn"], e


def test_psn_chain_per_ring(oracle):
    """Each WQE's first PSN is the previous WQE's plus ceil(len / mtu) of the
    previous, from the old PSN head to the new one; without an mtu byte 44
    stays zero."""
    rng = np.random.default_rng(44)
    world, n_qp, heap, cs, depth, mtu = 3, 2, 1 << 22, 12, 1 << 14, 1024
    n = 2000
    pe, qp = rng.integers(0, world, size=n), rng.integers(0, n_qp, size=n)
    off = 16 * rng.integers(0, heap // 16, size=n)
    nbytes = np.minimum(16 * rng.integers(1, 2000, size=n), heap - off)
    from synth import pack_put_requests
    req = pack_put_requests(off, nbytes, pe, qp)
    raddr, rkey, lkey = chunk_tables(rng, world, heap >> cs)
    head = rng.integers(0, 1 << 20, size=world * n_qp).astype(np.uint64)
    psn0 = rng.integers(0, 1 << 33, size=world * n_qp).astype(np.uint64)
    out = oracle.wqe_bucket_vmm(req, raddr, rkey, lkey, cs, world, n_qp, 0, heap, depth, head,
                                mtu=mtu, psn_head=psn0)
    f = wqe_fields(out["rings"])
    psn = out["rings"].view(np.uint32).reshape(world * n_qp, depth, 16)[..., 11]
    for r in range(world * n_qp):
        cnt = int(out["count"][r])
        want = int(psn0[r])
        for k in range(cnt):
            s = (int(head[r]) + k) % depth
            assert int(psn[r, s]) == want % (1 << 32)
            want += -(-int(f["len"][r, s]) // mtu)
        assert int(out["psn_head"][r]) == want
    plain = oracle.wqe_bucket_vmm(req, raddr, rkey, lkey, cs, world, n_qp, 0, heap, depth, head)
    assert (plain["rings"].view(np.uint32).reshape(world * n_qp, depth, 16)[..., 11] == 0).all()
    assert (plain["rings"] == np.where(np.arange(64) // 4 == 11, 0, out["rings"])).all()
