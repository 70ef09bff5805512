"""db_cq_mirror on the GPU: completions a controller writes into device
memory reach the host CQ whole and in order, bit for bit as the oracle's
mirror pass copies them (xNVMe "uPCIe CUDA" backend page, "Completions in
device memory").

The host stands in for the controller. It writes each batch of entries
into the device CQ twice, in stream order: first with the previous pass's
phase tag, then with the new one. An entry whose new tag the kernel sees
is therefore complete. Every wait here is bounded: the host polls with a
time limit, and each launch ends by itself after its own limit even if a
test fails before it raises `stop`.
"""

import ctypes
import time

import numpy as np
import pytest

from gpu_util import lib, need_gpu, torch

pytestmark = pytest.mark.gpu

PHASE_BIT = 1 << 16
ERR_TIMEOUT = 1


@pytest.fixture(scope="module")
def db():
    need_gpu()
    return lib()


class Controller:
    """A device-memory CQ written from the host, one batch at a time."""

    def __init__(self, depth, seed, stream):
        self.depth = depth
        self.rng = np.random.default_rng(seed)
        self.dev = torch.zeros((depth, 4), dtype=torch.int32, device="cuda")
        self.host = torch.zeros((depth, 4), dtype=torch.int32).pin_memory()
        self.stage_old = torch.zeros((depth, 4), dtype=torch.int32).pin_memory()
        self.stage_new = torch.zeros((depth, 4), dtype=torch.int32).pin_memory()
        self.replica = np.zeros((depth, 4), dtype=np.uint32)   # what the device CQ holds
        self.stream = stream
        self.produced = 0
        self.reaped = []            # entries the host has seen, in order
        self.head, self.phase = 0, 1

    def produce(self, k):
        """Write the next k completions (k < depth), then wait for the copies."""
        d = self.depth
        rows = []
        for j in range(k):
            i = self.produced + j
            body = self.rng.integers(0, 2**32, size=4, dtype=np.uint64).astype(np.uint32)
            tag = 1 - (i // d) % 2
            new = body.copy()
            new[3] = (int(body[3]) & ~PHASE_BIT) | (tag << 16)
            old = new.copy()
            old[3] ^= PHASE_BIT
            self.stage_old.numpy().view(np.uint32)[i % d] = old
            self.stage_new.numpy().view(np.uint32)[i % d] = new
            self.replica[i % d] = new
            rows.append(i % d)
        # contiguous segments (a batch may wrap once)
        segs = []
        start = self.produced % d
        first = min(k, d - start)
        if first:
            segs.append((start, start + first))
        if k > first:
            segs.append((0, k - first))
        with torch.cuda.stream(self.stream):
            for stage in (self.stage_old, self.stage_new):
                for a, b in segs:
                    self.dev[a:b].copy_(stage[a:b], non_blocking=True)
        self.stream.synchronize()
        self.produced += k
        return rows

    def reap_until(self, db, total, timeout=5.0):
        """Poll the host CQ until `total` completions have been seen."""
        t0 = time.monotonic()
        while len(self.reaped) < total and time.monotonic() - t0 < timeout:
            got, self.head, self.phase = db.cq_host_reap(self.host, self.head, self.phase)
            self.reaped.extend(got)
            if got.shape[0] == 0:
                time.sleep(20e-6)
        return len(self.reaped)


class Mirror:
    def __init__(self, db, n_slots, limit_s):
        self.db = db
        self.slots = db.cq_slots(n_slots)
        self.stop = torch.zeros(1, dtype=torch.int32).pin_memory()
        self.ctr = torch.zeros(4, dtype=torch.int64, device="cuda")
        self.stream = torch.cuda.Stream()
        self.limit_s = limit_s

    def launch(self):
        self.stop.zero_()
        self.db.cq_mirror(self.slots, self.stop, self.limit_s, ctr=self.ctr, stream=self.stream)

    def finish(self):
        self.db.cq_request_stop(self.stop)
        self.stream.synchronize()
        return self.ctr.cpu().numpy()

    @property
    def fields(self):
        return self.db.cq_slot_fields(self.slots)


@pytest.mark.parametrize("depth", [2, 7, 64, 1024])
def test_one_queue_against_the_oracle(db, oracle, depth):
    """Random batches (wrapping many times): the host sees every completion
    once, in order, and the host CQ equals the oracle's mirror of the
    device CQ after every batch."""
    m = Mirror(db, 1, limit_s=20.0)
    c = Controller(depth, depth, torch.cuda.Stream())
    o_host = np.zeros((depth, 4), dtype=np.uint32)
    o_head, o_phase = 0, 1
    history = []
    m.launch()
    try:
        g = db.cq_attach(m.slots, 0, c.dev, c.host)
        assert g == 1
        for _ in range(40 if depth > 2 else 80):
            k = int(c.rng.integers(1, depth))
            rows = c.produce(k)
            history.extend(c.replica[r].copy() for r in rows)
            assert c.reap_until(db, c.produced) == c.produced
            n, o_head, o_phase = oracle.cq_mirror_pass(c.replica, o_head, o_phase, o_host)
            assert n == k
            assert (c.host.numpy().view(np.uint32) == o_host).all()
        assert (np.array(c.reaped) == np.array(history)).all()
        f = m.fields[0]
        assert (int(f["head"]), int(f["phase"])) == (o_head, o_phase)
        assert int(f["copied"]) == c.produced and int(f["seen"]) == 1
        gd = db.cq_detach(m.slots, 0)
        assert db.cq_wait_ack(m.slots, 0, gd, 5.0)
    finally:
        ctr = m.finish()
    assert ctr.tolist() == [c.produced, 0, 0, 0]


def test_timed_slot_records_latency(db, oracle):
    """A slot attached with DB_CQ_TIMED: the copies are the oracle's, and
    after each batch the slot holds that batch's latency (lat_seq equal to
    the completions copied so far, lat_ns between 0 and 10 ms). An untimed
    slot served by the same launch leaves both fields as they were."""
    m = Mirror(db, 2, limit_s=20.0)
    cs = torch.cuda.Stream()
    timed, plain = Controller(64, 71, cs), Controller(64, 72, cs)
    o_host = np.zeros((64, 4), dtype=np.uint32)
    o_head, o_phase = 0, 1
    f = m.fields
    f["flags"][0] = db.CQ_TIMED
    m.launch()
    try:
        db.cq_attach(m.slots, 0, timed.dev, timed.host)
        db.cq_attach(m.slots, 1, plain.dev, plain.host)
        lat = []
        for _ in range(30):
            k = int(timed.rng.integers(1, 40))
            timed.produce(k)
            plain.produce(k)
            assert timed.reap_until(db, timed.produced) == timed.produced
            assert plain.reap_until(db, plain.produced) == plain.produced
            n, o_head, o_phase = oracle.cq_mirror_pass(timed.replica, o_head, o_phase, o_host)
            assert n == k
            assert (timed.host.numpy().view(np.uint32) == o_host).all()
            t0 = time.monotonic()  # the latency fields follow the host CQ writes
            while int(m.fields[0]["lat_seq"]) != timed.produced and time.monotonic() - t0 < 5.0:
                time.sleep(10e-6)
            g = m.fields[0]
            assert int(g["lat_seq"]) == timed.produced
            assert 0 < int(g["lat_ns"]) < 10_000_000
            lat.append(int(g["lat_ns"]))
        assert int(m.fields[1]["lat_seq"]) == 0 and int(m.fields[1]["lat_ns"]) == 0
        gens = [db.cq_detach(m.slots, i) for i in range(2)]
        assert all(db.cq_wait_ack(m.slots, i, g, 5.0) for i, g in enumerate(gens))
    finally:
        ctr = m.finish()
    assert int(ctr[0]) == timed.produced + plain.produced and int(ctr[3]) == 0


def test_sixty_four_queues(db, oracle):
    """64 queues of different depths, batches on random subsets of them."""
    m = Mirror(db, 64, limit_s=30.0)
    copy_stream = torch.cuda.Stream()
    rng = np.random.default_rng(64)
    depths = [int(x) for x in rng.integers(2, 400, size=64)]
    cs = [Controller(d, 1000 + i, copy_stream) for i, d in enumerate(depths)]
    hist = [[] for _ in cs]
    m.launch()
    try:
        for i, c in enumerate(cs):
            db.cq_attach(m.slots, i, c.dev, c.host)
        for _ in range(12):
            for i in np.flatnonzero(rng.random(64) < 0.5):
                c = cs[i]
                rows = c.produce(int(rng.integers(1, c.depth)))
                hist[i].extend(c.replica[r].copy() for r in rows)
            for c in cs:
                assert c.reap_until(db, c.produced) == c.produced
        for c, h in zip(cs, hist):
            assert (np.array(c.reaped).reshape(-1, 4) == np.array(h).reshape(-1, 4)).all()
        gens = [db.cq_detach(m.slots, i) for i in range(64)]
        assert all(db.cq_wait_ack(m.slots, i, g, 5.0) for i, g in enumerate(gens))
    finally:
        ctr = m.finish()
    assert int(ctr[0]) == sum(c.produced for c in cs) and int(ctr[3]) == 0


def test_generations_and_acknowledgements(db):
    m = Mirror(db, 3, limit_s=20.0)
    cs = torch.cuda.Stream()
    a, b = Controller(16, 1, cs), Controller(5, 2, cs)
    f = m.fields
    # slot 2: attached and detached before the mirror ran
    db.cq_attach(m.slots, 2, a.dev, a.host)
    assert db.cq_detach(m.slots, 2) == 1
    with pytest.raises(db.DescBuildError) as e:       # not acknowledged yet
        db.cq_attach(m.slots, 2, a.dev, a.host)
    assert e.value.code == -16
    m.launch()
    try:
        assert db.cq_wait_ack(m.slots, 2, 1, 5.0)     # the odd value before the even one
        g = db.cq_attach(m.slots, 0, a.dev, a.host)
        with pytest.raises(db.DescBuildError) as e:   # attached already
            db.cq_attach(m.slots, 0, b.dev, b.host)
        assert e.value.code == -16
        a.produce(10)
        assert a.reap_until(db, 10) == 10
        assert db.cq_detach(m.slots, 0) == g
        assert db.cq_wait_ack(m.slots, 0, g, 5.0)
        # the same slot takes another queue pair: a fresh head and phase
        g2 = db.cq_attach(m.slots, 0, b.dev, b.host)
        assert g2 == 3
        b.produce(4)
        assert b.reap_until(db, 4) == 4               # a controller waits for the host
        b.produce(4)                                  # wraps
        assert b.reap_until(db, 8) == 8
        assert int(f[0]["seen"]) == 3 and int(f[0]["copied"]) == 8
        assert (int(f[0]["head"]), int(f[0]["phase"])) == (3, 0)
        assert int(f[1]["ack"]) == 0 and int(f[1]["generation"]) == 0
    finally:
        ctr = m.finish()
    assert ctr.tolist() == [18, 0, 0, 0]


def test_limit_ends_a_launch_and_the_next_resumes(db):
    """A launch that nobody stops ends at its limit with DB_ERR_TIMEOUT;
    completions written meanwhile wait in the device CQ, and the next
    launch resumes from the head and phase kept in the slot."""
    m = Mirror(db, 1, limit_s=0.3)
    c = Controller(8, 3, torch.cuda.Stream())
    m.launch()
    db.cq_attach(m.slots, 0, c.dev, c.host)
    c.produce(6)
    assert c.reap_until(db, 6) == 6
    m.stream.synchronize()                  # ends by itself at the limit
    ctr = m.ctr.cpu().numpy()
    assert ctr.tolist() == [6, 0, 0, ERR_TIMEOUT]
    c.produce(7)                            # wraps; no mirror is running
    time.sleep(0.05)
    assert c.reap_until(db, 13, timeout=0.05) == 6
    m.limit_s = 20.0
    m.launch()
    try:
        assert c.reap_until(db, 13) == 13
        f = m.fields[0]
        assert (int(f["head"]), int(f["phase"]), int(f["copied"])) == (5, 0, 13)
    finally:
        ctr = m.finish()
    assert ctr.tolist() == [7, 0, 0, 0]


def test_slot_the_attach_would_refuse_is_not_served(db):
    """A slot written by hand with depth 0 is counted, never dereferenced,
    and still acknowledged when detached."""
    m = Mirror(db, 2, limit_s=20.0)
    f = m.fields
    f["depth"][1] = 0
    f["generation"][1] = 1
    m.launch()
    try:
        time.sleep(0.2)                     # the warp takes the slot up first
        g = db.cq_detach(m.slots, 1)
        assert db.cq_wait_ack(m.slots, 1, g, 5.0)
    finally:
        ctr = m.finish()
    assert ctr.tolist() == [0, 1, 0, 0]


def test_memory_kinds_are_checked(db):
    stop = torch.zeros(1, dtype=torch.int32).pin_memory()
    pageable = torch.zeros((1, 64), dtype=torch.uint8)
    with pytest.raises(db.DescBuildError) as e:
        db.cq_mirror(pageable, stop, 1.0)
    assert e.value.code == -19
    slots = db.cq_slots(1)
    dev = torch.zeros((8, 4), dtype=torch.int32, device="cuda")
    pinned = torch.zeros((8, 4), dtype=torch.int32).pin_memory()
    g = ctypes.c_uint32(0)
    # the C call itself checks (the binding refuses a device tensor as a host CQ first)
    assert db._lib.db_cq_attach(slots.data_ptr(), dev.data_ptr(), dev.data_ptr(), 8,
                                ctypes.byref(g)) == -19      # host CQ in device memory
    assert db._lib.db_cq_attach(slots.data_ptr(), pinned.data_ptr(), pinned.data_ptr(), 8,
                                ctypes.byref(g)) == -19      # device CQ in host memory
    assert db._lib.db_cq_attach(slots.data_ptr(), dev.data_ptr(), pinned.data_ptr(), 8,
                                ctypes.byref(g)) == 0 and g.value == 1
    with pytest.raises(db.DescBuildError):
        db.cq_mirror(slots, stop, 61.0)
