"""Host half of the CQ-mirror slot protocol, without a GPU: reaping a host
CQ, detaching, waiting for an acknowledgement, and the argument checks of
the launch (xNVMe "uPCIe CUDA" backend page, "Completions in device
memory")."""

import threading
import time

import numpy as np
import pytest
import torch

from conftest import ROOT  # noqa: F401  (puts the repository on sys.path)

PHASE_BIT = 1 << 16


@pytest.fixture(scope="module")
def db():
    import descriptor_build_gb300 as d
    return d


def controller_write(cq, first, count, rng):
    depth = cq.shape[0]
    for k in range(count):
        i = first + k
        body = rng.integers(0, 2**32, size=4, dtype=np.uint64).astype(np.uint32)
        body[3] = (int(body[3]) & ~PHASE_BIT) | ((1 - (i // depth) % 2) << 16)
        cq[i % depth] = body


@pytest.mark.parametrize("depth", [2, 5, 64, 257])
def test_reap_equals_the_oracle_pass(db, oracle, depth):
    """The host's reap follows the same phase rule as the mirror pass."""
    rng = np.random.default_rng(depth)
    cq = np.zeros((depth, 4), dtype=np.uint32)
    replica = np.zeros_like(cq)
    head = o_head = 0
    phase = o_phase = 1
    produced = 0
    for _ in range(40):
        k = int(rng.integers(0, depth))
        controller_write(cq, produced, k, rng)
        produced += k
        t = torch.from_numpy(cq.view(np.int32))
        got, head, phase = db.cq_host_reap(t, head, phase)
        n, o_head, o_phase = oracle.cq_mirror_pass(cq, o_head, o_phase, replica)
        assert got.shape[0] == n == k and (head, phase) == (o_head, o_phase)
        if k:
            idx = [(produced - k + j) % depth for j in range(k)]
            assert (got == replica[idx]).all()


def test_reap_respects_max_and_checks_arguments(db):
    cq = torch.zeros((8, 4), dtype=torch.int32)
    cq[:6, 3] = PHASE_BIT
    got, h, ph = db.cq_host_reap(cq, 0, 1, max_entries=4)
    assert got.shape[0] == 4 and (h, ph) == (4, 1)
    got, h, ph = db.cq_host_reap(cq, h, ph)
    assert got.shape[0] == 2 and (h, ph) == (6, 1)
    with pytest.raises(db.DescBuildError):
        db.cq_host_reap(cq, 8, 1)        # head outside the queue


def test_detach_and_wait_for_the_acknowledgement(db):
    slots = torch.zeros((2, 64), dtype=torch.uint8)
    f = db.cq_slot_fields(slots)
    with pytest.raises(db.DescBuildError):
        db.cq_detach(slots, 0)            # not attached
    f["generation"][1] = 3                # attached (as if by db_cq_attach)
    g = db.cq_detach(slots, 1)
    assert g == 3 and f["generation"][1] == 4
    assert not db.cq_wait_ack(slots, 1, g, 0.02)   # nobody acknowledges

    def device_side():                    # a stand-in for the warp
        time.sleep(0.02)
        f["ack"][1] = 3

    th = threading.Thread(target=device_side)
    th.start()
    assert db.cq_wait_ack(slots, 1, g, 5.0)
    th.join()


def test_request_stop(db):
    stop = torch.zeros(1, dtype=torch.int32)
    db.cq_request_stop(stop)
    assert int(stop[0]) == 1


def test_launch_argument_checks_need_no_gpu(db):
    """Checks that fail before any CUDA call."""
    import ctypes
    lib = ctypes.CDLL(db.lib_path)
    vp, u32, u64 = ctypes.c_void_p, ctypes.c_uint32, ctypes.c_uint64
    lib.db_cq_mirror.argtypes = [vp, u32, vp, u64, vp, vp]
    slots = np.zeros((65, 64), dtype=np.uint8)
    stop = np.zeros(1, dtype=np.uint32)
    p = slots.ctypes.data + (-slots.ctypes.data % 64)
    assert lib.db_cq_mirror(p, 0, stop.ctypes.data, 10**9, None, None) == -22
    assert lib.db_cq_mirror(p, 65, stop.ctypes.data, 10**9, None, None) == -22
    assert lib.db_cq_mirror(p, 1, stop.ctypes.data, 0, None, None) == -22
    assert lib.db_cq_mirror(p, 1, stop.ctypes.data, 61 * 10**9, None, None) == -22
    assert lib.db_cq_mirror(p + 8, 1, stop.ctypes.data, 10**9, None, None) == -22
    assert lib.db_cq_mirror(p, 1, None, 10**9, None, None) == -22


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the answer without a device")
def test_attach_needs_a_device_to_check_memory(db):
    slots = torch.zeros((1, 64), dtype=torch.uint8)
    cq = torch.zeros((4, 4), dtype=torch.int32)
    with pytest.raises(db.DescBuildError) as e:
        db.cq_attach(slots, 0, cq, cq)
    assert e.value.code == -19
