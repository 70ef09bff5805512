"""Pins for the CQ-mirror oracle.

Follows xNVMe "uPCIe CUDA" backend page, "Completions in device memory":
an entry is forwarded to the host CQ once its phase tag has flipped, and a
slot's generation (odd while attached) is acknowledged by the warp that
worked under it. The phase-tag rule restated here (completion i of a queue
goes to entry i mod depth, with tag 1 on the first pass through the queue,
0 on the second, and so on) is the NVMe completion-queue convention the
page relies on.
"""

import numpy as np
import pytest

PHASE_BIT = 1 << 16


def controller_write(cq: np.ndarray, first: int, count: int, rng) -> np.ndarray:
    """Write completions first .. first+count-1 the way a controller does;
    returns the entries written, [count, 4]."""
    depth = cq.shape[0]
    out = np.empty((count, 4), dtype=np.uint32)
    for k in range(count):
        i = first + k
        body = rng.integers(0, 2**32, size=4, dtype=np.uint64).astype(np.uint32)
        tag = 1 - (i // depth) % 2
        body[3] = (int(body[3]) & ~PHASE_BIT) | (tag << 16)
        cq[i % depth] = body
        out[k] = body
    return out


def test_hand_worked_wrap(oracle):
    """Depth 4: three completions, then two more that wrap. The second pass
    writes tag 0, so after the wrap the mirror expects 0."""
    dev = np.zeros((4, 4), dtype=np.uint32)
    host = np.zeros_like(dev)
    dev[0] = [10, 0, 0, 0x0001_0007]   # cid 7, tag 1
    dev[1] = [11, 0, 0, 0x0001_0008]
    dev[2] = [12, 0, 0, 0x0001_0009]
    assert oracle.cq_mirror_pass(dev, 0, 1, host) == (3, 3, 1)
    assert host[:3].tolist() == dev[:3].tolist() and host[3].tolist() == [0, 0, 0, 0]
    dev[3] = [13, 0, 0, 0x0001_000A]   # last of pass one, tag 1
    dev[0] = [14, 0, 0, 0x0000_000B]   # first of pass two, tag 0
    assert oracle.cq_mirror_pass(dev, 3, 1, host) == (2, 1, 0)
    assert host.tolist() == [[14, 0, 0, 0xB], [11, 0, 0, 0x0001_0008],
                             [12, 0, 0, 0x0001_0009], [13, 0, 0, 0x0001_000A]]
    # nothing new: entry 1 still carries tag 1
    assert oracle.cq_mirror_pass(dev, 1, 0, host) == (0, 1, 0)


def test_only_the_phase_bit_decides(oracle):
    """Other status bits set around bit 16 do not make an entry new."""
    dev = np.zeros((8, 4), dtype=np.uint32)
    host = np.zeros_like(dev)
    dev[0, 3] = 0xFFFE_FFFF            # every bit but the phase tag
    assert oracle.cq_mirror_pass(dev, 0, 1, host)[0] == 0
    dev[0, 3] = 0x0001_0000
    dev[1, 3] = 0x8000_0000 | 0x0000_8000
    assert oracle.cq_mirror_pass(dev, 0, 1, host)[0] == 1


@pytest.mark.parametrize("depth", [2, 3, 32, 33, 64, 1000])
def test_mirror_follows_the_controller(oracle, depth):
    """Random batches of completions, a pass after each: the pass copies
    exactly the new ones, head and phase follow the closed form, and the
    host CQ equals what the controller wrote at every entry."""
    rng = np.random.default_rng(depth)
    dev = np.zeros((depth, 4), dtype=np.uint32)
    host = np.zeros_like(dev)
    head, phase, produced = 0, 1, 0
    for _ in range(60):
        k = int(rng.integers(0, depth + 1))   # never more than a queue's worth ahead
        controller_write(dev, produced, k, rng)
        produced += k
        n, head, phase = oracle.cq_mirror_pass(dev, head, phase, host)
        assert n == k
        assert head == produced % depth
        assert phase == 1 - (produced // depth) % 2
        assert (host == dev).all() if produced >= depth else (host[:produced] == dev[:produced]).all()


def test_max_bounds_a_pass(oracle):
    rng = np.random.default_rng(1)
    dev = np.zeros((16, 4), dtype=np.uint32)
    host = np.zeros_like(dev)
    controller_write(dev, 0, 10, rng)
    assert oracle.cq_mirror_pass(dev, 0, 1, host, max_entries=4) == (4, 4, 1)
    assert oracle.cq_mirror_pass(dev, 4, 1, host, max_entries=100) == (6, 10, 1)


def test_stale_entry_stops_the_pass(oracle):
    """An entry the controller has not rewritten yet (old tag) ends the run
    even when later entries look new."""
    rng = np.random.default_rng(2)
    dev = np.zeros((8, 4), dtype=np.uint32)
    host = np.zeros_like(dev)
    controller_write(dev, 0, 8, rng)           # pass one complete: all tag 1
    n, head, phase = oracle.cq_mirror_pass(dev, 0, 1, host)
    assert (n, head, phase) == (8, 0, 0)
    controller_write(dev, 8, 3, rng)           # entries 0..2 tag 0
    dev[1, 3] |= PHASE_BIT                     # entry 1 not yet rewritten
    assert oracle.cq_mirror_pass(dev, 0, 0, host)[:2] == (1, 1)


@pytest.mark.parametrize("cur,now,keep,want", [
    (0, 0, 0, 0),     # never attached: nothing to acknowledge
    (0, 1, 0, 0),     # takes up generation 1: nothing yet
    (1, 1, 0, 0),     # still working under 1
    (1, 2, 0, 1),     # detached: the odd value worked under
    (0, 2, 0, 1),     # found detached before taking it up: the odd value before
    (2, 2, 1, 1),     # idle on an even generation: already acknowledged
    (3, 4, 1, 3),
    (0, 6, 0, 5),
    (5, 7, 4, 5),     # re-attached before the warp saw the detach: acknowledge 5
    (4, 5, 3, 3),     # takes up 5 after idling
])
def test_ack_rule(oracle, cur, now, keep, want):
    assert oracle.cq_ack(cur, now, keep) == want
