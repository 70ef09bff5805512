"""PRP build with no caller workspace, checked against the workspace version.

db_prp_build_static exists for callers that must not allocate device memory
while they submit I/O: cudaMalloc can wait for work already queued on the
device and takes driver locks, which a latency-bound submitter cannot afford,
and a process whose device memory is handed out up front by its own
allocator may have no room for one more allocation. Its scratch memory is a
static array inside the library instead.

The test calls it through the C ABI twice in a row, on two different
batches, and requires every output to equal what db_prp_build (with its own
workspace) produces for the same inputs -- bit for bit, like every PRP test.
The second call checks that the shared array was left ready by the first.
This file is collected last on purpose; it needs no state from other tests.
"""

import ctypes

import numpy as np
import pytest

from gpu_util import dev64, host64, lib, need_gpu, torch

pytestmark = pytest.mark.gpu

FILL = -0x2152411021524111


@pytest.fixture(scope="module")
def db():
    need_gpu()
    return lib()


def build(db, w, static: bool):
    n = w["req"].shape[0]
    req, lut = dev64(w["req"]), dev64(w["lut"])
    cap = 1 << 16
    arena = torch.full((cap, 512), FILL, dtype=torch.int64, device="cuda")
    prp = torch.full((n, 2), FILL, dtype=torch.int64, device="cuda")
    pb = torch.full((n,), FILL, dtype=torch.int64, device="cuda")
    st = torch.full((n,), 0xEE, dtype=torch.uint8, device="cuda")
    ctr = torch.full((4,), FILL, dtype=torch.int64, device="cuda")
    if static:
        db.prp_build_static(req, lut, w["heap_size"], w["arena_base"], cap, arena, prp,
                            page_base=pb, status=st, ctr=ctr)
    else:
        ws = db.workspace(db.prp_workspace_size(n))
        db.prp_build(req, lut, w["heap_size"], w["arena_base"], cap, arena, prp, ws,
                     page_base=pb, status=st, ctr=ctr)
    torch.cuda.synchronize()
    used = int(host64(ctr)[0])
    return dict(prp=host64(prp), page_base=host64(pb), status=st.cpu().numpy(),
                ctr=host64(ctr), arena=host64(arena[:min(used, cap) + 1]))


def test_static_scratch_matches_workspace_build_twice(db):
    import synth
    batches = [synth.prp_large(seed=101, n=60_000), synth.prp_tiny(seed=202)]
    for w in batches:  # two calls in a row on the shared static array
        got = build(db, w, static=True)
        want = build(db, w, static=False)
        for key in ("prp", "page_base", "status", "ctr", "arena"):
            assert (got[key] == want[key]).all(), key
        assert int(got["ctr"][3]) == 0 and int(got["ctr"][0]) > 0


def test_static_scratch_rejects_batches_over_its_limit(db):
    E2BIG = 7
    fake = 1 << 20  # never dereferenced: the size check comes first
    rc = db._lib.db_prp_build_static(fake, db.PRP_STATIC_MAX_REQUESTS + 1, fake, 1 << 20, 0, 1,
                                     fake, fake, None, None, None, 0, None)
    assert rc == -E2BIG
    assert "built-in workspace" in db.strerror(rc)
