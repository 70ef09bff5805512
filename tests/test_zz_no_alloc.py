"""PRP build with no caller workspace, checked against the oracle and against
the workspace version.

db_prp_build_static exists for callers that must not allocate device memory
while they submit I/O: cudaMalloc can wait for work already queued on the
device and takes driver locks, which a latency-bound submitter cannot afford,
and a process whose device memory is handed out up front by its own
allocator may have no room for one more allocation. Its scratch memory is a
static array inside the library instead.

The tests call it through the C ABI twice in a row, on two different
batches, and require every output to equal the oracle's -- bit for bit, like
every PRP test -- and what db_prp_build (with its own workspace) produces for
the same inputs. The second call checks that the shared array was left ready
by the first. One more batch holds exactly the array's limit of requests
(every status word of the array in use). A call whose wait for another tile
runs out cannot be made on purpose here: the array has no caller-side handle
to plant a stuck ticket in, and tickets go only to running CTAs; that
recovery is the workspace kernel's own end-of-call path, tested with a
planted ticket in tests/test_gpu_prp.py.
This file is collected last on purpose; it needs no state from other tests.
"""

import numpy as np
import pytest

from gpu_util import assert_arena_equal, dev64, host64, lib, need_gpu, torch

pytestmark = pytest.mark.gpu

FILL = -0x2152411021524111


@pytest.fixture(scope="module")
def db():
    need_gpu()
    return lib()


def build(db, w, static: bool, cap: int, per_request: bool = True, arena: bool = True):
    n = w["req"].shape[0]
    req, lut = dev64(w["req"]), dev64(w["lut"])
    ar = torch.full((max(cap, 1), 512), FILL, dtype=torch.int64, device="cuda") if arena else None
    prp = torch.full((n, 2), FILL, dtype=torch.int64, device="cuda")
    pb = torch.full((n,), FILL, dtype=torch.int64, device="cuda") if per_request else None
    st = torch.full((n,), 0xEE, dtype=torch.uint8, device="cuda") if per_request else None
    ctr = torch.full((4,), FILL, dtype=torch.int64, device="cuda")
    if static:
        db.prp_build_static(req, lut, w["heap_size"], w["arena_base"], cap, ar, prp,
                            page_base=pb, status=st, ctr=ctr)
    else:
        ws = db.workspace(db.prp_workspace_size(n))
        db.prp_build(req, lut, w["heap_size"], w["arena_base"], cap, ar, prp, ws,
                     page_base=pb, status=st, ctr=ctr)
    torch.cuda.synchronize()
    used = min(int(host64(ctr)[0]), cap)
    out = dict(prp=host64(prp), ctr=host64(ctr))
    if per_request:
        out.update(page_base=host64(pb), status=st.cpu().numpy())
    if arena:
        out["arena"] = host64(ar[:max(used, 1)])[:used]
    return out


def test_static_scratch_matches_oracle_twice(db, oracle):
    import synth
    batches = [synth.prp_large(seed=101, n=60_000), synth.prp_tiny(seed=202)]
    for w in batches:  # two calls in a row on the shared static array
        need = oracle.prp_build(w["req"], w["lut"], w["heap_size"], w["arena_base"], 1 << 40,
                                lists=False)
        cap = int(need["ctr"][0])
        assert cap > 0
        want = oracle.prp_build(w["req"], w["lut"], w["heap_size"], w["arena_base"], cap,
                                fill=FILL & (2**64 - 1))
        got = build(db, w, static=True, cap=cap)
        for key in ("prp", "page_base", "status", "ctr"):
            assert (got[key] == want[key]).all(), key
        assert_arena_equal(got["arena"], want["arena"][:cap], FILL, where="static call")
        # ... and the workspace call on the same inputs gives the same words.
        ref = build(db, w, static=False, cap=cap)
        for key in ("prp", "page_base", "status", "ctr", "arena"):
            assert (got[key] == ref[key]).all(), key
        assert int(got["ctr"][3]) == 0


def test_static_scratch_at_its_request_limit(db, oracle):
    """A batch of exactly DB_PRP_STATIC_MAX_REQUESTS small requests (no
    lists): every PRP pair and the counters against the oracle, twice."""
    import synth
    n = db.PRP_STATIC_MAX_REQUESTS
    w = synth.prp_small(n=n)
    assert w["req"].shape[0] == n
    want = oracle.prp_build(w["req"], w["lut"], w["heap_size"], w["arena_base"], 0, lists=False)
    assert int(want["ctr"][0]) == 0
    for _ in range(2):
        got = build(db, w, static=True, cap=0, per_request=False, arena=False)
        assert (got["prp"] == want["prp"]).all()
        assert (got["ctr"] == want["ctr"]).all()


def test_static_scratch_rejects_batches_over_its_limit(db):
    E2BIG = 7
    fake = 1 << 20  # never dereferenced: the size check comes first
    rc = db._lib.db_prp_build_static(fake, db.PRP_STATIC_MAX_REQUESTS + 1, fake, 1 << 20, 0, 1,
                                     fake, fake, None, None, None, 0, None)
    assert rc == -E2BIG
    assert "built-in workspace" in db.strerror(rc)
