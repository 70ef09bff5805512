"""Calls on the caller's own streams, against the oracle, bit for bit.

The MR lookup and the put bucketing launch their second and later kernels as
programmatic dependents of the kernel before them. These tests run them on
two side streams at once, twice in a row with the same workspaces, so each
call follows the previous call's last kernel on its stream while the other
stream's kernels share the GPU.
"""

import numpy as np
import pytest

from gpu_util import dev32, dev64, host32, host64, lib, need_gpu, torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def db():
    need_gpu()
    return lib()


def test_mr_lookup_and_put_bucketing_on_two_side_streams(db, oracle):
    import synth
    m = synth.mr_lookup(seed=0x5EED1, n_mr=20_000, n_q=300_000)
    # 200,000 puts over 32 rings of 8,192 WQEs: the second batch wraps the rings.
    p = synth.put_bucket(seed=0x5EED2, n=200_000, world=8, n_qp=4, depth=1 << 13)
    R = p["world"] * p["n_qp"]
    want_mr = oracle.mr_bsearch(m["queries"], m["mr_start"], m["mr_end"], m["mr_lkey"])
    want_1 = oracle.wqe_bucket(p["req"], p["peer_ptrs"], p["rkeys"], p["world"], p["n_qp"],
                               p["local_base"], p["lkey"], p["heap_size"], p["depth"], p["head"])
    want_2 = oracle.wqe_bucket(p["req"], p["peer_ptrs"], p["rkeys"], p["world"], p["n_qp"],
                               p["local_base"], p["lkey"], p["heap_size"], p["depth"],
                               want_1["head"], rings=want_1["rings"].copy())

    n_q = m["queries"].shape[0]
    q, start, end = dev64(m["queries"]), dev64(m["mr_start"]), dev64(m["mr_end"])
    lk_tab = dev32(m["mr_lkey"])
    mr_ws = db.workspace(db.mr_workspace_size(m["mr_start"].shape[0]))
    req, peer, rkeys = dev64(p["req"]), dev64(p["peer_ptrs"]), dev32(p["rkeys"])
    rings = torch.full((R, p["depth"], 64), 0, dtype=torch.uint8, device="cuda")
    head = dev64(p["head"])
    wqe_ws = db.workspace(db.wqe_workspace_size(p["req"].shape[0], R))
    s_mr, s_wqe = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    results = []
    for _ in range(2):
        idx = torch.full((n_q,), 0x55, dtype=torch.int32, device="cuda")
        lk = torch.full((n_q,), 0x55, dtype=torch.int32, device="cuda")
        kind = torch.full((n_q,), 0x55, dtype=torch.uint8, device="cuda")
        mr_ctr = torch.full((4,), -1, dtype=torch.int64, device="cuda")
        count = torch.full((R,), -1, dtype=torch.int32, device="cuda")
        wqe_ctr = torch.full((4,), -1, dtype=torch.int64, device="cuda")
        for s in (s_mr, s_wqe):
            s.wait_stream(torch.cuda.current_stream())
        db.mr_lookup(q, start, end, lk_tab, idx, lk, kind, mr_ws, ctr=mr_ctr,
                     stream=s_mr)
        db.wqe_bucket(req, peer, rkeys, p["world"], p["n_qp"], p["local_base"], p["lkey"],
                      p["heap_size"], rings, p["depth"], head, count, wqe_ws, ctr=wqe_ctr,
                      stream=s_wqe)
        torch.cuda.synchronize()
        results.append(dict(idx=idx.cpu().numpy(), lkey=host32(lk), kind=kind.cpu().numpy(),
                            mr_ctr=host64(mr_ctr), head=host64(head), count=host32(count),
                            wqe_ctr=host64(wqe_ctr), rings=rings.cpu().numpy()))
    for got, want in zip(results, (want_1, want_2)):
        assert (got["kind"] == want_mr["kind"]).all()
        assert (got["idx"] == want_mr["idx"]).all()
        assert (got["lkey"] == want_mr["lkey"]).all()
        assert got["mr_ctr"][0] == int((want_mr["kind"] == 1).sum() + (want_mr["kind"] == 2).sum())
        assert (got["head"] == want["head"]).all()
        assert (got["count"] == want["count"]).all()
        assert (got["wqe_ctr"] == want["ctr"]).all()
        assert (got["rings"] == want["rings"]).all()
