"""Throughput of batched GPU-range -> DMA-descriptor translation on one GB300.

One step runs every part of the hot path once, each on its full-size seeded
synthetic workload. The four batches are independent: each runs on its own
CUDA stream, forked together and joined at the end of the step (--serial:
one stream, in turn):

  prp_small   db_prp_build, 1,048,576 small requests (1 GiB heap)
  prp_large   db_prp_build, 4,194,304 requests, chained lists (16 GiB heap)
  mr_lookup   db_mr_lookup, 16,777,216 queries over 1,048,576 records
  put_bucket  db_wqe_bucket, 8,388,608 puts into 32 rings of 2^19 WQEs

``value`` is requests translated per second over the whole step (all four
batches), with inputs resident in HBM. Each call is also timed with CUDA
events alone on the stream, in the same steps run one call at a time after
the timed region; the dominant one (prp_large) gives the roofline line.
Beside each call, a plain device copy of the same algorithmic bytes timed the
same way (``size_matched_copy_ms``): small batches cannot reach the peak copy
rate, and the ratio shows how near a call is to a copy of its own size.
``output_GB_per_s`` counts the descriptor bytes written (PRP pairs, list
words, MR results, WQEs), for the step and per call. ``e2e`` repeats the
step through the same API with inputs in pinned host memory and every
descriptor copied back to the host. ``next``
times, on its own and outside the step, the rows built after the hot path:
the put batch on a heap of 2 MiB chunks (db_wqe_bucket_vmm, without and
with packet sequence numbers), the MR lookup on a table whose records
overlap (db_mr_lookup_overlap), the registration-cache batches
(db_mr_register, db_mr_deregister) and the completion-queue mirror
(db_cq_mirror: drain rate over 64 queues, latency at queue depth 1).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun each rank runs its own replica (the batches are independent);
the step time is the maximum over ranks.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "M requests/s translated + achieved HBM GB/s as % of GB300 peak"
UNIT = "M requests/s"
WORKLOAD = "descriptor batch: prp_small + prp_large + mr_lookup + put_bucket (full sizes)"
# Launch order of a step's calls on their own streams (measured best on GB300).
SCHEDULE = ("mr_lookup", "put_bucket", "prp_small", "prp_large")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-next", action="store_true",
                    help="skip the separately timed rows after the hot path")
    ap.add_argument("--only", choices=["prp_small", "prp_large", "mr_lookup", "put_bucket"],
                    help="profiling aid: run one workload only (not a bench line)")
    ap.add_argument("--fraction", type=float, default=1.0,
                    help="profiling aid: keep this leading fraction of each batch")
    ap.add_argument("--prp-sched", choices=["auto", "single", "split"], default="auto",
                    help="profiling aid: force a PRP schedule (a leading fraction of the large "
                         "batch would otherwise take the small-batch one)")
    ap.add_argument("--serial", action="store_true",
                    help="run a step's four calls one after another on one stream "
                         "(default: each on its own stream, all at once)")
    ap.add_argument("--next-only", choices=["mr_register", "mr_deregister", "put_bucket_vmm",
                                            "put_bucket_vmm_psn", "mr_lookup_overlap",
                                            "put_bucket_transport"],
                    help="profiling aid: time one of the rows after the hot path, alone")
    return ap.parse_args()


# --------------------------------------------------------------------- inputs
def make_inputs(only=None, fraction=1.0):
    import synth
    gens = {"prp_small": synth.prp_small, "prp_large": synth.prp_large,
            "mr_lookup": synth.mr_lookup, "put_bucket": synth.put_bucket}
    inp = {k: g() for k, g in gens.items() if only in (None, k)}
    if fraction < 1.0:
        for k, w in inp.items():
            key = "queries" if k == "mr_lookup" else "req"
            w[key] = w[key][: max(1, int(w[key].shape[0] * fraction))]
    return inp


def list_words(req: np.ndarray) -> int:
    """8-byte words a PRP batch writes into list pages (data entries plus
    chain pointers), counted from the requests -- measurement bookkeeping."""
    off = req[:, 0]
    ln = req[:, 1] & np.uint64(0xFFFFFFFF)
    n = ((off & np.uint64(4095)) + ln + np.uint64(4095)) >> np.uint64(12)
    n = n[n >= 3].astype(np.int64)
    entries = n - 1
    pages = -(-(entries - 1) // 511)
    return int((entries + pages - 1).sum())


def algorithmic_bytes(inp) -> dict:
    """Bytes each call must move at minimum (read inputs once, write outputs once):
    PRP 16 B request + 16 B PRP pair + 8 B per list word + the LUT once;
    MR 16 B query + 9 B result + the 20 B/record table once; put 16 B + 64 B WQE."""
    out = {}
    for k in ("prp_small", "prp_large"):
        if k in inp:
            w = inp[k]
            out[k] = 32 * w["req"].shape[0] + 8 * list_words(w["req"]) + 8 * w["lut"].shape[0]
    if "mr_lookup" in inp:
        m = inp["mr_lookup"]
        out["mr_lookup"] = 25 * m["queries"].shape[0] + 20 * m["mr_start"].shape[0]
    if "put_bucket" in inp:
        out["put_bucket"] = 80 * inp["put_bucket"]["req"].shape[0]
    return out


def output_bytes(inp) -> dict:
    """Descriptor bytes each call writes: the 16 B PRP pair and 8 B per list
    word; the 9 B MR result (index, lkey, kind); the 64 B WQE."""
    out = {}
    for k in ("prp_small", "prp_large"):
        if k in inp:
            out[k] = 16 * inp[k]["req"].shape[0] + 8 * list_words(inp[k]["req"])
    if "mr_lookup" in inp:
        out["mr_lookup"] = 9 * inp["mr_lookup"]["queries"].shape[0]
    if "put_bucket" in inp:
        out["put_bucket"] = 64 * inp["put_bucket"]["req"].shape[0]
    return out


def units(inp) -> dict:
    return {k: (w["queries"] if k == "mr_lookup" else w["req"]).shape[0]
            for k, w in inp.items()}


def max_over_ranks(dist, value: float, device=None) -> float:
    """The largest of every rank's value, on every rank (the value itself
    without a process group). NCCL wants a device tensor, gloo a host one."""
    if not dist:
        return value
    import torch
    tt = torch.tensor([value], dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def job_throughput(world: int, reqs_per_rank_step: int, ms_per_step: float) -> float:
    """Whole-job M requests/s: every rank's requests over the slowest rank's step."""
    return world * reqs_per_rank_step / (ms_per_step * 1e-3) / 1e6


def peak_gbs():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return 6800.0, "fallback"


def source_sha256(kernel_src: str) -> str:
    """Hash of what a kernel is built from: its file, the shared device
    header and the public header."""
    h = hashlib.sha256()
    for path in (os.path.join(ROOT, "descriptor_build_gb300", "csrc", kernel_src),
                 os.path.join(ROOT, "descriptor_build_gb300", "csrc", "common.cuh"),
                 os.path.join(ROOT, "include", "descbuild.h")):
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def recorded_traffic(workload: str):
    """The committed ncu figures of one call (DRAM bytes per call, L2 sectors
    and requests per request), if they were taken on the kernel sources as
    they are now (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)[workload]
        if source_sha256(rec["source"]) != rec["source_sha256"]:
            return None
        return rec
    except Exception:
        return None


def host_cpu() -> dict:
    """Host cores and CPU model (lscpu), recorded beside the CPU baseline."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":")[0].strip() in ("Model name", "Model"):
                model = line.split(":", 1)[1].strip()
                if not model.isdigit():
                    break
    except Exception:
        pass
    if not model:
        import platform
        model = platform.processor() or platform.machine()
    return {"nproc": os.cpu_count(), "cpu_model": model}


# -------------------------------------------------------------- clock sampler
class Clocks:
    def __init__(self, index: int):
        self.proc = None
        self.index = index

    def __enter__(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.rows = []
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) == 9:
                self.rows.append(parts)

    def summary(self):
        if not getattr(self, "rows", None):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in self.rows for k in range(4)
                          if r[5 + k].lower() == "active"})
        load = [x for x in sm if mx and x > 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(load) if load else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(self.rows)}


def smi_index(device) -> int:
    """nvidia-smi's index of a CUDA device (honours CUDA_VISIBLE_DEVICES)."""
    local = device.index or 0
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [x.strip() for x in vis.split(",")]
        if local < len(ids) and ids[local].isdigit():
            return int(ids[local])
    return local


# ----------------------------------------------------------------- our arm
class Step:
    """Device buffers for one replica and the calls of one step."""

    LAUNCHES = {"prp_small": 1, "prp_large": 1, "mr_lookup": 2, "put_bucket": 3}

    def launches(self, name: str) -> int:
        """Kernels one call launches. A PRP batch of at most one wave of the
        pair kernel (4 CTAs of 2,048 requests per SM) takes the two-kernel
        schedule unless a schedule is forced."""
        if name.startswith("prp"):
            n = self.inp[name]["req"].shape[0]
            sms = self.torch.cuda.get_device_properties(self.device).multi_processor_count
            split = -(-n // 2048) <= 4 * sms
            if self.prp_flags:
                split = self.prp_flags == self.db.PRP_SCHED_SPLIT
            return 2 if split else 1
        return self.LAUNCHES[name]

    def __init__(self, db, torch, inp, device, prp_sched="auto"):
        self.db, self.torch, self.inp, self.device = db, torch, inp, device
        self.prp_flags = {"auto": 0, "single": db.PRP_SCHED_SINGLE,
                          "split": db.PRP_SCHED_SPLIT}[prp_sched]
        t = torch
        d64 = lambda a: t.from_numpy(np.ascontiguousarray(a).view(np.int64)).to(device)
        d32 = lambda a: t.from_numpy(np.ascontiguousarray(a).view(np.int32)).to(device)
        self.bufs = {}
        for k in ("prp_small", "prp_large"):
            if k not in inp:
                continue
            w = inp[k]
            n = w["req"].shape[0]
            a = dict(req=d64(w["req"]), lut=d64(w["lut"]), heap=w["heap_size"],
                     base=w["arena_base"], cap=0, arena=None,
                     prp=t.empty((n, 2), dtype=t.int64, device=device),
                     ctr=t.zeros(4, dtype=t.int64, device=device),
                     ws=db.workspace(db.prp_workspace_size(n), device))
            # Size the list arena the way a caller would: a call with no arena
            # reports, in its counters, the list pages the batch needs.
            self.prp(a, t.cuda.current_stream(device))
            t.cuda.synchronize(device)
            a["cap"] = int(a["ctr"][0].item())
            a["arena"] = t.empty((max(a["cap"], 1), 512), dtype=t.int64, device=device)
            self.bufs[k] = a
        if "mr_lookup" in inp:
            m = inp["mr_lookup"]
            nq = m["queries"].shape[0]
            self.bufs["mr_lookup"] = dict(
                q=d64(m["queries"]), start=d64(m["mr_start"]), end=d64(m["mr_end"]),
                lkey=d32(m["mr_lkey"]), idx=t.empty(nq, dtype=t.int32, device=device),
                olkey=t.empty(nq, dtype=t.int32, device=device),
                kind=t.empty(nq, dtype=t.uint8, device=device),
                ctr=t.zeros(4, dtype=t.int64, device=device),
                ws=db.workspace(db.mr_workspace_size(m["mr_start"].shape[0]), device))
        if "put_bucket" in inp:
            p = inp["put_bucket"]
            R = p["world"] * p["n_qp"]
            self.bufs["put_bucket"] = dict(
                req=d64(p["req"]), peer=d64(p["peer_ptrs"]), rkeys=d32(p["rkeys"]),
                rings=t.empty((R, p["depth"], 64), dtype=t.uint8, device=device),
                head=d64(p["head"]), count=t.empty(R, dtype=t.int32, device=device),
                ctr=t.zeros(4, dtype=t.int64, device=device),
                ws=db.workspace(db.wqe_workspace_size(p["req"].shape[0], R), device))

    def prp(self, a, stream):
        self.db.prp_build(a["req"], a["lut"], a["heap"], a["base"], a["cap"], a["arena"],
                          a["prp"], a["ws"], ctr=a["ctr"], flags=self.prp_flags, stream=stream)

    def mr_call(self, stream):
        m = self.bufs["mr_lookup"]
        self.db.mr_lookup(m["q"], m["start"], m["end"], m["lkey"], m["idx"], m["olkey"],
                          m["kind"], m["ws"], ctr=m["ctr"], stream=stream)

    def put_call(self, stream):
        p, P = self.bufs["put_bucket"], self.inp["put_bucket"]
        self.db.wqe_bucket(p["req"], p["peer"], p["rkeys"], P["world"], P["n_qp"],
                           P["local_base"], P["lkey"], P["heap_size"], p["rings"], P["depth"],
                           p["head"], p["count"], p["ws"], ctr=p["ctr"], stream=stream)

    def calls(self):
        fns = {"prp_small": lambda s: self.prp(self.bufs["prp_small"], s),
               "prp_large": lambda s: self.prp(self.bufs["prp_large"], s),
               "mr_lookup": self.mr_call, "put_bucket": self.put_call}
        return [(k, fns[k]) for k in ("prp_small", "prp_large", "mr_lookup", "put_bucket")
                if k in self.bufs]

    def check_counters(self):
        for name, b in self.bufs.items():
            err = int(b["ctr"][3].item())
            if err:
                raise RuntimeError(f"{name}: device error bits {err}")
            if name.startswith("prp"):
                assert int(b["ctr"][2].item()) == 0, "arena overflow in the benchmark"


def run_next(args, device) -> dict:
    """The rows after the hot path, timed on their own (not part of a step):
    the put batch on a heap of 2 MiB chunks (db_wqe_bucket_vmm), without and
    with packet sequence numbers (mtu 4096), the MR lookup on a table whose
    records overlap (db_mr_lookup_overlap), the registration and
    deregistration batches (db_mr_register, db_mr_deregister) and the CQ
    mirror (db_cq_mirror)."""
    import torch as t
    stream = t.cuda.Stream(device=device)
    out = time_vmm(args, device, stream)
    out["put_bucket_transport"] = time_transport(args, device, stream)
    out["mr_lookup_overlap"] = time_mr_overlap(args, device, stream)
    out.update(time_mr_mutation(args, device, stream))
    out["cq_mirror"] = time_cq_mirror(args, device)
    return out


def time_vmm(args, device, stream, only=None) -> dict:
    """db_wqe_bucket_vmm on the put batch over 2 MiB chunks, without and with
    packet sequence numbers (mtu 4096)."""
    import torch as t
    import descriptor_build_gb300 as db
    import synth
    P = synth.put_bucket_vmm()
    d64 = lambda a: t.from_numpy(np.ascontiguousarray(a).view(np.int64)).to(device)
    d32 = lambda a: t.from_numpy(np.ascontiguousarray(a).view(np.int32)).to(device)
    R = P["world"] * P["n_qp"]
    n = P["req"].shape[0]
    b = dict(req=d64(P["req"]), raddr=d64(P["chunk_raddr"]), rkey=d32(P["chunk_rkey"]),
             lkey=d32(P["chunk_lkey"]),
             rings=t.empty((R, P["depth"], 64), dtype=t.uint8, device=device),
             head=d64(P["head"]), count=t.empty(R, dtype=t.int32, device=device),
             ctr=t.zeros(4, dtype=t.int64, device=device),
             psn=t.zeros(R, dtype=t.int64, device=device),
             ws=db.workspace(db.wqe_vmm_workspace_size(n, P["world"], P["n_qp"],
                                                       P["heap_size"], P["chunk_shift"]), device))
    out = {}
    for name, mtu in (("put_bucket_vmm", 0), ("put_bucket_vmm_psn", 4096)):
        if only and name != only:
            continue

        def call():
            db.wqe_bucket_vmm(b["req"], b["raddr"], b["rkey"], b["lkey"], P["chunk_shift"],
                              P["world"], P["n_qp"], P["local_base"], P["heap_size"], b["rings"],
                              P["depth"], b["head"], b["count"], b["ws"], ctr=b["ctr"],
                              stream=stream, mtu=mtu, psn_head=b["psn"] if mtu else None)

        for _ in range(args.warmup):
            call()
        t.cuda.synchronize(device)
        evs = [(t.cuda.Event(enable_timing=True), t.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        for a, z in evs:
            a.record(stream)
            call()
            z.record(stream)
        t.cuda.synchronize(device)
        ms = statistics.mean(a.elapsed_time(z) for a, z in evs)
        wqes = int(b["ctr"][0].item())
        if int(b["ctr"][3].item()):
            raise RuntimeError(f"{name}: device error bits")
        n_chunks = P["chunk_lkey"].shape[0]
        alg = 16 * n + 64 * wqes + P["world"] * n_chunks * 12 + n_chunks * 4
        peak, peak_kind = peak_gbs()
        gbs = alg / (ms * 1e-3) / 1e9
        out[name] = {
            "ms": round(ms, 4), "M_req_per_s": round(n / ms / 1e3, 2), "wqes": wqes,
            "chunk_bytes": 1 << P["chunk_shift"], "mtu": mtu, "algorithmic_bytes": alg,
            "GB_per_s": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4), "launches": 4,
            "note": "not part of the step: timed alone, same stream discipline"}
    return out


def time_transport(args, device, stream) -> dict:
    """db_wqe_bucket_transport on the put batch with PEs 1 and 2 on P2P: RDMA
    puts into the rings, the others as direct records."""
    import torch as t
    import descriptor_build_gb300 as db
    import synth
    P = synth.put_bucket_transport()
    d64 = lambda a: t.from_numpy(np.ascontiguousarray(a).view(np.int64)).to(device)
    d32 = lambda a: t.from_numpy(np.ascontiguousarray(a).view(np.int32)).to(device)
    R = P["world"] * P["n_qp"]
    n = P["req"].shape[0]
    b = dict(req=d64(P["req"]), peer=d64(P["peer_ptrs"]), rkeys=d32(P["rkeys"]),
             transport=t.from_numpy(P["transport"]).to(device),
             rings=t.empty((R, P["depth"], 64), dtype=t.uint8, device=device),
             head=d64(P["head"]), count=t.empty(R, dtype=t.int32, device=device),
             direct=t.empty((n, 32), dtype=t.uint8, device=device),
             n_direct=t.zeros(1, dtype=t.int64, device=device),
             ctr=t.zeros(4, dtype=t.int64, device=device),
             ws=db.workspace(db.wqe_workspace_size(n, R), device))

    def call():
        db.wqe_bucket_transport(b["req"], b["peer"], b["rkeys"], b["transport"], P["world"],
                                P["n_qp"], P["local_base"], P["lkey"], P["heap_size"],
                                b["rings"], P["depth"], b["head"], b["count"], b["direct"],
                                b["n_direct"], b["ws"], ctr=b["ctr"], stream=stream)

    ms = _event_ms(t, stream, call, args.warmup, args.steps)
    if int(b["ctr"][3].item()):
        raise RuntimeError("put_bucket_transport: device error bits")
    wqes, nd = int(b["ctr"][0].item()), int(b["n_direct"].item())
    alg = 16 * n + 64 * wqes + 32 * nd
    peak, _ = peak_gbs()
    gbs = alg / (ms * 1e-3) / 1e9
    return {"ms": round(ms, 4), "M_req_per_s": round(n / ms / 1e3, 2), "wqes": wqes,
            "direct": nd, "p2p_pes": [int(x) for x in np.flatnonzero(P["transport"] == 1)],
            "algorithmic_bytes": alg, "GB_per_s": round(gbs, 1),
            "frac_of_peak": round(gbs / peak, 4), "launches": 3,
            "note": "not part of the step: timed alone, same stream discipline"}


def _event_ms(t, stream, call, warmup, steps) -> float:
    for _ in range(warmup):
        call()
    t.cuda.synchronize()
    evs = [(t.cuda.Event(enable_timing=True), t.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for a, z in evs:
        a.record(stream)
        call()
        z.record(stream)
    t.cuda.synchronize()
    return statistics.mean(a.elapsed_time(z) for a, z in evs)


def time_mr_mutation(args, device, stream, only=None) -> dict:
    """db_mr_register on the mr_lookup table and queries taken as a
    registration batch (16,777,216 requests, 1,048,576 records, a fifth of
    the requests missing), and db_mr_deregister of 2,097,152 handles.
    Algorithmic bytes: per request 16 B range + 4 B new lkey in, 8 B handle
    + 1 B kind out; per record 24 B in and 24 B + 8 B remap out (registration
    also writes 24 B per new record); per handle 8 B in, 1 B out."""
    import torch as t
    import descriptor_build_gb300 as db
    import synth
    d64 = lambda a: t.from_numpy(np.ascontiguousarray(a).view(np.int64)).to(device)
    d32 = lambda a: t.from_numpy(np.ascontiguousarray(a).view(np.int32)).to(device)
    peak, _ = peak_gbs()
    out = {}
    if only == "mr_deregister":
        return _time_dereg(args, device, stream, db, synth, t, d64, d32, peak)
    r = synth.mr_register()
    nq, n = r["queries"].shape[0], r["mr_start"].shape[0]
    cap = n + nq
    rb = dict(q=d64(r["queries"]), nl=d32(r["new_lkey"]), s=d64(r["mr_start"]),
              e=d64(r["mr_end"]), lk=d32(r["mr_lkey"]), refs=d32(r["mr_refs"]),
              os=t.empty(cap, dtype=t.int64, device=device),
              oe=t.empty(cap, dtype=t.int64, device=device),
              olk=t.empty(cap, dtype=t.int32, device=device),
              orefs=t.empty(cap, dtype=t.int32, device=device),
              h=t.empty(nq, dtype=t.int64, device=device),
              k=t.empty(nq, dtype=t.uint8, device=device),
              remap=t.empty(n, dtype=t.int64, device=device),
              ctr=t.zeros(4, dtype=t.int64, device=device),
              ws=db.workspace(db.mr_register_workspace_size(nq, n), device))
    del r

    def reg():
        db.mr_register(rb["q"], rb["nl"], rb["s"], rb["e"], rb["lk"], rb["refs"], rb["os"],
                       rb["oe"], rb["olk"], rb["orefs"], rb["h"], rb["k"], rb["remap"], rb["ws"],
                       ctr=rb["ctr"], stream=stream)

    ms = _event_ms(t, stream, reg, args.warmup, args.steps)
    c = rb["ctr"].cpu().tolist()
    if c[2] or c[3]:
        raise RuntimeError(f"mr_register: counters {c}")
    u = c[0] - n
    alg = 29 * nq + 56 * n + 24 * u
    gbs = alg / (ms * 1e-3) / 1e9
    out["mr_register"] = {"ms": round(ms, 4), "M_req_per_s": round(nq / ms / 1e3, 2),
                          "records_before": n, "new_records": u, "algorithmic_bytes": alg,
                          "GB_per_s": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4),
                          "note": "not part of the step: timed alone; the requests' one-at-a-time "
                                  "result: lookup, one radix sort of the misses on a packed "
                                  "(start, length) key, two dominance passes (merge sorts on the "
                                  "end), merge; 153 launches, each a programmatic dependent of "
                                  "the one before"}
    del rb
    if only == "mr_register":
        return out
    return {**out, **_time_dereg(args, device, stream, db, synth, t, d64, d32, peak)}


def _time_dereg(args, device, stream, db, synth, t, d64, d32, peak) -> dict:
    g = synth.mr_deregister()
    nh, n = g["handles"].shape[0], g["mr_start"].shape[0]
    db_ = dict(hd=t.from_numpy(g["handles"]).to(device), s=d64(g["mr_start"]),
               e=d64(g["mr_end"]), lk=d32(g["mr_lkey"]), refs=d32(g["mr_refs"]),
               os=t.empty(n, dtype=t.int64, device=device),
               oe=t.empty(n, dtype=t.int64, device=device),
               olk=t.empty(n, dtype=t.int32, device=device),
               orefs=t.empty(n, dtype=t.int32, device=device),
               remap=t.empty(n, dtype=t.int64, device=device),
               st=t.empty(nh, dtype=t.uint8, device=device),
               ctr=t.zeros(4, dtype=t.int64, device=device),
               ws=db.workspace(db.mr_deregister_workspace_size(nh, n), device))

    def dereg():
        db.mr_deregister(db_["hd"], db_["s"], db_["e"], db_["lk"], db_["refs"], db_["os"],
                         db_["oe"], db_["olk"], db_["orefs"], db_["remap"], db_["st"], db_["ws"],
                         ctr=db_["ctr"], stream=stream)

    ms = _event_ms(t, stream, dereg, args.warmup, args.steps)
    c = db_["ctr"].cpu().tolist()
    alg = 9 * nh + 56 * n
    gbs = alg / (ms * 1e-3) / 1e9
    return {"mr_deregister": {"ms": round(ms, 4), "M_handles_per_s": round(nh / ms / 1e3, 2),
                            "records_before": n, "records_after": c[0], "stale": c[1],
                            "algorithmic_bytes": alg, "GB_per_s": round(gbs, 1),
                            "frac_of_peak": round(gbs / peak, 4),
                            "note": "not part of the step: timed alone; per-record counts, "
                                    "buckets of the contested records, statuses, "
                                    "compaction"}}


def time_cq_mirror(args, device) -> dict:
    """db_cq_mirror with the host standing in for a controller.

    drain: 64 queues of 4,096 entries, each with 4,095 completions already in
    its device CQ; the time from attaching the queues (the kernel running)
    until the kernel has copied all of them, averaged over --steps rounds.
    qd1: one queue, one completion at a time: the round trip from the host
    issuing the completion's two copies into the device CQ until its host CQ
    shows the new phase tag, median over 2,000 completions; beside it the
    same round trip with a copy engine (a 16-byte device-to-host copy queued
    after the write) doing the mirror's job. The queue is timed
    (DB_CQ_TIMED), so the slot also gives each completion's latency on the
    device: from the warp reading its new phase tag to its host-CQ writes
    being performed at system scope.
    Every copied entry is checked against what was written."""
    import torch as t
    import descriptor_build_gb300 as db
    PHASE = np.uint32(1 << 16)
    depth, nq, k = 4096, 64, 4095
    rng = np.random.default_rng(0xC0FFEE)
    copy_s, mir_s = t.cuda.Stream(device=device), t.cuda.Stream(device=device)
    slots = db.cq_slots(nq)
    f = db.cq_slot_fields(slots)
    stop = t.zeros(1, dtype=t.int32).pin_memory()
    ctr = t.zeros(4, dtype=t.int64, device=device)
    devs = [t.zeros((depth, 4), dtype=t.int32, device=device) for _ in range(nq)]
    hosts = [t.zeros((depth, 4), dtype=t.int32).pin_memory() for _ in range(nq)]
    body = rng.integers(0, 2**32, size=(nq, depth, 4), dtype=np.uint64).astype(np.uint32)
    body[:, :, 3] |= PHASE                       # first pass: tag 1
    stage = t.from_numpy(body.view(np.int32)).pin_memory()
    one_old = t.zeros((depth, 4), dtype=t.int32).pin_memory()
    one_new = t.zeros((depth, 4), dtype=t.int32).pin_memory()
    t.cuda.synchronize(device)
    db.cq_mirror(slots, stop, 20.0, ctr=ctr, stream=mir_s)
    rates, total = [], 0
    try:
        for rep in range(args.warmup + args.steps):
            if rep:
                gens = [db.cq_detach(slots, i) for i in range(nq)]
                if not all(db.cq_wait_ack(slots, i, g, 5.0) for i, g in enumerate(gens)):
                    raise RuntimeError("cq_mirror: no acknowledgement")
            with t.cuda.stream(copy_s):
                for i in range(nq):
                    devs[i].zero_()
                    hosts[i].zero_()
                    devs[i][:k].copy_(stage[i, :k], non_blocking=True)
            copy_s.synchronize()
            t0 = time.perf_counter()
            gnew = np.array([db.cq_attach(slots, i, devs[i], hosts[i]) for i in range(nq)])
            # a warp writes copied = 0 before it publishes the generation it took up
            while (not ((f["seen"] == gnew) & (f["copied"] == k)).all()
                   and time.perf_counter() - t0 < 5.0):
                pass
            dt = time.perf_counter() - t0
            for i in range(nq):
                got, _, _ = db.cq_host_reap(hosts[i], 0, 1)
                if got.shape[0] != k or not (got == body[i, :k]).all():
                    raise RuntimeError("cq_mirror: host CQ differs from the device CQ")
            total += nq * k
            if rep >= args.warmup:
                rates.append(nq * k / dt)
        # QD1 on queue 0: host issues one completion, polls its host CQ until
        # the tag shows. The same round trip with a copy engine in place of
        # the mirror (a 16-byte device-to-host copy queued after the write)
        # is timed beside it, on an unattached queue pair.
        gens = [db.cq_detach(slots, i) for i in range(nq)]
        if not all(db.cq_wait_ack(slots, i, g, 5.0) for i, g in enumerate(gens)):
            raise RuntimeError("cq_mirror: no acknowledgement")
        d, h, d2, h2 = devs[0], hosts[0], devs[1], hosts[1]
        with t.cuda.stream(copy_s):
            d.zero_()
            d2.zero_()
        h.zero_()
        h2.zero_()
        copy_s.synchronize()
        f["flags"][0] = db.CQ_TIMED  # the kernel records each batch's latency in the slot
        db.cq_attach(slots, 0, d, h)
        ov, nv = one_old.numpy().view(np.uint32), one_new.numpy().view(np.uint32)
        rts = {"mirror": [], "copy_engine": []}
        dev_lat = []
        for i in range(4000):
            leg = "mirror" if i % 2 == 0 else "copy_engine"
            j = i // 2
            pos, tag = j % depth, np.uint32(1 - (j // depth) % 2)
            dq, hq = (d, h) if leg == "mirror" else (d2, h2)
            hv = hq.numpy().view(np.uint32)
            e = rng.integers(0, 2**32, size=4, dtype=np.uint64).astype(np.uint32)
            e[3] = (e[3] & ~PHASE) | (tag << np.uint32(16))
            nv[pos] = e
            ov[pos] = e
            ov[pos, 3] ^= PHASE
            want = tag << np.uint32(16)
            ta = time.perf_counter()
            with t.cuda.stream(copy_s):
                dq[pos:pos + 1].copy_(one_old[pos:pos + 1], non_blocking=True)
                dq[pos:pos + 1].copy_(one_new[pos:pos + 1], non_blocking=True)
                if leg == "copy_engine":
                    hq[pos:pos + 1].copy_(dq[pos:pos + 1], non_blocking=True)
            while (hv[pos, 3] & PHASE) != want and time.perf_counter() - ta < 1.0:
                pass
            tc = time.perf_counter()
            copy_s.synchronize()
            got, _, _ = db.cq_host_reap(hq, pos, int(tag), max_entries=1)
            if got.shape[0] != 1 or not (got[0] == e).all():
                raise RuntimeError(f"cq_mirror: QD1 entry differs ({leg})")
            total += leg == "mirror"
            rts[leg].append(tc - ta)
            if leg == "mirror":
                tl = time.perf_counter()
                while int(f["lat_seq"][0]) != j + 1 and time.perf_counter() - tl < 1.0:
                    pass
                if int(f["lat_seq"][0]) != j + 1:
                    raise RuntimeError("cq_mirror: no latency record")
                dev_lat.append(int(f["lat_ns"][0]))
        g = db.cq_detach(slots, 0)
        db.cq_wait_ack(slots, 0, g, 5.0)
    finally:
        db.cq_request_stop(stop)
        mir_s.synchronize()
    c = ctr.cpu().numpy()
    if int(c[0]) != total or int(c[3]):
        raise RuntimeError(f"cq_mirror: counters {c.tolist()}, expected {total} copied")
    rate = statistics.mean(rates)
    return {"drain_M_cqe_per_s": round(rate / 1e6, 3), "queues": nq, "depth": depth,
            "cqes_per_round": nq * k,
            "ns_per_cqe_per_queue": round(nq / rate * 1e9, 1),
            "qd1_roundtrip_us_median": round(statistics.median(rts["mirror"]) * 1e6, 2),
            "qd1_roundtrip_us_copy_engine_median":
                round(statistics.median(rts["copy_engine"]) * 1e6, 2),
            "qd1_device_latency_us_median": round(statistics.median(dev_lat) / 1e3, 3),
            "qd1_device_latency_us_p99": round(float(np.percentile(dev_lat, 99)) / 1e3, 3),
            "device_latency": "per completion at queue depth 1, %globaltimer on the GPU: the "
                              "warp reads the new phase tag -> its host-CQ writes performed at "
                              "system scope (slot lat_ns, DB_CQ_TIMED)",
            "launches": 1, "bound": "latency: device CQ to host CQ over the CPU-GPU link",
            "note": "not part of the step: the host writes the device CQs (two stream-ordered "
                    "copies per batch) and polls host memory; times are host wall clock, "
                    "round trips include the host's copy issue and polling"}


def time_mr_overlap(args, device, stream) -> dict:
    """db_mr_lookup_overlap on a registration table whose records overlap
    (1,048,576 disjoint records plus 262,144 straddling ones), 16,777,216
    queries; algorithmic bytes as for mr_lookup."""
    import torch as t
    import descriptor_build_gb300 as db
    import synth
    m = synth.mr_lookup_overlap()
    d64 = lambda a: t.from_numpy(np.ascontiguousarray(a).view(np.int64)).to(device)
    d32 = lambda a: t.from_numpy(np.ascontiguousarray(a).view(np.int32)).to(device)
    nq, nr = m["queries"].shape[0], m["mr_start"].shape[0]
    b = dict(q=d64(m["queries"]), start=d64(m["mr_start"]), end=d64(m["mr_end"]),
             lkey=d32(m["mr_lkey"]), idx=t.empty(nq, dtype=t.int32, device=device),
             olkey=t.empty(nq, dtype=t.int32, device=device),
             kind=t.empty(nq, dtype=t.uint8, device=device),
             ctr=t.zeros(4, dtype=t.int64, device=device),
             ws=db.workspace(db.mr_workspace_size(nr), device))

    def call():
        db.mr_lookup_overlap(b["q"], b["start"], b["end"], b["lkey"], b["idx"], b["olkey"],
                             b["kind"], b["ws"], ctr=b["ctr"], stream=stream)

    for _ in range(args.warmup):
        call()
    t.cuda.synchronize(device)
    evs = [(t.cuda.Event(enable_timing=True), t.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    for a, z in evs:
        a.record(stream)
        call()
        z.record(stream)
    t.cuda.synchronize(device)
    ms = statistics.mean(a.elapsed_time(z) for a, z in evs)
    if int(b["ctr"][3].item()):
        raise RuntimeError("mr_lookup_overlap: device error bits")
    alg = 25 * nq + 20 * nr
    peak, _ = peak_gbs()
    gbs = alg / (ms * 1e-3) / 1e9
    return {"ms": round(ms, 4), "M_req_per_s": round(nq / ms / 1e3, 2), "records": nr,
            "hits": int(b["ctr"][0].item()), "algorithmic_bytes": alg,
            "GB_per_s": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4), "launches": 5,
            "note": "not part of the step: timed alone, same stream discipline"}


def run_ours(args, inp, world, device, dist):
    import torch
    import descriptor_build_gb300 as db

    torch.cuda.set_device(device)
    st = Step(db, torch, inp, device, args.prp_sched)
    stream = torch.cuda.Stream(device=device)
    ev = lambda: torch.cuda.Event(enable_timing=True)
    # The four calls are independent batches with their own buffers and
    # workspaces: each runs on its own stream and a step forks them together
    # and joins them (the MR lookup, bound by L2 requests, and the latency-bound
    # small PRP batch overlap the HBM-bound ones). --serial runs them in turn.
    calls = st.calls()
    if not args.serial:
        rank_of = {k: i for i, k in enumerate(SCHEDULE)}
        calls = sorted(calls, key=lambda c: rank_of[c[0]])
    streams = [stream if args.serial else torch.cuda.Stream(device=device) for _ in calls]

    def one_step(call_ev, fork, join):
        fork.record(stream)
        for j, (_, fn) in enumerate(calls):
            s = streams[j]
            if s is not stream:
                s.wait_event(fork)
            call_ev[j][0].record(s)
            fn(s)
            call_ev[j][1].record(s)
        for j in range(len(calls)):
            if streams[j] is not stream:
                stream.wait_event(call_ev[j][1])
        join.record(stream)

    for _ in range(args.warmup):
        one_step([(ev(), ev()) for _ in calls], ev(), ev())
    torch.cuda.synchronize(device)
    st.check_counters()

    K = args.steps
    evs = [[(ev(), ev()) for _ in calls] for _ in range(K)]
    step_ev = [(ev(), ev()) for _ in range(K)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize(device)
    with Clocks(smi_index(device)) as clk:
        t0 = ev()
        t1 = ev()
        t0.record(stream)
        for k in range(K):
            one_step(evs[k], step_ev[k][0], step_ev[k][1])
        t1.record(stream)
        torch.cuda.synchronize(device)
    total_ms = max_over_ranks(dist, t0.elapsed_time(t1), device)
    if dist:
        dist.barrier()
    st.check_counters()
    span_ms = {name: statistics.mean(evs[k][j][0].elapsed_time(evs[k][j][1]) for k in range(K))
               for j, (name, _) in enumerate(calls)}
    if args.serial:
        per_kernel_ms = span_ms
    else:
        # A concurrent call's span includes waiting for SMs the others hold, so
        # each call's own time comes from the same steps run one call at a time.
        sev = [[(ev(), ev()) for _ in calls] for _ in range(K)]
        torch.cuda.synchronize(device)
        for k in range(K):
            for j, (_, fn) in enumerate(calls):
                sev[k][j][0].record(stream)
                fn(stream)
                sev[k][j][1].record(stream)
        torch.cuda.synchronize(device)
        st.check_counters()
        per_kernel_ms = {name: statistics.mean(sev[k][j][0].elapsed_time(sev[k][j][1])
                                               for k in range(K))
                         for j, (name, _) in enumerate(calls)}

    u = units(inp)
    alg = algorithmic_bytes(inp)
    outb = output_bytes(inp)
    peak, peak_kind = peak_gbs()
    copy_ms = size_matched_copy_ms(torch, [n for n, _ in calls], alg, K, stream, device)
    reqs_per_step = sum(u.values())
    ms_per_step = total_ms / K
    value = job_throughput(world, reqs_per_step, ms_per_step)
    kernels = {}
    for name in u:
        ms = per_kernel_ms[name]
        gbs = alg[name] / (ms * 1e-3) / 1e9
        kernels[name] = {"ms": round(ms, 4), "M_req_per_s": round(u[name] / ms / 1e3, 2),
                         "algorithmic_bytes": alg[name], "GB_per_s": round(gbs, 1),
                         "frac_of_peak": round(gbs / peak, 4),
                         "output_bytes": outb[name],
                         "output_GB_per_s": round(outb[name] / (ms * 1e-3) / 1e9, 1),
                         "launches": st.launches(name),
                         "size_matched_copy_ms": round(copy_ms[name], 4),
                         "frac_of_size_matched_copy": round(copy_ms[name] / ms, 4)}
        if not args.serial:
            kernels[name]["concurrent_span_ms"] = round(span_ms[name], 4)
    for name in kernels:
        rec = recorded_traffic(name) if args.fraction >= 1.0 else None
        kernels[name]["traffic"] = rec["dram_bytes_per_call"] if rec else None
        kernels[name]["traffic_over_algorithmic"] = rec["traffic_over_algorithmic"] if rec else None
        kernels[name]["l2_sectors_per_request"] = rec["l2_sectors_per_request"] if rec else None
        kernels[name]["l2_requests_per_request"] = rec["l2_requests_per_request"] if rec else None
    dom = max(kernels, key=lambda k: kernels[k]["ms"])
    names = {"prp_small": "prp_pairs_kernel + prp_build_kernel<true>",
             "prp_large": "prp_build_kernel<false>",
             "mr_lookup": "mr_index_kernel + mr_lookup_kernel",
             "put_bucket": "wqe_count_kernel + wqe_scan_kernel + wqe_scatter_kernel"}
    roof = {"bound": "hbm", "kernel": names.get(dom, dom),
            "workload": dom, "achieved": kernels[dom]["GB_per_s"], "peak": peak,
            "peak_source": peak_kind, "unit": "GB/s",
            "frac": round(kernels[dom]["GB_per_s"] / peak, 4), "traffic": kernels[dom]["traffic"],
            "algorithmic_bytes_per_launch": alg[dom],
            # every call of the step, timed alone (the same figures as `kernels`)
            "calls": {n: {"ms": k["ms"], "GB_per_s": k["GB_per_s"], "frac": k["frac_of_peak"],
                          "frac_of_size_matched_copy": k["frac_of_size_matched_copy"],
                          "traffic": k["traffic"],
                          "traffic_over_algorithmic": k["traffic_over_algorithmic"],
                          "l2_sectors_per_request": k["l2_sectors_per_request"]}
                      for n, k in kernels.items()}}
    if not args.only and args.fraction >= 1.0:
        c1 = time_tiny(args, device)
        kernels["c1_tiny"] = c1
        roof["calls"]["c1_tiny"] = {"prp_us": c1["prp_us"], "mr_lookup_us": c1["mr_lookup_us"]}

    out = {"metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
           "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u64",
           "data": "synthetic (seeded generators of the five study workloads)",
           "config": workload_config(u, world, args.serial),
           "output_GB_per_s": round(world * sum(outb.values()) / (ms_per_step * 1e-3) / 1e9, 1),
           "kernels": kernels, "roofline": roof,
           "gpu_launches": K * sum(st.launches(k) for k in u),  # in the timed region
           "clocks": clk.summary()}
    if not args.no_e2e:
        out["e2e"] = run_e2e(st, stream, inp, max(3, min(K, 5)), device, dist, world,
                             serial=args.serial)
    return out


def workload_config(u: dict, world: int, serial: bool) -> dict:
    """The `config` of a bench line; both arms print the same one."""
    order = [n for n in SCHEDULE if n in u]
    return {"workload": WORKLOAD, "requests_per_step": sum(u.values()),
            "per_workload_requests": u,
            "l2": "inputs larger than L2: each step streams ~6 GB, so every "
                  "kernel's inputs are evicted before its next launch",
            "parallelism": f"replicas x{world}",
            "schedule": ("one stream, the four calls in turn" if serial else
                         "four streams, forked and joined each step; launch order "
                         + ", ".join(order)
                         + "; per-call times and the roofline from the same steps "
                           "run one call at a time after the timed region")}


def time_tiny(args, device) -> dict:
    """Latency of the tiny workload (4,096 requests): the PRP build and the
    lookup of the same ranges against its 64-record table, each call timed
    alone with CUDA events after an L2 flush, mean of 50 calls."""
    import torch as t
    import descriptor_build_gb300 as db
    import synth
    w = synth.prp_tiny()
    n = w["req"].shape[0]
    d64 = lambda a: t.from_numpy(np.ascontiguousarray(a).view(np.int64)).to(device)
    req, lut = d64(w["req"]), d64(w["lut"])
    prp = t.empty((n, 2), dtype=t.int64, device=device)
    ctr = t.zeros(4, dtype=t.int64, device=device)
    ws = db.workspace(db.prp_workspace_size(n), device)
    stream = t.cuda.Stream(device=device)
    db.prp_build(req, lut, w["heap_size"], w["arena_base"], 0, None, prp, ws, ctr=ctr,
                 stream=stream)
    stream.synchronize()
    cap = int(ctr[0].item())
    arena = t.empty((max(cap, 1), 512), dtype=t.int64, device=device)
    q, ms_, me = d64(w["queries"]), d64(w["mr_start"]), d64(w["mr_end"])
    mk = t.from_numpy(w["mr_lkey"].view(np.int32)).to(device)
    idx = t.empty(n, dtype=t.int32, device=device)
    lk = t.empty(n, dtype=t.int32, device=device)
    kind = t.empty(n, dtype=t.uint8, device=device)
    mws = db.workspace(db.mr_workspace_size(w["mr_start"].shape[0]), device)
    flush = t.empty(256 << 20, dtype=t.uint8, device=device)
    calls = {"prp_us": lambda: db.prp_build(req, lut, w["heap_size"], w["arena_base"], cap, arena,
                                            prp, ws, ctr=ctr, stream=stream),
             "mr_lookup_us": lambda: db.mr_lookup(q, ms_, me, mk, idx, lk, kind, mws,
                                                  stream=stream)}
    res = {}
    for name, fn in calls.items():
        evs = []
        with t.cuda.stream(stream):
            for r in range(55):
                flush.fill_(r & 0xFF)
                a, b = t.cuda.Event(enable_timing=True), t.cuda.Event(enable_timing=True)
                a.record(stream)
                fn()
                b.record(stream)
                if r >= 5:
                    evs.append((a, b))
        stream.synchronize()
        res[name] = round(1000 * statistics.mean(a.elapsed_time(b) for a, b in evs), 2)
    assert int(ctr[3].item()) == 0 and int(ctr[0].item()) == cap
    return {"requests": n, "mr_records": int(w["mr_start"].shape[0]), **res,
            "note": "latency of one call, inputs resident; CUDA event intervals come in steps "
                    "of about 2 us here, so these are means of 50 calls"}


def size_matched_copy_ms(torch, names, alg, K, stream, device) -> dict:
    """Per workload, the mean time of a plain device copy that moves the same
    algorithmic bytes (half read, half written), timed like the calls: CUDA
    events on the launching stream, the workloads' copies in the step's order
    so that each one starts with the others' data in L2. A kernel cannot move
    its bytes faster than such a copy, and for small batches the copy itself is
    far below the peak copy rate (launch and DRAM latency dominate), so the
    ratio says how close a call is to the HBM bound at its own size."""
    half = {n: (alg[n] // 2 + 255) & ~255 for n in names}
    off, o = {}, 0
    for n in names:  # disjoint regions: no copy finds another's lines in L2
        off[n] = o
        o += half[n]
    src = torch.empty(o, dtype=torch.uint8, device=device)
    dst = torch.empty_like(src)
    src.fill_(1)
    view = lambda b, n: b[off[n]: off[n] + half[n]]
    ev = lambda: torch.cuda.Event(enable_timing=True)
    t = {n: [] for n in names}
    with torch.cuda.stream(stream):
        for _ in range(2):  # warm-up
            for n in names:
                view(dst, n).copy_(view(src, n))
        pairs = []
        for _ in range(K):
            for n in names:
                e0, e1 = ev(), ev()
                e0.record(stream)
                view(dst, n).copy_(view(src, n))
                e1.record(stream)
                pairs.append((n, e0, e1))
    torch.cuda.synchronize(device)
    for n, e0, e1 in pairs:
        t[n].append(e0.elapsed_time(e1))
    del src, dst
    return {n: statistics.mean(v) for n, v in t.items()}


def run_e2e(st, stream, inp, K, device, dist, world, serial=False):
    """The same step through the API with host buffers: pinned host inputs are
    copied in, every descriptor the step produces ends in host memory. The
    PRP lists are written by the kernel straight into a pinned host arena
    (the host-memory list region of the source page), so only the words a
    list holds cross the link; everything else is copied back. Each workload
    runs on its own stream (copy in, call, copy out), the four forked together
    as in the device-resident step; an output above 1 GiB is copied back in
    four pieces on streams of their own, so that more than one copy engine
    moves it."""
    import torch
    t = torch
    pin = lambda a: t.from_numpy(np.ascontiguousarray(a).view(np.int64)).pin_memory()
    pin32 = lambda a: t.from_numpy(np.ascontiguousarray(a).view(np.int32)).pin_memory()
    groups, host_calls = {}, {}
    list_bytes = 0
    alg = algorithmic_bytes(inp)
    for k in ("prp_small", "prp_large"):
        if k in st.bufs:
            b, w = st.bufs[k], inp[k]
            groups[k] = ([(pin(w["req"]), b["req"]), (pin(w["lut"]), b["lut"])],
                         [b["prp"], b["ctr"]])
            if b["cap"]:
                hb = dict(b, arena=t.empty((b["cap"], 512), dtype=t.int64, pin_memory=True))
                host_calls[k] = (lambda hb: lambda s_: st.prp(hb, s_))(hb)
                # list words the kernel writes into host memory (algorithmic
                # bytes less the 16-byte request and 16-byte PRP pair)
                list_bytes += alg[k] - 32 * w["req"].shape[0] - w["lut"].shape[0] * 8
    if "mr_lookup" in st.bufs:
        b, m = st.bufs["mr_lookup"], inp["mr_lookup"]
        groups["mr_lookup"] = ([(pin(m["queries"]), b["q"]), (pin(m["mr_start"]), b["start"]),
                                (pin(m["mr_end"]), b["end"]), (pin32(m["mr_lkey"]), b["lkey"])],
                               [b["idx"], b["olkey"], b["kind"], b["ctr"]])
    if "put_bucket" in st.bufs:
        b, p = st.bufs["put_bucket"], inp["put_bucket"]
        groups["put_bucket"] = ([(pin(p["req"]), b["req"]), (pin(p["peer_ptrs"]), b["peer"]),
                                 (pin32(p["rkeys"]), b["rkeys"])],
                                [b["rings"], b["head"], b["count"], b["ctr"]])
    h_out = {k: [t.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outs]
             for k, (_, outs) in groups.items()}
    bi = sum(h.numel() * h.element_size() for h_in, _ in groups.values() for h, _ in h_in)
    bo = sum(o.numel() * o.element_size() for _, outs in groups.values() for o in outs)
    calls = dict(st.calls())
    calls.update(host_calls)
    order = [k for k in SCHEDULE if k in groups]
    streams = {k: (stream if serial else t.cuda.Stream(device=device)) for k in order}
    pieces = [t.cuda.Stream(device=device) for _ in range(4)]
    big = 1 << 30

    def one():
        fork = t.cuda.Event()
        fork.record(stream)
        done = []
        for k in order:
            s = streams[k]
            if s is not stream:
                s.wait_event(fork)
            with t.cuda.stream(s):
                for h, d in groups[k][0]:
                    d.copy_(h, non_blocking=True)
                calls[k](s)
                for o, h in zip(groups[k][1], h_out[k]):
                    n = o.numel() * o.element_size()
                    if n < big or serial:
                        h.copy_(o, non_blocking=True)
                        continue
                    ready = t.cuda.Event()
                    ready.record(s)
                    rows = o.shape[0]
                    for i, ps in enumerate(pieces):
                        lo, hi = rows * i // len(pieces), rows * (i + 1) // len(pieces)
                        ps.wait_event(ready)
                        with t.cuda.stream(ps):
                            h[lo:hi].copy_(o[lo:hi], non_blocking=True)
                        e = t.cuda.Event()
                        e.record(ps)
                        done.append(e)
            e = t.cuda.Event()
            e.record(s)
            done.append(e)
        for e in done:
            stream.wait_event(e)

    one()
    t.cuda.synchronize(device)
    if dist:
        dist.barrier()
    a, b = t.cuda.Event(enable_timing=True), t.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(K):
        one()
    b.record(stream)
    t.cuda.synchronize(device)
    ms = max_over_ranks(dist, a.elapsed_time(b) / K, device)
    reqs = sum(units(inp).values())
    return {"value": round(job_throughput(world, reqs, ms), 2), "unit": UNIT,
            "ms_per_step": round(ms, 3), "steps": K, "h2d_bytes_per_step": bi,
            "d2h_bytes_per_step": bo + list_bytes,
            "d2h_detail": {"copied_back": bo, "lists_written_to_host_arena": list_bytes}}


# ------------------------------------------------------------ CPU baseline
def cpu_baseline(inp, repeats: int = 3) -> dict:
    """The oracle as it stands (single-threaded C++) on a bounded sample of
    each workload: every request of prp_small, mr_lookup and put_bucket and
    the first 524,288 of prp_large (their lists, 2 GB, are written into a
    host arena), each timed `repeats` times (median); the value is one full
    step's requests over the time those rates give for it. Output buffers
    that scale with the ring or arena size are allocated outside the timed
    calls."""
    import oracle
    oracle.build()  # compiled (if need be) before anything is timed
    s, l, m, p = inp["prp_small"], inp["prp_large"], inp["mr_lookup"], inp["put_bucket"]
    u = units(inp)
    samples = {"prp_small": u["prp_small"], "prp_large": min(524_288, u["prp_large"]),
               "mr_lookup": u["mr_lookup"], "put_bucket": u["put_bucket"]}
    req = l["req"][:samples["prp_large"]]
    need = int(oracle.prp_build(req, l["lut"], l["heap_size"], l["arena_base"], 1 << 40,
                                lists=False)["ctr"][0])
    arena = np.zeros((need, 512), dtype=np.uint64)
    rings = np.zeros((p["world"] * p["n_qp"], p["depth"], 64), dtype=np.uint8)
    arena.fill(0)  # fault the pages in before the timed calls
    rings.fill(0)
    calls = {
        "prp_small": lambda: oracle.prp_build(s["req"][:samples["prp_small"]], s["lut"],
                                              s["heap_size"], s["arena_base"], 1, lists=False),
        "prp_large": lambda: oracle.prp_build(req, l["lut"], l["heap_size"], l["arena_base"],
                                              need, arena=arena),
        "mr_lookup": lambda: oracle.mr_bsearch(m["queries"][:samples["mr_lookup"]], m["mr_start"],
                                               m["mr_end"], m["mr_lkey"]),
        "put_bucket": lambda: oracle.wqe_bucket(p["req"][:samples["put_bucket"]], p["peer_ptrs"],
                                                p["rkeys"], p["world"], p["n_qp"], p["local_base"],
                                                p["lkey"], p["heap_size"], p["depth"], p["head"],
                                                rings=rings),
    }
    secs = {}
    for k, fn in calls.items():
        ts = []
        for _ in range(repeats):
            t = time.perf_counter()
            fn()
            ts.append(time.perf_counter() - t)
        secs[k] = statistics.median(ts)
    # Time for one full step's requests at the sampled per-request rates.
    step_s = sum(secs[k] * u[k] / samples[k] for k in u)
    return {"value": round(sum(u.values()) / step_s / 1e6, 3), "unit": UNIT, "cores": 1,
            **host_cpu(), "kind": "oracle",
            "sample": "all %d prp_small, the first %d prp_large (lists written), all %d "
                      "mr_lookup (binary-search oracle) and all %d put_bucket requests, each "
                      "timed %d times (median); per-workload rates scaled to one full step"
                      % (samples["prp_small"], samples["prp_large"], samples["mr_lookup"],
                         samples["put_bucket"], repeats),
            "seconds": {k: round(v, 4) for k, v in secs.items()}}


# ------------------------------------------------------------ reference arm
def run_reference(args):
    """The oracle as the reference arm: each step a bounded sample of the
    workload on the host cores, same metric and unit as our arm."""
    inp = make_inputs()
    for _ in range(args.warmup):
        cpu_baseline(inp, repeats=1)
    vals = []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        vals.append(cpu_baseline(inp, repeats=1))
    wall = time.perf_counter() - t0
    v = round(statistics.median(x["value"] for x in vals), 3)
    reqs = sum(units(inp).values())
    ms = reqs / (v * 1e6) * 1e3
    cb = dict(vals[0])
    cb["value"] = v
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u64",
            "data": "synthetic (seeded generators of the five study workloads)",
            "config": workload_config(units(inp), int(os.environ.get("WORLD_SIZE", "1")), False),
            "cpu_baseline": cb, "wall_s": round(wall, 2),
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    dist = None
    import torch
    local = int(os.environ.get("LOCAL_RANK", "0"))
    device = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(device)
        dist.init_process_group("nccl", device_id=device)
    if args.next_only:
        if rank == 0:
            import torch as t
            s = t.cuda.Stream(device=device)
            if args.next_only.startswith("put_bucket_vmm"):
                res = time_vmm(args, device, s, only=args.next_only)
            elif args.next_only == "mr_lookup_overlap":
                res = {"mr_lookup_overlap": time_mr_overlap(args, device, s)}
            elif args.next_only == "put_bucket_transport":
                res = {"put_bucket_transport": time_transport(args, device, s)}
            else:
                res = time_mr_mutation(args, device, s, only=args.next_only)
            print(json.dumps({"next_only": args.next_only, **res,
                              "note": "profiling aid: not a bench line"}), flush=True)
        return
    inp = make_inputs(args.only, args.fraction)
    out = run_ours(args, inp, world, device, dist)
    if rank == 0:
        if args.only or args.fraction < 1.0:
            out["note"] = "profiling run on a subset: not a bench line"
        if not args.no_cpu and not args.only and args.fraction >= 1.0:
            out["cpu_baseline"] = cpu_baseline(inp)
        if not args.only and args.fraction >= 1.0 and not args.no_next:
            out["next"] = run_next(args, device)
        print(json.dumps(out), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
