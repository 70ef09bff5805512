"""The pins must catch plausible mistakes in the oracle.

Each case plants one mistake in a copy of oracle.cpp (a dropped term, a wrong
index, an off-by-one, a transposed operand), builds it on the CPU, and runs
the oracle pin tests against it in a subprocess: they must fail.
"""

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.cpp")

MUTANTS = [
    ("prp2 drops the in-chunk offset",
     "prp[1] = bus_address(lut, n_lut, first_page + kPage);",
     "prp[1] = lut[(first_page + kPage) / kChunk];"),
    ("prp1 loses its in-page offset",
     "prp[0] = bus_address(lut, n_lut, off);",
     "prp[0] = bus_address(lut, n_lut, first_page);"),
    ("chain pointer names the current page",
     "arena_base + (page_base + page + 1) * kPage;",
     "arena_base + (page_base + page) * kPage;"),
    ("list page holds 512 data entries before chaining",
     "left -= kListSlots - 1;", "left -= kListSlots;"),
    ("page count off by one at the end",
     "uint64_t last = (off + len - 1) / kPage;", "uint64_t last = (off + len) / kPage;"),
    ("list used from two pages on",
     "if (n < 3) return 0;\n  return list_pages_for(n - 1);",
     "if (n < 2) return 0;\n  return list_pages_for(n - 1);"),
    ("list entries start at the first page",
     "bus_address(lut, n_lut, first_page + k * kPage);",
     "bus_address(lut, n_lut, first_page + (k - 1) * kPage);"),
    ("mr containment uses a strict end",
     "if (start[i] <= base && aend <= end[i]) {", "if (start[i] <= base && aend < end[i]) {"),
    ("mr rounding truncates the end",
     "uint64_t pages = (uint64_t)((stop - b + kPage - 1) / kPage);",
     "uint64_t pages = (uint64_t)((stop - b) / kPage);"),
    ("mr exact compares one end only",
     "kind[k] = (start[i] == base && end[i] == aend) ? 1 : 2;",
     "kind[k] = (start[i] == base) ? 1 : 2;"),
    ("mr prefix max: exact compares one end only",
     "const bool same_ends = start[i] == base && end[i] == aend;",
     "const bool same_ends = start[i] == base;"),
    ("mr prefix max searches past the last start at or below base",
     "std::lower_bound(pm.begin(), pm.begin() + cnt, aend)",
     "std::lower_bound(pm.begin(), pm.begin() + std::min<uint64_t>(cnt + 1, n_mr), aend)"),
    ("mr prefix max keeps each end alone",
     "pm[i] = i ? std::max(pm[i - 1], end[i]) : end[i];", "pm[i] = end[i];"),
    ("mr bsearch takes lower_bound",
     "std::upper_bound(start, start + n_mr, base);", "std::lower_bound(start, start + n_mr, base);"),
    ("wqe ring order is qp-major",
     "return (int)(f.pe * n_qp + f.qp);", "return (int)(f.qp * world + f.pe);"),
    ("wqe seq ignores the head",
     "uint64_t seq = head[r] + taken[r];", "uint64_t seq = taken[r];"),
    ("wqe rkey of the local PE",
     "put_u32(wqe + 24, rkeys[f.pe]);", "put_u32(wqe + 24, rkeys[0]);"),
    ("wqe ring full one early",
     "if (demand[r] > depth) {", "if (demand[r] >= depth) {"),
    ("wqe raddr from the local base",
     "put_u64(wqe + 0, peer_ptrs[f.pe] + f.off);", "put_u64(wqe + 0, local_base + f.off);"),
    ("vmm raddr adds the heap offset, not the chunk offset",
     "chunk_raddr[pe * n_chunks + dst_chunk] + (dst % C);",
     "chunk_raddr[pe * n_chunks + dst_chunk] + dst;"),
    ("vmm lkey of chunk 0",
     "const uint32_t lkey = chunk_lkey[src_chunk];", "const uint32_t lkey = chunk_lkey[0];"),
    ("vmm rkey of the PE's first chunk",
     "const uint32_t rkey = chunk_rkey[pe * n_chunks + dst_chunk];",
     "const uint32_t rkey = chunk_rkey[pe * n_chunks];"),
    ("vmm laddr does not advance per fragment",
     "put_u64(wqe + 8, local_base + src);", "put_u64(wqe + 8, local_base + off);"),
    ("psn counts round down",
     "if (mtu) psns += (t + mtu - 1) / mtu;", "if (mtu) psns += t / mtu;"),
    ("psn taken after its own WQE",
     "put_u32(wqe + 44, (uint32_t)(psn_head[r] + psn_taken[r]));  // first PSN\n        psn_taken[r] += (t + mtu - 1) / mtu;",
     "psn_taken[r] += (t + mtu - 1) / mtu;\n        put_u32(wqe + 44, (uint32_t)(psn_head[r] + psn_taken[r]));"),
    ("register: holder must start below the base, not at it",
     "const uint64_t starting = (uint64_t)(std::upper_bound(start, start + n, base) - start);",
     "const uint64_t starting = (uint64_t)(std::lower_bound(start, start + n, base) - start);"),
    ("register: prefix maximum of the ends restarts", "reach = std::max(reach, end[i]);",
     "reach = end[i];"),
    ("prp: tail slots cleared without the zero-tail option", "  if (zero_tail) {\n    for (; slot",
     "  if (true) {\n    for (; slot"),
    ("prp: zero tail stops one slot short", "for (; slot < kListSlots; ++slot)",
     "for (; slot + 1 < kListSlots; ++slot)"),
    ("transport: direct dst from the local base", "put_u64(d + 0, peer_ptrs[f.pe] + f.off);",
     "put_u64(d + 0, local_base + f.off);"),
    ("transport: direct src from the peer", "put_u64(d + 8, local_base + f.off);",
     "put_u64(d + 8, peer_ptrs[f.pe] + f.off);"),
    ("transport: direct puts counted in their ring", "ring_of[i] = -2;\n      continue;",
     "ring_of[i] = -2;\n      demand[ring_index(f, world, n_qp)] += 1;\n      continue;"),
    ("transport: unknown codes taken as RDMA", " || transport[f.pe] > 2) {", ") {"),
    ("transport: direct index counts descriptors", "put_u32(d + 20, (uint32_t)i);",
     "put_u32(d + 20, (uint32_t)nd);"),
    ("transport: SDMA puts become WQEs", "if (transport[f.pe] != 0) {",
     "if (transport[f.pe] == 1) {"),
    ("register: a hit takes no reference", "more[i] += 1;", "more[i] += 0;"),
    ("register: new record before an old one with the same start",
     "start[i] <= nit->first.first);", "start[i] < nit->first.first);"),
    ("register: new record keyed by the wrong request",
     "o_lkey[w] = new_lkey[nit->second.first];",
     "o_lkey[w] = new_lkey[nit->second.first + nit->second.second - 1];"),
    ("register: granule rounding drops the tail",
     "const uint64_t units = (uint64_t)((stop - b + g - 1) / g);",
     "const uint64_t units = (uint64_t)((stop - b) / g);"),
    ("register: repeats are not merged", "if (it == fresh.end()) {", "if (true) {"),
    ("register one at a time: insert before equal starts",
     "while (at < t.size() && t[at].s <= b) ++at;", "while (at < t.size() && t[at].s < b) ++at;"),
    ("register indexed: a created record beats an old one of equal start",
     "if (c < nc && (o < 0 || cand[c].first < start[o])) {",
     "if (c < nc && (o < 0 || cand[c].first <= start[o])) {"),
    ("register indexed: created holders may start past the base",
     "std::make_pair(b, UINT64_MAX)) -", "std::make_pair(b + g, UINT64_MAX)) -"),
    ("register indexed: holder search ignores the end",
     "if (lo >= hi || tree[x] < e) return nc;", "if (lo >= hi || tree[x] == 0) return nc;"),
    ("register indexed: prefix maximum of the ends restarts",
     "pm[i] = (i && pm[i - 1] > end[i]) ? pm[i - 1] : end[i];", "pm[i] = end[i];"),
    ("register one at a time: overflow not reported",
     "ctr[2] = t.size() > o_cap ? 1 : 0;", "ctr[2] = 0;"),
    ("deregister: released one reference early",
     "status[k] = left[i] == 0 ? 1 : 0;", "status[k] = left[i] <= 1 ? 1 : 0;"),
    ("deregister: a released record takes more",
     "if (i < 0 || (uint64_t)i >= n || left[i] == 0) {", "if (i < 0 || (uint64_t)i >= n) {"),
    ("deregister: survivors keep their old references",
     "o_refs[w] = (uint32_t)left[i];", "o_refs[w] = refs[i];"),
    ("deregister: a removed record keeps its place",
     "      remap[i] = -1;\n      continue;", "      remap[i] = -1;\n      ++w;\n      continue;"),
    ("deregister: stale handles not counted",
     "      status[k] = 2;\n      n_stale += 1;", "      status[k] = 2;\n      n_stale += 0;"),
    ("cq phase tag read from bit 15",
     "const uint32_t tag = (entry[3] >> 16) & 1u;", "const uint32_t tag = (entry[3] >> 15) & 1u;"),
    ("cq phase kept across the wrap",
     "      *head = 0;\n      *phase ^= 1u;", "      *head = 0;"),
    ("cq copies three dwords",
     "for (int w = 0; w < 4; ++w) host_cq", "for (int w = 0; w < 3; ++w) host_cq"),
    ("cq even generation acknowledged as itself",
     "if ((now & 1u) == 0 && now > 0) return now - 1;", "if ((now & 1u) == 0 && now > 0) return now;"),
    ("cq acknowledges the new generation",
     "if ((cur & 1u) && now != cur) return cur;", "if ((cur & 1u) && now != cur) return now;"),
    ("vmm fragment runs 16 bytes past its chunk",
     "const uint64_t t = std::min(std::min(src_left, dst_left), remaining);\n      const uint64_t post",
     "const uint64_t t = std::min(src_left + 16, remaining);\n      const uint64_t post"),
]


PIN_FILES = ("test_oracle_prp.py", "test_oracle_mr.py", "test_oracle_wqe.py",
             "test_oracle_vmm.py", "test_oracle_cq.py", "test_oracle_mr_cache.py",
             "test_oracle_transport.py")
# The pin file a mutant's name points at runs first (every file still runs
# until one fails), so most mutants stop after one file.
FIRST = (("transport", "test_oracle_transport.py"), ("register", "test_oracle_mr_cache.py"),
         ("deregister", "test_oracle_mr_cache.py"), ("vmm", "test_oracle_vmm.py"),
         ("psn", "test_oracle_vmm.py"), ("wqe", "test_oracle_wqe.py"), ("cq", "test_oracle_cq.py"),
         ("mr", "test_oracle_mr.py"))


def pin_order(name):
    first = next((f for key, f in FIRST if name.startswith(key)), PIN_FILES[0])
    return [first] + [f for f in PIN_FILES if f != first]


def run_mutant(workdir, name, old, new):
    """Build the mutant and run the pins against it: (returncode, output tail)."""
    src = open(SRC).read()
    if src.count(old) != 1:
        return None, f"mutation anchor not unique: {old!r}"
    mutated = os.path.join(workdir, "oracle_mutant.cpp")
    with open(mutated, "w") as f:
        f.write(src.replace(old, new))
    lib = os.path.join(workdir, "liboracle_mutant.so")
    subprocess.run(["g++", "-O1", "-std=c++17", "-shared", "-fPIC", "-o", lib, mutated],
                   check=True)
    env = dict(os.environ, DB_ORACLE_LIB=lib)
    tests = [os.path.join(ROOT, "tests", f) for f in pin_order(name)]
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", *tests],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=600)
    return r.returncode, r.stdout[-2000:]


@pytest.fixture(scope="module")
def verdicts(tmp_path_factory):
    """Every mutant built and run once, several at a time (each run is its
    own process with its own library)."""
    assert len({m[0] for m in MUTANTS}) == len(MUTANTS), "mutant names must be unique"
    jobs = {}
    with ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as pool:
        for i, (name, old, new) in enumerate(MUTANTS):
            d = str(tmp_path_factory.mktemp(f"mutant{i}"))
            jobs[name] = pool.submit(run_mutant, d, name, old, new)
        return {name: job.result() for name, job in jobs.items()}


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(verdicts, name, old, new):
    rc, out = verdicts[name]
    assert rc is not None, out
    assert rc != 0, f"pins did not catch: {name}\n{out}"
