// CPU oracle for batched descriptor building -- TEST INFRASTRUCTURE ONLY.
//
// A plain, single-threaded statement of the three definitions that the CUDA
// library computes, written for a reader to check by eye against the source
// pages. Only the tests and the benchmark's CPU-baseline leg load it. It
// shares no code, header, table or constant with the CUDA library.
//
// Sources (page title, section):
//  * PRP building -- xNVMe "uPCIe CUDA" backend page: the introduction (the
//    CUDA driver exports device memory at 64 KiB granularity, the physical
//    address of each 64 KiB chunk sits in a lookup table, PRP entries are
//    built at 4 KiB from sub-page offsets within a chunk), "Memory
//    Architecture" (PRP lists live in a separate host-memory region) and
//    "Limitations" (one 4 KiB list page holds 512 entries; with PRP1 that is
//    513 x 4 KiB per command).
//  * MR lookup -- "NCCL expert course 26: GPUDirect RDMA, DMA-BUF, MR and the
//    registration cache": "IB Backend MR Cache" (rounding a range down/up to
//    whole pages, worked table; reuse only if an existing MR fully contains
//    the range, partial overlap is no hit) and "Communicator User
//    Registration Cache" (page_floor / page_cover, sorted records).
//  * Put translation -- "mori communication library analysis (1)": static
//    heap address/key computation (raddr = peerPtrs[pe] + offset,
//    rkey = peerRkeys[pe], lkey = the source object's lkey), the VMM-heap
//    branch (one WQE per chunk: min of the source and destination chunk
//    remainders and the bytes left) and the warp-level WQE slot reservation
//    (a post index per send queue).
//  * MR cache mutation -- the same NCCL page: a hit takes one more
//    reference, a miss is registered anew and inserted in address order,
//    deregistration drops a reference and removes the MR at zero, a handle
//    not in the cache is an error (the ncclCommRegister experiment: the same
//    range twice and a range inside it share one record, refs 3; three
//    deregistrations delete it; then a stale handle is invalid usage); and
//    the xNVMe "uPCIe CUDA" page: xnvme_buf_register refcounts whole 64 KiB
//    device pages.
//  * CQ mirror -- xNVMe "uPCIe CUDA" backend page, "Completions in device
//    memory": completion queues live in device memory and a GPU kernel
//    forwards each new completion (recognised by its flipped phase tag) to
//    the host CQ, one warp per queue; each queue's slot holds a generation
//    (odd while attached) and an acknowledgement.
//
// Readings where the pages are silent are listed with each function.
//
// Parity status: every function here is pinned by tests under tests/
// (worked examples from the pages, brute force on tiny inputs, invariants,
// library-routine equivalences).

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <functional>
#include <map>
#include <utility>
#include <vector>

namespace {

typedef unsigned __int128 u128;

const uint64_t kPage = 4096;        // NVMe memory page (host page size used for PRPs)
const uint64_t kChunk = 65536;      // dma-buf export granule, one LUT entry each
const uint64_t kListSlots = 512;    // 8-byte entries in one 4 KiB PRP list page

[[noreturn]] void fail(const char* what) {
  std::fprintf(stderr, "oracle: %s\n", what);
  std::abort();
}

// Bus address of heap offset x: the LUT entry of the 64 KiB chunk that holds
// x, plus x's offset inside that chunk.
uint64_t bus_address(const uint64_t* lut, uint64_t n_lut, uint64_t x) {
  uint64_t chunk = x / kChunk;
  if (chunk >= n_lut) fail("heap offset beyond the LUT");
  uint64_t chunk_base = lut[chunk];
  if (chunk_base == 0 || chunk_base % kChunk != 0)
    fail("LUT entry is not a non-zero 64 KiB-aligned address");
  uint64_t inside = x % kChunk;
  if (chunk_base + inside < chunk_base) fail("bus address wraps");
  return chunk_base + inside;
}

// A request is well formed when it moves at least one byte, starts on a
// dword boundary, and ends inside the heap.
bool prp_request_valid(uint64_t off, uint64_t len, uint64_t heap_size) {
  if (len == 0) return false;
  if (off % 4 != 0) return false;
  if ((u128)off + (u128)len > (u128)heap_size) return false;
  return true;
}

// Number of 4 KiB memory pages that [off, off + len) touches.
uint64_t pages_touched(uint64_t off, uint64_t len) {
  uint64_t first = off / kPage;
  uint64_t last = (off + len - 1) / kPage;
  return last - first + 1;
}

// List pages needed for `entries` list entries when every page but the last
// gives its final slot to a pointer to the next page.
uint64_t list_pages_for(uint64_t entries) {
  if (entries == 0) return 0;
  uint64_t pages = 0;
  uint64_t left = entries;
  while (left > kListSlots) {   // this page cannot be the last one
    pages += 1;
    left -= kListSlots - 1;     // 511 entries + the chain pointer
  }
  return pages + 1;
}

}  // namespace

extern "C" {

// Per-request list-page count (0 when no list is used or when invalid).
// PRP1 covers the first page; a second page goes in PRP2; three or more
// pages put every page after the first into a PRP list.
uint64_t oracle_prp_list_pages(uint64_t off, uint64_t len, uint64_t heap_size) {
  if (!prp_request_valid(off, len, heap_size)) return 0;
  uint64_t n = pages_touched(off, len);
  if (n < 3) return 0;
  return list_pages_for(n - 1);
}

// Descriptors of ONE request whose list (if any) starts at list page
// `page_base` of the arena. `list` receives the request's list pages
// (list_pages * 512 words, laid out as they sit in the arena); untouched
// slots are left as they are unless `zero_tail`. A NULL `list` computes
// PRP1/PRP2 only. Returns the list-page count.
uint64_t oracle_prp_one(uint64_t off, uint64_t len, const uint64_t* lut, uint64_t n_lut,
                        uint64_t heap_size, uint64_t arena_base, uint64_t page_base,
                        uint64_t* prp /*[2]*/, uint64_t* list, int zero_tail) {
  prp[0] = 0;
  prp[1] = 0;
  if (!prp_request_valid(off, len, heap_size)) return 0;
  uint64_t n = pages_touched(off, len);
  uint64_t first_page = off - off % kPage;        // heap offset of the first page
  prp[0] = bus_address(lut, n_lut, off);          // PRP1 keeps the in-page offset
  if (n == 1) return 0;
  if (n == 2) {
    prp[1] = bus_address(lut, n_lut, first_page + kPage);
    return 0;
  }
  // n >= 3: PRP2 points at the first list page; the list holds pages 1..n-1.
  if (arena_base % kPage != 0) fail("arena base not page aligned");
  uint64_t n_list = list_pages_for(n - 1);
  prp[1] = arena_base + page_base * kPage;
  if (!list) return n_list;
  uint64_t page = 0;   // list page being filled, relative to page_base
  uint64_t slot = 0;   // next free slot on it
  for (uint64_t k = 1; k < n; ++k) {
    bool more_after_this = (k + 1 < n);
    if (slot == kListSlots - 1 && more_after_this) {
      // Last slot of a full page with entries still to come: chain.
      list[page * kListSlots + slot] = arena_base + (page_base + page + 1) * kPage;
      page += 1;
      slot = 0;
    }
    list[page * kListSlots + slot] = bus_address(lut, n_lut, first_page + k * kPage);
    slot += 1;
  }
  if (page + 1 != n_list) fail("list page count mismatch");
  // Reading: the pages say nothing of the slots after a list's last entry,
  // so they are left as they were; the zero-tail option clears them.
  if (zero_tail) {
    for (; slot < kListSlots; ++slot) list[page * kListSlots + slot] = 0;
  }
  return n_list;
}

// Whole batch, in request order.
//  req        [n][2]: word 0 = heap offset, word 1 low 32 bits = length
//  arena      host copy of the list arena, arena_cap_pages * 512 words, or
//             NULL to compute everything but the list pages
//  prp        [n][2] out: PRP1, PRP2
//  page_base  [n] out (nullable): first list page of each request (exclusive
//             running sum of list pages, in request order)
//  status     [n] out (nullable): 0 ok, 1 invalid, 2 list would not fit
//  ctr        [4] out: total list pages, invalid count, overflow count, error bits (0)
// A request whose list would end past the arena gets status 2, PRP {0,0}
// and no list; it still advances the running page count.
void oracle_prp_build(const uint64_t* req, uint64_t n, const uint64_t* lut, uint64_t n_lut,
                      uint64_t heap_size, uint64_t arena_base, uint64_t arena_cap_pages,
                      uint64_t* arena, uint64_t* prp, uint64_t* page_base, uint8_t* status,
                      uint64_t* ctr, int zero_tail) {
  uint64_t running = 0;
  uint64_t n_invalid = 0, n_overflow = 0;
  std::vector<uint64_t> scratch;
  for (uint64_t i = 0; i < n; ++i) {
    uint64_t off = req[2 * i];
    uint64_t len = req[2 * i + 1] & 0xFFFFFFFFull;
    uint8_t st = 0;
    uint64_t pages = 0;
    prp[2 * i] = 0;
    prp[2 * i + 1] = 0;
    if (page_base) page_base[i] = running;
    if (!prp_request_valid(off, len, heap_size)) {
      st = 1;
      n_invalid += 1;
    } else {
      pages = oracle_prp_list_pages(off, len, heap_size);
      // Only a request that needs list pages can run out of arena.
      if (pages > 0 && running + pages > arena_cap_pages) {
        st = 2;
        n_overflow += 1;
      } else {
        uint64_t* list = (pages && arena) ? arena + running * kListSlots : nullptr;
        uint64_t got = oracle_prp_one(off, len, lut, n_lut, heap_size, arena_base, running,
                                      prp + 2 * i, list, zero_tail);
        if (got != pages) fail("list page count disagrees");
      }
    }
    if (status) status[i] = st;
    running += pages;
  }
  ctr[0] = running;
  ctr[1] = n_invalid;
  ctr[2] = n_overflow;
  ctr[3] = 0;
}

// ---------------------------------------------------------------------------
// MR lookup.
//
// Rounding: the range [addr, addr + size) widens to whole 4 KiB pages,
// base = page floor of addr, aend = base + pages * 4096 with
// pages = ceil((addr + size - base) / 4096).
// Reading: a range is INVALID (kind 3) when size == 0 or when the rounded end
// would not fit in 64 bits (addr + size > 2^64 - 4096).
// Classification: the lowest-index registered range [start_i, end_i) with
// start_i <= base and aend <= end_i is the hit; EXACT (1) when both ends
// match, CONTAINED (2) otherwise. No such range: MISS (0). Partial overlap
// is a miss. Ranges are end-exclusive.

static bool mr_round(uint64_t addr, uint64_t size, uint64_t* base, uint64_t* aend) {
  if (size == 0) return false;
  u128 stop = (u128)addr + (u128)size;
  if (stop > (u128)(UINT64_MAX - kPage + 1)) return false;
  uint64_t b = addr - addr % kPage;
  uint64_t pages = (uint64_t)((stop - b + kPage - 1) / kPage);
  *base = b;
  *aend = b + pages * kPage;
  return true;
}

void oracle_mr_round(uint64_t addr, uint64_t size, uint64_t* out /*[3]: valid, base, aend*/) {
  uint64_t b = 0, e = 0;
  out[0] = mr_round(addr, size, &b, &e) ? 1 : 0;
  out[1] = b;
  out[2] = e;
}

// The definition: a scan over the whole table for every query.
void oracle_mr_linear(const uint64_t* q, uint64_t n_q, const uint64_t* start,
                      const uint64_t* end, const uint32_t* lkey, uint64_t n_mr,
                      int32_t* idx, uint32_t* lkey_out, uint8_t* kind) {
  for (uint64_t k = 0; k < n_q; ++k) {
    uint64_t base, aend;
    idx[k] = -1;
    lkey_out[k] = 0;
    if (!mr_round(q[2 * k], q[2 * k + 1], &base, &aend)) {
      kind[k] = 3;
      continue;
    }
    kind[k] = 0;
    for (uint64_t i = 0; i < n_mr; ++i) {
      if (start[i] <= base && aend <= end[i]) {
        idx[k] = (int32_t)i;
        lkey_out[k] = lkey[i];
        kind[k] = (start[i] == base && end[i] == aend) ? 1 : 2;
        break;
      }
    }
  }
}

// For tables sorted by start whose ranges may overlap: the lowest index
// containing [base, aend) has start <= base, so it lies in [0, j] with j the
// last range starting at or below base; among those it is the first whose
// end reaches aend, found by binary search on the prefix maximum of the ends
// (non-decreasing). Pinned against oracle_mr_linear, the definition.
void oracle_mr_prefix_max(const uint64_t* q, uint64_t n_q, const uint64_t* start,
                          const uint64_t* end, const uint32_t* lkey, uint64_t n_mr,
                          int32_t* idx, uint32_t* lkey_out, uint8_t* kind) {
  std::vector<uint64_t> pm(n_mr);
  for (uint64_t i = 0; i < n_mr; ++i) pm[i] = i ? std::max(pm[i - 1], end[i]) : end[i];
  for (uint64_t k = 0; k < n_q; ++k) {
    uint64_t base, aend;
    idx[k] = -1;
    lkey_out[k] = 0;
    if (!mr_round(q[2 * k], q[2 * k + 1], &base, &aend)) {
      kind[k] = 3;
      continue;
    }
    kind[k] = 0;
    const uint64_t cnt = (uint64_t)(std::upper_bound(start, start + n_mr, base) - start);
    if (cnt == 0) continue;
    const uint64_t i = (uint64_t)(std::lower_bound(pm.begin(), pm.begin() + cnt, aend) - pm.begin());
    if (i == cnt) continue;
    idx[k] = (int32_t)i;
    lkey_out[k] = lkey[i];
    const bool same_ends = start[i] == base && end[i] == aend;
    kind[k] = same_ends ? 1 : 2;
  }
}

// For tables sorted by start with no two ranges overlapping: the only range
// that can contain [base, aend) is the last one starting at or below base.
void oracle_mr_bsearch(const uint64_t* q, uint64_t n_q, const uint64_t* start,
                       const uint64_t* end, const uint32_t* lkey, uint64_t n_mr,
                       int32_t* idx, uint32_t* lkey_out, uint8_t* kind) {
  for (uint64_t k = 0; k < n_q; ++k) {
    uint64_t base, aend;
    idx[k] = -1;
    lkey_out[k] = 0;
    if (!mr_round(q[2 * k], q[2 * k + 1], &base, &aend)) {
      kind[k] = 3;
      continue;
    }
    kind[k] = 0;
    const uint64_t* it = std::upper_bound(start, start + n_mr, base);
    if (it == start) continue;
    uint64_t j = (uint64_t)(it - start) - 1;
    if (aend <= end[j]) {
      idx[k] = (int32_t)j;
      lkey_out[k] = lkey[j];
      kind[k] = (start[j] == base && end[j] == aend) ? 1 : 2;
    }
  }
}

// ---------------------------------------------------------------------------
// Put translation and stable bucketing into per-queue WQE rings.
//
// Request word 0 = heap offset, word 1 = bytes | pe << 32 | qp << 48.
// A request is valid when pe < world, qp < n_qp, bytes >= 1 and
// offset + bytes <= heap_size. Valid requests go to ring r = pe * n_qp + qp
// (PE-major), in request order; the k-th one of ring r (k from 0) takes
// sequence number seq = head[r] + k and slot seq mod depth.
// A ring asked to take more than `depth` entries in one batch overflows: it
// gets no entry, its head stays, its requests count in ctr[2] and ctr[3]
// gets bit 2. count[r] is the number of valid requests routed to ring r.
// ctr = {entries posted, invalid count, overflow count, error bits}.
//
// WQE (64 bytes, little-endian): +0 raddr, +8 laddr, +16 u32 len,
// +20 u32 lkey, +24 u32 rkey, +28 u32 flags (0), +32 u64 seq,
// +40 u32 request index, +44..63 zero.
// raddr = peer_ptrs[pe] + offset, rkey = rkeys[pe];
// laddr = local_base + offset (the source sits at the same symmetric offset
// in the local heap), lkey = the local object's single lkey.

static void put_u64(uint8_t* p, uint64_t v) { std::memcpy(p, &v, 8); }
static void put_u32(uint8_t* p, uint32_t v) { std::memcpy(p, &v, 4); }

struct PutFields {
  uint64_t off, bytes, pe, qp;
};
static PutFields put_fields(const uint64_t* req, uint64_t i) {
  uint64_t w1 = req[2 * i + 1];
  return PutFields{req[2 * i], w1 & 0xFFFFFFFFull, (w1 >> 32) & 0xFFFF, (w1 >> 48) & 0xFFFF};
}

// The validity rule of a put (the same for every transport).
static bool put_valid(const PutFields& f, uint32_t world, uint32_t n_qp, uint64_t heap_size) {
  return f.pe < world && f.qp < n_qp && f.bytes >= 1 &&
         (u128)f.off + (u128)f.bytes <= (u128)heap_size;
}

// Ring of a valid put.
static int ring_index(const PutFields& f, uint32_t world, uint32_t n_qp) {
  (void)world;
  return (int)(f.pe * n_qp + f.qp);
}

// Steps 2-4 of the bucketing, given each put's ring (negative: none) and
// each ring's demand: overflowing rings take nothing, the others get their
// puts in request order, heads advance. Fills ctr[0], ctr[2], ctr[3].
static void post_into_rings(const uint64_t* req, uint64_t n, const std::vector<int>& ring_of,
                            const std::vector<uint64_t>& demand, const uint64_t* peer_ptrs,
                            const uint32_t* rkeys, uint64_t local_base, uint32_t lkey,
                            uint8_t* rings, uint64_t depth, uint64_t* head, uint32_t* count,
                            uint64_t* ctr) {
  uint64_t n_rings = demand.size();
  // 2. Overflowing rings take nothing.
  uint64_t n_overflow = 0, posted = 0, err = 0;
  std::vector<bool> full(n_rings, false);
  for (uint64_t r = 0; r < n_rings; ++r) {
    if (demand[r] > depth) {
      full[r] = true;
      n_overflow += demand[r];
      err |= 2;
    }
  }
  // 3. Post in request order.
  std::vector<uint64_t> taken(n_rings, 0);
  for (uint64_t i = 0; i < n; ++i) {
    int r = ring_of[i];
    if (r < 0 || full[r]) continue;
    PutFields f = put_fields(req, i);
    uint64_t seq = head[r] + taken[r];
    taken[r] += 1;
    uint8_t* wqe = rings + ((uint64_t)r * depth + (seq % depth)) * 64;
    std::memset(wqe, 0, 64);
    put_u64(wqe + 0, peer_ptrs[f.pe] + f.off);
    put_u64(wqe + 8, local_base + f.off);
    put_u32(wqe + 16, (uint32_t)f.bytes);
    put_u32(wqe + 20, lkey);
    put_u32(wqe + 24, rkeys[f.pe]);
    put_u32(wqe + 28, 0);
    put_u64(wqe + 32, seq);
    put_u32(wqe + 40, (uint32_t)i);
    posted += 1;
  }
  // 4. Advance heads of the rings that took their batch.
  for (uint64_t r = 0; r < n_rings; ++r) {
    count[r] = (uint32_t)demand[r];
    if (!full[r]) head[r] += demand[r];
  }
  ctr[0] = posted;
  ctr[2] = n_overflow;
  ctr[3] = err;
}

void oracle_wqe_bucket(const uint64_t* req, uint64_t n, const uint64_t* peer_ptrs,
                       const uint32_t* rkeys, uint32_t world, uint32_t n_qp,
                       uint64_t local_base, uint32_t lkey, uint64_t heap_size,
                       uint8_t* rings, uint64_t depth, uint64_t* head, uint32_t* count,
                       uint64_t* ctr) {
  uint64_t n_rings = (uint64_t)world * n_qp;
  std::vector<uint64_t> demand(n_rings, 0);
  std::vector<int> ring_of(n);
  uint64_t n_invalid = 0;
  // 1. Validate and count per ring.
  for (uint64_t i = 0; i < n; ++i) {
    PutFields f = put_fields(req, i);
    if (!put_valid(f, world, n_qp, heap_size)) {
      ring_of[i] = -1;
      n_invalid += 1;
      continue;
    }
    ring_of[i] = ring_index(f, world, n_qp);
    demand[ring_of[i]] += 1;
  }
  post_into_rings(req, n, ring_of, demand, peer_ptrs, rkeys, local_base, lkey, rings, depth,
                  head, count, ctr);
  ctr[1] = n_invalid;
}

// Put translation with a transport per PE -- "mori communication library
// analysis (1)", the transport dispatch of the put path and the symmetric
// object set-up before it: every PE is marked once with a transport type
// (RDMA, P2P or SDMA) and each put branches on its target's type; for a PE
// that is not reached over RDMA the peer pointer is replaced by the address
// at which this process maps that PE's heap, so the destination is always
// peer_ptrs[pe] + offset.
//
// transport[pe]: 0 RDMA, 1 P2P, 2 SDMA. Readings:
//  - An RDMA put is translated and bucketed exactly as by oracle_wqe_bucket
//    (its ring, seq, slot, fields, overflow rule); puts to other PEs take no
//    ring slot and do not count in any ring.
//  - A P2P or SDMA put makes no WQE: it is a copy this process issues itself
//    (loads/stores through the mapping, or a DMA engine). It becomes a
//    32-byte direct descriptor, appended in request order to `direct`:
//    +0 u64 dst = peer_ptrs[pe] + offset, +8 u64 src = local_base + offset,
//    +16 u32 len, +20 u32 request index, +24 u16 pe, +26 u8 transport,
//    +27..31 zero.
//  - Validity is the same rule for every transport (pe < world, qp < n_qp,
//    bytes >= 1, offset + bytes <= heap_size), and a PE whose transport code
//    is none of the three makes its puts invalid.
//  - ctr = {WQEs posted, invalid puts, puts of overflowing rings, error
//    bits}; *n_direct = direct descriptors written.
void oracle_wqe_bucket_transport(const uint64_t* req, uint64_t n, const uint64_t* peer_ptrs,
                                 const uint32_t* rkeys, const uint8_t* transport,
                                 uint32_t world, uint32_t n_qp, uint64_t local_base,
                                 uint32_t lkey, uint64_t heap_size, uint8_t* rings,
                                 uint64_t depth, uint64_t* head, uint32_t* count, uint64_t* ctr,
                                 uint8_t* direct, uint64_t* n_direct) {
  uint64_t n_rings = (uint64_t)world * n_qp;
  std::vector<uint64_t> demand(n_rings, 0);
  std::vector<int> ring_of(n);     // -1 invalid, -2 direct
  uint64_t n_invalid = 0;
  // 1. Validate, dispatch on the target's transport, count per ring.
  for (uint64_t i = 0; i < n; ++i) {
    PutFields f = put_fields(req, i);
    if (!put_valid(f, world, n_qp, heap_size) || transport[f.pe] > 2) {
      ring_of[i] = -1;
      n_invalid += 1;
      continue;
    }
    if (transport[f.pe] != 0) {
      ring_of[i] = -2;
      continue;
    }
    ring_of[i] = ring_index(f, world, n_qp);
    demand[ring_of[i]] += 1;
  }
  // 2-4. The RDMA puts, into their rings.
  post_into_rings(req, n, ring_of, demand, peer_ptrs, rkeys, local_base, lkey, rings, depth,
                  head, count, ctr);
  ctr[1] = n_invalid;
  // The direct puts, appended in request order.
  uint64_t nd = 0;
  for (uint64_t i = 0; i < n; ++i) {
    if (ring_of[i] != -2) continue;
    PutFields f = put_fields(req, i);
    uint8_t* d = direct + nd * 32;
    std::memset(d, 0, 32);
    put_u64(d + 0, peer_ptrs[f.pe] + f.off);
    put_u64(d + 8, local_base + f.off);
    put_u32(d + 16, (uint32_t)f.bytes);
    put_u32(d + 20, (uint32_t)i);
    d[24] = (uint8_t)(f.pe & 0xFF);
    d[25] = (uint8_t)(f.pe >> 8);
    d[26] = transport[f.pe];
    nd += 1;
  }
  *n_direct = nd;
}

// Put translation on a VMM heap -- "mori communication library analysis
// (1)", the VMM-heap branch of the put path: while bytes remain, look up the
// chunk holding the current source address (its lkey and how many bytes of
// it remain) and the chunk holding the current destination address on the
// target PE (its remote address, rkey and remainder); send
// min(source remainder, destination remainder, remaining) bytes as one WQE;
// advance. Readings (the page does not give the chunk layout):
//  * the heap is cut into chunks of 2^chunk_shift bytes at the same offsets
//    on every PE; local chunk c has lkey chunk_lkey[c]; chunk c of PE pe sits
//    at remote address chunk_raddr[pe * n_chunks + c] with rkey
//    chunk_rkey[pe * n_chunks + c] (n_chunks = ceil(heap_size / 2^chunk_shift));
//  * a put covers the same symmetric range [off, off + bytes) on both sides,
//    and laddr is local_base + the fragment's offset;
//  * a put's fragments take consecutive post indices in its ring, in address
//    order, each carrying the put's batch index; validity and ring order are
//    those of the static heap;
//  * a ring asked for more than `depth` WQEs by the batch takes none;
//    counters: WQEs posted, invalid puts, WQEs of overflowing rings, err.
// Packet sequence numbers (same page, the BNXT branch), when mtu != 0: a WQE
// of `len` bytes uses psnCnt = ceil(len / mtu) PSNs; its first PSN is the
// ring's PSN counter plus the psnCnt of the ring's earlier WQEs (the page's
// exclusive prefix over active lanes, here over the batch in order), written
// as a u32 at byte 44 of the WQE. The SQ index still advances by one per WQE
// (the page's code adds the lane count to the MSN and the PSN total to the
// PSN). A ring that takes its batch advances psn_head by its PSN total.
void oracle_wqe_bucket_vmm(const uint64_t* req, uint64_t n, const uint64_t* chunk_raddr,
                           const uint32_t* chunk_rkey, const uint32_t* chunk_lkey,
                           uint32_t chunk_shift, uint32_t world, uint32_t n_qp,
                           uint64_t local_base, uint64_t heap_size, uint8_t* rings,
                           uint64_t depth, uint64_t* head, uint32_t mtu, uint64_t* psn_head,
                           uint32_t* count, uint64_t* ctr) {
  const uint64_t C = 1ull << chunk_shift;
  const uint64_t n_chunks = (heap_size + C - 1) / C;
  uint64_t n_rings = (uint64_t)world * n_qp;
  std::vector<uint64_t> demand(n_rings, 0), psn_demand(n_rings, 0);
  std::vector<int> ring_of(n);
  uint64_t n_invalid = 0;
  // One pass of the page's loop, emitting nothing: how many WQEs a put makes
  // (and, with an mtu, how many PSNs they use).
  auto fragments = [&](uint64_t off, uint64_t bytes, uint64_t& psns) {
    uint64_t cur = 0, remaining = bytes, k = 0;
    psns = 0;
    while (remaining > 0) {
      const uint64_t src = off + cur, dst = off + cur;
      const uint64_t src_left = C - (src % C), dst_left = C - (dst % C);
      const uint64_t t = std::min(std::min(src_left, dst_left), remaining);
      if (mtu) psns += (t + mtu - 1) / mtu;
      cur += t;
      remaining -= t;
      k += 1;
    }
    return k;
  };
  // 1. Validate and count WQEs per ring.
  for (uint64_t i = 0; i < n; ++i) {
    uint64_t off = req[2 * i];
    uint64_t w1 = req[2 * i + 1];
    uint64_t bytes = w1 & 0xFFFFFFFFull;
    uint64_t pe = (w1 >> 32) & 0xFFFF;
    uint64_t qp = (w1 >> 48) & 0xFFFF;
    bool ok = pe < world && qp < n_qp && bytes >= 1 &&
              (u128)off + (u128)bytes <= (u128)heap_size;
    if (!ok) {
      ring_of[i] = -1;
      n_invalid += 1;
      continue;
    }
    const int ring = (int)(pe * n_qp + qp);  // PE-major, as for the static heap
    ring_of[i] = ring;
    uint64_t psns = 0;
    demand[ring] += fragments(off, bytes, psns);
    psn_demand[ring] += psns;
  }
  // 2. Overflowing rings take nothing.
  uint64_t n_overflow = 0, posted = 0, err = 0;
  std::vector<bool> full(n_rings, false);
  for (uint64_t r = 0; r < n_rings; ++r) {
    if (depth < demand[r]) {
      full[r] = true;
      n_overflow += demand[r];
      err |= 2;
    }
  }
  // 3. Post in request order, each put's fragments in address order.
  std::vector<uint64_t> taken(n_rings, 0), psn_taken(n_rings, 0);
  for (uint64_t i = 0; i < n; ++i) {
    int r = ring_of[i];
    if (r < 0 || full[r]) continue;
    uint64_t off = req[2 * i];
    uint64_t w1 = req[2 * i + 1];
    uint64_t bytes = w1 & 0xFFFFFFFFull;
    uint32_t pe = (uint32_t)((w1 >> 32) & 0xFFFF);
    uint64_t cur = 0, remaining = bytes;
    while (remaining > 0) {
      const uint64_t src = off + cur, dst = off + cur;
      const uint64_t src_chunk = src / C, dst_chunk = dst / C;
      if (src_chunk >= n_chunks || dst_chunk >= n_chunks) std::abort();  // inside the heap
      const uint32_t lkey = chunk_lkey[src_chunk];
      const uint64_t raddr = chunk_raddr[pe * n_chunks + dst_chunk] + (dst % C);
      const uint32_t rkey = chunk_rkey[pe * n_chunks + dst_chunk];
      const uint64_t src_left = C - (src % C), dst_left = C - (dst % C);
      const uint64_t t = std::min(std::min(src_left, dst_left), remaining);
      const uint64_t post = head[r] + taken[r];  // the ring's next post index
      taken[r] += 1;
      uint8_t* wqe = rings + ((uint64_t)r * depth + (post % depth)) * 64;
      std::memset(wqe, 0, 64);
      put_u64(wqe + 0, raddr);
      put_u64(wqe + 8, local_base + src);
      put_u32(wqe + 16, (uint32_t)t);
      put_u32(wqe + 20, lkey);
      put_u32(wqe + 24, rkey);
      put_u32(wqe + 28, 0);
      put_u64(wqe + 32, post);
      put_u32(wqe + 40, (uint32_t)i);
      if (mtu) {
        put_u32(wqe + 44, (uint32_t)(psn_head[r] + psn_taken[r]));  // first PSN
        psn_taken[r] += (t + mtu - 1) / mtu;
      }
      posted += 1;
      cur += t;
      remaining -= t;
    }
  }
  // 4. Advance heads of the rings that took their batch.
  for (uint64_t r = 0; r < n_rings; ++r) {
    count[r] = (uint32_t)std::min<uint64_t>(demand[r], 0xFFFFFFFFull);
    if (!full[r]) head[r] += demand[r];
    if (mtu && !full[r]) psn_head[r] += psn_demand[r];
  }
  ctr[0] = posted;
  ctr[1] = n_invalid;
  ctr[2] = n_overflow;
  ctr[3] = err;
}

// ---------------------------------------------------------- MR cache mutation
// Readings (a batch form of the pages' one-call-at-a-time operations):
//  * Registration batch. Every request is rounded to whole granules (4 KiB,
//    or 64 KiB for the xNVMe registry) and looked up in the table as it
//    stood before the batch: a hit takes one more reference on the
//    lowest-index record holding it. The requests that missed become one
//    new record per distinct rounded range, with as many references as
//    requests for it and the new_lkey of its first request. A new record
//    goes after every old record with the same start; new records among
//    themselves are in (start, end) order. This is one-at-a-time
//    registration whenever no new range of the batch lies inside another
//    one (then the later one would have been a hit).
//  * Handles are record indices; remap[i] is old record i's index after the
//    batch (-1 once removed). A handle of a request is its record's index in
//    the table after the batch.
//  * Deregistration batch: in batch order, each handle takes one reference
//    off its record; the one that takes the last reference releases it; a
//    handle naming no record, or a record already released, is stale. The
//    records whose references reach 0 are removed.
// Kinds: 1 hit (same range), 2 hit (contained), 3 invalid, 4 new record,
// 5 same range as a new record of this batch. Deregistration status: 0 a
// reference dropped, 1 released, 2 stale.

// [base, aend): the range widened to whole granules of g bytes; false for an
// empty range or one whose widened end would not fit in 64 bits.
static bool round_to_granule(uint64_t addr, uint64_t size, uint64_t g, uint64_t* base,
                             uint64_t* aend) {
  if (size == 0) return false;
  const u128 stop = (u128)addr + (u128)size;
  if (stop > (u128)(UINT64_MAX - g + 1)) return false;
  const uint64_t b = addr - addr % g;
  const uint64_t units = (uint64_t)((stop - b + g - 1) / g);
  *base = b;
  *aend = b + units * g;
  return true;
}

// Lowest index i with start[i] <= base and aend <= end[i] in a table sorted
// by start, or -1: records after the last start <= base start too late, and
// among the others the first whose prefix maximum of ends reaches aend.
static int64_t lowest_holder(const uint64_t* start, const std::vector<uint64_t>& pm, uint64_t n,
                             uint64_t base, uint64_t aend) {
  const uint64_t starting = (uint64_t)(std::upper_bound(start, start + n, base) - start);
  const auto first_reach = std::lower_bound(pm.begin(), pm.begin() + (ptrdiff_t)starting, aend);
  const uint64_t i = (uint64_t)(first_reach - pm.begin());
  return i < starting ? (int64_t)i : -1;
}

void oracle_mr_register(const uint64_t* q, uint64_t n_q, const uint32_t* new_lkey,
                        uint32_t granule_shift, const uint64_t* start, const uint64_t* end,
                        const uint32_t* lkey, const uint32_t* refs, uint64_t n,
                        uint64_t* o_start, uint64_t* o_end, uint32_t* o_lkey, uint32_t* o_refs,
                        uint64_t o_cap, int64_t* handle, uint8_t* kind, int64_t* remap,
                        uint64_t* ctr) {
  const uint64_t g = 1ull << granule_shift;
  uint64_t err = 0;
  for (uint64_t i = 0; i < n; ++i)
    if (!(start[i] < end[i]) || (i > 0 && start[i - 1] > start[i])) err = 4;
  std::vector<uint64_t> pm(n);  // prefix maximum of the ends
  uint64_t reach = 0;
  for (uint64_t i = 0; i < n; ++i) {
    reach = std::max(reach, end[i]);
    pm[i] = reach;
  }
  // 1. look every request up in the table as it stood before the batch
  std::vector<uint64_t> more(n, 0);                 // references each old record gains
  std::vector<int64_t> holder(n_q, -1);
  std::vector<std::pair<uint64_t, uint64_t>> range(n_q);
  std::map<std::pair<uint64_t, uint64_t>, std::pair<uint64_t, uint64_t>> fresh;  // -> (first, count)
  uint64_t n_invalid = 0;
  for (uint64_t k = 0; k < n_q; ++k) {
    uint64_t b, e;
    if (!round_to_granule(q[2 * k], q[2 * k + 1], g, &b, &e)) {
      kind[k] = 3;
      n_invalid += 1;
      continue;
    }
    range[k] = {b, e};
    const int64_t i = lowest_holder(start, pm, n, b, e);
    if (i >= 0) {
      holder[k] = i;
      more[i] += 1;
      kind[k] = (start[i] == b && end[i] == e) ? 1 : 2;
    } else {
      auto it = fresh.find({b, e});
      if (it == fresh.end()) {
        fresh[{b, e}] = {k, 1};
        kind[k] = 4;
      } else {
        it->second.second += 1;
        kind[k] = 5;
      }
    }
  }
  const uint64_t n_out = n + fresh.size();
  ctr[0] = n_out;
  ctr[1] = n_invalid;
  ctr[2] = n_out > o_cap ? 1 : 0;
  ctr[3] = err;
  if (n_out > o_cap) return;  // nothing else is written
  // 2. merge: an old record goes before new records with the same start
  std::map<std::pair<uint64_t, uint64_t>, uint64_t> placed;  // new range -> index after the batch
  auto nit = fresh.begin();
  uint64_t i = 0, w = 0;
  while (i < n || nit != fresh.end()) {
    const bool take_old = i < n && (nit == fresh.end() || start[i] <= nit->first.first);
    if (take_old) {
      o_start[w] = start[i];
      o_end[w] = end[i];
      o_lkey[w] = lkey[i];
      o_refs[w] = (uint32_t)(refs[i] + more[i]);
      remap[i] = (int64_t)w;
      ++i;
    } else {
      o_start[w] = nit->first.first;
      o_end[w] = nit->first.second;
      o_lkey[w] = new_lkey[nit->second.first];
      o_refs[w] = (uint32_t)nit->second.second;
      placed[nit->first] = w;
      ++nit;
    }
    ++w;
  }
  // 3. handles
  for (uint64_t k = 0; k < n_q; ++k) {
    if (kind[k] == 3) handle[k] = -1;
    else if (kind[k] <= 2) handle[k] = remap[holder[k]];
    else handle[k] = (int64_t)placed[range[k]];
  }
}

// One registration at a time, as the pages describe it: look the range up
// in the table as it is now (lowest index holding it); a hit takes a
// reference, a miss inserts a record after every record starting at or
// before it. Kind 5 marks a hit on a record this batch created. Handles and
// remap are indices in the final table.
void oracle_mr_register_seq(const uint64_t* q, uint64_t n_q, const uint32_t* new_lkey,
                            uint32_t granule_shift, const uint64_t* start, const uint64_t* end,
                            const uint32_t* lkey, const uint32_t* refs, uint64_t n,
                            uint64_t* o_start, uint64_t* o_end, uint32_t* o_lkey,
                            uint32_t* o_refs, uint64_t o_cap, int64_t* handle, uint8_t* kind,
                            int64_t* remap, uint64_t* ctr) {
  struct Rec { uint64_t s, e; uint32_t lk, refs; int64_t id; };  // id: old index, or -1 - request
  const uint64_t g = 1ull << granule_shift;
  std::vector<Rec> t;
  for (uint64_t i = 0; i < n; ++i) t.push_back({start[i], end[i], lkey[i], refs[i], (int64_t)i});
  std::vector<int64_t> got(n_q, 0);  // record id each request ends up on
  uint64_t n_invalid = 0;
  for (uint64_t k = 0; k < n_q; ++k) {
    uint64_t b, e;
    if (!round_to_granule(q[2 * k], q[2 * k + 1], g, &b, &e)) {
      kind[k] = 3;
      n_invalid += 1;
      continue;
    }
    bool hit = false;
    for (auto& r : t) {
      if (r.s <= b && e <= r.e) {
        r.refs += 1;
        got[k] = r.id;
        kind[k] = r.id >= 0 ? ((r.s == b && r.e == e) ? 1 : 2) : 5;
        hit = true;
        break;
      }
    }
    if (hit) continue;
    size_t at = 0;
    while (at < t.size() && t[at].s <= b) ++at;
    t.insert(t.begin() + at, Rec{b, e, new_lkey[k], 1, -1 - (int64_t)k});
    got[k] = -1 - (int64_t)k;
    kind[k] = 4;
  }
  uint64_t err = 0;
  for (uint64_t i = 0; i < n; ++i)
    if (!(start[i] < end[i]) || (i > 0 && start[i - 1] > start[i])) err = 4;
  ctr[0] = t.size();
  ctr[1] = n_invalid;
  ctr[2] = t.size() > o_cap ? 1 : 0;
  ctr[3] = err;
  if (t.size() > o_cap) return;  // as in the batch reading: only counters and kinds
  std::map<int64_t, int64_t> final_index;
  for (size_t w = 0; w < t.size(); ++w) {
    o_start[w] = t[w].s;
    o_end[w] = t[w].e;
    o_lkey[w] = t[w].lk;
    o_refs[w] = t[w].refs;
    final_index[t[w].id] = (int64_t)w;
  }
  for (uint64_t i = 0; i < n; ++i) remap[i] = final_index[(int64_t)i];
  for (uint64_t k = 0; k < n_q; ++k) handle[k] = kind[k] == 3 ? -1 : final_index[got[k]];
}

// The same one-at-a-time registration with an index, for batches too large
// for the scan above (pinned equal to it by the tests). At request k the
// table holds the old records and the records created by requests before k,
// in start order (a record goes after every record starting at or before
// it, so the old records come first on equal starts and created records of
// equal start follow in creation order). The lowest-index record holding
// [b, e) is then the old one found as in the batch reading, or the created
// one of least start holding it, whichever comes first in that order. Two
// created records of equal start hold no common later request in a
// different order: the later one was created only because the earlier did
// not hold it, so it ends later, and creation order is end order. So the
// created records are kept at their (start, end) rank among every range
// that could be created (the requests that miss the old table); the
// created holder of least table index is the leftmost rank with start <= b
// whose end reaches e (a max-tree over ranks).
void oracle_mr_register_seq_indexed(const uint64_t* q, uint64_t n_q, const uint32_t* new_lkey,
                                    uint32_t granule_shift, const uint64_t* start,
                                    const uint64_t* end, const uint32_t* lkey,
                                    const uint32_t* refs, uint64_t n, uint64_t* o_start,
                                    uint64_t* o_end, uint32_t* o_lkey, uint32_t* o_refs,
                                    uint64_t o_cap, int64_t* handle, uint8_t* kind,
                                    int64_t* remap, uint64_t* ctr) {
  const uint64_t g = 1ull << granule_shift;
  uint64_t err = 0;
  for (uint64_t i = 0; i < n; ++i)
    if (!(start[i] < end[i]) || (i > 0 && start[i - 1] > start[i])) err = 4;
  std::vector<uint64_t> pm(n);  // prefix maximum of the ends
  for (uint64_t i = 0; i < n; ++i) pm[i] = (i && pm[i - 1] > end[i]) ? pm[i - 1] : end[i];
  // 1. widen; the old holder of every request (the table before the batch)
  std::vector<std::pair<uint64_t, uint64_t>> range(n_q);
  std::vector<int64_t> old(n_q, -1);
  std::vector<char> valid(n_q, 0);
  std::vector<std::pair<uint64_t, uint64_t>> cand;  // ranges that miss the old table
  for (uint64_t k = 0; k < n_q; ++k) {
    uint64_t b, e;
    if (!round_to_granule(q[2 * k], q[2 * k + 1], g, &b, &e)) continue;
    valid[k] = 1;
    range[k] = {b, e};
    old[k] = lowest_holder(start, pm, n, b, e);
    if (old[k] < 0) cand.push_back({b, e});
  }
  std::sort(cand.begin(), cand.end());
  cand.erase(std::unique(cand.begin(), cand.end()), cand.end());
  const uint64_t nc = cand.size();
  // max-tree over ranks: the end of the record created at that rank (0: none)
  uint64_t size = 1;
  while (size < nc) size <<= 1;
  std::vector<uint64_t> tree(2 * size, 0);
  auto set_end = [&](uint64_t r, uint64_t e) {
    uint64_t x = r + size;
    tree[x] = e;
    for (x >>= 1; x > 0; x >>= 1) tree[x] = std::max(tree[2 * x], tree[2 * x + 1]);
  };
  // leftmost rank in [0, hi) whose end is >= e, or nc
  std::function<uint64_t(uint64_t, uint64_t, uint64_t, uint64_t, uint64_t)> leftmost =
      [&](uint64_t x, uint64_t lo, uint64_t width, uint64_t hi, uint64_t e) -> uint64_t {
    if (lo >= hi || tree[x] < e) return nc;
    if (width == 1) return lo;
    const uint64_t half = width / 2;
    const uint64_t a = leftmost(2 * x, lo, half, hi, e);
    return a < nc ? a : leftmost(2 * x + 1, lo + half, half, hi, e);
  };
  // 2. the requests in order
  std::vector<int64_t> creator(nc, -1);  // request that created the record at each rank
  std::vector<uint64_t> crefs(nc, 0);
  std::vector<uint64_t> more(n, 0);
  std::vector<int64_t> got_old(n_q, -1), got_new(n_q, -1);
  uint64_t n_invalid = 0, n_new = 0;
  for (uint64_t k = 0; k < n_q; ++k) {
    if (!valid[k]) {
      kind[k] = 3;
      n_invalid += 1;
      continue;
    }
    const uint64_t b = range[k].first, e = range[k].second;
    const uint64_t hi = (uint64_t)(std::upper_bound(cand.begin(), cand.end(),
                                                    std::make_pair(b, UINT64_MAX)) -
                                   cand.begin());
    const uint64_t c = nc ? leftmost(1, 0, size, hi, e) : nc;
    const int64_t o = old[k];
    if (c < nc && (o < 0 || cand[c].first < start[o])) {
      crefs[c] += 1;
      got_new[k] = (int64_t)c;
      kind[k] = 5;
    } else if (o >= 0) {
      more[o] += 1;
      got_old[k] = o;
      kind[k] = (start[o] == b && end[o] == e) ? 1 : 2;
    } else {
      const uint64_t r = (uint64_t)(std::lower_bound(cand.begin(), cand.end(), range[k]) -
                                    cand.begin());
      set_end(r, e);
      creator[r] = (int64_t)k;
      crefs[r] = 1;
      got_new[k] = (int64_t)r;
      kind[k] = 4;
      n_new += 1;
    }
  }
  const uint64_t n_out = n + n_new;
  ctr[0] = n_out;
  ctr[1] = n_invalid;
  ctr[2] = n_out > o_cap ? 1 : 0;
  ctr[3] = err;
  if (n_out > o_cap) return;
  // 3. merge: old records first on equal starts; created ones in rank order
  std::vector<int64_t> placed(nc, -1);
  uint64_t i = 0, r = 0, w = 0;
  while (r < nc && creator[r] < 0) ++r;
  while (i < n || r < nc) {
    const bool take_old = i < n && (r >= nc || start[i] <= cand[r].first);
    if (take_old) {
      o_start[w] = start[i];
      o_end[w] = end[i];
      o_lkey[w] = lkey[i];
      o_refs[w] = (uint32_t)(refs[i] + more[i]);
      remap[i] = (int64_t)w;
      ++i;
    } else {
      o_start[w] = cand[r].first;
      o_end[w] = cand[r].second;
      o_lkey[w] = new_lkey[creator[r]];
      o_refs[w] = (uint32_t)crefs[r];
      placed[r] = (int64_t)w;
      ++r;
      while (r < nc && creator[r] < 0) ++r;
    }
    ++w;
  }
  for (uint64_t k = 0; k < n_q; ++k) {
    if (kind[k] == 3) handle[k] = -1;
    else if (got_new[k] >= 0) handle[k] = placed[got_new[k]];
    else handle[k] = remap[got_old[k]];
  }
}

void oracle_mr_deregister(const int64_t* h, uint64_t n_h, const uint64_t* start,
                          const uint64_t* end, const uint32_t* lkey, const uint32_t* refs,
                          uint64_t n, uint64_t* o_start, uint64_t* o_end, uint32_t* o_lkey,
                          uint32_t* o_refs, int64_t* remap, uint8_t* status, uint64_t* ctr) {
  std::vector<uint64_t> left(refs, refs + n);
  uint64_t n_stale = 0;
  for (uint64_t k = 0; k < n_h; ++k) {
    const int64_t i = h[k];
    if (i < 0 || (uint64_t)i >= n || left[i] == 0) {
      status[k] = 2;
      n_stale += 1;
      continue;
    }
    left[i] -= 1;
    status[k] = left[i] == 0 ? 1 : 0;
  }
  uint64_t w = 0;
  for (uint64_t i = 0; i < n; ++i) {
    if (left[i] == 0) {
      remap[i] = -1;
      continue;
    }
    o_start[w] = start[i];
    o_end[w] = end[i];
    o_lkey[w] = lkey[i];
    o_refs[w] = (uint32_t)left[i];
    remap[i] = (int64_t)w;
    ++w;
  }
  ctr[0] = w;
  ctr[1] = n_stale;
  ctr[2] = 0;
  ctr[3] = 0;
}

// ---------------------------------------------------------------- CQ mirror
// Readings: a completion entry is 16 bytes (four dwords) in the NVMe layout,
// whose phase tag is bit 16 of the fourth dword; a fresh queue expects
// phase 1, and the expected phase flips each time the head wraps to 0; an
// entry is copied whole to the same position of the host CQ.
//
// One pass of the mirror over one queue: starting at (head, phase), every
// entry whose phase tag is the expected one is copied, in queue order,
// stopping at the first entry that is not, or after `max` entries. Returns
// how many were copied; head and phase are advanced past them.
uint32_t oracle_cq_mirror_pass(const uint32_t* dev_cq, uint32_t depth, uint32_t* head,
                               uint32_t* phase, uint32_t* host_cq, uint32_t max) {
  uint32_t copied = 0;
  while (copied < max) {
    const uint32_t* entry = dev_cq + 4 * (uint64_t)*head;
    const uint32_t tag = (entry[3] >> 16) & 1u;
    if (tag != *phase) break;
    for (int w = 0; w < 4; ++w) host_cq[4 * (uint64_t)*head + w] = entry[w];
    copied += 1;
    *head += 1;
    if (*head == depth) {
      *head = 0;
      *phase ^= 1u;
    }
  }
  return copied;
}

// The acknowledgement written by a warp that last worked under generation
// `cur` (0 if under none) and now finds generation `now`: once the
// generation has moved on from an odd value, that odd value; on finding an
// even generation, the odd value before it (a queue detached before the
// warp took it up has nothing to drain). Otherwise `keep` (no write).
uint32_t oracle_cq_ack(uint32_t cur, uint32_t now, uint32_t keep) {
  if ((cur & 1u) && now != cur) return cur;
  if ((now & 1u) == 0 && now > 0) return now - 1;
  return keep;
}

}  // extern "C"
