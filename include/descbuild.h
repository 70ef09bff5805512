/*
 * descbuild.h -- batched translation of GPU buffer ranges into DMA descriptors.
 *
 * C ABI of libdescbuild.so (CUDA, sm_103a). Three batched operations:
 *
 *   db_prp_build   NVMe PRP1/PRP2 and chained 4 KiB PRP lists from heap
 *                  offsets and a 64 KiB-granular bus-address LUT.
 *   db_mr_lookup   classify ranges against a sorted registration (MR) table
 *                  after rounding them to whole 4 KiB pages
 *                  (db_mr_lookup_overlap: records may overlap).
 *   db_wqe_bucket  translate symmetric-heap puts and stable-partition them
 *                  into per-queue rings of 64-byte work-queue entries.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Every data pointer is a DEVICE pointer (cudaMalloc / torch), owned by the
 *    caller, unless its comment says "host". The library allocates nothing
 *    and keeps no state between calls other than what it leaves in the
 *    caller's workspace.
 *  - `stream` is a cudaStream_t passed as void*. Work is enqueued on it and the
 *    call returns without waiting: results are valid once the caller has
 *    synchronised with that stream. Inputs must stay alive and unchanged
 *    until then.
 *  - Return value: 0 on success, or a negative errno:
 *      -EINVAL  a null or misaligned pointer, or an argument outside its range
 *      -ENOSPC  the workspace is smaller than *_workspace_size reports
 *      -EIO     the CUDA launch failed (db_last_cuda_error() gives the code)
 *    The return covers argument checks and the launch only. Errors that
 *    depend on the data are reported in device memory (per-request status,
 *    db_counters) and are read after synchronising.
 *  - n == 0 is a successful call that only zeroes the counters it would
 *    otherwise fill.
 *  - Workspaces: `ws` is device memory of at least *_workspace_size() bytes,
 *    256-byte aligned, ZERO-FILLED when first allocated. Each call leaves it
 *    ready for the next one, so it is never cleared again. One workspace
 *    serves one call at a time: calls sharing a workspace must be ordered on
 *    one stream.
 */
#ifndef DESCBUILD_H
#define DESCBUILD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- records ------------------------------------------------------------ */

/* One NVMe transfer: `len` bytes at byte offset `off` of the device heap. */
typedef struct db_prp_req {
  uint64_t off;
  uint32_t len;
  uint32_t rsvd; /* ignored */
} db_prp_req;    /* 16 bytes */

typedef struct db_prp_out {
  uint64_t prp1;
  uint64_t prp2;
} db_prp_out;    /* 16 bytes */

/* A byte range [addr, addr + size). */
typedef struct db_range {
  uint64_t addr;
  uint64_t size;
} db_range;      /* 16 bytes */

/* One put: `bytes` bytes at symmetric-heap offset `off` to PE `pe` on its
 * queue pair `qp`. */
typedef struct db_put_req {
  uint64_t off;
  uint32_t bytes;
  uint16_t pe;
  uint16_t qp;
} db_put_req;    /* 16 bytes */

/* A work-queue entry as written into a ring. */
typedef struct db_wqe {
  uint64_t raddr;     /* peer_ptrs[pe] + off               */
  uint64_t laddr;     /* local_base + off                  */
  uint32_t len;       /* bytes                             */
  uint32_t lkey;      /* the local object's lkey           */
  uint32_t rkey;      /* rkeys[pe]                         */
  uint32_t flags;     /* 0                                 */
  uint64_t seq;       /* post index in its ring            */
  uint32_t req_index; /* position of the put in the batch  */
  uint32_t rsvd[5];   /* 0                                 */
} db_wqe;             /* 64 bytes */

/* A put to a PE reached without RDMA (db_wqe_bucket_transport): the copy
 * this process issues itself, through its mapping of the peer's heap. */
typedef struct db_direct {
  uint64_t dst;       /* peer_ptrs[pe] + off (the mapped peer heap) */
  uint64_t src;       /* local_base + off                           */
  uint32_t len;       /* bytes                                      */
  uint32_t req_index; /* position of the put in the batch           */
  uint16_t pe;
  uint8_t transport;  /* DB_XPORT_P2P or DB_XPORT_SDMA              */
  uint8_t rsvd0;      /* 0                                          */
  uint32_t rsvd1;     /* 0                                          */
} db_direct;          /* 32 bytes */

/* Batch counters, written by the device at the end of a call. */
typedef struct db_counters {
  uint64_t total;      /* prp: list pages the batch needs; wqe: entries posted */
  uint64_t n_invalid;  /* malformed requests                                  */
  uint64_t n_overflow; /* prp: lists that did not fit; wqe: puts refused      */
  uint64_t err;        /* DB_ERR_* bits                                       */
} db_counters;

/* ---- codes ----------------------------------------------------------------*/

#define DB_PRP_OK 0
#define DB_PRP_INVALID 1  /* len == 0, off % 4 != 0, or off + len > heap_size */
#define DB_PRP_OVERFLOW 2 /* the request's list pages would end past the arena */

#define DB_MR_MISS 0
#define DB_MR_EXACT 1
#define DB_MR_CONTAINED 2
#define DB_MR_INVALID 3

#define DB_ERR_TIMEOUT 1u       /* a bounded wait for another CTA ran out; outputs undefined */
#define DB_ERR_RING_OVERFLOW 2u /* a ring was asked for more than `depth` entries            */
#define DB_ERR_TABLE_ORDER 4u   /* the MR table is not sorted and non-overlapping            */

#define DB_PRP_ZERO_TAIL 1u     /* db_prp_build: zero the unused slots of each last list page */
/* db_prp_build schedule (results are the same either way; by default a batch
 * that one wave of the pair kernel holds takes two kernels, a larger one one): */
#define DB_PRP_SCHED_SINGLE 2u  /* one persistent kernel, tiles by ticket, decoupled lookback */
#define DB_PRP_SCHED_SPLIT 4u   /* a pair kernel, then a list kernel for the tiles with lists */

#define DB_XPORT_RDMA 0 /* db_wqe_bucket_transport: how each PE is reached */
#define DB_XPORT_P2P 1
#define DB_XPORT_SDMA 2

/* ---- PRP build ------------------------------------------------------------
 * Source: xNVMe "uPCIe CUDA" backend page. Introduction: the CUDA driver
 * exports device memory at 64 KiB granularity; the bus address of each
 * 64 KiB chunk sits in a LUT indexed by chunk, and PRP entries are built at
 * 4 KiB from sub-page offsets inside a chunk. "Memory Architecture": PRP
 * lists live in their own memory region. "Limitations": one 4 KiB list page
 * holds 512 entries (513 x 4 KiB with PRP1); longer lists chain through the
 * last slot of each full page (NVMe convention, required by the large
 * workload). List pages are placed by an exclusive scan of per-request
 * list-page counts in request order.
 *
 * For request i (off, len), n = pages of 4 KiB that [off, off+len) touches,
 * bus(x) = lut[x >> 16] + (x & 0xFFFF):
 *   prp1 = bus(off)
 *   n == 1: prp2 = 0
 *   n == 2: prp2 = bus(page_floor(off) + 4096)
 *   n >= 3: prp2 = arena_base + 4096 * page_base[i], and list pages
 *           page_base[i] .. page_base[i] + L_i - 1 of the arena hold the
 *           n - 1 entries bus(page_floor(off) + 4096 k), k = 1 .. n-1;
 *           every page but the last holds 511 entries and, in slot 511,
 *           the bus address of the next page; the last holds up to 512.
 *   page_base[i] = sum of L_j over j < i (valid requests only).
 *
 * Arguments
 *   req              [n] requests (16-byte aligned)
 *   lut              [heap_size / 65536] bus addresses, 64 KiB-aligned, non-zero
 *   heap_size        bytes of device heap; a multiple of 65536
 *   arena_base       bus address of list page 0; a multiple of 4096
 *   arena_cap_pages  pages the arena holds
 *   arena            [arena_cap_pages][512] uint64: the arena's contents (32-byte aligned),
 *                    in device memory or in pinned host memory (the host-memory
 *                    region the lists live in on the source page; the kernel
 *                    then writes the lists across the CPU-GPU link).
 *                    Unused slots of a list's last page are undefined: the
 *                    library leaves them as they were, except that it may write
 *                    0 into the ones sharing the last entry's 32-byte sector (at
 *                    most three; this kernel does, so that every list ends on a
 *                    whole sector). DB_PRP_ZERO_TAIL writes 0 into all of them.
 *   prp              [n] output (16-byte aligned)
 *   page_base        [n] output or NULL
 *   status           [n] output (DB_PRP_*) or NULL
 *   ctr              output counters or NULL: total list pages (including
 *                    those of requests that did not fit), n_invalid,
 *                    n_overflow, err
 *   flags            DB_PRP_ZERO_TAIL, and at most one of DB_PRP_SCHED_SINGLE /
 *                    DB_PRP_SCHED_SPLIT (the schedule; the outputs do not depend
 *                    on it). By default a batch of at most one wave of the pair
 *                    kernel's tiles (4 CTAs x 2048 requests per SM) takes the
 *                    two-kernel schedule: all its requests are loaded at once,
 *                    and only tiles that own lists (or all, when page_base is
 *                    asked for) go through the list kernel. Larger batches take
 *                    the single persistent kernel, which overlaps the scan of
 *                    later tiles with the lists of earlier ones.
 * A request that is invalid or whose list does not fit gets prp = {0, 0}
 * and writes no list; one that does not fit still advances page_base.
 * Limits: n <= 2^28, arena_cap_pages <= 2^40.
 */
int db_prp_workspace_size(uint64_t n, size_t* bytes);
int db_prp_build(const db_prp_req* req, uint64_t n, const uint64_t* lut, uint64_t heap_size,
                 uint64_t arena_base, uint64_t arena_cap_pages, uint64_t* arena,
                 db_prp_out* prp, uint64_t* page_base, uint8_t* status, db_counters* ctr,
                 uint32_t flags, void* ws, size_t ws_bytes, void* stream);

/* ---- MR lookup ------------------------------------------------------------
 * Source: "NCCL expert course 26: GPUDirect RDMA, DMA-BUF, MR and the
 * registration cache". "IB Backend MR Cache": a range is widened to whole
 * pages (addr = data & -pageSize; pages = ceil((data + size - addr) /
 * pageSize)); an existing MR is reused only if it fully contains the widened
 * range; partial overlap is not a hit. "Communicator User Registration
 * Cache": the same rounding over records kept sorted by address.
 *
 * For query k: base = addr & ~4095, aend = base + 4096 * pages.
 *   invalid (size == 0, or addr + size > 2^64 - 4096): kind = DB_MR_INVALID
 *   the lowest i with mr_start[i] <= base and aend <= mr_end[i]:
 *     kind = DB_MR_EXACT if both ends are equal, else DB_MR_CONTAINED;
 *     idx = i, lkey = mr_lkey[i]
 *   none: kind = DB_MR_MISS, idx = -1, lkey = 0
 *
 * Arguments
 *   q         [n_q] query ranges (16-byte aligned)
 *   mr_start  [n_mr] record starts, sorted ascending
 *   mr_end    [n_mr] record ends (exclusive); records must not overlap and
 *             must not be empty (mr_start[i] < mr_end[i] <= mr_start[i+1])
 *   mr_lkey   [n_mr]
 *   idx, lkey, kind  [n_q] outputs
 *   ctr       NULL or counters: err gets DB_ERR_TABLE_ORDER when the table
 *             breaks the ordering rule (results are then undefined);
 *             n_invalid counts invalid queries; total = hits
 * Limits: n_mr < 2^31.
 */
int db_mr_workspace_size(uint64_t n_mr, size_t* bytes);
int db_mr_lookup(const db_range* q, uint64_t n_q, const uint64_t* mr_start,
                 const uint64_t* mr_end, const uint32_t* mr_lkey, uint64_t n_mr, int32_t* idx,
                 uint32_t* lkey, uint8_t* kind, db_counters* ctr, void* ws, size_t ws_bytes,
                 void* stream);

/* db_mr_lookup_overlap: the same classification on a table whose records
 * may overlap. Source: the same page, "IB Backend MR Cache": a range that
 * only partly overlaps a cached MR is no hit and is registered anew, so the
 * cache comes to hold MRs that overlap one another, and "Communicator User
 * Registration Cache" inserts each new record in address order.
 *
 * The answer is the same as db_mr_lookup's rule above: the LOWEST i with
 * mr_start[i] <= base and aend <= mr_end[i]. Records must be non-empty and
 * sorted by start (mr_start[i] < mr_end[i], mr_start[i] <= mr_start[i+1]);
 * ends are free. Every record at or after the last one starting at or
 * below base starts too late, so the answer is the first i <= j whose
 * prefix maximum of ends reaches aend (the prefix maximum is kept in the
 * workspace, rebuilt on every call).
 *
 * Arguments, workspace (db_mr_workspace_size), counters and limits as for
 * db_mr_lookup; err gets DB_ERR_TABLE_ORDER when starts are not sorted or
 * a record is empty.
 */
int db_mr_lookup_overlap(const db_range* q, uint64_t n_q, const uint64_t* mr_start,
                         const uint64_t* mr_end, const uint32_t* mr_lkey, uint64_t n_mr,
                         int32_t* idx, uint32_t* lkey, uint8_t* kind, db_counters* ctr,
                         void* ws, size_t ws_bytes, void* stream);

/* ---- put translation and WQE bucketing ------------------------------------
 * Source: "mori communication library analysis (1)". Static-heap put:
 * raddr = peerPtrs[pe] + offset with rkey = peerRkeys[pe] and the source
 * object's lkey, the whole transfer in one WQE. Warp-level WQE slot
 * reservation: each entry takes the next post index of its send queue.
 *
 * Put i is valid when pe < world, qp < n_qp, bytes >= 1 and
 * off + bytes <= heap_size. Valid puts go to ring r = pe * n_qp + qp in
 * batch order: the k-th of ring r takes seq = head[r] + k and lands in
 * slot seq & (depth - 1) of ring r, i.e. at
 * rings + (r * depth + (seq & (depth - 1))) * 64.
 * A ring asked for more than `depth` entries by one batch takes none of
 * them: its head stays, its puts count in n_overflow and err gets
 * DB_ERR_RING_OVERFLOW. Otherwise head[r] += count[r].
 *
 * Arguments
 *   req         [n] puts (16-byte aligned)
 *   peer_ptrs   [world] heap base of each PE
 *   rkeys       [world]
 *   world, n_qp PEs and queue pairs per PE; 1 <= world * n_qp <= 1024
 *   local_base, lkey, heap_size  the local object
 *   rings       [world * n_qp][depth] db_wqe (64-byte aligned), in device memory or
 *               in pinned host memory (a send queue the NIC reads may sit in either;
 *               the kernel then writes each WQE across the CPU-GPU link). Only the
 *               entries of this batch are written; the kernel reads none.
 *   depth       entries per ring, a power of two
 *   head        [world * n_qp] in/out post indices
 *   count       [world * n_qp] output: valid puts per ring in this batch
 *   ctr         NULL or counters: total = entries posted
 * Limits: n < 2^32.
 */
int db_wqe_workspace_size(uint64_t n, uint32_t n_rings, size_t* bytes);
int db_wqe_bucket(const db_put_req* req, uint64_t n, const uint64_t* peer_ptrs,
                  const uint32_t* rkeys, uint32_t world, uint32_t n_qp, uint64_t local_base,
                  uint32_t lkey, uint64_t heap_size, db_wqe* rings, uint64_t depth,
                  uint64_t* head, uint32_t* count, db_counters* ctr, void* ws,
                  size_t ws_bytes, void* stream);

/* ---- put translation with a transport per PE --------------------------------
 * Source: "mori communication library analysis (1)": the put path branches
 * on its target PE's transport type (RDMA, P2P or SDMA), fixed per PE when
 * the connections are set up; for a PE that is not reached over RDMA the
 * symmetric object's peer pointer holds the address at which this process
 * maps that PE's heap, so the destination is peer_ptrs[pe] + off whatever
 * the transport.
 *
 * Put i is valid under db_wqe_bucket's rule and when transport[pe] is one of
 * DB_XPORT_RDMA / _P2P / _SDMA (any other code makes the PE's puts invalid).
 *   transport[pe] == DB_XPORT_RDMA: a WQE, exactly as db_wqe_bucket (ring
 *     r = pe * n_qp + qp, seq = head[r] + earlier RDMA puts of ring r, the
 *     overflow rule); puts to other PEs take no ring slot and do not count
 *     in count[] or in any ring's overflow decision.
 *   P2P or SDMA: no WQE; a db_direct record, the k-th valid such put of the
 *     batch (batch order) at direct[k]: dst = peer_ptrs[pe] + off,
 *     src = local_base + off, len = bytes, req_index, pe, transport.
 *
 * Arguments as for db_wqe_bucket, and
 *   transport  [world] DB_XPORT_* per PE (device memory)
 *   direct     [n] output, 32-byte aligned: room for every put of the batch
 *   n_direct   one uint64_t output (8-byte aligned): records written
 *   ctr        NULL or counters: total = WQEs posted, n_invalid, n_overflow
 *              = puts of overflowing rings
 * Workspace: db_wqe_workspace_size(n, world * n_qp) bytes, as for
 * db_wqe_bucket. Only the static heap has this variant.
 */
int db_wqe_bucket_transport(const db_put_req* req, uint64_t n, const uint64_t* peer_ptrs,
                            const uint32_t* rkeys, const uint8_t* transport, uint32_t world,
                            uint32_t n_qp, uint64_t local_base, uint32_t lkey,
                            uint64_t heap_size, db_wqe* rings, uint64_t depth, uint64_t* head,
                            uint32_t* count, db_direct* direct, uint64_t* n_direct,
                            db_counters* ctr, void* ws, size_t ws_bytes, void* stream);

/* ---- put translation on a VMM heap ------------------------------------------
 * Source: "mori communication library analysis (1)", the VMM-heap branch of
 * the put path: while bytes remain, the WQE covers the rest of the chunk
 * holding the current source address, the rest of the chunk holding the
 * current destination address, or what remains, whichever is least, with the
 * source chunk's lkey and the destination chunk's remote address and rkey.
 *
 * The heap is cut into chunks of C = 2^chunk_shift bytes at the same offsets
 * on every PE (n_chunks = ceil(heap_size / C)). A valid put (as for
 * db_wqe_bucket) covering [off, off + bytes) makes one WQE for each chunk c
 * it touches, in address order; for the part [s, e) of chunk c:
 *   raddr = chunk_raddr[pe * n_chunks + c] + (s - c * C)
 *   rkey  = chunk_rkey[pe * n_chunks + c]
 *   laddr = local_base + s,  lkey = chunk_lkey[c],  len = e - s
 *   seq, req_index as for db_wqe_bucket; a put's WQEs take consecutive post
 *   indices of its ring.
 * count[r] is the WQEs ring r was asked for (saturating at 2^32 - 1); a ring
 * asked for more than `depth` takes none. ctr: total = WQEs posted,
 * n_invalid = invalid puts, n_overflow = WQEs of overflowing rings.
 * With one chunk as large as the heap this is db_wqe_bucket with
 * peer_ptrs[pe] = chunk_raddr[pe], rkeys[pe] = chunk_rkey[pe] and
 * lkey = chunk_lkey[0].
 *
 * Packet sequence numbers (same page, the BNXT branch), when mtu != 0: a WQE
 * of len bytes uses ceil(len / mtu) PSNs; its first PSN, psn_head[r] plus
 * the PSNs of ring r's earlier WQEs in the batch, is stored as a u32 at byte
 * 44 (rsvd[0]). A ring that takes its batch advances psn_head[r] by its PSN
 * total. The post index still advances by one per WQE. With mtu == 0 byte
 * 44 stays 0 and psn_head is not used.
 *
 * Arguments as for db_wqe_bucket, and
 *   chunk_raddr  [world][n_chunks] remote address of each chunk (8-byte aligned)
 *   chunk_rkey   [world][n_chunks]
 *   chunk_lkey   [n_chunks]
 *   chunk_shift  4 <= chunk_shift <= 48
 *   mtu          0, or 512 <= mtu <= 2^20 with chunk_shift >= 12
 *   psn_head     [world * n_qp] in/out PSN counters (8-byte aligned); NULL if mtu == 0
 * Limits: n < 2^32, depth <= 2^31, n_chunks <= 2^32, heap_size >= 1.
 * Workspace: db_wqe_vmm_workspace_size(n, world, n_qp, heap_size, chunk_shift)
 * bytes: the bucketing columns plus a per-call packed copy of the chunk tables
 * (16 bytes per PE and chunk, so that a WQE reads its chunk's remote address,
 * rkey and lkey at once); -ENOSPC below that.
 */
int db_wqe_vmm_workspace_size(uint64_t n, uint32_t world, uint32_t n_qp, uint64_t heap_size,
                              uint32_t chunk_shift, size_t* bytes);
int db_wqe_bucket_vmm(const db_put_req* req, uint64_t n, const uint64_t* chunk_raddr,
                      const uint32_t* chunk_rkey, const uint32_t* chunk_lkey,
                      uint32_t chunk_shift, uint32_t world, uint32_t n_qp, uint64_t local_base,
                      uint64_t heap_size, db_wqe* rings, uint64_t depth, uint64_t* head,
                      uint32_t* count, uint32_t mtu, uint64_t* psn_head, db_counters* ctr,
                      void* ws, size_t ws_bytes, void* stream);

/* ---- PRP build with no caller workspace ------------------------------------
 * The source pages have no counterpart to this entry point; it is an addition
 * for callers that must not allocate device memory on their submission path:
 * cudaMalloc can wait for work already queued on the device and takes driver
 * locks, so a latency-bound I/O submitter cannot afford it, and a process
 * whose device memory is handed out up front by its own allocator may have no
 * room for an extra cudaMalloc at all.
 *
 * Same arguments and results as db_prp_build, without `ws`/`ws_bytes`: the
 * scratch memory (a header and one status word per tile of requests) is a
 * static device array inside libdescbuild.so, sized for at most
 * DB_PRP_STATIC_MAX_REQUESTS (16,777,216) requests per call: 256 B of header
 * plus 8 B per tile of 2048 requests, 64.25 KiB in all. Every GPU that loads
 * the library holds that array until the process exits.
 *
 *  - n > DB_PRP_STATIC_MAX_REQUESTS returns -E2BIG before any GPU work.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current) and keeps it with the
 *    ID of the device's current CUDA context; make that first call before
 *    any stream capture on the device. Later calls compare the context ID
 *    (one driver query) and look the address up again when it differs, as
 *    after cudaDeviceReset, which unloads the array with its context. A new
 *    context's copy of the array starts zeroed.
 *  - The array starts zeroed and every call leaves it ready for the next one,
 *    so no call has to clear it. All calls share it: calls whose work can
 *    overlap on the GPU (different streams without ordering between them, or
 *    different host threads) race on it and must be serialised by the caller.
 *  - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 */
#define DB_PRP_STATIC_MAX_REQUESTS (1u << 24)
int db_prp_build_static(const db_prp_req* req, uint64_t n, const uint64_t* lut,
                        uint64_t heap_size, uint64_t arena_base, uint64_t arena_cap_pages,
                        uint64_t* arena, db_prp_out* prp, uint64_t* page_base, uint8_t* status,
                        db_counters* ctr, uint32_t flags, void* stream);

/* ---- misc ----------------------------------------------------------------- */
const char* db_strerror(int code);
/* The cudaError_t of the last -EIO on this thread (0 if none). */
int db_last_cuda_error(void);

#ifdef __cplusplus
}
#endif
#endif /* DESCBUILD_H */
