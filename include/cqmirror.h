/*
 * cqmirror.h -- the completion-queue mirror of libdescbuild.so (CUDA, sm_103a).
 *
 * Source: xNVMe "uPCIe CUDA" backend page, section "Completions in device
 * memory". That section moves an NVMe completion queue (CQ) out of host
 * memory into device memory, next to the data the controller writes, and
 * has a GPU kernel forward each completion to the host CQ that the CPU keeps
 * polling as before.
 *
 * This header's contract, as invariants the library keeps:
 *  - One kernel launch serves up to 64 queues, one warp per queue, on a
 *    stream of its own.
 *  - Host and kernel share a table of 64-byte slots, one per queue: the
 *    device CQ, the host CQ, the depth, a generation counter and an
 *    acknowledgement.
 *  - The generation is odd exactly while the slot describes a live queue.
 *    db_cq_attach fills the slot first and bumps the generation to odd last;
 *    db_cq_detach bumps it to even.
 *  - The warp mirrors a queue only under the odd generation it read. When
 *    it sees any other value, it stops touching that queue's CQs and stores
 *    the odd generation it was serving into `ack`. A warp serving no queue
 *    that sees an even, non-zero generation stores the odd value just below
 *    it (the queue was detached before the warp took it up).
 *  - The host reuses or releases a slot's CQ memory only after `ack` holds
 *    the slot's last odd generation (db_cq_wait_ack); db_cq_attach refuses a
 *    slot whose last generation is not acknowledged yet (-EBUSY).
 *
 * What differs from the page: the kernel is never resident without a limit.
 * A launch ends when the host raises `stop` or after `limit_ns`, whichever
 * comes first. Each warp keeps its progress (head, phase) in its slot, so a
 * new launch resumes every attached queue where the last one left off.
 *
 * Entry format (NVMe completion queue entry, 16 bytes): four little-endian
 * dwords; the phase tag is bit 16 of the fourth. Entry i of a queue is
 * written with phase tag 1 on the first pass through the queue, 0 on the
 * second, and so on. The mirror copies an entry whole, to the same position
 * of the host CQ: the first three dwords, then (ordered after them at
 * system scope) the fourth, so a host that sees the new phase tag sees the
 * whole entry.
 *
 * Memory: the slot table, `stop` and every host CQ are pinned host memory
 * (cudaHostAlloc / cudaMallocHost, or registered with cudaHostRegister),
 * used through the same pointer on both sides (unified addressing). Device
 * CQs are device memory. The slot table starts zero-filled. The library
 * allocates nothing.
 *
 * Ordering the writer of a device CQ must keep: an entry's first three
 * dwords must be in memory no later than the fourth dword that carries the
 * new phase tag. (A controller writes an entry in one posted write. A host
 * standing in for one, as the tests do, copies the entries with the old
 * tag and then again with the new one, in stream order.)
 */
#ifndef CQMIRROR_H
#define CQMIRROR_H

#include <stdint.h>

#include "descbuild.h" /* db_counters, DB_ERR_TIMEOUT, db_strerror */

#ifdef __cplusplus
extern "C" {
#endif

#define DB_CQ_MAX_SLOTS 64
#define DB_CQ_MAX_DEPTH 65536
#define DB_CQ_MAX_LIMIT_NS 60000000000ull /* one launch stays resident 60 s at most */

typedef struct db_cq_slot {
  /* Written by the host (db_cq_attach, db_cq_detach). */
  uint64_t dev_cq;     /* device CQ: depth x 16 bytes of device memory, 16-byte aligned */
  uint64_t host_cq;    /* host CQ: depth x 16 bytes of pinned host memory, 16-byte aligned */
  uint32_t depth;      /* entries, 2 .. DB_CQ_MAX_DEPTH */
  uint32_t generation; /* odd while the queue is attached; starts at 0 */
  /* Written by the kernel. */
  uint32_t ack;        /* the last odd generation the kernel is done with */
  uint32_t seen;       /* the generation that head, phase and copied belong to */
  uint32_t head;       /* next entry to copy */
  uint32_t phase;      /* phase tag expected at head */
  uint64_t copied;     /* completions copied under `seen` */
  /* Written by the host before db_cq_attach, read when the kernel takes the
   * generation up. */
  uint32_t flags;      /* 0, or DB_CQ_TIMED */
  /* Written by the kernel, for a slot attached with DB_CQ_TIMED. */
  uint32_t lat_ns;     /* the last batch: new tags seen -> its entries visible at system scope */
  uint64_t lat_seq;    /* `copied` after that batch (written after lat_ns, release order) */
} db_cq_slot;          /* 64 bytes */

/* A timed slot: after each batch the warp waits for its host-CQ writes to
 * be performed at system scope (a fence.sc.sys per lane) and records the
 * time from reading the batch's new phase tags in the device CQ to that
 * point (%globaltimer, ns) in lat_ns, then the batch's `copied` value in
 * lat_seq. The wait costs the warp that time per batch, so only queues
 * being measured should be timed. */
#define DB_CQ_TIMED 1u

/* Launch the mirror for slots[0 .. n_slots) on `stream`: warp i serves
 * slot i. The launch returns at once (the kernel stays resident).
 *   slots     pinned host memory, n_slots entries, 64-byte aligned
 *   n_slots   1 .. DB_CQ_MAX_SLOTS
 *   stop      pinned host memory; the kernel ends once *stop != 0
 *             (db_cq_request_stop)
 *   limit_ns  1 .. DB_CQ_MAX_LIMIT_NS: the kernel ends by itself after this
 *   ctr       NULL or device memory, zeroed by the call on `stream`, then:
 *             total = completions copied by this launch; n_invalid = slots
 *             found attached with a depth or address db_cq_attach would
 *             refuse (such a slot is not served, only acknowledged);
 *             err = DB_ERR_TIMEOUT when the limit, not `stop`, ended it.
 * While the kernel runs, cudaDeviceSynchronize() and cudaFree() wait for
 * it: synchronise on streams instead. Returns 0, -EINVAL, -ENODEV (no
 * CUDA device, or a pointer that is not pinned host memory) or -EIO. */
int db_cq_mirror(db_cq_slot* slots, uint32_t n_slots, const uint32_t* stop, uint64_t limit_ns,
                 db_counters* ctr, void* stream);

/* Host side of the slot protocol (host code only; callable while the
 * kernel runs; no GPU work). */

/* Attach a queue pair to a detached slot: fills the addresses and depth,
 * then raises the generation to the next odd value (release order), which
 * goes to *generation. -EBUSY if the slot is attached or its previous
 * generation has not been acknowledged; -EINVAL for a depth outside
 * 2 .. DB_CQ_MAX_DEPTH, a null or misaligned address; -ENODEV when
 * dev_cq is not CUDA device memory or host_cq is not pinned host memory
 * (or no CUDA device can say). */
int db_cq_attach(db_cq_slot* slot, uint64_t dev_cq, uint64_t host_cq, uint32_t depth,
                 uint32_t* generation);

/* Detach: raises an odd generation to the even value after it; the odd
 * value goes to *generation. The queue's memory may be freed once
 * db_cq_wait_ack has seen that value. -EINVAL if the slot is not attached. */
int db_cq_detach(db_cq_slot* slot, uint32_t* generation);

/* Wait until slot->ack == generation (acquire order), polling for at most
 * timeout_ns. 0, or -ETIMEDOUT (for example when no mirror is running). */
int db_cq_wait_ack(const db_cq_slot* slot, uint32_t generation, uint64_t timeout_ns);

/* Reap a host CQ the way its owner polls it: from (*head, *phase), copy
 * each entry whose phase tag is the expected one to out (host memory,
 * max x 16 bytes), in order, stopping at the first stale entry. Advances
 * *head and *phase (the phase flips when the head wraps). Returns the
 * count, or -EINVAL. */
int db_cq_host_reap(const void* host_cq, uint32_t depth, uint32_t* head, uint32_t* phase,
                    void* out, uint32_t max);

/* Ask a running mirror to end (release order). */
void db_cq_request_stop(uint32_t* stop);

#ifdef __cplusplus
}
#endif

#endif /* CQMIRROR_H */
