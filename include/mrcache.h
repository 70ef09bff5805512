/*
 * mrcache.h -- registration-cache mutation batches of libdescbuild.so
 * (CUDA, sm_103a): register and deregister many ranges in one call.
 *
 * Sources: "NCCL expert course 26: GPUDirect RDMA, DMA-BUF, MR and the
 * registration cache". "IB Backend MR Cache": an MR that fully contains the
 * widened range is reused and takes one more reference; partial overlap is
 * no hit and the range is registered anew; the cache grows from 0 to 32
 * entries, then doubles; deregistration drops a reference and deregisters
 * the MR at zero; a handle not in the cache is an error. "Communicator User
 * Registration Cache": the new record is inserted in address order. The
 * ncclCommRegister experiment: the same range twice and a range inside it
 * share one record (refs 3); three deregistrations delete it; the stale
 * handle is then invalid usage. xNVMe "uPCIe CUDA" backend page:
 * xnvme_buf_register covers whole 64 KiB device pages and refcounts what it
 * covers, so registering twice is cheap.
 *
 * Conventions are those of descbuild.h (device pointers owned by the caller,
 * asynchronous on `stream`, negative errno returns, data-dependent results
 * in db_counters). A table is four device arrays of n records sorted by
 * start (ties allowed, records may overlap, start < end):
 *   start, end  u64 (end exclusive), lkey u32, refs u32.
 * A handle is a record index. A call writes the table after the batch into
 * separate output arrays and `remap[i]`, the index record i has after the
 * batch (-1 once removed), so the caller can carry its handles forward.
 *
 * A batch gives the result of the pages' one-call-at-a-time operations
 * applied to its requests in order:
 *  - Registration. Each request is widened to whole granules (4 KiB, or 64 KiB
 *    for the xNVMe registry) and looked up in the table as the requests
 *    before it in the batch left it: the old records and the records those
 *    requests created, in table order (start; an old record before a new one
 *    of the same start; new records of one start in the order they were
 *    made). The lowest-index record holding it takes one more reference:
 *    an old record (kind DB_MR_EXACT or DB_MR_CONTAINED) or one an earlier
 *    request of the batch created (DB_MR_NEW_DUP, whether the same range, a
 *    wider one, or one that starts before the old record that also holds
 *    it). A request that no record holds creates a record with one
 *    reference and its new_lkey (DB_MR_NEW), placed after every record
 *    starting at or before it.
 *  - Deregistration, in batch order: each handle drops one reference of its
 *    record; the handle that drops the last one releases the record
 *    (DB_DEREG_RELEASED); a handle naming no record or a released one is
 *    stale (DB_DEREG_STALE, the experiment's invalid usage). Records left
 *    with no reference are removed.
 */
#ifndef MRCACHE_H
#define MRCACHE_H

#include <stddef.h>
#include <stdint.h>

#include "descbuild.h"

#ifdef __cplusplus
extern "C" {
#endif

#define DB_MR_NEW 4u     /* the request made a new record                                 */
#define DB_MR_NEW_DUP 5u /* a hit on a record an earlier request of the batch made        */

#define DB_DEREG_OK 0u       /* one reference dropped                      */
#define DB_DEREG_RELEASED 1u /* the last reference: the record is removed  */
#define DB_DEREG_STALE 2u    /* no such record, or already released        */

/* Table capacity after growth to hold n records: 0, then 32, then doubling
 * (the IB MR cache's growth). Host only. */
uint64_t db_mr_capacity_for(uint64_t n);

int db_mr_register_workspace_size(uint64_t n_q, uint64_t n_mr, size_t* bytes);

/* A batch of registrations.
 *   q             [n_q] ranges (16-byte aligned)
 *   new_lkey      [n_q] the lkey a new registration for request k would get
 *   granule_shift 12 (4 KiB pages) or 16 (64 KiB granules)
 *   start, end, lkey, refs  the table before the batch, n_mr records
 *   out_*         the table after the batch, room for out_cap records
 *   handle        [n_q] out: record index after the batch (-1 if invalid)
 *   kind          [n_q] out: DB_MR_EXACT / DB_MR_CONTAINED / DB_MR_NEW /
 *                 DB_MR_NEW_DUP / DB_MR_INVALID
 *   remap         [n_mr] out
 *   ctr           NULL or counters: total = records after the batch,
 *                 n_invalid, n_overflow = 1 when total > out_cap (then only
 *                 ctr and kind are written), err = DB_ERR_TABLE_ORDER when
 *                 the table is not sorted by start or holds an empty record
 *                 (results undefined).
 * Limits: n_q < 2^31, n_mr < 2^31, out_cap < 2^31; the arrays may not
 * overlap; out_* must not alias the input table. */
int db_mr_register(const db_range* q, uint64_t n_q, const uint32_t* new_lkey,
                   uint32_t granule_shift, const uint64_t* start, const uint64_t* end,
                   const uint32_t* lkey, const uint32_t* refs, uint64_t n_mr,
                   uint64_t* out_start, uint64_t* out_end, uint32_t* out_lkey,
                   uint32_t* out_refs, uint64_t out_cap, int64_t* handle, uint8_t* kind,
                   int64_t* remap, db_counters* ctr, void* ws, size_t ws_bytes, void* stream);

int db_mr_deregister_workspace_size(uint64_t n_h, uint64_t n_mr, size_t* bytes);

/* A batch of deregistrations.
 *   handle   [n_h] record indices (any value; out of range is stale)
 *   start, end, lkey, refs  the table before the batch, n_mr records
 *   out_*    the table after the batch (room for n_mr records)
 *   remap    [n_mr] out
 *   status   [n_h] out: DB_DEREG_*
 *   ctr      NULL or counters: total = records after the batch,
 *            n_invalid = stale handles.
 * Limits: n_h < 2^31, n_mr < 2^31. */
int db_mr_deregister(const int64_t* handle, uint64_t n_h, const uint64_t* start,
                     const uint64_t* end, const uint32_t* lkey, const uint32_t* refs,
                     uint64_t n_mr, uint64_t* out_start, uint64_t* out_end, uint32_t* out_lkey,
                     uint32_t* out_refs, int64_t* remap, uint8_t* status, db_counters* ctr,
                     void* ws, size_t ws_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MRCACHE_H */
