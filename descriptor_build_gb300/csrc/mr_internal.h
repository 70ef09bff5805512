// Internal entry points of the MR lookup, shared with the registration
// batches (not part of the C ABI).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "descbuild.h"

namespace db {
namespace mr {

// db_mr_lookup / db_mr_lookup_overlap with the granule as a parameter:
// granule_shift 12 widens queries to 4 KiB pages, 16 to 64 KiB granules
// (the latter always on the overlap path).
int lookup(const db_range* q, uint64_t n_q, const uint64_t* mr_start, const uint64_t* mr_end,
           const uint32_t* mr_lkey, uint64_t n_mr, int32_t* idx, uint32_t* lkey, uint8_t* kind,
           db_counters* ctr, void* ws, size_t ws_bytes, cudaStream_t s, bool overlap,
           int granule_shift);

// Workspace bytes the lookup needs for a table of n_mr records.
size_t workspace_bytes(uint64_t n_mr);

}  // namespace mr
}  // namespace db
