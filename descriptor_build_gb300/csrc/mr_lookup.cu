// Registration (MR) cache lookup (sm_103a).
//
// Source: "NCCL expert course 26: GPUDirect RDMA, DMA-BUF, MR and the
// registration cache" -- "IB Backend MR Cache" (widen a range to whole
// pages; reuse an MR only if it fully contains the widened range; partial
// overlap is not a hit) and "Communicator User Registration Cache" (the same
// rounding over records kept sorted by address).
//
// Two launches per call:
//   index build  copies (start, end, lkey) into 32-byte records (one L2
//                sector each), checks the table is sorted and disjoint, and
//                fills a directory D[b] = number of records starting below
//                lo + b * 2^shift (2^shift chosen so that the records' span
//                fits nb buckets) by a merge path over records and buckets.
//   lookup       kQPT queries per thread: round to pages, read D[b], D[b+1]
//                (adjacent words), binary-search the few records of the
//                bucket, read the one candidate record, classify. Queries of
//                a thread advance in lockstep so their L2 misses overlap.
// For a sorted table of disjoint non-empty records the only record that can
// contain [base, aend) is the last one starting at or below base, so the
// lowest containing index is that record or none.
#include "common.cuh"

namespace db {
namespace mr {

constexpr int kBuildThreads = 256;
constexpr int kThreads = 256;
constexpr int kQPT = 4;

struct Header {        // first 256 bytes of the workspace
  uint64_t lo;         // start of record 0
  uint32_t shift;      // bucket width is 2^shift bytes
  uint32_t nb;         // buckets (a power of two)
  unsigned int done;   // lookup CTAs finished
  unsigned int err;    // DB_ERR_TABLE_ORDER from the build
  unsigned long long hits;
  unsigned long long invalid;
};
struct alignas(32) Rec {
  uint64_t start, end;
  uint32_t lkey, pad0;
  uint64_t pad1;
};
constexpr size_t kHeaderBytes = 256;

inline uint32_t buckets_for(uint64_t n_mr) {
  uint64_t nb = 1024;
  while (nb < n_mr && nb < (1u << 22)) nb <<= 1;
  return (uint32_t)nb;
}
inline size_t dir_bytes(uint32_t nb) { return (((size_t)nb + 1) * 4 + 255) & ~(size_t)255; }
inline size_t ws_bytes_for(uint64_t n_mr) {
  return kHeaderBytes + dir_bytes(buckets_for(n_mr)) + (size_t)n_mr * sizeof(Rec);
}

struct BuildParams {
  const uint64_t* start;
  const uint64_t* end;
  const uint32_t* lkey;
  uint64_t n_mr;
  Header* hdr;
  uint32_t* dir;
  Rec* rec;
  uint32_t nb;
  uint32_t log_nb;
};

__device__ __forceinline__ uint64_t bucket_of(uint64_t x, uint64_t lo, uint32_t shift,
                                              uint32_t nb) {
  if (x < lo) return 0;
  const uint64_t b = (x - lo) >> shift;
  return b < nb ? b : nb;
}

constexpr int kMergeChunk = 32;  // merged elements per thread in the directory build

// Records: 32-byte copies and the ordering check. Directory: D[b] = number of
// records whose bucket key is below b, for b = 0..nb -- the merge of the
// (sorted) record keys with the bucket numbers, split into equal chunks of
// the merged sequence ("merge path"), so every thread does the same work
// however the records fall into buckets.
__global__ void __launch_bounds__(kBuildThreads) mr_index_kernel(const BuildParams p) {
  const uint64_t lo = p.start[0];
  const uint64_t hi = p.start[p.n_mr - 1];
  const uint64_t span = hi > lo ? hi - lo : 0;
  const uint32_t bits = span ? 64u - (uint32_t)__clzll((long long)span) : 0u;
  const uint32_t shift = bits > p.log_nb ? bits - p.log_nb : 0u;
  const uint64_t nb = p.nb;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    p.hdr->lo = lo;
    p.hdr->shift = shift;
    p.hdr->nb = p.nb;
  }
  const uint64_t tid = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const uint64_t nthreads = (uint64_t)gridDim.x * blockDim.x;

  bool bad = false;
  for (uint64_t i = tid; i < p.n_mr; i += nthreads) {
    const uint64_t s = p.start[i], e = p.end[i];
    Rec r;
    r.start = s;
    r.end = e;
    r.lkey = p.lkey[i];
    r.pad0 = 0;
    r.pad1 = 0;
    p.rec[i] = r;
    if (!(s < e) || (i > 0 && p.end[i - 1] > s)) bad = true;
  }
  if (bad) atomicOr(&p.hdr->err, DB_ERR_TABLE_ORDER);

  // Merge order: record i comes before bucket number b iff key(i) < b.
  const uint64_t n = p.n_mr;
  const uint64_t merged = n + nb + 1;
  for (uint64_t k = tid * kMergeChunk; k < merged; k += nthreads * kMergeChunk) {
    // m = records among the first k merged elements: the largest m with
    // key(m - 1) < k - m.
    uint64_t mlo = k > nb + 1 ? k - (nb + 1) : 0;
    uint64_t mhi = k < n ? k : n;
    while (mlo < mhi) {
      const uint64_t mid = (mlo + mhi + 1) >> 1;
      if (bucket_of(p.start[mid - 1], lo, shift, p.nb) < k - mid)
        mlo = mid;
      else
        mhi = mid - 1;
    }
    uint64_t i = mlo, b = k - mlo;
    for (int step = 0; step < kMergeChunk && (i < n || b <= nb); ++step) {
      if (i < n && (b > nb || bucket_of(p.start[i], lo, shift, p.nb) < b))
        ++i;
      else
        p.dir[b++] = (uint32_t)i;
    }
  }
}

struct LookupParams {
  const ulonglong2* q;
  uint64_t n_q;
  uint64_t n_mr;
  const Header* hdr_ro;
  Header* hdr;
  const uint32_t* dir;
  const Rec* rec;
  int32_t* idx;
  uint32_t* lkey;
  uint8_t* kind;
  db_counters* ctr;
};

__global__ void __launch_bounds__(kThreads) mr_lookup_kernel(const LookupParams p) {
  const uint64_t pol_first = policy_evict_first();
  const uint64_t pol_last = policy_evict_last();
  const uint64_t lo = p.hdr_ro->lo;
  const uint32_t shift = p.hdr_ro->shift;
  const uint32_t nb = p.hdr_ro->nb;
  const uint64_t n_mr = p.n_mr;
  const uint64_t first = (uint64_t)blockIdx.x * (kThreads * kQPT) + threadIdx.x;

  uint64_t base[kQPT], aend[kQPT];
  uint32_t a[kQPT], z[kQPT];
  uint8_t state[kQPT];  // 0 done (miss), 1 searching, 2 invalid, 3 out of range
  // Load and round.
#pragma unroll
  for (int k = 0; k < kQPT; ++k) {
    const uint64_t i = first + (uint64_t)k * kThreads;
    state[k] = 3;
    base[k] = 0;
    aend[k] = 0;
    if (i < p.n_q) {
      const ulonglong2 r = ld_stream16(p.q + i, pol_first);
      const uint64_t addr = r.x, size = r.y;
      // valid iff size >= 1 and addr + size <= 2^64 - 4096 (the widened end fits)
      constexpr uint64_t kTop = ~0ull - 4095ull;
      const bool ok = size != 0 && size <= kTop && addr <= kTop - size;
      if (!ok) {
        state[k] = 2;
      } else {
        base[k] = addr & ~4095ull;
        aend[k] = (addr + size + 4095ull) & ~4095ull;
        state[k] = (n_mr == 0 || base[k] < lo) ? 0 : 1;
      }
    }
  }
  // Directory: candidate records [a, z).
#pragma unroll
  for (int k = 0; k < kQPT; ++k) {
    a[k] = 0;
    z[k] = 0;
    if (state[k] == 1) {
      const uint64_t b = (base[k] - lo) >> shift;
      if (b >= nb) {
        a[k] = (uint32_t)n_mr;
        z[k] = (uint32_t)n_mr;
      } else {
        uint32_t x = ld_table4(p.dir + b, pol_last), y = ld_table4(p.dir + b + 1, pol_last);
        x = x < n_mr ? x : (uint32_t)n_mr;
        y = y < n_mr ? y : (uint32_t)n_mr;
        a[k] = x;
        z[k] = y > x ? y : x;
      }
    }
  }
  // Binary search, all queries of the thread in lockstep: first record in
  // [a, z) starting above base.
  bool more = true;
  while (more) {
    more = false;
#pragma unroll
    for (int k = 0; k < kQPT; ++k) {
      if (state[k] == 1 && a[k] < z[k]) {
        const uint32_t mid = (a[k] + z[k]) >> 1;
        const uint64_t s = ld_table8(&p.rec[mid].start, pol_last);
        if (s <= base[k])
          a[k] = mid + 1;
        else
          z[k] = mid;
        more |= a[k] < z[k];
      }
    }
  }
  // The candidate is record a - 1: the last one starting at or below base.
  uint32_t hits = 0, invalid = 0;
#pragma unroll
  for (int k = 0; k < kQPT; ++k) {
    const uint64_t i = first + (uint64_t)k * kThreads;
    if (state[k] == 3) continue;
    int32_t out_idx = -1;
    uint32_t out_lkey = 0;
    uint8_t out_kind = state[k] == 2 ? DB_MR_INVALID : DB_MR_MISS;
    invalid += state[k] == 2;
    if (state[k] == 1 && a[k] > 0) {
      const uint32_t j = a[k] - 1;
      const ulonglong2 se = ld_table16(&p.rec[j], pol_last);
      if (se.x <= base[k] && aend[k] <= se.y) {
        out_idx = (int32_t)j;
        out_lkey = ld_table4(&p.rec[j].lkey, pol_last);
        out_kind = (se.x == base[k] && se.y == aend[k]) ? DB_MR_EXACT : DB_MR_CONTAINED;
        hits += 1;
      }
    }
    __stcs(p.idx + i, out_idx);
    __stcs(reinterpret_cast<unsigned int*>(p.lkey + i), out_lkey);
    __stcs(reinterpret_cast<unsigned char*>(p.kind + i), out_kind);
  }
  // Counters and hand-off to the next call.
  if (p.ctr) {
    hits = warp_sum32(hits);
    invalid = warp_sum32(invalid);
    if ((threadIdx.x & 31) == 0 && (hits | invalid)) {
      atomicAdd(&p.hdr->hits, (unsigned long long)hits);
      atomicAdd(&p.hdr->invalid, (unsigned long long)invalid);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned int d = atomicAdd(&p.hdr->done, 1u);
    if (d == gridDim.x - 1) {
      __threadfence();
      const unsigned long long h = atomicExch(&p.hdr->hits, 0ull);
      const unsigned long long v = atomicExch(&p.hdr->invalid, 0ull);
      const unsigned int err = atomicExch(&p.hdr->err, 0u);
      if (p.ctr) {
        p.ctr->total = h;
        p.ctr->n_invalid = v;
        p.ctr->n_overflow = 0;
        p.ctr->err = err;
      }
      p.hdr->done = 0;
      __threadfence();
    }
  }
}

}  // namespace mr
}  // namespace db

using namespace db;

extern "C" int db_mr_workspace_size(uint64_t n_mr, size_t* bytes) {
  if (!bytes || n_mr >= (1ull << 31)) return -EINVAL;
  *bytes = mr::ws_bytes_for(n_mr);
  return 0;
}

extern "C" int db_mr_lookup(const db_range* q, uint64_t n_q, const uint64_t* mr_start,
                            const uint64_t* mr_end, const uint32_t* mr_lkey, uint64_t n_mr,
                            int32_t* idx, uint32_t* lkey, uint8_t* kind, db_counters* ctr,
                            void* ws, size_t ws_bytes, void* stream) {
  cudaStream_t s = (cudaStream_t)stream;
  if (n_mr >= (1ull << 31)) return -EINVAL;
  if (ctr && !aligned(ctr, 8)) return -EINVAL;
  if (n_q == 0) {
    if (ctr) cudaMemsetAsync(ctr, 0, sizeof(db_counters), s);
    return launch_result();
  }
  if (!q || !idx || !lkey || !kind || !ws) return -EINVAL;
  if (n_mr && (!mr_start || !mr_end || !mr_lkey)) return -EINVAL;
  if (!aligned(q, 16) || !aligned(idx, 4) || !aligned(lkey, 4) || !aligned(ws, 256))
    return -EINVAL;
  if (n_mr && (!aligned(mr_start, 8) || !aligned(mr_end, 8) || !aligned(mr_lkey, 4)))
    return -EINVAL;
  if (ws_bytes < mr::ws_bytes_for(n_mr)) return -ENOSPC;
  if (n_q > (1ull << 40)) return -EINVAL;

  const uint32_t nb = mr::buckets_for(n_mr);
  uint32_t log_nb = 0;
  while ((1u << log_nb) < nb) ++log_nb;
  char* w = static_cast<char*>(ws);
  mr::Header* hdr = reinterpret_cast<mr::Header*>(w);
  uint32_t* dir = reinterpret_cast<uint32_t*>(w + mr::kHeaderBytes);
  mr::Rec* rec = reinterpret_cast<mr::Rec*>(w + mr::kHeaderBytes + mr::dir_bytes(nb));

  if (n_mr > 0) {
    mr::BuildParams b{mr_start, mr_end, mr_lkey, n_mr, hdr, dir, rec, nb, log_nb};
    const uint64_t merged = n_mr + nb + 1;
    const uint64_t threads = (merged + mr::kMergeChunk - 1) / mr::kMergeChunk;
    uint64_t grid = (threads + mr::kBuildThreads - 1) / mr::kBuildThreads;
    const uint64_t cap = (uint64_t)num_sms() * 16;
    if (grid > cap) grid = cap;
    mr::mr_index_kernel<<<(unsigned)grid, mr::kBuildThreads, 0, s>>>(b);
    int rc = launch_result();
    if (rc) return rc;
  }
  mr::LookupParams l{reinterpret_cast<const ulonglong2*>(q), n_q, n_mr, hdr, hdr, dir, rec,
                     idx, lkey, kind, ctr};
  const uint64_t per_cta = (uint64_t)mr::kThreads * mr::kQPT;
  const uint64_t grid = (n_q + per_cta - 1) / per_cta;
  if (grid > 0x7FFFFFFFull) return -EINVAL;
  mr::mr_lookup_kernel<<<(unsigned)grid, mr::kThreads, 0, s>>>(l);
  return launch_result();
}
