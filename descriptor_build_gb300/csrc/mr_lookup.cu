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
//                fills a directory of 32-byte entries (one sector each):
//                D[b] = number of records starting below lo + b * 2^shift
//                (2^shift chosen so that the records' span fits nb buckets)
//                and the page offsets, from the bucket's first page, of the
//                starts of records D[b] .. D[b] + 6. Each record fills the
//                buckets between its predecessor's and its own.
//   lookup       persistent CTAs, 4 queries per thread per step: round to
//                pages; the directory entry of the base's bucket names the
//                candidate unless seven or more records start in the bucket
//                at or below the base (then binary steps over the records up
//                to D[b+1]); read the candidate's 32-byte record and classify.
//                The next step's queries load meanwhile.
// For a sorted table of disjoint non-empty records the only record that can
// contain [base, aend) is the last one starting at or below base, so the
// lowest containing index is that record or none.
#include "common.cuh"
#include "mr_internal.h"

namespace db {
namespace mr {

// Launch shape of the lookup (tunable at build time; the defaults are the
// measured best on GB300): threads per CTA, queries per thread, minimum CTAs
// per SM for the register budget, and log2 of buckets per record.
#ifndef DB_MR_THREADS
#define DB_MR_THREADS 256
#endif
#ifndef DB_MR_QPT
#define DB_MR_QPT 3
#endif
#ifndef DB_MR_MIN_CTAS
#define DB_MR_MIN_CTAS 4
#endif
#ifndef DB_MR_BUCKET_SHIFT
#define DB_MR_BUCKET_SHIFT 0
#endif
#ifndef DB_MR_BUCKET_DOWN
#define DB_MR_BUCKET_DOWN 1  // log2 of the fewest records per bucket (measured best: two)
#endif
// Directory and record reads of the lookup: 1 skips the L1 allocation (the
// reads are random and never reused by the same SM).
#ifndef DB_MR_GATHER_NOALLOC
#define DB_MR_GATHER_NOALLOC 1
#endif
// 1: the lookup is launched as a programmatic dependent of the index build,
// so its CTAs start and load their first queries while the build finishes.
#ifndef DB_MR_PDL
#define DB_MR_PDL 1
#endif
// Index build grid: at most this many CTAs per SM (threads loop over records).
#ifndef DB_MR_BUILD_CTAS_PER_SM
#define DB_MR_BUILD_CTAS_PER_SM 4
#endif
constexpr int kBuildThreads = 256;
constexpr int kThreads = DB_MR_THREADS;
constexpr int kQPT = DB_MR_QPT;


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
  uint64_t before;  // tables that may overlap: the largest end of records 0 .. i-1 (0 for i = 0)
};
constexpr size_t kHeaderBytes = 256;

inline uint32_t buckets_for(uint64_t n_mr) {
  uint64_t nb = 1024;
  // The largest power of two at most n_mr / 2 (at least 1024): a directory
  // rounded up instead can be nearly twice as large, and tables plus
  // directory then no longer stay in L2.
  while (nb * 2 <= ((n_mr << DB_MR_BUCKET_SHIFT) >> DB_MR_BUCKET_DOWN) && nb < (1u << 22)) nb <<= 1;
  return (uint32_t)nb;
}
// Directory entry of bucket b: the records starting below the bucket
// (D[b]) and where records D[b] .. D[b] + 6 start, as page offsets from the
// bucket's first page, rounded up (a start s lies at or below a
// page-aligned base exactly when ceil(s / 4096) <= base / 4096). The starts
// are increasing, so the offsets at or below a base's offset form a prefix
// and their count says which record is the candidate; kNoOff stands for a
// record that does not exist or starts more than 2^32 - 2 pages on. One
// 32-byte load settles every query whose bucket holds fewer than seven
// record starts at or below it.
constexpr int kOffs = 7;
struct alignas(32) Dir {
  uint32_t first;        // D[b]
  uint32_t off[kOffs];   // page offsets of records D[b] .. D[b] + 6
};
constexpr uint32_t kNoOff = 0xFFFFFFFFu;
constexpr uint32_t kMaxOffsetShift = 43;  // bucket widths up to 2^43 bytes keep offsets in 32 bits
inline size_t dir_bytes(uint32_t nb) { return (((size_t)nb + 1) * sizeof(Dir) + 255) & ~(size_t)255; }
static_assert(sizeof(Dir) == 32, "one L2 sector per directory entry");
// Tables that may overlap: Rec::before is the prefix maximum of the ends of
// the records before it, built first in an array of its own (blocks of 1024
// records, whose maxima sit after the records).
constexpr int kPmBlock = 1024;
inline size_t pm_blocks(uint64_t n_mr) { return (n_mr + kPmBlock - 1) / kPmBlock; }
inline size_t rec_bytes(uint64_t n_mr) { return ((size_t)n_mr * sizeof(Rec) + 255) & ~(size_t)255; }
inline size_t ws_bytes_for(uint64_t n_mr) {
  const uint32_t nb = buckets_for(n_mr);
  return kHeaderBytes + dir_bytes(nb) + rec_bytes(n_mr) +
         ((pm_blocks(n_mr) * 8 + 255) & ~(size_t)255) + (size_t)n_mr * 8;
}

struct BuildParams {
  const uint64_t* start;
  const uint64_t* end;
  const uint32_t* lkey;
  uint64_t n_mr;
  Header* hdr;
  Dir* dir;  // [nb + 1]
  Rec* rec;
  uint32_t nb;
  uint32_t log_nb;
  bool overlap;        // ranges may overlap: only starts must be sorted
  const uint64_t* pm;  // overlap: prefix maximum of the ends, pm[i] = max(end[0..i])
};

__device__ __forceinline__ uint64_t bucket_of(uint64_t x, uint64_t lo, uint32_t shift,
                                              uint32_t nb) {
  if (x < lo) return 0;
  const uint64_t b = (x - lo) >> shift;
  return b < nb ? b : nb;
}

// Records: 32-byte copies and the ordering check. Directory: D[b] = number
// of records whose bucket key is below b, for b = 0..nb. Record i owns the
// buckets (key(i-1), key(i)] (all with D = i); a short range is written by
// its thread, a longer one (a wide gap before the record) by its whole warp.
// The buckets after the last record's (D = n) are written by a grid-stride
// loop of their own. Each entry is written whole, by one 32-byte store, by
// its owner: the starts of records D[b] .. D[b] + 6 are all it needs.
// ss[k] is the start of record x + k, or ~0 when that record does not exist.
__device__ __forceinline__ uint32_t page_offset(uint64_t s, uint64_t bpage0) {
  if (s == ~0ull) return kNoOff;
  const uint64_t sp = (s >> 12) + ((s & 4095u) ? 1 : 0);  // ceil(s / 4096), s < 2^64
  const uint64_t d = sp - bpage0;  // the record starts in or after the bucket: d >= 0
  return d < kNoOff ? (uint32_t)d : kNoOff;
}
__device__ __forceinline__ void set_dir(const BuildParams& p, uint64_t b, uint32_t x,
                                        const uint64_t (&ss)[kOffs], uint64_t lo, uint32_t shift) {
  const uint64_t bpage0 = (lo + (b << shift)) >> 12;
  const bool offs = shift <= kMaxOffsetShift;
  uint32_t o[kOffs];
#pragma unroll
  for (int k = 0; k < kOffs; ++k) o[k] = offs ? page_offset(ss[k], bpage0) : kNoOff;
  const uint64_t w0 = (uint64_t)x | ((uint64_t)o[0] << 32);
  const uint64_t w1 = (uint64_t)o[1] | ((uint64_t)o[2] << 32);
  const uint64_t w2 = (uint64_t)o[3] | ((uint64_t)o[4] << 32);
  const uint64_t w3 = (uint64_t)o[5] | ((uint64_t)o[6] << 32);
  asm volatile("st.global.v4.u64 [%0], {%1, %2, %3, %4};" ::"l"(p.dir + b), "l"(w0), "l"(w1),
               "l"(w2), "l"(w3)
               : "memory");
}

#ifndef DB_MR_BUILD_MIN_CTAS
#define DB_MR_BUILD_MIN_CTAS 4
#endif
__global__ void __launch_bounds__(kBuildThreads, DB_MR_BUILD_MIN_CTAS) mr_index_kernel(const BuildParams p) {
  if (DB_MR_PDL) {
    wait_for_prerequisites();  // launched as a dependent after the prefix-maximum kernels
    dependents_may_launch();
  }
  const uint64_t lo = p.start[0];
  const uint64_t hi = p.start[p.n_mr - 1];
  const uint64_t span = hi > lo ? hi - lo : 0;
  const uint32_t bits = span ? 64u - (uint32_t)__clzll((long long)span) : 0u;
  const uint32_t shift = bits > p.log_nb ? bits - p.log_nb : 0u;
  const uint64_t nb = p.nb, n = p.n_mr;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    p.hdr->lo = lo;
    p.hdr->shift = shift;
    p.hdr->nb = p.nb;
  }
  const int lane = threadIdx.x & 31;
  const uint64_t nthreads = (uint64_t)gridDim.x * blockDim.x;
  const uint64_t tid = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const uint64_t n_round = (n + 31) & ~31ull;  // whole warps stay in the loop together

  bool bad = false;
  for (uint64_t i = tid; i < n_round; i += nthreads) {
    uint64_t b0 = 1, b1 = 0, s = 0;  // buckets [b0, b1] get D = i
    uint64_t ss[kOffs];              // starts of records i .. i + 6
#pragma unroll
    for (int k = 0; k < kOffs; ++k) ss[k] = i + k < n ? p.start[i + k] : ~0ull;
    if (i < n) {
      s = ss[0];
      const uint64_t e = p.end[i];
      Rec r;
      r.start = s;
      r.end = e;
      r.lkey = p.lkey[i];
      r.pad0 = 0;
      r.before = (p.overlap && i > 0) ? p.pm[i - 1] : 0;
      p.rec[i] = r;
      if (!(s < e) || (i > 0 && (p.overlap ? p.start[i - 1] > s : p.end[i - 1] > s))) bad = true;
      b0 = i == 0 ? 0 : bucket_of(p.start[i - 1], lo, shift, p.nb) + 1;
      b1 = bucket_of(s, lo, shift, p.nb);
    }
    const bool wide = b1 >= b0 && b1 - b0 >= 32;
    if (!wide)
      for (uint64_t b = b0; b <= b1 && b1 >= b0; ++b) set_dir(p, b, (uint32_t)i, ss, lo, shift);
    uint32_t todo = __ballot_sync(kFull, wide);
    while (todo) {
      const int l = __ffs(todo) - 1;
      todo &= todo - 1;
      const uint64_t wb0 = __shfl_sync(kFull, b0, l), wb1 = __shfl_sync(kFull, b1, l);
      const uint64_t wi = __shfl_sync(kFull, i, l);
      uint64_t wss[kOffs];
#pragma unroll
      for (int k = 0; k < kOffs; ++k) wss[k] = __shfl_sync(kFull, ss[k], l);
      for (uint64_t b = wb0 + lane; b <= wb1; b += 32) set_dir(p, b, (uint32_t)wi, wss, lo, shift);
    }
  }
  if (bad) atomicOr(&p.hdr->err, DB_ERR_TABLE_ORDER);
  // Buckets after the last record's: D = n, no record starts in or after them.
  const uint64_t tail0 = bucket_of(hi, lo, shift, p.nb) + 1;
  uint64_t none[kOffs];
#pragma unroll
  for (int k = 0; k < kOffs; ++k) none[k] = ~0ull;
  for (uint64_t b = tail0 + tid; b <= nb; b += nthreads) set_dir(p, b, (uint32_t)n, none, lo, shift);
}

struct LookupParams {
  const ulonglong2* q;
  uint64_t n_q;
  uint64_t n_mr;
  const Header* hdr_ro;
  Header* hdr;
  const Dir* dir;
  const Rec* rec;
  int32_t* idx;
  uint32_t* lkey;
  uint8_t* kind;
  db_counters* ctr;
};

// Tables that may overlap: the first record i <= j whose prefix maximum of
// ends, pm(i) = rec[i + 1].before, reaches aend, given pm(j - 1) >= aend.
// Galloping back from j - 1 (overlaps are usually short), then a binary
// search between the last miss and the first hit.
__device__ __forceinline__ uint32_t first_reaching(const Rec* rec, uint32_t j, uint64_t aend,
                                                   uint64_t pol) {
  int64_t hi = (int64_t)j - 1, step = 1;  // pm(hi) >= aend
  while (hi - step >= 0 && ld_table8(&rec[hi - step + 1].before, pol) >= aend) {
    hi -= step;
    step <<= 1;
  }
  int64_t lo = hi - step;  // pm(lo) < aend, or lo = -1
  if (lo < -1) lo = -1;
  while (hi - lo > 1) {
    const int64_t mid = lo + (hi - lo) / 2;
    if (ld_table8(&rec[mid + 1].before, pol) >= aend) hi = mid;
    else lo = mid;
  }
  return (uint32_t)hi;
}

__device__ __forceinline__ void ld_gather32(const void* a, uint64_t pol, uint64_t& x, uint64_t& y,
                                            uint64_t& z, uint64_t& w) {
  if (DB_MR_GATHER_NOALLOC)
    asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u64 {%0, %1, %2, %3}, [%4], %5;"
        : "=l"(x), "=l"(y), "=l"(z), "=l"(w)
        : "l"(a), "l"(pol));
  else
    ld_table32(a, pol, x, y, z, w);
}

// kGranuleShift: queries are widened to whole granules of 2^kGranuleShift
// bytes (12: 4 KiB pages; 16: the 64 KiB registry granule). The directory
// works in 4 KiB pages either way, since every granule boundary is one.
template <bool kOverlap, int kGranuleShift>
__global__ void __launch_bounds__(kThreads, DB_MR_MIN_CTAS) mr_lookup_kernel(const LookupParams p) {
  constexpr uint64_t kGran = 1ull << kGranuleShift;
  const uint64_t pol_first = policy_evict_first();
  const uint64_t pol_last = policy_evict_last();
  const uint64_t n_mr = p.n_mr;
  constexpr uint64_t kGroup = (uint64_t)kThreads * kQPT;  // queries per CTA step
  const uint64_t n_groups = (p.n_q + kGroup - 1) / kGroup;
  uint32_t hits = 0, invalid = 0;

  // Persistent: CTAs stride over groups of queries; the next group's queries
  // are loaded while the current group's table lookups are in flight.
  ulonglong2 nq[kQPT];
  uint64_t g = blockIdx.x;
#pragma unroll
  for (int k = 0; k < kQPT; ++k) {
    const uint64_t i = g * kGroup + (uint64_t)k * kThreads + threadIdx.x;
    nq[k] = (g < n_groups && i < p.n_q) ? ld_stream16(p.q + i, pol_first) : make_ulonglong2(0, 0);
  }
  // Launched as a dependent of the index build: everything the build writes
  // (header, directory, records) is read only after this wait. The queries
  // above are the caller's input, complete before the build started. Without
  // a programmatic launch the wait returns at once.
  wait_for_prerequisites();
  const uint64_t lo = p.hdr_ro->lo;
  const uint32_t shift = p.hdr_ro->shift;
  const uint32_t nb = p.hdr_ro->nb;
  const bool offsets_kept = shift <= kMaxOffsetShift;
  for (; g < n_groups; g += gridDim.x) {
    const uint64_t first = g * kGroup + threadIdx.x;
    uint64_t base[kQPT], aend[kQPT];
    uint32_t a[kQPT], z[kQPT];
    uint8_t state[kQPT];  // 0 miss, 1 searching, 2 invalid, 3 outside the batch
    // Round.
#pragma unroll
    for (int k = 0; k < kQPT; ++k) {
      const uint64_t i = first + (uint64_t)k * kThreads;
      state[k] = 3;
      base[k] = 0;
      aend[k] = 0;
      if (i < p.n_q) {
        const uint64_t addr = nq[k].x, size = nq[k].y;
        // valid iff size >= 1 and addr + size <= 2^64 - 4096 (the widened end fits)
        constexpr uint64_t kTop = ~0ull - (kGran - 1);
        const bool ok = size != 0 && size <= kTop && addr <= kTop - size;
        if (!ok) {
          state[k] = 2;
        } else {
          base[k] = addr & ~(kGran - 1);
          aend[k] = (addr + size + kGran - 1) & ~(kGran - 1);
          state[k] = (n_mr == 0 || base[k] < lo) ? 0 : 1;
        }
      }
    }
    // Directory: the number of records starting at or below base is
    // D[b] plus the count of start offsets at or below base's offset; only
    // when all seven are (or the offsets are not kept) does it take binary
    // steps over records up to D[b+1]. [a, z) is the range still open.
    bool wide_search = false;
#pragma unroll
    for (int k = 0; k < kQPT; ++k) {
      a[k] = 0;
      z[k] = 0;
      if (state[k] == 1) {
        uint64_t b = (base[k] - lo) >> shift;
        b = b < nb ? b : nb;
        uint64_t w0, w1, w2, w3;
        ld_gather32(p.dir + b, pol_last, w0, w1, w2, w3);
        uint32_t x = (uint32_t)w0;
        x = x < n_mr ? x : (uint32_t)n_mr;
        // base's page offset in the bucket, capped below kNoOff
        const uint64_t bo64 = (base[k] >> 12) - ((lo + (b << shift)) >> 12);
        const uint32_t bo = bo64 < kNoOff - 1 ? (uint32_t)bo64 : kNoOff - 1;
        const uint32_t o[kOffs] = {(uint32_t)(w0 >> 32), (uint32_t)w1, (uint32_t)(w1 >> 32),
                                   (uint32_t)w2, (uint32_t)(w2 >> 32), (uint32_t)w3,
                                   (uint32_t)(w3 >> 32)};
        uint32_t c = 0;
#pragma unroll
        for (int j = 0; j < kOffs; ++j) c += o[j] <= bo;
        if (offsets_kept && c < kOffs) {
          x += c;
          x = x < n_mr ? x : (uint32_t)n_mr;
          a[k] = x;
          z[k] = x;
        } else {
          a[k] = offsets_kept ? x + kOffs : x;   // the rest lies in [a, D[b+1])
          a[k] = a[k] < n_mr ? a[k] : (uint32_t)n_mr;
          z[k] = b < nb ? ~0u : (uint32_t)n_mr;  // D[b+1], read below
          wide_search = true;
        }
      }
    }
    // Prefetch the next group's queries.
    const uint64_t gn = g + gridDim.x;
#pragma unroll
    for (int k = 0; k < kQPT; ++k) {
      const uint64_t i = gn * kGroup + (uint64_t)k * kThreads + threadIdx.x;
      nq[k] = (gn < n_groups && i < p.n_q) ? ld_stream16(p.q + i, pol_first)
                                            : make_ulonglong2(0, 0);
    }
    // Rare: the upper bound D[b+1] of a bucket holding many record starts.
    if (wide_search) {
#pragma unroll
      for (int k = 0; k < kQPT; ++k) {
        if (state[k] == 1 && z[k] == ~0u) {
          const uint64_t b = (base[k] - lo) >> shift;
          uint32_t y = ld_table4(&p.dir[b + 1].first, pol_last);
          y = y < n_mr ? y : (uint32_t)n_mr;
          z[k] = y > a[k] ? y : a[k];
        }
      }
    }
    // Binary steps over any records still undecided (a bucket with two or
    // more record starts; all queries of the thread in lockstep).
    bool more = true;
    while (more) {
      more = false;
#pragma unroll
      for (int k = 0; k < kQPT; ++k) {
        if (state[k] == 1 && a[k] < z[k]) {
          const uint32_t mid = (a[k] + z[k]) >> 1;
          if (ld_table8(&p.rec[mid].start, pol_last) <= base[k])
            a[k] = mid + 1;
          else
            z[k] = mid;
          more |= a[k] < z[k];
        }
      }
    }
    // The candidate is record j = a - 1: the last one starting at or below
    // base. On a table that may overlap, an earlier record whose end
    // reaches aend (Rec::before of j says whether one exists) comes first.
#pragma unroll
    for (int k = 0; k < kQPT; ++k) {
      const uint64_t i = first + (uint64_t)k * kThreads;
      if (state[k] == 3) continue;
      int32_t out_idx = -1;
      uint32_t out_lkey = 0;
      uint8_t out_kind = state[k] == 2 ? DB_MR_INVALID : DB_MR_MISS;
      invalid += state[k] == 2;
      if (state[k] == 1 && a[k] > 0) {
        uint32_t j = a[k] - 1;
        uint64_t rs, re, rk, before;
        ld_gather32(&p.rec[j], pol_last, rs, re, rk, before);
        if (kOverlap && before >= aend[k]) {
          j = first_reaching(p.rec, j, aend[k], pol_last);
          ld_gather32(&p.rec[j], pol_last, rs, re, rk, before);
        }
        if (rs <= base[k] && aend[k] <= re) {
          out_idx = (int32_t)j;
          out_lkey = (uint32_t)rk;
          out_kind = (rs == base[k] && re == aend[k]) ? DB_MR_EXACT : DB_MR_CONTAINED;
          hits += 1;
        }
      }
      if (DB_STORE_HINT) {
        __stcs(p.idx + i, out_idx);
        __stcs(reinterpret_cast<unsigned int*>(p.lkey + i), out_lkey);
        __stcs(reinterpret_cast<unsigned char*>(p.kind + i), out_kind);
      } else {
        p.idx[i] = out_idx;
        p.lkey[i] = out_lkey;
        p.kind[i] = out_kind;
      }
    }
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

// ------------------------------------------------------ overlapping tables
// The prefix maximum of the ends, pm(i) = max(end[0..i]), into an array of
// its own: a block-local inclusive max-scan, a scan of the block maxima (one
// CTA), then each block takes the maximum of the blocks before it. The index
// build then writes Rec::before = pm(i - 1) with the rest of record i, in one
// whole-sector store. A record read then says whether an earlier one may contain
// the query, so the common case costs the same single 32-byte record load
// as on a disjoint table.
__device__ __forceinline__ uint64_t warp_max_scan(uint64_t x, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint64_t y = __shfl_up_sync(kFull, x, o);
    if (lane >= o && y > x) x = y;
  }
  return x;
}
// Inclusive max-scan of one value per thread over a CTA of kPmBlock threads.
__device__ __forceinline__ uint64_t block_max_scan(uint64_t x, uint64_t* s_w) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  x = warp_max_scan(x, lane);
  if (lane == 31) s_w[warp] = x;
  __syncthreads();
  if (warp == 0) s_w[lane] = warp_max_scan(s_w[lane], lane);  // kPmBlock / 32 == 32 warps
  __syncthreads();
  const uint64_t before = warp ? s_w[warp - 1] : 0ull;
  return before > x ? before : x;
}
__global__ void __launch_bounds__(kPmBlock) mr_pm_block_kernel(const uint64_t* end, uint64_t n,
                                                               uint64_t* pm, uint64_t* bmax) {
  wait_for_prerequisites();
  dependents_may_launch();
  __shared__ uint64_t s_w[32];
  const uint64_t i = (uint64_t)blockIdx.x * kPmBlock + threadIdx.x;
  const uint64_t x = block_max_scan(i < n ? end[i] : 0ull, s_w);
  if (i < n) pm[i] = x;  // block-local for now
  if (threadIdx.x == kPmBlock - 1) bmax[blockIdx.x] = x;
}
__global__ void __launch_bounds__(kPmBlock) mr_pm_scan_kernel(uint64_t* bmax, uint64_t nblk) {
  wait_for_prerequisites();
  dependents_may_launch();
  __shared__ uint64_t s_w[32];
  uint64_t carry = 0;
  for (uint64_t b0 = 0; b0 < nblk; b0 += kPmBlock) {
    const uint64_t b = b0 + threadIdx.x;
    uint64_t x = block_max_scan(b < nblk ? bmax[b] : 0ull, s_w);
    x = x > carry ? x : carry;
    if (b < nblk) bmax[b] = x;
    __syncthreads();  // block_max_scan's reads of s_w are done
    if (threadIdx.x == kPmBlock - 1) s_w[0] = x;  // this round's maximum carries to the next
    __syncthreads();
    carry = s_w[0];
    __syncthreads();
  }
}
__global__ void __launch_bounds__(kPmBlock) mr_pm_apply_kernel(uint64_t* pm, uint64_t n,
                                                               const uint64_t* bmax) {
  wait_for_prerequisites();
  dependents_may_launch();
  const uint64_t i = (uint64_t)blockIdx.x * kPmBlock + threadIdx.x;
  if (blockIdx.x == 0 || i >= n) return;
  const uint64_t prior = bmax[blockIdx.x - 1];
  if (prior > pm[i]) pm[i] = prior;
}

int lookup_ctas_per_sm() {
  static int per_sm[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  int& occ = per_sm[dev & 63];
  if (occ == 0) {
    int o = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, mr_lookup_kernel<false, 12>, kThreads, 0) !=
            cudaSuccess ||
        o < 1)
      o = 1;
    occ = o;
  }
  return occ;
}

}  // namespace mr
}  // namespace db

using namespace db;

extern "C" int db_mr_workspace_size(uint64_t n_mr, size_t* bytes) {
  if (!bytes || n_mr >= (1ull << 31)) return -EINVAL;
  *bytes = mr::ws_bytes_for(n_mr);
  return 0;
}

namespace db {
namespace mr {

int lookup(const db_range* q, uint64_t n_q, const uint64_t* mr_start, const uint64_t* mr_end,
           const uint32_t* mr_lkey, uint64_t n_mr, int32_t* idx, uint32_t* lkey, uint8_t* kind,
           db_counters* ctr, void* ws, size_t ws_bytes, cudaStream_t s, bool overlap,
           int granule_shift) {
  if (granule_shift != 12 && granule_shift != 16) return -EINVAL;
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
  mr::Dir* dir = reinterpret_cast<mr::Dir*>(w + mr::kHeaderBytes);
  char* recs = w + mr::kHeaderBytes + mr::dir_bytes(nb);
  mr::Rec* rec = reinterpret_cast<mr::Rec*>(recs);
  uint64_t* bmax = reinterpret_cast<uint64_t*>(recs + mr::rec_bytes(n_mr));
  uint64_t* pm = reinterpret_cast<uint64_t*>(
      recs + mr::rec_bytes(n_mr) + ((mr::pm_blocks(n_mr) * 8 + 255) & ~(size_t)255));

  if (n_mr > 0) {
    int rc = 0;
    if (overlap) {  // the prefix maximum first, so the index build writes whole records
      const uint64_t nblk = mr::pm_blocks(n_mr);
      mr::mr_pm_block_kernel<<<(unsigned)nblk, mr::kPmBlock, 0, s>>>(mr_end, n_mr, pm, bmax);
      if ((rc = launch_result())) return rc;
      launch_dep(mr::mr_pm_scan_kernel, 1, mr::kPmBlock, 0, s, bmax, nblk);
      if ((rc = launch_result())) return rc;
      launch_dep(mr::mr_pm_apply_kernel, (unsigned)nblk, mr::kPmBlock, 0, s, pm, n_mr, bmax);
      if ((rc = launch_result())) return rc;
    }
    mr::BuildParams b{mr_start, mr_end, mr_lkey, n_mr, hdr, dir, rec, nb, log_nb, overlap, pm};
    uint64_t grid = (n_mr + mr::kBuildThreads - 1) / mr::kBuildThreads;
    const uint64_t cap = (uint64_t)num_sms() * DB_MR_BUILD_CTAS_PER_SM;
    if (grid > cap) grid = cap;
    if (DB_MR_PDL && overlap)
      launch_dep(mr::mr_index_kernel, (unsigned)grid, mr::kBuildThreads, 0, s, b);
    else
      mr::mr_index_kernel<<<(unsigned)grid, mr::kBuildThreads, 0, s>>>(b);
    if ((rc = launch_result())) return rc;
  }
  mr::LookupParams l{reinterpret_cast<const ulonglong2*>(q), n_q, n_mr, hdr, hdr, dir, rec,
                     idx, lkey, kind, ctr};
  const uint64_t per_cta = (uint64_t)mr::kThreads * mr::kQPT;
  uint64_t grid = (n_q + per_cta - 1) / per_cta;
  const uint64_t resident = (uint64_t)num_sms() * mr::lookup_ctas_per_sm();
  if (grid > resident) grid = resident;
  void (*kern)(const mr::LookupParams) = granule_shift == 16 ? mr::mr_lookup_kernel<true, 16>
                                         : overlap            ? mr::mr_lookup_kernel<true, 12>
                                                              : mr::mr_lookup_kernel<false, 12>;
  if (DB_MR_PDL && n_mr > 0)  // a dependent of the index build just launched on `s`
    return launch_dependent(kern, (unsigned)grid, mr::kThreads, 0, s, l);
  kern<<<(unsigned)grid, mr::kThreads, 0, s>>>(l);
  return launch_result();
}

size_t workspace_bytes(uint64_t n_mr) { return ws_bytes_for(n_mr); }

}  // namespace mr
}  // namespace db

extern "C" int db_mr_lookup(const db_range* q, uint64_t n_q, const uint64_t* mr_start,
                            const uint64_t* mr_end, const uint32_t* mr_lkey, uint64_t n_mr,
                            int32_t* idx, uint32_t* lkey, uint8_t* kind, db_counters* ctr,
                            void* ws, size_t ws_bytes, void* stream) {
  return mr::lookup(q, n_q, mr_start, mr_end, mr_lkey, n_mr, idx, lkey, kind, ctr, ws, ws_bytes,
                    (cudaStream_t)stream, false, 12);
}

extern "C" int db_mr_lookup_overlap(const db_range* q, uint64_t n_q, const uint64_t* mr_start,
                                    const uint64_t* mr_end, const uint32_t* mr_lkey,
                                    uint64_t n_mr, int32_t* idx, uint32_t* lkey, uint8_t* kind,
                                    db_counters* ctr, void* ws, size_t ws_bytes, void* stream) {
  return mr::lookup(q, n_q, mr_start, mr_end, mr_lkey, n_mr, idx, lkey, kind, ctr, ws, ws_bytes,
                    (cudaStream_t)stream, true, 12);
}
