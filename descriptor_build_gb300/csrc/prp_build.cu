// NVMe PRP construction from a 64 KiB-granular bus-address LUT (sm_103a).
//
// Source: xNVMe "uPCIe CUDA" backend page -- introduction (bus address per
// 64 KiB chunk in a LUT, PRP entries at 4 KiB from sub-page offsets),
// "Memory Architecture" (PRP lists in their own region) and "Limitations"
// (512 entries per 4 KiB list page; 513 x 4 KiB with PRP1). Lists longer than
// one page chain through slot 511 (NVMe convention).
//
// Two schedules with the same results (the host picks one by batch size):
//
// Single kernel (large batches): one persistent kernel, one pass over the
// requests:
//   1. a CTA takes a tile of 2,048 requests by atomic ticket and loads four
//      16-byte requests per thread;
//   2. page count n and list-page count L per request, block scan of L;
//   3. decoupled lookback over the tiles before it (one status word per
//      tile in the workspace, bounded wait) gives the tile's first list page;
//      a tile with no list, in a call without page_base output, skips the
//      scan and the wait and takes its next ticket at once;
//   4. PRP1/PRP2, page_base and status go out as 16/8/1-byte stores;
//   5. the tile's lists are written by warps that take one request at a time
//      from a shared-memory queue: each list is a contiguous run of 8-byte
//      words starting on a 4 KiB page, written as 32-byte stores and ended on
//      a whole 32-byte sector.
// The last CTA to finish publishes the counters and readies the workspace
// for the next call (new epoch, ticket back to 0).
//
// Two kernels (batches that fit one wave of the first): a light pair kernel,
// one CTA per tile and four CTAs per SM, loads every request at once,
// publishes each tile's list-page total, and writes the PRP pairs of the
// tiles that own no list (when page_base is not asked for). The list kernel
// then runs the steps above on the remaining tiles, taken by index, with the
// tile's first list page summed from the published totals instead of a
// lookback. A small-I/O batch so spends one wave of loads, gathers and
// stores rather than two rounds of a latency chain per CTA.
#include "common.cuh"

namespace db {
namespace prp {

// Build-time tuning: gather the PRP1/PRP2 LUT entries before the tile's
// scan and lookback (1) or after them (0).
#ifndef DB_PRP_EARLY_LUT
#define DB_PRP_EARLY_LUT 0
#endif
// List words: 32-byte stores with the evict-first L2 hint (1) or plain (0).
#ifndef DB_PRP_LIST_HINT
#define DB_PRP_LIST_HINT 0
#endif

// Tile shape (tunable at build time; defaults measured best on GB300):
// threads per CTA, requests per thread, minimum resident CTAs per SM.
#ifndef DB_PRP_THREADS
#define DB_PRP_THREADS 512
#endif
#ifndef DB_PRP_ITEMS
#define DB_PRP_ITEMS 4
#endif
#ifndef DB_PRP_MIN_CTAS
#define DB_PRP_MIN_CTAS 2
#endif
constexpr int kThreads = DB_PRP_THREADS;
constexpr int kWarps = kThreads / 32;
constexpr int kItems = DB_PRP_ITEMS;       // requests per thread per tile
constexpr int kTile = kThreads * kItems;   // requests per tile

// Workspace: ScanHeader (acc[0] invalid, acc[1] overflow, acc[2] list pages), then one status
// word per tile.
constexpr uint64_t tiles_for(uint64_t n) { return (n + kTile - 1) / kTile; }
constexpr uint64_t kMaxRequests = 1ull << 28;
constexpr size_t ws_bytes_for(uint64_t n) {
  return kScanHeaderBytes + ((tiles_for(n) * 8 + 255) & ~(uint64_t)255);
}

struct Params {
  const ulonglong2* req;
  uint64_t n;
  uint64_t n_tiles;
  const uint64_t* lut;
  uint64_t heap_size;
  uint64_t arena_base;
  uint64_t cap;
  uint64_t* arena;
  ulonglong2* prp;
  uint64_t* page_base;
  uint8_t* status;
  db_counters* ctr;
  uint32_t zero_tail;
  uint32_t parts;  // list kernel of the two-kernel schedule: CTAs per tile (1..kWarps)
  ScanHeader* hdr;
  unsigned long long* tile_status;  // [cap_tiles]
  uint64_t cap_tiles;
};

// A request that owns list pages, as the emission phase sees it.
struct ListItem {
  uint64_t pb;    // first list page (arena page index)
  uint64_t hb;    // heap offset of the request's first 4 KiB page
  uint32_t words; // data entries + chain pointers
  uint32_t pages; // list pages (0: skip, the list did not fit)
};

// Queued form, 16 bytes: w0 = hb | pages (hb is page aligned, pages < 4096),
// w1 = pb | n << 40 (pb < 2^40 by the host check, n < 2^21).
__device__ __forceinline__ ulonglong2 pack_item(uint64_t hb, uint32_t pages, uint64_t pb,
                                                uint32_t npg) {
  return make_ulonglong2(hb | pages, (pb & ((1ull << 40) - 1)) | ((uint64_t)npg << 40));
}
__device__ __forceinline__ ListItem unpack_item(ulonglong2 q) {
  ListItem it;
  it.hb = q.x & ~4095ull;
  it.pages = (uint32_t)(q.x & 4095ull);
  it.pb = q.y & ((1ull << 40) - 1);
  const uint32_t npg = (uint32_t)(q.y >> 40);
  it.words = it.pages ? (npg - 1) + (it.pages - 1) : 0;
  return it;
}

__device__ __forceinline__ uint64_t bus(const uint64_t* lut, uint64_t x, uint64_t pol) {
  return ld_table8(lut + (x >> 16), pol) + (x & 0xFFFFull);
}

// LUT window of a warp: lane l holds lut[c0 + wrel + l] (0 past the
// request's last chunk). Issued as a volatile load so that it is not moved
// behind the stores of the previous request (it is the prefetch of the next).
__device__ __forceinline__ uint64_t lut_window(const uint64_t* lut, uint64_t c, uint64_t c_last,
                                               uint64_t pol) {
  uint64_t v = 0;
  if (c <= c_last)
    asm volatile("ld.global.nc.L2::cache_hint.u64 %0, [%1], %2;" : "=l"(v) : "l"(lut + c), "l"(pol));
  return v;
}

// Page positions are counted from the start of the request's first 64 KiB
// chunk c0: data entry e (0-based) names heap page hb + 4096 (e + 1), which
// is page t = p0 + e + 1 of that count (p0 = position of hb in its chunk),
// i.e. chunk c0 + (t >> 4) at offset (t & 15) * 4096.
__device__ __forceinline__ uint32_t first_pos(const ListItem& it) {
  return (uint32_t)((it.hb >> 12) & 15u);
}
__device__ __forceinline__ uint64_t last_chunk(const ListItem& it) {
  const uint32_t m = it.words - (it.pages - 1);  // data entries
  return (it.hb >> 16) + ((first_pos(it) + m) >> 4);
}

// Four consecutive data words of a lane, from the page position t of the
// first: words s < 16 - (t & 15) lie in the chunk whose LUT value is
// (hi_a, lo_a), the others in the next chunk (hi_b, lo_b). LUT values are
// 64 KiB aligned, so adding the in-chunk offset to the low word never carries.
__device__ __forceinline__ void four_words(uint32_t t, uint32_t lo_a, uint32_t hi_a, uint32_t lo_b,
                                           uint32_t hi_b, uint64_t (&v)[4]) {
  const uint32_t off0 = (t & 15u) << 12;
  const uint32_t nsame = 16u - (t & 15u);
  const uint32_t A = lo_a + off0, B = lo_b + off0 - 65536u;
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const bool same = (uint32_t)s < nsame;
    const uint32_t lo = (same ? A : B) + ((uint32_t)s << 12);
    v[s] = ((uint64_t)(same ? hi_a : hi_b) << 32) | lo;
  }
}

// List-word stores. Plain stores measured faster than evict-first hinted
// ones for this pattern (runs at page starts across the whole arena).
__device__ __forceinline__ void st_list32(void* a, uint64_t x, uint64_t y, uint64_t z, uint64_t w,
                                          uint64_t pol) {
  if (DB_PRP_LIST_HINT) {
    st_stream32(a, x, y, z, w, pol);
  } else {
    asm volatile("st.global.v4.u64 [%0], {%1, %2, %3, %4};" ::"l"(a), "l"(x), "l"(y), "l"(z),
                 "l"(w)
                 : "memory");
  }
}
__device__ __forceinline__ void st_list8(void* a, uint64_t x, uint64_t pol) {
  if (DB_PRP_LIST_HINT)
    st_stream8(a, x, pol);
  else
    asm volatile("st.global.u64 [%0], %1;" ::"l"(a), "l"(x) : "memory");
}

// One long request's list, written by a whole warp a list page (512 words)
// at a time, in four steps of 128 words: lane l writes words 4l .. 4l+3 of a
// step with one 32-byte store, so a warp store covers 1 KiB of contiguous
// arena. Word w of list page j is data entry 511 j + w, which names page
// position t = p0 + 1 + 511 j + w (w = 511 of a page with a successor is the
// chain pointer instead). Step k moves a lane's words 128 k positions on,
// exactly 8 chunks, so a lane's chunk offset and where its four words cross
// into the next chunk are worked out once per page. The page's LUT values
// come by shuffle from two windows of 32 chunks anchored at the page's first
// chunk (lane l holds chunks anchor + l and anchor + 32 + l; the first page
// is anchored at c0); a page spans at most 34 of them, and the next page's
// windows load while this one is written.
__device__ __forceinline__ void emit_list(const Params& p, const ListItem& it, uint64_t win0,
                                          uint64_t win1, int lane, uint64_t pol_lut,
                                          uint64_t pol_out) {
  uint64_t* const dst0 = p.arena + (it.pb << 9) + 4 * lane;
  const uint32_t W = it.words;
  // Words written: the list, then 0 up to the end of its last 32-byte sector
  // (no partial-sector writes), or the whole last page with zeroed tails.
  const uint32_t total = p.zero_tail ? (it.pages << 9) : ((W + 3u) & ~3u);
  const uint64_t c0 = it.hb >> 16;
  const uint64_t c_last = last_chunk(it);
  const uint32_t p0 = first_pos(it);
  for (uint32_t j = 0; j < it.pages; ++j) {
    const uint32_t tp = p0 + 1 + 511 * j;            // position of the page's word 0
    const uint32_t anchor = j == 0 ? 0u : (tp >> 4);  // chunk of window lane 0, from c0
    const bool last = j + 1 == it.pages;              // uniform across the warp
    uint64_t nwin0 = 0, nwin1 = 0;
    if (!last) {
      const uint64_t na = c0 + ((tp + 511) >> 4);
      nwin0 = lut_window(p.lut, na + lane, c_last, pol_lut);
      nwin1 = lut_window(p.lut, na + 32 + lane, c_last, pol_lut);
    }
    const uint32_t tl = tp + 4 * lane;
    const uint32_t ql = tl & 15;
    const uint32_t al = (tl >> 4) - anchor;  // at most 8
    // LUT values are 64 KiB aligned: the in-chunk offset is OR-ed into the low word.
    uint32_t offs[4];
    bool useb[4];
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      offs[s] = ((ql + s) & 15u) << 12;
      useb[s] = ql + s >= 16;
    }
    const uint32_t wpage = j << 9;
    uint64_t* const dst = dst0 + wpage;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (last && wpage + 128 * k >= total) break;  // uniform
      const uint32_t ca = al + 8 * k, cb = ca + 1;   // ca <= 32, cb <= 33
      uint32_t alo, ahi, blo, bhi;
      if (k < 3) {                                   // ca <= 24, cb <= 25: first window
        alo = __shfl_sync(kFull, (uint32_t)win0, ca);
        ahi = __shfl_sync(kFull, (uint32_t)(win0 >> 32), ca);
        blo = __shfl_sync(kFull, (uint32_t)win0, cb);
        bhi = __shfl_sync(kFull, (uint32_t)(win0 >> 32), cb);
      } else {
        const uint32_t alo0 = __shfl_sync(kFull, (uint32_t)win0, ca & 31);
        const uint32_t ahi0 = __shfl_sync(kFull, (uint32_t)(win0 >> 32), ca & 31);
        const uint32_t blo0 = __shfl_sync(kFull, (uint32_t)win0, cb & 31);
        const uint32_t bhi0 = __shfl_sync(kFull, (uint32_t)(win0 >> 32), cb & 31);
        const uint32_t alo1 = __shfl_sync(kFull, (uint32_t)win1, ca & 31);
        const uint32_t ahi1 = __shfl_sync(kFull, (uint32_t)(win1 >> 32), ca & 31);
        const uint32_t blo1 = __shfl_sync(kFull, (uint32_t)win1, cb & 31);
        const uint32_t bhi1 = __shfl_sync(kFull, (uint32_t)(win1 >> 32), cb & 31);
        alo = ca < 32 ? alo0 : alo1;
        ahi = ca < 32 ? ahi0 : ahi1;
        blo = cb < 32 ? blo0 : blo1;
        bhi = cb < 32 ? bhi0 : bhi1;
      }
      uint64_t v[4];
#pragma unroll
      for (int s = 0; s < 4; ++s)
        v[s] = ((uint64_t)(useb[s] ? bhi : ahi) << 32) | ((useb[s] ? blo : alo) | offs[s]);
      if (!last) {
        if (k == 3 && lane == 31) v[3] = p.arena_base + ((it.pb + j + 1) << 12);  // chain pointer
        st_list32(dst + 128 * k, v[0], v[1], v[2], v[3], pol_out);
      } else {
        const uint32_t w = wpage + 128 * k + 4 * lane;
        if (wpage + 128 * k + 128 <= W) {            // a full step of data (uniform)
          st_list32(dst + 128 * k, v[0], v[1], v[2], v[3], pol_out);
        } else {
#pragma unroll
          for (int s = 0; s < 4; ++s)
            if (w + s >= W) v[s] = 0;  // zeroed tail
          if (w + 3 < total) {
            st_list32(dst + 128 * k, v[0], v[1], v[2], v[3], pol_out);
          } else {
#pragma unroll
            for (int s = 0; s < 4; ++s)
              if (w + s < total) st_list8(dst + 128 * k + s, v[s], pol_out);
          }
        }
      }
    }
    win0 = nwin0;
    win1 = nwin1;
  }
}

// Short lists (at most kShortWords entries, one list page) are written by
// 8-lane groups, four lists per warp step: lane g of a group writes words
// 4g .. 4g+3 (one 32-byte store). Such a list touches at most 3 LUT chunks,
// loaded by lanes 0..2 of the group. With zeroed tails every list fills its
// whole page, 32 words per group step.
constexpr uint32_t kShortWords = 32;
// Marker a thread adds to its part of a prefix sum when one of its status
// words is not what it should be. Real sums stay below 2^40 (list pages of at
// most 2^28 requests); 512 markers stay below 2^60.
constexpr uint64_t kSplitBad = 1ull << 50;
__device__ __forceinline__ uint64_t short_window(const Params& p, const ListItem& it, bool valid,
                                                 int lane, uint64_t pol_lut) {
  return valid ? lut_window(p.lut, (it.hb >> 16) + (uint64_t)(lane & 7), last_chunk(it), pol_lut)
               : 0;
}
__device__ __forceinline__ void emit_short(const Params& p, const ListItem& it, bool valid,
                                           uint64_t lutv, int lane, uint64_t pol_out) {
  const int g = lane & 7, g0 = lane & ~7;
  const uint32_t p0 = first_pos(it);
  uint64_t* dst = p.arena + (it.pb << 9);
  const uint32_t total = p.zero_tail ? 512u : ((it.words + 3u) & ~3u);  // whole sectors
  const uint32_t steps = p.zero_tail ? 16u : 1u;  // the same for every group of the warp
  for (uint32_t st = 0; st < steps; ++st) {
    const uint32_t w = st * 32 + 4 * g;
    const uint32_t t = p0 + 1 + w;
    const int sa = g0 + (int)((t >> 4) & 7u), sb = g0 + (int)(((t + 3) >> 4) & 7u);
    const uint32_t lo_a = __shfl_sync(kFull, (uint32_t)lutv, sa);
    const uint32_t hi_a = __shfl_sync(kFull, (uint32_t)(lutv >> 32), sa);
    const uint32_t lo_b = __shfl_sync(kFull, (uint32_t)lutv, sb);
    const uint32_t hi_b = __shfl_sync(kFull, (uint32_t)(lutv >> 32), sb);
    uint64_t v[4];
    four_words(t, lo_a, hi_a, lo_b, hi_b, v);
#pragma unroll
    for (int s = 0; s < 4; ++s)
      if (w + s >= it.words) v[s] = 0;  // zeroed tail
    if (valid) {
      if (w + 3 < total) {
        st_list32(dst + w, v[0], v[1], v[2], v[3], pol_out);
      } else {
#pragma unroll
        for (int s = 0; s < 4; ++s)
          if (w + s < total) st_list8(dst + w + s, v[s], pol_out);
      }
    }
  }
}

// Validity, pages touched (n) and list pages (L) of one request; the same
// arithmetic in every kernel that reads requests.
__device__ __forceinline__ void classify(const Params& p, uint64_t i, uint64_t off, uint32_t len,
                                         bool& valid, uint32_t& npg, uint32_t& L) {
  valid = i < p.n && len != 0 && (off & 3) == 0 && off <= p.heap_size &&
          (uint64_t)len <= p.heap_size - off;
  npg = valid ? (uint32_t)(((off & 4095) + len + 4095) >> 12) : 0;
  L = npg >= 3 ? (npg - 2 + 510) / 511 : 0;  // ceil((list entries - 1) / 511)
}

// Whether any of a thread's requests owns list pages.
__device__ __forceinline__ bool any_list_rows(const uint32_t (&L)[kItems]) {
  uint32_t a = 0;
#pragma unroll
  for (int k = 0; k < kItems; ++k) a |= L[k];
  return a != 0;
}

// Exclusive scan over a tile held as kItems rows of kThreads values, in
// request order (row-major: request k * kThreads + thread). s_scan holds
// kItems * kWarps values.
__device__ __forceinline__ void tile_excl_scan(const uint64_t (&v)[kItems], uint64_t (&excl)[kItems],
                                               uint64_t& total, uint64_t* s_scan) {
  static_assert(kItems * kWarps <= 64, "at most two scan totals per lane");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint64_t x[kItems];
#pragma unroll
  for (int k = 0; k < kItems; ++k) {
    x[k] = v[k];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint64_t y = __shfl_up_sync(kFull, x[k], o);
      if (lane >= o) x[k] += y;
    }
    if (lane == 31) s_scan[k * kWarps + warp] = x[k];
  }
  __syncthreads();
  if (warp == 0) {
    const uint64_t a = 2 * lane < kItems * kWarps ? s_scan[2 * lane] : 0;
    const uint64_t b = 2 * lane + 1 < kItems * kWarps ? s_scan[2 * lane + 1] : 0;
    uint64_t t = a + b;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint64_t y = __shfl_up_sync(kFull, t, o);
      if (lane >= o) t += y;
    }
    const uint64_t before = t - a - b;
    if (2 * lane < kItems * kWarps) s_scan[2 * lane] = before;
    if (2 * lane + 1 < kItems * kWarps) s_scan[2 * lane + 1] = before + a;
    if (lane == 31) s_scan[kItems * kWarps] = t;
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < kItems; ++k) excl[k] = s_scan[k * kWarps + warp] + x[k] - v[k];
  total = s_scan[kItems * kWarps];
}

// Decoupled lookback for tile t (warp 0 only). Publishes the tile's
// aggregate, then sums predecessors 128 at a time (4 per lane, nearest
// first) until an inclusive prefix (or the start of the batch) is found,
// then publishes its own prefix.
__device__ __forceinline__ void lookback(const Params& p, uint64_t t, uint32_t epoch, uint64_t agg,
                                         uint64_t& excl_out, bool& failed) {
  const int lane = threadIdx.x & 31;
  unsigned long long* mine = p.tile_status + t;
  failed = false;
  if (t == 0) {
    if (lane == 0) st_relaxed(mine, status_word(kPrefix, epoch, agg));
    excl_out = 0;
    return;
  }
  if (lane == 0) st_relaxed(mine, status_word(kAggregate, epoch, agg));
  uint64_t excl = 0;
  int64_t top = (int64_t)t - 1;  // newest tile of the window
  Backoff backoff;
  while (true) {
    // This lane's four tiles, nearest first: top - 4 lane - s.
    uint32_t stop_s = 4;           // first of them holding a prefix (or a failure)
    bool empty_before = false;     // an unpublished tile before that
    bool stop_failed = false;
    uint64_t sum = 0;              // values up to and including the stop
#pragma unroll
    for (int sidx = 0; sidx < 4; ++sidx) {
      const int64_t u = top - 4 * lane - sidx;
      uint32_t flag = kPrefix;     // before tile 0: an inclusive prefix of 0
      uint64_t val = 0;
      if (u >= 0) {
        const uint64_t w = ld_relaxed(p.tile_status + u);
        flag = status_flag(w, epoch);
        val = w & kValueMask;
      }
      if (stop_s == 4) {
        if (flag == kEmpty) empty_before = true;
        sum += val;
        if (flag == kPrefix || flag == kFailed) {
          stop_s = (uint32_t)sidx;
          stop_failed = flag == kFailed;
        }
      }
    }
    const uint32_t stop_mask = __ballot_sync(kFull, stop_s < 4);
    const int stop_lane = stop_mask ? __ffs(stop_mask) - 1 : 31;
    const bool counts = lane <= stop_lane;
    if (__ballot_sync(kFull, counts && empty_before)) {
      if (!backoff.wait()) {
        failed = true;
        break;
      }
      continue;
    }
    if (__shfl_sync(kFull, stop_failed ? 1 : 0, stop_lane) && stop_mask) {
      failed = true;
      break;
    }
    excl += warp_sum64(counts ? sum : 0);
    if (stop_mask) break;
    top -= 128;
  }
  if (lane == 0)
    st_relaxed(mine, failed ? status_word(kFailed, epoch, 0)
                            : status_word(kPrefix, epoch, excl + agg));
  excl_out = excl;
}

// kSplit: the list kernel of the two-kernel schedule (tiles by index, first
// list pages from the pair kernel's totals); otherwise the single kernel.
template <bool kSplit>
__global__ void __launch_bounds__(kThreads, DB_PRP_MIN_CTAS) prp_build_kernel(const Params p) {
  __shared__ unsigned long long s_ticket[2];  // this tile's ticket, the next one's
  __shared__ uint64_t s_scan[kItems * kWarps + 1];
  __shared__ unsigned long long s_excl;
  __shared__ int s_failed;
  __shared__ uint32_t s_next, s_next_short, s_warps_done;
  __shared__ uint64_t s_split[kWarps];  // two-kernel schedule: list pages before the tile, by warp
  __shared__ ulonglong2 s_list[kTile];

  // In the two-kernel schedule this kernel runs as a programmatic dependent
  // of the pair kernel and reads what that kernel wrote: wait for it first.
  // If the pair kernel completed the call (epoch E recorded in acc[4], epoch
  // now E + 1, tile 0's word still tagged E), there is nothing to do. Every
  // thread reads the same settled values, so the exit is uniform.
  if (kSplit) {
    wait_for_prerequisites();
    const uint32_t now = *(volatile unsigned int*)&p.hdr->epoch;
    const uint32_t done_epoch = (uint32_t)*(volatile unsigned long long*)&p.hdr->acc[4];
    if (done_epoch + 1 == now && status_flag(ld_relaxed(p.tile_status), done_epoch) == kAggregate)
      return;
  }

  const int lane = threadIdx.x & 31;
  const uint64_t pol_first = policy_evict_first();
  const uint64_t pol_last = policy_evict_last();
  const uint32_t epoch = *(volatile unsigned int*)&p.hdr->epoch;
  uint32_t my_invalid = 0, my_overflow = 0;
  uint64_t my_pages = 0;  // list pages of this CTA's tiles (thread 0's count is used)
  bool any_failed = false;

  if (threadIdx.x == 0) {
    if (!kSplit) s_ticket[0] = atomicAdd(&p.hdr->ticket, 1ull);
    s_warps_done = 0;
  }
  for (uint32_t round = 0;; ++round) {
    // Every thread is past the previous tile (its lists included) here, so
    // the tile's shared memory is free again.
    __syncthreads();
    // Two-kernel schedule: tiles by index (nothing waits on another tile),
    // each split into p.parts parts taken by different CTAs (part `part`
    // writes the requests of warps w with w % parts == part and the lists
    // the tile queues at positions j with j % parts == part); otherwise by
    // ticket, one part.
    uint64_t tile;
    uint32_t part = 0, parts = 1;
    if (kSplit) {  // fewer than 2^32 parts in all: n < 2^28 requests, parts <= 16
      const uint32_t vt = blockIdx.x + round * gridDim.x;
      parts = p.parts;
      tile = vt / parts;
      part = vt % parts;
    } else {
      tile = s_ticket[round & 1];
    }
    if (tile >= p.n_tiles) break;
    if (kSplit) {
      // The pair kernel published every tile's list-page total and wrote the
      // tile in full unless it owns lists or page_base is asked for. Every
      // thread reads the same settled word, so the skip is uniform.
      const uint64_t w = ld_relaxed(p.tile_status + tile);
      if (status_flag(w, epoch) == kAggregate && (w & kValueMask) == 0 && !p.page_base) continue;
    }

    // 1-2. Four requests per thread (rows of the tile): validity, pages
    //      touched, list pages; one scan in request order of the list pages
    //      (bits 0..22), short lists (bits 23..34) and long lists (35..46).
    uint64_t off[kItems];
    uint32_t len[kItems], npg[kItems], L[kItems];
    bool valid[kItems];
    uint64_t v[kItems], ex[kItems], tile_v;
#pragma unroll
    for (int k = 0; k < kItems; ++k) {
      const uint64_t i = tile * kTile + (uint64_t)k * kThreads + threadIdx.x;
      off[k] = 0;
      len[k] = 0;
      if (i < p.n) {
        const ulonglong2 r = ld_stream16(p.req + i, pol_first);
        off[k] = r.x;
        len[k] = (uint32_t)r.y;
      }
    }
#pragma unroll
    for (int k = 0; k < kItems; ++k) {
      const uint64_t i = tile * kTile + (uint64_t)k * kThreads + threadIdx.x;
      classify(p, i, off[k], len[k], valid[k], npg[k], L[k]);
      const bool is_short = L[k] != 0 && npg[k] - 1 <= kShortWords;  // then L = 1, words = n - 1
      v[k] = (uint64_t)L[k] | ((uint64_t)(is_short ? 1 : 0) << 23) |
             ((uint64_t)(L[k] != 0 && !is_short ? 1 : 0) << 35);
    }
    // A tile none of whose requests owns a list, in a call that writes no
    // page_base, needs neither the scan nor its predecessors: it publishes a
    // zero aggregate, takes its next ticket at once (the atomic's latency
    // hides behind the tile's LUT gathers and stores; it holds that ticket
    // only for this short tile, so no later tile waits on it for long) and
    // writes its PRP pairs.
    const bool lists = __syncthreads_or(any_list_rows(L)) != 0;
    if (!kSplit && !lists && !p.page_base) {
      unsigned long long next_ticket = 0;
      if (threadIdx.x == 0) {
        next_ticket = atomicAdd(&p.hdr->ticket, 1ull);
        st_relaxed(p.tile_status + tile, status_word(tile == 0 ? kPrefix : kAggregate, epoch, 0));
      }
#pragma unroll
      for (int k = 0; k < kItems; ++k) {
        const uint64_t i = tile * kTile + (uint64_t)k * kThreads + threadIdx.x;
        uint64_t prp1 = 0, prp2 = 0;
        if (valid[k]) {
          prp1 = bus(p.lut, off[k], pol_last);
          if (npg[k] == 2) prp2 = bus(p.lut, (off[k] & ~4095ull) + 4096, pol_last);
        }
        if (i < p.n) {
          st_stream16(p.prp + i, prp1, prp2, pol_first);
          if (p.status) p.status[i] = valid[k] ? DB_PRP_OK : DB_PRP_INVALID;
          my_invalid += !valid[k];
        }
      }
      if (threadIdx.x == 0) s_ticket[(round + 1) & 1] = next_ticket;
      continue;
    }
    // The PRP1 / PRP2 gathers do not depend on the scan: optionally start
    // them before it (DB_PRP_EARLY_LUT).
    uint64_t g1[kItems], g2[kItems];
#pragma unroll
    for (int k = 0; k < kItems; ++k) {
      g1[k] = (DB_PRP_EARLY_LUT && valid[k]) ? lut_window(p.lut, off[k] >> 16, ~0ull, pol_last) : 0;
      g2[k] = (DB_PRP_EARLY_LUT && npg[k] == 2)
                  ? lut_window(p.lut, ((off[k] & ~4095ull) + 4096) >> 16, ~0ull, pol_last)
                  : 0;
    }
    // Two-kernel schedule: the tile's first list page is the sum of the
    // totals the pair kernel published for the tiles before it (a word that
    // is not this call's aggregate fails the tile).
    if (kSplit) {
      uint64_t psum = 0;
      bool bad = false;
      for (uint64_t u = threadIdx.x; u < tile; u += kThreads) {
        const uint64_t w = ld_relaxed(p.tile_status + u);
        bad |= status_flag(w, epoch) != kAggregate;
        psum += w & kValueMask;
      }
      psum = warp_sum64(psum + (bad ? kSplitBad : 0));
      if (lane == 0) s_split[threadIdx.x >> 5] = psum;  // read after the scan's barriers
    }
    tile_excl_scan(v, ex, tile_v, s_scan);
    const uint64_t tile_L = tile_v & ((1ull << 23) - 1);
    const uint32_t n_short = (uint32_t)(tile_v >> 23) & 4095u;
    const uint32_t n_long = (uint32_t)(tile_v >> 35) & 4095u;

    // 3. First list page of this tile. A tile that owns no list and writes
    //    no page_base never uses it: it publishes its (zero) aggregate and
    //    goes on without waiting for its predecessors.
    if (threadIdx.x < 32) {
      uint64_t excl = 0;
      bool failed = false;
      if (kSplit) {
        const uint64_t w = ld_relaxed(p.tile_status + tile);
        excl = warp_sum64(lane < kWarps ? s_split[lane] : 0);
        failed = excl >= kSplitBad || status_flag(w, epoch) != kAggregate ||
                 (w & kValueMask) != tile_L;
        if (failed) excl = 0;
      } else if (tile_L != 0 || p.page_base)
        lookback(p, tile, epoch, tile_L, excl, failed);
      else if (lane == 0)
        st_relaxed(p.tile_status + tile, status_word(tile == 0 ? kPrefix : kAggregate, epoch, 0));
      if (lane == 0) {
        s_excl = excl;
        s_failed = failed;
        s_next = 0;
        s_next_short = 0;
      }
    }
    __syncthreads();
    const bool failed = s_failed != 0;
    any_failed |= failed;

    // 4. PRP1 / PRP2, page_base, status (this part's warps); queue the lists.
    const bool mine = !kSplit || (uint32_t)(threadIdx.x >> 5) % parts == part;
#pragma unroll
    for (int k = 0; k < kItems; ++k) {
      const uint64_t i = tile * kTile + (uint64_t)k * kThreads + threadIdx.x;
      const uint64_t pb = s_excl + (ex[k] & ((1ull << 23) - 1));
      const bool ovf = L[k] != 0 && pb + L[k] > p.cap;
      uint64_t prp1 = 0, prp2 = 0;
      if (valid[k] && !ovf && !failed) {
        const uint64_t x2 = (off[k] & ~4095ull) + 4096;  // the second page
        prp1 = DB_PRP_EARLY_LUT ? g1[k] + (off[k] & 0xFFFFull) : bus(p.lut, off[k], pol_last);
        if (npg[k] == 2)
          prp2 = DB_PRP_EARLY_LUT ? g2[k] + (x2 & 0xFFFFull) : bus(p.lut, x2, pol_last);
        else if (npg[k] >= 3)
          prp2 = p.arena_base + (pb << 12);
      }
      if (i < p.n && mine) {
        st_stream16(p.prp + i, prp1, prp2, pol_first);
        if (p.page_base) p.page_base[i] = pb;
        if (p.status)
          p.status[i] = !valid[k] ? DB_PRP_INVALID : (ovf ? DB_PRP_OVERFLOW : DB_PRP_OK);
        my_invalid += !valid[k];
        my_overflow += ovf;
      }
      if (L[k]) {  // long lists from the front of the queue, short ones from the back
        const bool is_short = npg[k] - 1 <= kShortWords;
        const uint32_t q = is_short ? kTile - 1 - ((uint32_t)(ex[k] >> 23) & 4095u)
                                    : (uint32_t)(ex[k] >> 35) & 4095u;
        s_list[q] = pack_item(off[k] & ~4095ull, (ovf || failed) ? 0 : L[k], pb, npg[k]);
      }
    }
    if (part == 0) my_pages += tile_L;
    __syncthreads();

    // 5. Lists. Long ones: a warp takes the next queued request and writes
    //    its run, with the LUT window of the request after it already in
    //    flight. Then short ones, four per warp.
    uint32_t j = 0;
    if (lane == 0) j = kSplit ? part + parts * atomicAdd(&s_next, 1u) : atomicAdd(&s_next, 1u);
    j = __shfl_sync(kFull, j, 0);
    ListItem it{};
    uint64_t win0 = 0, win1 = 0;
    if (j < n_long) {
      it = unpack_item(s_list[j]);
      if (it.pages) {
        win0 = lut_window(p.lut, (it.hb >> 16) + lane, last_chunk(it), pol_last);
        win1 = lut_window(p.lut, (it.hb >> 16) + 32 + lane, last_chunk(it), pol_last);
      }
    }
    while (j < n_long) {
      uint32_t jn = 0;
      if (lane == 0) jn = kSplit ? part + parts * atomicAdd(&s_next, 1u) : atomicAdd(&s_next, 1u);
      jn = __shfl_sync(kFull, jn, 0);
      ListItem nx{};
      uint64_t nwin0 = 0, nwin1 = 0;
      if (jn < n_long) {
        nx = unpack_item(s_list[jn]);
        if (nx.pages) {
          nwin0 = lut_window(p.lut, (nx.hb >> 16) + lane, last_chunk(nx), pol_last);
          nwin1 = lut_window(p.lut, (nx.hb >> 16) + 32 + lane, last_chunk(nx), pol_last);
        }
      }
      if (it.pages) emit_list(p, it, win0, win1, lane, pol_last, pol_first);
      j = jn;
      it = nx;
      win0 = nwin0;
      win1 = nwin1;
    }
    // Short lists, four per warp step, the next four already loading.
    uint32_t q0 = 0;
    if (lane == 0)
      q0 = kSplit ? 4u * (part + parts * atomicAdd(&s_next_short, 1u)) : atomicAdd(&s_next_short, 4u);
    q0 = __shfl_sync(kFull, q0, 0);
    ListItem sh{};
    bool sv = false;
    uint64_t swin = 0;
    if (q0 < n_short) {
      const uint32_t q = q0 + (uint32_t)(lane >> 3);
      if (q < n_short) sh = unpack_item(s_list[kTile - 1 - q]);
      sv = q < n_short && sh.pages != 0;
      swin = short_window(p, sh, sv, lane, pol_last);
    }
    while (q0 < n_short) {
      uint32_t q1 = 0;
      if (lane == 0)
        q1 = kSplit ? 4u * (part + parts * atomicAdd(&s_next_short, 1u))
                    : atomicAdd(&s_next_short, 4u);
      q1 = __shfl_sync(kFull, q1, 0);
      ListItem nsh{};
      bool nsv = false;
      uint64_t nswin = 0;
      if (q1 < n_short) {
        const uint32_t q = q1 + (uint32_t)(lane >> 3);
        if (q < n_short) nsh = unpack_item(s_list[kTile - 1 - q]);
        nsv = q < n_short && nsh.pages != 0;
        nswin = short_window(p, nsh, nsv, lane, pol_last);
      }
      emit_short(p, sh, sv, swin, lane, pol_first);
      q0 = q1;
      sh = nsh;
      sv = nsv;
      swin = nswin;
    }
    // The last warp to finish the tile's lists takes the next ticket, so no
    // ticket is held while lists of this tile are still being written.
    if (!kSplit && lane == 0 && atomicAdd(&s_warps_done, 1u) == kWarps - 1) {
      s_warps_done = 0;
      s_ticket[(round + 1) & 1] = atomicAdd(&p.hdr->ticket, 1ull);
    }
  }

  // Counters and hand-off to the next call.
  __shared__ int s_last;
  my_invalid = warp_sum32(my_invalid);
  my_overflow = warp_sum32(my_overflow);
  if (lane == 0 && (my_invalid | my_overflow)) {
    atomicAdd(&p.hdr->acc[0], (unsigned long long)my_invalid);
    atomicAdd(&p.hdr->acc[1], (unsigned long long)my_overflow);
  }
  if (threadIdx.x == 0 && any_failed) atomicOr(&p.hdr->err, DB_ERR_TIMEOUT);
  if (threadIdx.x == 0 && my_pages) atomicAdd(&p.hdr->acc[2], (unsigned long long)my_pages);
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = atomicAdd(&p.hdr->done, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (s_last) {
    __threadfence();
    if (threadIdx.x == 0) {
      const unsigned long long inv = atomicExch(&p.hdr->acc[0], 0ull);
      const unsigned long long ovf = atomicExch(&p.hdr->acc[1], 0ull);
      const unsigned long long pages = atomicExch(&p.hdr->acc[2], 0ull);
      const unsigned int err = atomicExch(&p.hdr->err, 0u);
      if (p.ctr) {
        p.ctr->total = err ? 0 : pages;
        p.ctr->n_invalid = inv;
        p.ctr->n_overflow = ovf;
        p.ctr->err = err;
      }
    }
    end_of_call(p.hdr, p.tile_status, p.n_tiles, p.cap_tiles, true);
  }
}

// Pair kernel of the two-kernel schedule (batches that fit one wave of it):
// one CTA per tile, by index, with nothing to wait for; light enough for four
// CTAs of 512 threads per SM, so a batch of up to 4 x 2048 x SMs requests has
// all its requests in flight at once. A warp none of whose requests owns a
// list writes their PRP pairs and statuses at once (when page_base is not
// asked for). Each tile's list-page total is published; a tile with lists,
// or every tile when page_base is asked for, is left to the list kernel,
// which writes the whole tile again (the same values for these warps). The
// last CTA to finish completes the call itself when no tile was left over:
// it publishes the counters, records the call's epoch in acc[4] and
// advances the epoch, and the list kernel, finding that record, exits.
// (At an epoch wrap it leaves the call to the list kernel, which clears the
// status words.)
constexpr int kPairCtasPerSm = 4;
__global__ void __launch_bounds__(kThreads, kPairCtasPerSm) prp_pairs_kernel(const Params p) {
  __shared__ uint32_t s_part[kWarps], s_inv[kWarps];
  dependents_may_launch();  // the list kernel may take SMs as these CTAs finish
  const uint64_t tile = blockIdx.x;
  const int lane = threadIdx.x & 31;
  const uint64_t pol_first = policy_evict_first();
  const uint64_t pol_last = policy_evict_last();
  uint64_t off[kItems];
  uint32_t len[kItems];
#pragma unroll
  for (int k = 0; k < kItems; ++k) {
    const uint64_t i = tile * kTile + (uint64_t)k * kThreads + threadIdx.x;
    off[k] = 0;
    len[k] = 0;
    if (i < p.n) {
      const ulonglong2 r = ld_stream16(p.req + i, pol_first);
      off[k] = r.x;
      len[k] = (uint32_t)r.y;
    }
  }
  uint32_t my_L = 0, two = 0, ok = 0, my_invalid = 0;  // bit k: request k has two pages / is valid
#pragma unroll
  for (int k = 0; k < kItems; ++k) {
    const uint64_t i = tile * kTile + (uint64_t)k * kThreads + threadIdx.x;
    bool valid;
    uint32_t npg, L;
    classify(p, i, off[k], len[k], valid, npg, L);
    my_L += L;  // at most 4 x 2053
    ok |= (valid ? 1u : 0u) << k;
    two |= (npg == 2 ? 1u : 0u) << k;
    my_invalid += (i < p.n && !valid) ? 1u : 0u;
  }
  if (!p.page_base && !__any_sync(kFull, my_L != 0)) {
#pragma unroll
    for (int k = 0; k < kItems; ++k) {
      const uint64_t i = tile * kTile + (uint64_t)k * kThreads + threadIdx.x;
      const bool valid = (ok >> k) & 1u;
      uint64_t prp1 = 0, prp2 = 0;
      if (valid) {
        prp1 = bus(p.lut, off[k], pol_last);
        if ((two >> k) & 1u) prp2 = bus(p.lut, (off[k] & ~4095ull) + 4096, pol_last);
      }
      if (i < p.n) {
        st_stream16(p.prp + i, prp1, prp2, pol_first);
        if (p.status) p.status[i] = valid ? DB_PRP_OK : DB_PRP_INVALID;
      }
    }
  }
  my_L = warp_sum32(my_L);  // at most 2^23 per tile
  my_invalid = warp_sum32(my_invalid);
  if (lane == 0) {
    s_part[threadIdx.x >> 5] = my_L;
    s_inv[threadIdx.x >> 5] = my_invalid;
  }
  __syncthreads();
  if (threadIdx.x != 0) return;
  uint64_t agg = 0, inv = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    agg += s_part[w];
    inv += s_inv[w];
  }
  const uint32_t epoch = *(volatile unsigned int*)&p.hdr->epoch;
  st_relaxed(p.tile_status + tile, status_word(kAggregate, epoch, agg));
  if (agg != 0 || p.page_base)
    atomicAdd(&p.hdr->acc[3], 1ull);  // left to the list kernel
  else if (inv)
    atomicAdd(&p.hdr->acc[0], inv);
  __threadfence();
  if (atomicAdd(&p.hdr->done, 1u) != gridDim.x - 1) return;
  // Last CTA: every other CTA's counts and words are in place.
  __threadfence();
  ScanHeader* h = p.hdr;
  const unsigned long long left = atomicExch(&h->acc[3], 0ull);
  const unsigned long long n_inv = atomicExch(&h->acc[0], 0ull);  // in the same round trip
  if (left != 0 || ((epoch + 1) & kEpochMask) == 0) {
    if (n_inv) atomicAdd(&h->acc[0], n_inv);  // the list kernel publishes it
    h->done = 0;                              // and counts its own CTAs
    return;
  }
  if (p.ctr) {
    p.ctr->total = 0;
    p.ctr->n_invalid = n_inv;
    p.ctr->n_overflow = 0;
    p.ctr->err = 0;
  }
  h->acc[4] = epoch;  // this call is complete
  if (h->hw_words < p.n_tiles) h->hw_words = p.n_tiles;
  h->epoch = epoch + 1;
  h->ticket = 0;
  h->done = 0;
}

template <bool kSplit>
int grid_for(uint64_t n_tiles) {
  static int per_sm[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  int& occ = per_sm[dev & 63];
  if (occ == 0) {
    int o = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, prp_build_kernel<kSplit>, kThreads, 0) !=
            cudaSuccess ||
        o < 1)
      o = 1;
    occ = o;
  }
  const uint64_t g = (uint64_t)num_sms() * (uint64_t)occ;
  return (int)(n_tiles < g ? n_tiles : g);
}

// Tiles one wave of the pair kernel holds on this device: batches of at most
// this many tiles take the two-kernel schedule.
uint64_t pair_wave_tiles() {
  static int per_sm[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  int& occ = per_sm[dev & 63];
  if (occ == 0) {
    int o = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, prp_pairs_kernel, kThreads, 0) !=
            cudaSuccess ||
        o < 1)
      o = 1;
    occ = o;
  }
  return (uint64_t)num_sms() * (uint64_t)occ;
}

}  // namespace prp
}  // namespace db

using namespace db;

extern "C" int db_prp_workspace_size(uint64_t n, size_t* bytes) {
  if (!bytes) return -EINVAL;
  if (n > prp::kMaxRequests) return -EINVAL;
  *bytes = prp::ws_bytes_for(n);
  return 0;
}

extern "C" int db_prp_build(const db_prp_req* req, uint64_t n, const uint64_t* lut,
                            uint64_t heap_size, uint64_t arena_base, uint64_t arena_cap_pages,
                            uint64_t* arena, db_prp_out* prp, uint64_t* page_base,
                            uint8_t* status, db_counters* ctr, uint32_t flags, void* ws,
                            size_t ws_bytes, void* stream) {
  cudaStream_t s = (cudaStream_t)stream;
  if (n > prp::kMaxRequests) return -EINVAL;
  if (heap_size == 0 || heap_size % 65536 != 0) return -EINVAL;
  if (arena_base % 4096 != 0) return -EINVAL;
  if (arena_cap_pages > ((~0ull - arena_base) >> 12)) return -EINVAL;  // bus addresses must not wrap
  if (arena_cap_pages > (1ull << 40)) return -EINVAL;
  if (flags & ~(DB_PRP_ZERO_TAIL | DB_PRP_SCHED_SINGLE | DB_PRP_SCHED_SPLIT)) return -EINVAL;
  if ((flags & DB_PRP_SCHED_SINGLE) && (flags & DB_PRP_SCHED_SPLIT)) return -EINVAL;
  if (ctr && !aligned(ctr, 8)) return -EINVAL;
  if (n == 0) {
    if (ctr) cudaMemsetAsync(ctr, 0, sizeof(db_counters), s);
    return launch_result();
  }
  if (!req || !lut || !prp || !ws) return -EINVAL;
  if (arena_cap_pages != 0 && !arena) return -EINVAL;
  if (!aligned(req, 16) || !aligned(prp, 16) || !aligned(lut, 8) || !aligned(ws, 256))
    return -EINVAL;
  if (arena && !aligned(arena, 32)) return -EINVAL;
  if (page_base && !aligned(page_base, 8)) return -EINVAL;
  if (ws_bytes < prp::ws_bytes_for(n)) return -ENOSPC;

  prp::Params p;
  p.req = reinterpret_cast<const ulonglong2*>(req);
  p.n = n;
  p.n_tiles = prp::tiles_for(n);
  p.lut = lut;
  p.heap_size = heap_size;
  p.arena_base = arena_base;
  p.cap = arena_cap_pages;
  p.arena = arena;
  p.prp = reinterpret_cast<ulonglong2*>(prp);
  p.page_base = page_base;
  p.status = status;
  p.ctr = ctr;
  p.zero_tail = (flags & DB_PRP_ZERO_TAIL) ? 1u : 0u;
  p.hdr = reinterpret_cast<ScanHeader*>(ws);
  p.tile_status = reinterpret_cast<unsigned long long*>(static_cast<char*>(ws) + kScanHeaderBytes);
  p.cap_tiles = (ws_bytes - kScanHeaderBytes) / 8;
  p.parts = 1;
  bool split = p.n_tiles <= prp::pair_wave_tiles();
  if (flags & DB_PRP_SCHED_SINGLE) split = false;
  if (flags & DB_PRP_SCHED_SPLIT) split = true;
  if (!split) {
    prp::prp_build_kernel<false>
        <<<prp::grid_for<false>(p.n_tiles), prp::kThreads, 0, s>>>(p);
    return launch_result();
  }
  // List kernel: with few tiles, several CTAs share each tile's lists.
  const uint64_t resident = (uint64_t)prp::grid_for<true>(~0ull);
  uint64_t parts = resident / p.n_tiles;
  parts = parts < 1 ? 1 : (parts > (uint64_t)prp::kWarps ? (uint64_t)prp::kWarps : parts);
  p.parts = (uint32_t)parts;
  prp::prp_pairs_kernel<<<(unsigned)p.n_tiles, prp::kThreads, 0, s>>>(p);
  const int rc = launch_result();
  if (rc) return rc;
  return launch_dependent(prp::prp_build_kernel<true>,
                          (unsigned)prp::grid_for<true>(p.n_tiles * parts), prp::kThreads, 0, s,
                          p);
}

// ---------------------------------------------------------------------------
// db_prp_build_static: the same build with its scratch in a static device
// array instead of a caller workspace (for callers that must not allocate).
#include <cuda.h>

#include <mutex>

namespace db {
namespace prp {

constexpr size_t kStaticWsBytes = ws_bytes_for(DB_PRP_STATIC_MAX_REQUESTS);

// Zero when the module loads; every call leaves it ready for the next call.
static __device__ __align__(256) unsigned char g_static_ws[kStaticWsBytes];

// Device address of g_static_ws in the current context. Host code cannot use
// the symbol itself (on the host it names a stand-in, not device memory), so
// the address is looked up with the device current and kept per device with
// the ID of the context it belongs to. A device reset destroys that context
// (the module, and the array, load again elsewhere in the next one), so a
// call whose context ID differs looks the address up again. The context
// queries come from the driver through the runtime's entry-point lookup.
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

int current_context_id(CtxGetCurrentFn get_current, CtxGetIdFn get_id, unsigned long long* id) {
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return -1;
  return get_id(ctx, id) == CUDA_SUCCESS ? 0 : -1;
}

int static_ws_address(void** out) {
  struct Entry {
    unsigned long long ctx_id;
    void* addr;
  };
  static std::mutex mu;
  static Entry cache[64] = {};
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_failure(e);
  if (dev < 0 || dev >= 64) return -EINVAL;
  std::lock_guard<std::mutex> lock(mu);
  if (!get_current || !get_id) {
    cudaDriverEntryPointQueryResult q1 = cudaDriverEntryPointSymbolNotFound, q2 = q1;
    void *f1 = nullptr, *f2 = nullptr;
    e = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1);
    if (e != cudaSuccess) return cuda_failure(e);
    e = cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2);
    if (e != cudaSuccess) return cuda_failure(e);
    if (q1 != cudaDriverEntryPointSuccess || q2 != cudaDriverEntryPointSuccess || !f1 || !f2)
      return -EIO;
    get_current = reinterpret_cast<CtxGetCurrentFn>(f1);
    get_id = reinterpret_cast<CtxGetIdFn>(f2);
  }
  unsigned long long id = 0;
  if (cache[dev].addr && current_context_id(get_current, get_id, &id) == 0 &&
      id == cache[dev].ctx_id) {
    *out = cache[dev].addr;
    return 0;
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_static_ws);  // makes the device's context current if need be
  if (e != cudaSuccess) return cuda_failure(e);
  if (current_context_id(get_current, get_id, &id) != 0) return -EIO;
  cache[dev].ctx_id = id;
  cache[dev].addr = p;
  *out = p;
  return 0;
}

}  // namespace prp
}  // namespace db

extern "C" int db_prp_build_static(const db_prp_req* req, uint64_t n, const uint64_t* lut,
                                   uint64_t heap_size, uint64_t arena_base,
                                   uint64_t arena_cap_pages, uint64_t* arena, db_prp_out* prp,
                                   uint64_t* page_base, uint8_t* status, db_counters* ctr,
                                   uint32_t flags, void* stream) {
  if (n > DB_PRP_STATIC_MAX_REQUESTS) return -E2BIG;
  void* ws = nullptr;
  const int rc = prp::static_ws_address(&ws);
  if (rc) return rc;
  return db_prp_build(req, n, lut, heap_size, arena_base, arena_cap_pages, arena, prp, page_base,
                      status, ctr, flags, ws, prp::kStaticWsBytes, stream);
}
