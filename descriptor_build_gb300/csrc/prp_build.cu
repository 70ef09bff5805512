// NVMe PRP construction from a 64 KiB-granular bus-address LUT (sm_103a).
//
// Source: xNVMe "uPCIe CUDA" backend page -- introduction (bus address per
// 64 KiB chunk in a LUT, PRP entries at 4 KiB from sub-page offsets),
// "Memory Architecture" (PRP lists in their own region) and "Limitations"
// (512 entries per 4 KiB list page; 513 x 4 KiB with PRP1). Lists longer than
// one page chain through slot 511 (NVMe convention).
//
// One persistent kernel, single pass over the requests:
//   1. a CTA takes a tile of 512 requests by atomic ticket and loads one
//      16-byte request per thread;
//   2. page count n and list-page count L per request, block scan of L;
//   3. decoupled lookback over the tiles before it (one status word per
//      tile in the workspace, bounded wait) gives the tile's first list page;
//   4. PRP1/PRP2, page_base and status go out as 16/8/1-byte stores;
//   5. the tile's lists are written by warps that take one request at a time
//      from a shared-memory queue: each list is a contiguous run of 8-byte
//      words starting on a 4 KiB page, written as 16-byte stores.
// The last CTA to finish publishes the counters and readies the workspace
// for the next call (new epoch, ticket back to 0).
#include "common.cuh"

namespace db {
namespace prp {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kTile = kThreads;  // requests per tile
constexpr uint32_t kPackShift = 21;  // list pages of a tile < 2^21

// Workspace: ScanHeader (acc[0] invalid, acc[1] overflow), then one status
// word per tile.
constexpr uint64_t tiles_for(uint64_t n) { return (n + kTile - 1) / kTile; }
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
  ScanHeader* hdr;
  unsigned long long* tile_status;  // [cap_tiles]
  uint64_t cap_tiles;
};

// A request that owns list pages, queued for the emission phase.
struct ListItem {
  uint64_t pb;    // first list page (arena page index)
  uint64_t hb;    // heap offset of the request's first 4 KiB page
  uint32_t words; // data entries + chain pointers
  uint32_t pages; // list pages (0: skip, the list did not fit)
};

__device__ __forceinline__ uint64_t bus(const uint64_t* lut, uint64_t x, uint64_t pol) {
  return ld_table8(lut + (x >> 16), pol) + (x & 0xFFFFull);
}

// Word w of a list: slot 511 of every page but the last points at the next
// page; every other word is data entry e = w - (pointers before w), which
// names the heap page hb + 4096 (e + 1).
__device__ __forceinline__ uint64_t list_word(const Params& p, const ListItem& it, uint32_t w,
                                              uint64_t pol) {
  if (w >= it.words) return 0;  // zeroed tail
  const uint32_t j = w >> 9;
  if ((w & 511u) == 511u && j + 1 < it.pages) return p.arena_base + ((it.pb + j + 1) << 12);
  const uint64_t x = it.hb + ((uint64_t)(w - j + 1) << 12);
  return bus(p.lut, x, pol);
}

// Decoupled lookback for tile t (warp 0 only). Publishes the tile's
// aggregate, then sums predecessors 32 at a time until an inclusive prefix
// (or the start of the batch) is found, then publishes its own prefix.
__device__ __forceinline__ void lookback(const Params& p, uint64_t t, uint32_t epoch, uint64_t agg,
                                         uint64_t& excl_out, bool& failed) {
  const int lane = threadIdx.x & 31;
  unsigned long long* mine = p.tile_status + t;
  failed = false;
  if (t == 0) {
    if (lane == 0) st_release(mine, status_word(kPrefix, epoch, agg));
    excl_out = 0;
    return;
  }
  if (lane == 0) st_release(mine, status_word(kAggregate, epoch, agg));
  uint64_t excl = 0;
  int64_t top = (int64_t)t - 1;  // newest tile of the window
  Backoff backoff;
  while (true) {
    const int64_t u = top - lane;
    uint32_t flag = kPrefix;  // before tile 0: an inclusive prefix of 0
    uint64_t val = 0;
    if (u >= 0) {
      const uint64_t w = ld_acquire(p.tile_status + u);
      flag = status_flag(w, epoch);
      val = w & kValueMask;
    }
    const uint32_t stop_mask = __ballot_sync(kFull, flag == kPrefix || flag == kFailed);
    const int stop = stop_mask ? __ffs(stop_mask) - 1 : 31;
    const uint32_t upto = stop == 31 ? kFull : ((2u << stop) - 1u);
    if (__ballot_sync(kFull, flag == kEmpty) & upto) {
      if (!backoff.wait()) {
        failed = true;
        break;
      }
      continue;
    }
    if (__ballot_sync(kFull, flag == kFailed) & upto) {
      failed = true;
      break;
    }
    excl += warp_sum64(lane <= stop ? val : 0);
    if (stop_mask) break;
    top -= 32;
  }
  if (lane == 0)
    st_release(mine, failed ? status_word(kFailed, epoch, 0)
                            : status_word(kPrefix, epoch, excl + agg));
  excl_out = excl;
}

__global__ void __launch_bounds__(kThreads, 2) prp_build_kernel(const Params p) {
  __shared__ unsigned long long s_ticket;
  __shared__ uint32_t s_scan[kWarps];
  __shared__ unsigned long long s_excl;
  __shared__ int s_failed;
  __shared__ uint32_t s_next;
  __shared__ ListItem s_list[kTile];

  const int lane = threadIdx.x & 31;
  const uint64_t pol_first = policy_evict_first();
  const uint64_t pol_last = policy_evict_last();
  const uint32_t epoch = *(volatile unsigned int*)&p.hdr->epoch;
  uint32_t my_invalid = 0, my_overflow = 0;
  bool any_failed = false;

  for (;;) {
    if (threadIdx.x == 0) s_ticket = atomicAdd(&p.hdr->ticket, 1ull);
    __syncthreads();
    const uint64_t tile = s_ticket;
    if (tile >= p.n_tiles) break;

    // 1-2. One request per thread: validity, pages touched, list pages.
    const uint64_t i = tile * kTile + threadIdx.x;
    const bool in = i < p.n;
    uint64_t off = 0;
    uint32_t len = 0;
    if (in) {
      const ulonglong2 r = ld_stream16(p.req + i, pol_first);
      off = r.x;
      len = (uint32_t)r.y;
    }
    const bool valid = in && len != 0 && (off & 3) == 0 && off <= p.heap_size &&
                       (uint64_t)len <= p.heap_size - off;
    const uint32_t npg = valid ? (uint32_t)(((off & 4095) + len + 4095) >> 12) : 0;
    const uint32_t L = npg >= 3 ? (npg - 2 + 510) / 511 : 0;  // ceil((list entries - 1) / 511)
    uint32_t excl_pack, tile_pack;
    block_excl_scan<kWarps>(L | ((L ? 1u : 0u) << kPackShift), excl_pack, tile_pack, s_scan);
    const uint32_t tile_L = tile_pack & ((1u << kPackShift) - 1);
    const uint32_t n_list = tile_pack >> kPackShift;

    // 3. First list page of this tile.
    if (threadIdx.x < 32) {
      uint64_t excl;
      bool failed;
      lookback(p, tile, epoch, tile_L, excl, failed);
      if (lane == 0) {
        s_excl = excl;
        s_failed = failed;
        s_next = 0;
      }
    }
    __syncthreads();
    const bool failed = s_failed != 0;
    any_failed |= failed;
    const uint64_t pb = s_excl + (excl_pack & ((1u << kPackShift) - 1));

    // 4. PRP1 / PRP2.
    const bool ovf = L != 0 && pb + L > p.cap;
    uint64_t prp1 = 0, prp2 = 0;
    if (valid && !ovf && !failed) {
      prp1 = bus(p.lut, off, pol_last);
      if (npg == 2)
        prp2 = bus(p.lut, (off & ~4095ull) + 4096, pol_last);
      else if (npg >= 3)
        prp2 = p.arena_base + (pb << 12);
    }
    if (in) {
      st_stream16(p.prp + i, prp1, prp2, pol_first);
      if (p.page_base) p.page_base[i] = pb;
      if (p.status) p.status[i] = !valid ? DB_PRP_INVALID : (ovf ? DB_PRP_OVERFLOW : DB_PRP_OK);
      my_invalid += !valid;
      my_overflow += ovf;
    }
    if (L) {
      ListItem it;
      it.pb = pb;
      it.hb = off & ~4095ull;
      it.words = (npg - 1) + (L - 1);
      it.pages = (ovf || failed) ? 0 : L;
      s_list[excl_pack >> kPackShift] = it;
    }
    if (tile + 1 == p.n_tiles && threadIdx.x == 0 && p.ctr && !failed)
      p.ctr->total = s_excl + tile_L;
    __syncthreads();

    // 5. Lists: a warp takes the next queued request and writes its run.
    for (;;) {
      uint32_t j = 0;
      if (lane == 0) j = atomicAdd(&s_next, 1u);
      j = __shfl_sync(kFull, j, 0);
      if (j >= n_list) break;
      const ListItem it = s_list[j];
      if (it.pages == 0) continue;
      uint64_t* dst = p.arena + (it.pb << 9);
      const uint32_t total = p.zero_tail ? (it.pages << 9) : it.words;
      for (uint32_t w = 2 * lane; w < total; w += 64) {
        const uint64_t v0 = list_word(p, it, w, pol_last);
        if (w + 1 < total) {
          const uint64_t v1 = list_word(p, it, w + 1, pol_last);
          st_stream16(dst + w, v0, v1, pol_first);
        } else {
          st_stream8(dst + w, v0, pol_first);
        }
      }
    }
    __syncthreads();
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
      const unsigned int err = atomicExch(&p.hdr->err, 0u);
      if (p.ctr) {
        p.ctr->n_invalid = inv;
        p.ctr->n_overflow = ovf;
        p.ctr->err = err;
        if (err) p.ctr->total = 0;
      }
    }
    end_of_call(p.hdr, p.tile_status, p.n_tiles, p.cap_tiles, true);
  }
}

int grid_for(uint64_t n_tiles) {
  static int per_sm[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  int& occ = per_sm[dev & 63];
  if (occ == 0) {
    int o = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, prp_build_kernel, kThreads, 0) !=
            cudaSuccess ||
        o < 1)
      o = 1;
    occ = o;
  }
  const uint64_t g = (uint64_t)num_sms() * (uint64_t)occ;
  return (int)(n_tiles < g ? n_tiles : g);
}

}  // namespace prp
}  // namespace db

using namespace db;

extern "C" int db_prp_workspace_size(uint64_t n, size_t* bytes) {
  (void)n;
  if (!bytes) return -EINVAL;
  if (n > (1ull << 29)) return -EINVAL;
  *bytes = prp::ws_bytes_for(n);
  return 0;
}

extern "C" int db_prp_build(const db_prp_req* req, uint64_t n, const uint64_t* lut,
                            uint64_t heap_size, uint64_t arena_base, uint64_t arena_cap_pages,
                            uint64_t* arena, db_prp_out* prp, uint64_t* page_base,
                            uint8_t* status, db_counters* ctr, uint32_t flags, void* ws,
                            size_t ws_bytes, void* stream) {
  cudaStream_t s = (cudaStream_t)stream;
  if (n > (1ull << 29)) return -EINVAL;
  if (heap_size == 0 || heap_size % 65536 != 0) return -EINVAL;
  if (arena_base % 4096 != 0) return -EINVAL;
  if (arena_cap_pages > ((~0ull - arena_base) >> 12)) return -EINVAL;  // bus addresses must not wrap
  if (arena_cap_pages > (1ull << 40)) return -EINVAL;
  if (flags & ~DB_PRP_ZERO_TAIL) return -EINVAL;
  if (ctr && !aligned(ctr, 8)) return -EINVAL;
  if (n == 0) {
    if (ctr) cudaMemsetAsync(ctr, 0, sizeof(db_counters), s);
    return launch_result();
  }
  if (!req || !lut || !prp || !ws) return -EINVAL;
  if (arena_cap_pages != 0 && !arena) return -EINVAL;
  if (!aligned(req, 16) || !aligned(prp, 16) || !aligned(lut, 8) || !aligned(ws, 256))
    return -EINVAL;
  if (arena && !aligned(arena, 16)) return -EINVAL;
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
  prp::prp_build_kernel<<<prp::grid_for(p.n_tiles), prp::kThreads, 0, s>>>(p);
  return launch_result();
}

// ---------------------------------------------------------------------------
// db_prp_build_static: the same build with its scratch in a static device
// array instead of a caller workspace (for callers that must not allocate).
#include <mutex>

namespace db {
namespace prp {

constexpr size_t kStaticWsBytes = ws_bytes_for(DB_PRP_STATIC_MAX_REQUESTS);

// Zero when the module loads; every call leaves it ready for the next call.
static __device__ __align__(256) unsigned char g_static_ws[kStaticWsBytes];

// Device address of g_static_ws on the current device. Host code cannot use
// the symbol itself (on the host it names a stand-in, not device memory), so
// the address is looked up once per device, with that device current.
int static_ws_address(void** out) {
  static std::mutex mu;
  static void* addr[64] = {nullptr};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_failure(e);
  if (dev < 0 || dev >= 64) return -EINVAL;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_ws);
    if (e != cudaSuccess) return cuda_failure(e);
    addr[dev] = p;
  }
  *out = addr[dev];
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
