// Symmetric-heap put translation and stable bucketing into WQE rings (sm_103a).
//
// Source: "mori communication library analysis (1)". Static-heap put:
// raddr = peerPtrs[pe] + offset, rkey = peerRkeys[pe], lkey of the source
// object, one WQE for the whole transfer. Warp-level slot reservation: each
// entry takes the next post index of its send queue, which here is
// head[ring] + (valid puts of the same ring earlier in the batch).
//
// A ring asked for more than `depth` entries takes none of the batch, so the
// per-ring totals must be known before any entry is written. Three launches,
// reduce-then-scan:
//   count    warps stride over tiles of 1024 puts: a per-warp shared-memory
//            histogram over the R rings plus one bin for invalid puts,
//            written column-major: counts[ring][tile].
//   scan     one CTA per ring: exclusive scan of its column in place (staged
//            through shared memory), the ring's batch total, count[], the
//            overflow decision, the head; the last CTA publishes the counters.
//   scatter  persistent CTAs, a tile at a time (the next tile's puts load
//            meanwhile): stable rank of each put inside its warp with
//            __match_any_sync, then across the tile's 32 warp-rows (a warp
//            scan per ring); the first 48 bytes of each WQE are built into
//            shared memory in ring order (48-byte stride, conflict-free
//            read-out) and each ring's run is written out contiguously with
//            16-byte stores, the zero last quarter straight from registers.
// No kernel waits on another CTA.
#include "common.cuh"

namespace db {
namespace wqe {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kItems = 2;
constexpr int kTile = kThreads * kItems;  // 1024 puts per tile
constexpr int kUnits = kItems * kWarps;   // warp-rows of 32 puts, in batch order
constexpr uint32_t kMaxRings = 1024;

// Build-time tuning (defaults measured best on GB300): how the count pass
// histograms a row of 32 puts (0: __match_any_sync + one shared atomic per
// distinct ring, 1: one shared atomic per put), and whether the scatter pass
// runs persistent CTAs (3 per SM) that load their next tile early.
#ifndef DB_WQE_COUNT_MODE
#define DB_WQE_COUNT_MODE 1
#endif
#ifndef DB_WQE_SCATTER_PERSIST
#define DB_WQE_SCATTER_PERSIST 1
#endif

// Workspace: Header, old heads [1024] u64, overflow flags [1024] u32,
// counts [R + 1][tiles] u32 (per-tile counts, then their exclusive prefixes).
struct Header {
  unsigned int done;           // scan CTAs finished in the current call
  unsigned int pad;
  unsigned long long posted;   // accumulators, zero between calls
  unsigned long long invalid;
  unsigned long long overflow;
};
constexpr size_t kHeadOldOff = 256;
constexpr size_t kFullOff = kHeadOldOff + 8 * kMaxRings;
constexpr size_t kCountsOff = kFullOff + 4 * kMaxRings;
inline uint64_t tiles_for(uint64_t n) { return (n + kTile - 1) / kTile; }
inline size_t ws_bytes_for(uint64_t n, uint32_t R) {
  return kCountsOff + ((tiles_for(n) * ((uint64_t)R + 1) * 4 + 255) & ~(uint64_t)255);
}

struct Params {
  const ulonglong2* req;
  uint64_t n;
  uint64_t n_tiles;
  const uint64_t* peer_ptrs;
  const uint32_t* rkeys;
  uint32_t world, n_qp, R, V;
  uint64_t local_base;
  uint32_t lkey;
  uint64_t heap_size;
  unsigned char* rings;
  uint64_t depth;
  uint64_t* head;
  uint32_t* count;
  db_counters* ctr;
  Header* hdr;
  uint64_t* head_old;
  uint32_t* full;
  uint32_t* counts;  // [V][n_tiles]
};

// Ring of a put, or R for an invalid one.
__device__ __forceinline__ uint32_t bin_of(const Params& p, const ulonglong2 r) {
  const uint64_t off = r.x;
  const uint32_t bytes = (uint32_t)r.y;
  const uint32_t pe = (uint32_t)(r.y >> 32) & 0xFFFFu;
  const uint32_t qp = (uint32_t)(r.y >> 48);
  const bool ok = pe < p.world && qp < p.n_qp && bytes != 0 && off <= p.heap_size &&
                  (uint64_t)bytes <= p.heap_size - off;
  return ok ? pe * p.n_qp + qp : p.R;
}

// ---------------------------------------------------------------- count pass
// One warp counts a whole tile (32 rows of 32 puts) into its own shared
// histogram; warps stride over tiles, so no block-wide barrier is needed.
constexpr int kCountThreads = 256;
constexpr int kCountWarps = kCountThreads / 32;
constexpr int kCountUnroll = 4;  // rows of 32 puts loaded at once

__global__ void __launch_bounds__(kCountThreads) wqe_count_kernel(const Params p) {
  extern __shared__ uint32_t s_hist_all[];  // [kCountWarps][V]
  const uint32_t V = p.V;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t* s_hist = s_hist_all + (size_t)warp * V;
  const uint64_t pol_first = policy_evict_first();
  const uint64_t n_warps = (uint64_t)gridDim.x * kCountWarps;
  for (uint64_t tile = (uint64_t)blockIdx.x * kCountWarps + warp; tile < p.n_tiles;
       tile += n_warps) {
    for (uint32_t v = lane; v < V; v += 32) s_hist[v] = 0;
    __syncwarp();
    for (int row = 0; row < kTile / 32; row += kCountUnroll) {
      ulonglong2 r[kCountUnroll];
#pragma unroll
      for (int u = 0; u < kCountUnroll; ++u) {
        const uint64_t i = tile * kTile + (uint64_t)(row + u) * 32 + lane;
        r[u] = i < p.n ? ld_stream16(p.req + i, pol_first) : make_ulonglong2(0, 0);
      }
#pragma unroll
      for (int u = 0; u < kCountUnroll; ++u) {
        const uint64_t i = tile * kTile + (uint64_t)(row + u) * 32 + lane;
        const uint32_t bin = i < p.n ? bin_of(p, r[u]) : V;
        if (DB_WQE_COUNT_MODE == 1) {
          if (bin < V) atomicAdd(&s_hist[bin], 1u);
        } else {
          const uint32_t peers = __match_any_sync(kFull, bin);
          if (bin < V && (peers & lanemask_lt()) == 0) atomicAdd(&s_hist[bin], __popc(peers));
        }
      }
    }
    __syncwarp();
    for (uint32_t v = lane; v < V; v += 32) p.counts[v * p.n_tiles + tile] = s_hist[v];
    __syncwarp();
  }
}

// ----------------------------------------------------------------- scan pass
constexpr int kScanThreads = 1024;
constexpr int kScanSeg = 4 * kScanThreads;  // column entries staged per round

__global__ void __launch_bounds__(kScanThreads) wqe_scan_kernel(const Params p) {
  constexpr int kW = kScanThreads / 32;
  __shared__ uint32_t s_scan[kW];
  __shared__ uint32_t s_col[kScanSeg];
  __shared__ int s_last;
  const uint32_t v = blockIdx.x;
  uint32_t* col = p.counts + (uint64_t)v * p.n_tiles;
  const uint64_t T = p.n_tiles;
  uint64_t carry = 0;
  for (uint64_t s0 = 0; s0 < T; s0 += kScanSeg) {
    const uint32_t len = (uint32_t)(T - s0 < (uint64_t)kScanSeg ? T - s0 : kScanSeg);
    for (uint32_t x = threadIdx.x; x < len; x += kScanThreads) s_col[x] = col[s0 + x];
    __syncthreads();
    uint32_t c[4], mine = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t x = 4 * threadIdx.x + q;
      c[q] = x < len ? s_col[x] : 0u;
      mine += c[q];
    }
    uint32_t excl, seg_total;
    block_excl_scan<kW>(mine, excl, seg_total, s_scan);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t x = 4 * threadIdx.x + q;
      if (x < len) s_col[x] = (uint32_t)carry + excl;
      excl += c[q];
    }
    __syncthreads();
    for (uint32_t x = threadIdx.x; x < len; x += kScanThreads) col[s0 + x] = s_col[x];
    carry += seg_total;
    __syncthreads();
  }
  const uint64_t total = carry;
  if (threadIdx.x == 0) {
    if (v < p.R) {
      const uint64_t h = p.head[v];
      const bool over = total > p.depth;
      p.count[v] = (uint32_t)total;
      p.head_old[v] = h;
      p.full[v] = over ? 1u : 0u;
      if (!over) p.head[v] = h + total;
      if (over)
        atomicAdd(&p.hdr->overflow, (unsigned long long)total);
      else if (total)
        atomicAdd(&p.hdr->posted, (unsigned long long)total);
    } else if (total) {
      atomicAdd(&p.hdr->invalid, (unsigned long long)total);
    }
    __threadfence();
    s_last = atomicAdd(&p.hdr->done, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (s_last && threadIdx.x == 0) {
    __threadfence();
    const unsigned long long posted = atomicExch(&p.hdr->posted, 0ull);
    const unsigned long long invalid = atomicExch(&p.hdr->invalid, 0ull);
    const unsigned long long overflow = atomicExch(&p.hdr->overflow, 0ull);
    if (p.ctr) {
      p.ctr->total = posted;
      p.ctr->n_invalid = invalid;
      p.ctr->n_overflow = overflow;
      p.ctr->err = overflow ? DB_ERR_RING_OVERFLOW : 0u;
    }
    p.hdr->done = 0;
    __threadfence();
  }
}

// -------------------------------------------------------------- scatter pass
inline size_t scatter_smem(uint32_t V) {
  size_t b = (size_t)kTile * 48;    // staged WQEs (bytes 48..63 are zero: not staged)
  b += (size_t)kTile * 8;           // destination of each staged WQE
  b += (size_t)V * 8;               // old heads
  b += (size_t)V * 4 * 4;           // run start, tile count, tile prefix, full flag
  b += (size_t)kUnits * V * 2;      // per warp-row counts
  return (b + 15) & ~(size_t)15;
}

__device__ __forceinline__ void scatter_tile(const Params& p, uint64_t tile, const ulonglong2 (&r)[kItems],
                                             unsigned char* smem, uint32_t* s_scan);

__global__ void __launch_bounds__(kThreads, 3) wqe_scatter_kernel(const Params p) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ uint32_t s_scan[kWarps];
  const uint64_t pol_first = policy_evict_first();
  auto load = [&](uint64_t tile, ulonglong2 (&r)[kItems]) {
#pragma unroll
    for (int k = 0; k < kItems; ++k) {
      const uint64_t i = tile * kTile + (uint64_t)k * kThreads + threadIdx.x;
      r[k] = (tile < p.n_tiles && i < p.n) ? ld_stream16(p.req + i, pol_first)
                                             : make_ulonglong2(0, 0);
    }
  };
  ulonglong2 cur[kItems];
  load(blockIdx.x, cur);
  const uint64_t stride = DB_WQE_SCATTER_PERSIST ? gridDim.x : p.n_tiles;
  for (uint64_t tile = blockIdx.x; tile < p.n_tiles; tile += stride) {
    ulonglong2 nxt[kItems];
    if (DB_WQE_SCATTER_PERSIST) load(tile + stride, nxt);
    scatter_tile(p, tile, cur, smem, s_scan);
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kItems; ++k) cur[k] = DB_WQE_SCATTER_PERSIST ? nxt[k] : cur[k];
  }
}

__device__ __forceinline__ void scatter_tile(const Params& p, uint64_t tile,
                                             const ulonglong2 (&rin)[kItems], unsigned char* smem,
                                             uint32_t* s_scan) {
  const uint32_t V = p.V, R = p.R;
  ulonglong2* s_stage = reinterpret_cast<ulonglong2*>(smem);  // WQE pos, part k at 3 pos + k
  uint64_t* s_dst = reinterpret_cast<uint64_t*>(smem + (size_t)kTile * 48);
  uint64_t* s_head = s_dst + kTile;
  uint32_t* s_run = reinterpret_cast<uint32_t*>(s_head + V);
  uint32_t* s_tot = s_run + V;
  uint32_t* s_pre = s_tot + V;
  uint32_t* s_full = s_pre + V;
  uint16_t* s_cnt = reinterpret_cast<uint16_t*>(s_full + V);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint64_t pol_first = policy_evict_first();

  for (uint32_t x = threadIdx.x; x < kUnits * V; x += kThreads) s_cnt[x] = 0;
  for (uint32_t v = threadIdx.x; v < V; v += kThreads) {
    s_pre[v] = p.counts[v * p.n_tiles + tile];
    if (v < R) {
      s_head[v] = p.head_old[v];
      s_full[v] = p.full[v];
    }
  }
  ulonglong2 r[kItems];
  uint32_t bin[kItems];
#pragma unroll
  for (int k = 0; k < kItems; ++k) {
    const uint64_t i = tile * kTile + (uint64_t)k * kThreads + threadIdx.x;
    r[k] = rin[k];
    bin[k] = i < p.n ? bin_of(p, r[k]) : V;  // outside the batch: no bin
  }
  __syncthreads();

  // Rank inside each warp-row (stable: lower lanes are earlier puts).
  uint32_t lrank[kItems];
#pragma unroll
  for (int k = 0; k < kItems; ++k) {
    const uint32_t peers = __match_any_sync(kFull, bin[k]);
    const uint32_t before = peers & lanemask_lt();
    lrank[k] = __popc(before);
    if (bin[k] < V && before == 0) s_cnt[(k * kWarps + warp) * V + bin[k]] = (uint16_t)__popc(peers);
  }
  __syncthreads();
  // Across warp-rows, in batch order: one warp per ring, lane u = warp-row u.
  static_assert(kUnits == 32, "one lane per warp-row");
  for (uint32_t v = warp; v < V; v += kWarps) {
    const uint32_t c = s_cnt[lane * V + v];
    uint32_t x = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(kFull, x, o);
      if (lane >= o) x += y;
    }
    s_cnt[lane * V + v] = (uint16_t)(x - c);
    if (lane == 31) s_tot[v] = x;
  }
  __syncthreads();
  // Where each ring's run starts in the staging buffer (ring order; the
  // invalid bin is left out). Thread t owns a chunk of consecutive rings.
  const uint32_t chunk = (R + kThreads - 1) / kThreads;
  const uint32_t r0 = threadIdx.x * chunk;
  uint32_t mine = 0;
  for (uint32_t v = r0; v < r0 + chunk && v < R; ++v) mine += s_tot[v];
  uint32_t excl, n_staged;
  block_excl_scan<kWarps>(mine, excl, n_staged, s_scan);
  for (uint32_t v = r0; v < r0 + chunk && v < R; ++v) {
    s_run[v] = excl;
    excl += s_tot[v];
  }
  __syncthreads();

  // Build the first 48 bytes of each WQE in ring order.
#pragma unroll
  for (int k = 0; k < kItems; ++k) {
    const uint32_t v = bin[k];
    if (v >= R) continue;
    const uint64_t i = tile * kTile + (uint64_t)k * kThreads + threadIdx.x;
    const uint32_t local = s_cnt[(k * kWarps + warp) * V + v] + lrank[k];
    const uint32_t pos = s_run[v] + local;
    const uint64_t seq = s_head[v] + s_pre[v] + local;
    const uint64_t off = r[k].x;
    const uint32_t bytes = (uint32_t)r[k].y;
    const uint32_t pe = (uint32_t)(r[k].y >> 32) & 0xFFFFu;
    const uint64_t raddr = __ldg(p.peer_ptrs + pe) + off;
    const uint32_t rkey = __ldg(p.rkeys + pe);
    s_stage[pos * 3 + 0] = make_ulonglong2(raddr, p.local_base + off);
    s_stage[pos * 3 + 1] = make_ulonglong2((uint64_t)bytes | ((uint64_t)p.lkey << 32), (uint64_t)rkey);
    s_stage[pos * 3 + 2] = make_ulonglong2(seq, (uint64_t)(uint32_t)i);
    s_dst[pos] = s_full[v] ? 0ull
                           : (uint64_t)(p.rings + (((uint64_t)v * p.depth + (seq & (p.depth - 1))) << 6));
  }
  __syncthreads();

  // Each ring's run is contiguous in the ring (up to one wrap): 16-byte stores.
  for (uint32_t f = threadIdx.x; f < n_staged * 4; f += kThreads) {
    const uint32_t q = f >> 2, part = f & 3;
    const uint64_t d = s_dst[q];
    if (d) {
      const ulonglong2 x = part < 3 ? s_stage[q * 3 + part] : make_ulonglong2(0, 0);
      st_stream16(reinterpret_cast<void*>(d + part * 16), x.x, x.y, pol_first);
    }
  }
}

// Allow the scatter kernel its largest shared-memory footprint (once per device).
int prepare_scatter() {
  static bool done_for[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (!done_for[dev & 63]) {
    const cudaError_t e = cudaFuncSetAttribute(
        wqe_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
        (int)scatter_smem(kMaxRings + 1));
    if (e != cudaSuccess) return cuda_failure(e);
    done_for[dev & 63] = true;
  }
  return 0;
}

}  // namespace wqe
}  // namespace db

using namespace db;

extern "C" int db_wqe_workspace_size(uint64_t n, uint32_t n_rings, size_t* bytes) {
  if (!bytes || n_rings == 0 || n_rings > wqe::kMaxRings || n >= (1ull << 32)) return -EINVAL;
  *bytes = wqe::ws_bytes_for(n, n_rings);
  return 0;
}

extern "C" int db_wqe_bucket(const db_put_req* req, uint64_t n, const uint64_t* peer_ptrs,
                             const uint32_t* rkeys, uint32_t world, uint32_t n_qp,
                             uint64_t local_base, uint32_t lkey, uint64_t heap_size,
                             db_wqe* rings, uint64_t depth, uint64_t* head, uint32_t* count,
                             db_counters* ctr, void* ws, size_t ws_bytes, void* stream) {
  cudaStream_t s = (cudaStream_t)stream;
  if (world == 0 || n_qp == 0 || (uint64_t)world * n_qp > wqe::kMaxRings) return -EINVAL;
  if (depth == 0 || (depth & (depth - 1)) != 0) return -EINVAL;
  if (n >= (1ull << 32)) return -EINVAL;
  const uint32_t R = world * n_qp;
  if (!count || !aligned(count, 4)) return -EINVAL;
  if (ctr && !aligned(ctr, 8)) return -EINVAL;
  if (n == 0) {
    cudaMemsetAsync(count, 0, (size_t)R * 4, s);
    if (ctr) cudaMemsetAsync(ctr, 0, sizeof(db_counters), s);
    return launch_result();
  }
  if (!req || !peer_ptrs || !rkeys || !rings || !head || !ws) return -EINVAL;
  if (!aligned(req, 16) || !aligned(peer_ptrs, 8) || !aligned(rkeys, 4) || !aligned(rings, 64) ||
      !aligned(head, 8) || !aligned(ws, 256))
    return -EINVAL;
  const uint64_t n_tiles = wqe::tiles_for(n);
  if (ws_bytes < wqe::ws_bytes_for(n, R)) return -ENOSPC;

  char* w = static_cast<char*>(ws);
  wqe::Params p;
  p.req = reinterpret_cast<const ulonglong2*>(req);
  p.n = n;
  p.n_tiles = n_tiles;
  p.peer_ptrs = peer_ptrs;
  p.rkeys = rkeys;
  p.world = world;
  p.n_qp = n_qp;
  p.R = R;
  p.V = R + 1;
  p.local_base = local_base;
  p.lkey = lkey;
  p.heap_size = heap_size;
  p.rings = reinterpret_cast<unsigned char*>(rings);
  p.depth = depth;
  p.head = head;
  p.count = count;
  p.ctr = ctr;
  p.hdr = reinterpret_cast<wqe::Header*>(w);
  p.head_old = reinterpret_cast<uint64_t*>(w + wqe::kHeadOldOff);
  p.full = reinterpret_cast<uint32_t*>(w + wqe::kFullOff);
  p.counts = reinterpret_cast<uint32_t*>(w + wqe::kCountsOff);

  int rc = wqe::prepare_scatter();
  if (rc) return rc;
  uint64_t count_grid = (uint64_t)num_sms() * 8;
  const uint64_t count_need = (n_tiles + wqe::kCountWarps - 1) / wqe::kCountWarps;
  if (count_grid > count_need) count_grid = count_need;
  wqe::wqe_count_kernel<<<(unsigned)count_grid, wqe::kCountThreads,
                          (size_t)wqe::kCountWarps * p.V * 4, s>>>(p);
  rc = launch_result();
  if (rc) return rc;
  wqe::wqe_scan_kernel<<<p.V, wqe::kScanThreads, 0, s>>>(p);
  rc = launch_result();
  if (rc) return rc;
  uint64_t scatter_grid = n_tiles;
  if (DB_WQE_SCATTER_PERSIST && scatter_grid > (uint64_t)num_sms() * 3)
    scatter_grid = (uint64_t)num_sms() * 3;
  wqe::wqe_scatter_kernel<<<(unsigned)scatter_grid, wqe::kThreads, wqe::scatter_smem(p.V), s>>>(p);
  return launch_result();
}
