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
// reduce-then-scan over tiles of 256 puts (8 rows of 32):
//   count    a warp per tile: a warp-private shared-memory histogram over
//            the R rings plus one bin for invalid puts, written column-major:
//            counts[ring][tile].
//   scan     one CTA per ring: exclusive scan of its column in place (each
//            warp a contiguous span), the ring's batch total, count[], the
//            overflow decision, the head; the last CTA publishes the counters.
//   scatter  a warp per tile, with no CTA-wide barrier: the tile's puts go to
//            warp-private shared memory; stable rank of each put inside its
//            row with __match_any_sync and across the 8 rows by a per-ring
//            prefix; a 2-byte permutation puts the tile in ring order, and
//            each ring's run is written out contiguously, a lane writing a
//            WQE's two 32-byte halves.
// No kernel waits on another CTA.
#include "common.cuh"

namespace db {
namespace wqe {

constexpr int kRows = 8;
constexpr int kTile = kRows * 32;  // 256 puts per tile, one warp each
constexpr uint32_t kMaxRings = 1024;
// Warps per scatter CTA (build-time tunable; fewer when many rings make a
// warp's shared memory large).
#ifndef DB_WQE_SCATTER_WARPS
#define DB_WQE_SCATTER_WARPS 4
#endif
constexpr int kSWarps = DB_WQE_SCATTER_WARPS;
constexpr size_t kMaxSmem = 227 * 1024;  // opt-in shared memory per CTA

// Build-time tuning (defaults measured best on GB300): how the count pass
// histograms a row of 32 puts (0: __match_any_sync + one shared atomic per
// distinct ring, 1: one shared atomic per put).
#ifndef DB_WQE_COUNT_MODE
#define DB_WQE_COUNT_MODE 1
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
constexpr size_t kPsnOldOff = kFullOff + 4 * kMaxRings;  // PSN heads before the call
constexpr size_t kPsnTotOff = kPsnOldOff + 8 * kMaxRings;  // PSNs each ring was asked for
constexpr size_t kCountsOff = kPsnTotOff + 8 * kMaxRings;
inline uint64_t tiles_for(uint64_t n) { return (n + kTile - 1) / kTile; }
// Column stride of counts: tiles rounded up to 8 (32-byte aligned columns).
inline uint64_t stride_for(uint64_t n) { return (tiles_for(n) + 7) & ~7ull; }
inline size_t column_bytes(uint64_t n, uint32_t R) {
  return (stride_for(n) * ((uint64_t)R + 1) * 4 + 255) & ~(uint64_t)255;
}
// WQE counts, then PSN counts (used when PSNs are asked for).
inline size_t ws_bytes_for(uint64_t n, uint32_t R) {
  return kCountsOff + 2 * column_bytes(n, R);
}
// A VMM heap's chunk tables, packed after the columns: one 16-byte record
// {remote address, rkey | lkey << 32} per (PE, chunk).
inline size_t vmm_table_off(uint64_t n, uint32_t R) { return (ws_bytes_for(n, R) + 255) & ~(size_t)255; }
inline size_t vmm_ws_bytes_for(uint64_t n, uint32_t R, uint32_t world, uint64_t n_chunks) {
  return vmm_table_off(n, R) + (size_t)world * n_chunks * 16;
}

struct Params {
  const ulonglong2* req;
  uint64_t n;
  uint64_t n_tiles;
  uint64_t stride;  // column stride of counts
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
  uint32_t* counts;  // [V][stride], first n_tiles of each column used
  // VMM heap: chunks of 2^cshift bytes; a put makes one WQE per chunk.
  bool vmm;
  uint32_t cshift;
  uint64_t n_chunks;
  const uint64_t* chunk_raddr;  // [world][n_chunks]
  const uint32_t* chunk_rkey;   // [world][n_chunks]
  const uint32_t* chunk_lkey;   // [n_chunks]
  ulonglong2* chunk_pack;       // [world][n_chunks]: the three, one record each
  // Packet sequence numbers (mtu != 0): one column of per-tile PSN counts
  // per bin, the PSN heads before the call and each ring's PSN total.
  uint32_t mtu;
  uint64_t mtu_magic;      // ceil(2^64 / mtu): floor(x / mtu) of a 32-bit x by one multiply
  uint64_t psn_per_chunk;  // ceil(chunk bytes / mtu)
  uint64_t* psn_head;
  uint32_t* psn_counts;  // [V][stride]
  uint64_t* psn_old;
  uint64_t* psn_tot;
  // Transport per PE (db_wqe_bucket_transport): bin R + 1 collects the puts
  // to P2P and SDMA PEs, which become direct descriptors in batch order.
  const uint8_t* transport;  // [world]
  unsigned char* direct;     // [n] 32-byte descriptors
  uint64_t* n_direct;
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

// With a transport table: an RDMA put keeps its ring, a P2P or SDMA put goes
// to the direct bin R + 1, and a PE with any other code makes its puts
// invalid (bin R).
template <bool kXport>
__device__ __forceinline__ uint32_t bin_for(const Params& p, const ulonglong2 r) {
  const uint32_t b = bin_of(p, r);
  if (!kXport || b >= p.R) return b;
  const uint32_t t = __ldg(p.transport + ((uint32_t)(r.y >> 32) & 0xFFFFu));
  return t == 0 ? b : (t <= 2 ? p.R + 1 : p.R);
}

// WQEs a valid put makes: one, or on a VMM heap one per chunk it touches.
__device__ __forceinline__ uint32_t wqes_of(const Params& p, const ulonglong2 r) {
  if (!p.vmm) return 1;
  const uint64_t off = r.x, last = r.x + (uint32_t)r.y - 1;
  return (uint32_t)((last >> p.cshift) - (off >> p.cshift)) + 1;
}

// ceil(x / mtu) for a 32-bit x: the quotient is the high half of the 96-bit
// product x * ceil(2^64 / mtu), exact for every 32-bit x and divisor
// (Lemire, Kaser and Kurz, "Faster remainder by direct computation", 2019),
// then one up unless the remainder is zero. Every length divided here is at
// most a put's byte count, so it fits in 32 bits.
__device__ __forceinline__ uint32_t ceil_mtu(const Params& p, uint32_t x) {
  const uint32_t q = (uint32_t)__umul64hi(p.mtu_magic, (uint64_t)x);
  return q + (x != q * p.mtu ? 1u : 0u);
}
// PSNs a valid put's WQEs use: ceil(len / mtu) per WQE, summed over its
// chunks (a first partial chunk, full chunks, a last partial one; the two
// partial ones are shorter than the put).
__device__ __forceinline__ uint32_t psns_of(const Params& p, const ulonglong2 r) {
  const uint64_t off = r.x;
  const uint32_t bytes = (uint32_t)r.y;
  const uint32_t k = wqes_of(p, r);
  if (k == 1) return ceil_mtu(p, bytes);
  const uint64_t C = 1ull << p.cshift;
  const uint32_t first = (uint32_t)(C - (off & (C - 1)));
  const uint32_t last = (uint32_t)(((off + bytes - 1) & (C - 1)) + 1);
  return (uint32_t)(ceil_mtu(p, first) + (uint64_t)(k - 2) * p.psn_per_chunk + ceil_mtu(p, last));
}
// PSNs of the fragments before fragment f of a put (f >= 1: the put crosses
// its first chunk's end, so that chunk's part is shorter than the put).
__device__ __forceinline__ uint32_t psns_before(const Params& p, uint64_t off, uint32_t f) {
  if (f == 0) return 0;
  const uint64_t C = 1ull << p.cshift;
  const uint32_t first = (uint32_t)(C - (off & (C - 1)));
  return (uint32_t)(ceil_mtu(p, first) + (uint64_t)(f - 1) * p.psn_per_chunk);
}

// ---------------------------------------------------------------- count pass
// One warp counts a whole tile (8 rows of 32 puts) into its own shared
// histogram; warps stride over tiles, so no block-wide barrier is needed.
constexpr int kCountThreads = 256;
constexpr int kCountWarps = kCountThreads / 32;
// 1: the scan and scatter passes are launched as programmatic dependents of
// the pass before them: their CTAs start while that pass finishes, and the
// scatter loads its tile of puts (the caller's input) before it waits.
#ifndef DB_WQE_PDL
#define DB_WQE_PDL 1
#endif
#ifndef DB_WQE_COUNT_UNROLL
#define DB_WQE_COUNT_UNROLL 8
#endif
constexpr int kCountUnroll = DB_WQE_COUNT_UNROLL;  // rows of 32 puts loaded at once

// kVmm / kPsn: the call's heap kind and whether PSNs are counted, fixed at
// compile time so that the common static-heap pass carries no per-put tests.
template <bool kVmm, bool kPsn, bool kXport = false>
__global__ void __launch_bounds__(kCountThreads) wqe_count_kernel(const Params p) {
  extern __shared__ uint32_t s_hist_all[];  // [kCountWarps][V] WQEs, then PSNs if asked
  if (DB_WQE_PDL) {
    wait_for_prerequisites();  // a dependent of the chunk-record pack on a VMM heap
    dependents_may_launch();
  }
  const uint32_t V = p.V;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t* s_hist = s_hist_all + (size_t)warp * V;
  uint32_t* s_psn = s_hist_all + (size_t)(kCountWarps + warp) * V;
  const uint64_t pol_first = policy_evict_first();
  const uint64_t n_warps = (uint64_t)gridDim.x * kCountWarps;
  for (uint64_t tile = (uint64_t)blockIdx.x * kCountWarps + warp; tile < p.n_tiles;
       tile += n_warps) {
    for (uint32_t v = lane; v < V; v += 32) {
      s_hist[v] = 0;
      if (kPsn) s_psn[v] = 0;
    }
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
        const uint32_t bin = i < p.n ? bin_for<kXport>(p, r[u]) : V;
        if (kPsn && bin < p.R) atomicAdd(&s_psn[bin], psns_of(p, r[u]));
        if (DB_WQE_COUNT_MODE == 1) {
          if (bin < p.R) atomicAdd(&s_hist[bin], kVmm ? wqes_of(p, r[u]) : 1u);
          else if (bin < V) atomicAdd(&s_hist[bin], 1u);
        } else {
          const uint32_t peers = __match_any_sync(kFull, bin);
          if (kVmm) {  // weights differ per put
            if (bin < p.R) atomicAdd(&s_hist[bin], wqes_of(p, r[u]));
            else if (bin == p.R) atomicAdd(&s_hist[bin], 1u);
          } else if (bin < V && (peers & lanemask_lt()) == 0) {
            atomicAdd(&s_hist[bin], __popc(peers));
          }
        }
      }
    }
    __syncwarp();
    for (uint32_t v = lane; v < V; v += 32) {
      p.counts[v * p.stride + tile] = s_hist[v];
      if (kPsn) p.psn_counts[v * p.stride + tile] = s_psn[v];
    }
    __syncwarp();
  }
}

// ----------------------------------------------------------------- scan pass
// One CTA per bin column. A round covers 32,768 column entries: warp w takes
// the 1,024 contiguous entries at w * 1,024 and its lane l the four at
// j * 128 + 4 l (j = 0..7), so every load and store of a warp covers 512
// contiguous bytes; a column of up to 32,768 tiles is one round. Sums are
// 64-bit; the prefixes are stored in 32 bits, exact for any ring whose batch
// total fits the ring (depth <= 2^31), which are the only ones written.
constexpr int kScanThreads = 1024;
constexpr int kScanGroups = 8;  // four-entry groups per thread per round
constexpr uint64_t kScanWarpSpan = 32ull * 4 * kScanGroups;
constexpr uint64_t kScanSeg = (uint64_t)(kScanThreads / 32) * kScanWarpSpan;

__global__ void __launch_bounds__(kScanThreads) wqe_scan_kernel(const Params p) {
  constexpr int kW = kScanThreads / 32;
  __shared__ uint64_t s_scan[kW];
  __shared__ int s_last;
  // CTAs 0 .. V-1 scan the WQE columns, V .. 2V-1 (when PSNs are asked for)
  // the PSN columns.
  if (DB_WQE_PDL) {
    dependents_may_launch();
    wait_for_prerequisites();  // the count pass's columns
  }
  const bool psn_col = blockIdx.x >= p.V;
  const uint32_t v = psn_col ? blockIdx.x - p.V : blockIdx.x;
  uint32_t* col = (psn_col ? p.psn_counts : p.counts) + (uint64_t)v * p.stride;
  const uint64_t T = p.n_tiles;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint64_t carry = 0;
  for (uint64_t s0 = 0; s0 < T; s0 += kScanSeg) {
    const uint64_t wb = s0 + (uint64_t)warp * kScanWarpSpan + 4u * lane;
    uint4 c[kScanGroups];
    uint64_t mine = 0;
#pragma unroll
    for (int j = 0; j < kScanGroups; ++j) {
      const uint64_t b = wb + (uint64_t)j * 128;
      uint4 x = make_uint4(0u, 0u, 0u, 0u);
      if (b < T) {  // columns are padded to 8 entries, so b + 4 <= stride
        x = *reinterpret_cast<const uint4*>(col + b);
        if (b + 1 >= T) x.y = 0;
        if (b + 2 >= T) x.z = 0;
        if (b + 3 >= T) x.w = 0;
      }
      c[j] = x;
      mine += (uint64_t)x.x + x.y + x.z + x.w;
    }
    // Lane 0's exclusive prefix (lanes in order) is the total of the warps
    // before this one.
    uint64_t excl, seg_total;
    block_excl_scan64<kW>(mine, excl, seg_total, s_scan);
    uint64_t run = carry + __shfl_sync(kFull, excl, 0);
#pragma unroll
    for (int j = 0; j < kScanGroups; ++j) {
      const uint4 x = c[j];
      const uint64_t g = (uint64_t)x.x + x.y + x.z + x.w;
      uint64_t incl = g;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint64_t y = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += y;
      }
      const uint32_t e0 = (uint32_t)(run + incl - g);
      c[j] = make_uint4(e0, e0 + x.x, e0 + x.x + x.y, e0 + x.x + x.y + x.z);
      run += __shfl_sync(kFull, incl, 31);
    }
#pragma unroll
    for (int j = 0; j < kScanGroups; ++j) {
      const uint64_t b = wb + (uint64_t)j * 128;
      if (b + 4 <= T) {
        *reinterpret_cast<uint4*>(col + b) = c[j];
      } else if (b < T) {
        col[b] = c[j].x;
        if (b + 1 < T) col[b + 1] = c[j].y;
        if (b + 2 < T) col[b + 2] = c[j].z;
      }
    }
    carry += seg_total;
    __syncthreads();  // s_scan is reused by the next round
  }
  const uint64_t total = carry;
  if (threadIdx.x == 0 && psn_col) {
    if (v < p.R) {  // the head moves once the ring's overflow decision is known
      p.psn_old[v] = p.psn_head[v];
      p.psn_tot[v] = total;
    }
    __threadfence();
    s_last = atomicAdd(&p.hdr->done, 1u) == gridDim.x - 1;
  } else if (threadIdx.x == 0) {
    if (v < p.R) {
      const uint64_t h = p.head[v];
      const bool over = total > p.depth;
      p.count[v] = total < 0xFFFFFFFFull ? (uint32_t)total : 0xFFFFFFFFu;
      p.head_old[v] = h;
      p.full[v] = over ? 1u : 0u;
      if (!over) p.head[v] = h + total;
      if (over)
        atomicAdd(&p.hdr->overflow, (unsigned long long)total);
      else if (total)
        atomicAdd(&p.hdr->posted, (unsigned long long)total);
    } else if (v == p.R) {
      if (total) atomicAdd(&p.hdr->invalid, (unsigned long long)total);
    } else {  // the direct bin of a transport call
      *p.n_direct = total;
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
    if (p.mtu)
      for (uint32_t r = 0; r < p.R; ++r)
        if (!*(volatile uint32_t*)&p.full[r])
          p.psn_head[r] = *(volatile uint64_t*)&p.psn_old[r] + *(volatile uint64_t*)&p.psn_tot[r];
    p.hdr->done = 0;
    __threadfence();
  }
}

// -------------------------------------------------------------- scatter pass
// Shared memory of a scatter CTA: per CTA, for each ring its slot array (0
// when the ring overflowed) and for each PE its peer pointer and rkey; per
// warp, the tile's puts, the ring-order permutation, the per-row ring counts
// (then their prefixes over rows), and per ring the tile's first sequence
// number and where its run starts.
__host__ __device__ inline size_t warp_smem(uint32_t V) {
  size_t b = (size_t)kTile * 16;      // puts
  b += (size_t)V * 8;                 // first sequence number per ring
  b += (size_t)V * 4;                 // run start per ring
  b += (size_t)kRows * V * 2;         // per-row counts
  b += (size_t)kTile * 2;             // permutation
  return (b + 15) & ~(size_t)15;
}
__host__ __device__ inline size_t cta_smem(uint32_t V) { return ((size_t)V * 20 + 15) & ~(size_t)15; }
// Warps of a scatter CTA for V bins, and its shared memory.
inline int scatter_warps(uint32_t V) {
  const size_t fit = (kMaxSmem - cta_smem(V)) / warp_smem(V);
  return (int)(fit < (size_t)kSWarps ? fit : (size_t)kSWarps);
}
inline size_t scatter_smem(uint32_t V) { return cta_smem(V) + scatter_warps(V) * warp_smem(V); }

template <bool kXport>
__global__ void __launch_bounds__(kSWarps * 32) wqe_scatter_kernel(const Params p) {
  extern __shared__ __align__(16) unsigned char smem[];
  const uint32_t V = p.V, R = p.R;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint64_t pol_first = policy_evict_first();
  uint64_t* s_slots = reinterpret_cast<uint64_t*>(smem);
  uint64_t* s_peer = s_slots + V;
  uint32_t* s_rkey = reinterpret_cast<uint32_t*>(s_peer + V);
  unsigned char* w = smem + cta_smem(V) + warp * warp_smem(V);
  ulonglong2* s_put = reinterpret_cast<ulonglong2*>(w);
  uint64_t* s_seq0 = reinterpret_cast<uint64_t*>(s_put + kTile);
  uint32_t* s_run = reinterpret_cast<uint32_t*>(s_seq0 + V);
  uint16_t* s_cnt = reinterpret_cast<uint16_t*>(s_run + V);  // [kRows][V]
  uint16_t* s_perm = s_cnt + kRows * V;

  // 1. Load the tile (all rows in flight at once): the puts are the
  //    caller's input, so this comes before the wait for the scan pass.
  const uint64_t tile = (uint64_t)blockIdx.x * (blockDim.x >> 5) + warp;
  const uint64_t t0 = tile * kTile;
  ulonglong2 r[kRows];
#pragma unroll
  for (int u = 0; u < kRows; ++u) {
    const uint64_t i = t0 + (uint64_t)u * 32 + lane;
    r[u] = (tile < p.n_tiles && i < p.n) ? ld_stream16(p.req + i, pol_first)
                                         : make_ulonglong2(0, 0);
  }
  if (DB_WQE_PDL) wait_for_prerequisites();  // slots, heads and prefixes of the scan pass
  for (uint32_t v = threadIdx.x; v < R; v += blockDim.x) {
    s_slots[v] = p.full[v] ? 0ull : (uint64_t)(p.rings + (((uint64_t)v * p.depth) << 6));
    if (v < p.world) {
      s_peer[v] = __ldg(p.peer_ptrs + v);
      s_rkey[v] = __ldg(p.rkeys + v);
    }
  }
  __syncthreads();  // the only CTA-wide barrier
  if (tile >= p.n_tiles) return;

  //    Ring of each put; rank inside its row; per-row counts by the row's
  //    first put of each ring.
  for (uint32_t x = lane; x < kRows * V; x += 32) s_cnt[x] = 0;
  __syncwarp();
  uint32_t bin_rank[kRows];  // ring | rank << 16
#pragma unroll
  for (int u = 0; u < kRows; ++u) {
    const uint64_t i = t0 + (uint64_t)u * 32 + lane;
    const uint32_t bin = i < p.n ? bin_for<kXport>(p, r[u]) : V;  // outside the batch: no bin
    s_put[u * 32 + lane] = r[u];
    const uint32_t peers = __match_any_sync(kFull, bin);
    const uint32_t before = peers & lanemask_lt();
    if (bin < V && before == 0) s_cnt[u * V + bin] = (uint16_t)__popc(peers);
    bin_rank[u] = bin | ((uint32_t)__popc(before) << 16);
  }
  __syncwarp();
  // 2. Per ring: prefix of its counts over the rows, the tile's total, where
  //    its run starts (rings in order, the invalid bin left out) and the
  //    tile's first sequence number (the count pass's scan).
  uint32_t carry = 0;
  for (uint32_t v0 = 0; v0 < R; v0 += 32) {
    const uint32_t v = v0 + lane;
    uint32_t tot = 0;
    if (v < R) {
#pragma unroll
      for (int u = 0; u < kRows; ++u) {
        const uint32_t c = s_cnt[u * V + v];
        s_cnt[u * V + v] = (uint16_t)tot;
        tot += c;
      }
    }
    uint32_t x = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(kFull, x, o);
      if (lane >= o) x += y;
    }
    if (v < R) {
      s_run[v] = carry + x - tot;
      s_seq0[v] = p.head_old[v] + p.counts[(uint64_t)v * p.stride + tile];
    }
    carry += __shfl_sync(kFull, x, 31);
  }
  if (kXport && lane == 0) {  // the direct bin: prefix of its counts over the rows
    uint32_t tot = 0;
#pragma unroll
    for (int u = 0; u < kRows; ++u) {
      const uint32_t c = s_cnt[u * V + R + 1];
      s_cnt[u * V + R + 1] = (uint16_t)tot;
      tot += c;
    }
  }
  __syncwarp();
  if (kXport) {
    // Direct descriptors, in batch order from the tile's first slot (the
    // count pass's scan of the direct bin): one 32-byte store per put.
    const uint64_t d0 = p.counts[(uint64_t)(R + 1) * p.stride + tile];
#pragma unroll
    for (int u = 0; u < kRows; ++u) {
      if ((bin_rank[u] & 0xFFFFu) != R + 1) continue;
      const ulonglong2 x = r[u];
      const uint32_t pe = (uint32_t)(x.y >> 32) & 0xFFFFu;
      const uint64_t at = d0 + s_cnt[u * V + R + 1] + (bin_rank[u] >> 16);
      const uint32_t t = __ldg(p.transport + pe);
      st_stream32(p.direct + (at << 5), s_peer[pe] + x.x, p.local_base + x.x,
                  (uint64_t)(uint32_t)x.y | ((t0 + (uint64_t)u * 32 + lane) << 32),
                  (uint64_t)pe | ((uint64_t)t << 16), pol_first);
    }
  }
  // 3. Ring-order permutation of the valid puts.
#pragma unroll
  for (int u = 0; u < kRows; ++u) {
    const uint32_t bin = bin_rank[u] & 0xFFFFu;
    if (bin < R) s_perm[s_run[bin] + s_cnt[u * V + bin] + (bin_rank[u] >> 16)] = (uint16_t)(u * 32 + lane);
  }
  __syncwarp();
  // 4. Write-out, each ring's run contiguous in its ring (up to one wrap):
  //    lane l writes the WQEs of positions l, l + 32, ..., both halves.
  const uint64_t slot_mask = p.depth - 1;
  for (uint32_t q = lane; q < carry; q += 32) {
    const uint32_t o = s_perm[q];
    const ulonglong2 x = s_put[o];
    const uint32_t pe = (uint32_t)(x.y >> 32) & 0xFFFFu, qp = (uint32_t)(x.y >> 48);
    const uint32_t v = pe * p.n_qp + qp;
    const uint64_t slots = s_slots[v];
    if (!slots) continue;
    const uint64_t seq = s_seq0[v] + (q - s_run[v]);
    unsigned char* d = reinterpret_cast<unsigned char*>(slots + ((seq & slot_mask) << 6));
    st_stream32(d, s_peer[pe] + x.x, p.local_base + x.x,
                (uint64_t)(uint32_t)x.y | ((uint64_t)p.lkey << 32), (uint64_t)s_rkey[pe], pol_first);
    st_stream32(d + 32, seq, t0 + o, 0ull, 0ull, pol_first);
  }
}

// ------------------------------------------------------ scatter, VMM heap
// As wqe_scatter_kernel, but a put makes one WQE per chunk it touches. The
// tile's puts are put in ring order as before (a put-count permutation);
// then an exclusive prefix of WQE counts over that order gives each put's
// first WQE, and the write-out walks the tile's WQEs in that order (each
// ring's WQEs contiguous in its ring), finding a WQE's put by binary search.
// Per warp: puts, per-ring first sequence number, run start in puts and in
// WQEs, per-row ring counts, the permutation and the WQE prefix.
// (With PSNs the two prefix arrays are padded to 16-byte multiples.)
__host__ __device__ inline size_t vmm_warp_smem(uint32_t V, bool psn) {
  size_t b = (size_t)kTile * 16;      // puts
  b += (size_t)V * 8;                 // first sequence number per ring
  b += (size_t)V * 4 * 2;             // run start (puts), run start (WQEs)
  b += (size_t)kRows * V * 2;         // per-row counts
  b += (size_t)kTile * 2;             // permutation
  b += (size_t)(kTile + (psn ? 4 : 1)) * 4;  // WQE prefix over the ring order
  b += (size_t)(kTile + (psn ? 4 : 1)) * 4;  // PSN prefix over the ring order
  b += (size_t)V * 4 * 2;             // first PSN of the tile, PSN run start
  return (b + 15) & ~(size_t)15;
}
inline int vmm_scatter_warps(uint32_t V, bool psn) {
  const size_t fit = (kMaxSmem - cta_smem(V)) / vmm_warp_smem(V, psn);
  return (int)(fit < (size_t)kSWarps ? fit : (size_t)kSWarps);
}
inline size_t vmm_scatter_smem(uint32_t V, bool psn) {
  return cta_smem(V) + vmm_scatter_warps(V, psn) * vmm_warp_smem(V, psn);
}

// The chunk tables packed per call: record (pe, c) = {chunk_raddr[pe][c],
// chunk_rkey[pe][c] | chunk_lkey[c] << 32}, so a WQE reads its chunk's three
// values with one L2 request instead of three.
__global__ void vmm_pack_kernel(const Params p) {
  if (DB_WQE_PDL) dependents_may_launch();
  const uint64_t total = (uint64_t)p.world * p.n_chunks;
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (uint64_t)gridDim.x * blockDim.x) {
    const uint64_t c = i % p.n_chunks;
    p.chunk_pack[i] = make_ulonglong2(p.chunk_raddr[i],
                                      (uint64_t)p.chunk_rkey[i] | ((uint64_t)p.chunk_lkey[c] << 32));
  }
}

// kPsn: the call asks for PSNs (p.mtu != 0), fixed at compile time.
template <bool kPsn>
__global__ void __launch_bounds__(kSWarps * 32) wqe_scatter_vmm_kernel(const Params p) {
  extern __shared__ __align__(16) unsigned char smem[];
  const uint32_t V = p.V, R = p.R;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint64_t pol_first = policy_evict_first();
  const uint64_t pol_last = policy_evict_last();
  uint64_t* s_slots = reinterpret_cast<uint64_t*>(smem);
  unsigned char* w = smem + cta_smem(V) + warp * vmm_warp_smem(V, kPsn);
  ulonglong2* s_put = reinterpret_cast<ulonglong2*>(w);
  uint64_t* s_seq0 = reinterpret_cast<uint64_t*>(s_put + kTile);
  uint32_t* s_run = reinterpret_cast<uint32_t*>(s_seq0 + V);
  uint32_t* s_wrun = s_run + V;
  uint16_t* s_cnt = reinterpret_cast<uint16_t*>(s_wrun + V);  // [kRows][V]
  uint16_t* s_perm = s_cnt + kRows * V;
  uint32_t* s_wstart = reinterpret_cast<uint32_t*>(s_perm + kTile);  // [kTile + 1]
  constexpr uint32_t kPad = kPsn ? 4 : 1;                             // 16-byte multiples
  uint32_t* s_pstart = s_wstart + kTile + kPad;                       // [kTile + 1]
  uint32_t* s_psn0 = s_pstart + kTile + kPad;                         // [V]
  uint32_t* s_prun = s_psn0 + V;                                      // [V]

  // 1. Load the tile (the caller's input: before the wait for the scan pass).
  const uint64_t tile = (uint64_t)blockIdx.x * (blockDim.x >> 5) + warp;
  const uint64_t t0 = tile * kTile;
  ulonglong2 r[kRows];
#pragma unroll
  for (int u = 0; u < kRows; ++u) {
    const uint64_t i = t0 + (uint64_t)u * 32 + lane;
    r[u] = (tile < p.n_tiles && i < p.n) ? ld_stream16(p.req + i, pol_first)
                                         : make_ulonglong2(0, 0);
  }
  if (DB_WQE_PDL) wait_for_prerequisites();  // slots, heads, prefixes and chunk records
  for (uint32_t v = threadIdx.x; v < R; v += blockDim.x)
    s_slots[v] = p.full[v] ? 0ull : (uint64_t)(p.rings + (((uint64_t)v * p.depth) << 6));
  __syncthreads();  // the only CTA-wide barrier
  if (tile >= p.n_tiles) return;

  //    Ring of each put; rank inside its row; per-row counts.
  for (uint32_t x = lane; x < kRows * V; x += 32) s_cnt[x] = 0;
  __syncwarp();
  uint32_t bin_rank[kRows];  // ring | rank << 16
#pragma unroll
  for (int u = 0; u < kRows; ++u) {
    const uint64_t i = t0 + (uint64_t)u * 32 + lane;
    const uint32_t bin = i < p.n ? bin_of(p, r[u]) : V;
    s_put[u * 32 + lane] = r[u];
    const uint32_t peers = __match_any_sync(kFull, bin);
    const uint32_t before = peers & lanemask_lt();
    if (bin < V && before == 0) s_cnt[u * V + bin] = (uint16_t)__popc(peers);
    bin_rank[u] = bin | ((uint32_t)__popc(before) << 16);
  }
  __syncwarp();
  // 2. Per ring: prefix of its put counts over the rows, where its run of
  //    puts starts, and the tile's first sequence number.
  uint32_t carry = 0;
  for (uint32_t v0 = 0; v0 < R; v0 += 32) {
    const uint32_t v = v0 + lane;
    uint32_t tot = 0;
    if (v < R) {
#pragma unroll
      for (int u = 0; u < kRows; ++u) {
        const uint32_t c = s_cnt[u * V + v];
        s_cnt[u * V + v] = (uint16_t)tot;
        tot += c;
      }
    }
    uint32_t x = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(kFull, x, o);
      if (lane >= o) x += y;
    }
    if (v < R) {
      s_run[v] = carry + x - tot;
      s_seq0[v] = p.head_old[v] + p.counts[(uint64_t)v * p.stride + tile];
      if (kPsn) s_psn0[v] = (uint32_t)(p.psn_old[v] + p.psn_counts[(uint64_t)v * p.stride + tile]);
    }
    carry += __shfl_sync(kFull, x, 31);
  }
  const uint32_t n_valid = carry;
  __syncwarp();
  // 3. Ring-order permutation of the valid puts (with PSNs, each put's WQE
  //    and PSN counts are stored at its ring-order position as well).
#pragma unroll
  for (int u = 0; u < kRows; ++u) {
    const uint32_t bin = bin_rank[u] & 0xFFFFu;
    if (bin < R) {
      const uint32_t at = s_run[bin] + s_cnt[u * V + bin] + (bin_rank[u] >> 16);
      s_perm[at] = (uint16_t)(u * 32 + lane);
      if (kPsn) {
        s_wstart[at] = wqes_of(p, r[u]);
        s_pstart[at] = psns_of(p, r[u]);
      }
    }
  }
  __syncwarp();
  // 4. Exclusive prefix of WQE counts over the ring order (lane l takes
  //    positions 8l .. 8l + 7), and where each ring's WQEs start; with PSNs
  //    the same over PSN counts (mod 2^32, as the WQE keeps 32 bits), both in
  //    place from the counts of step 3, two 16-byte words a lane.
  constexpr int kPer = kTile / 32;
  static_assert(kPer == 8, "two 16-byte words per lane");
  uint32_t n_wqe;
  if (kPsn) {
    auto prefix8 = [&](uint32_t* a) {  // returns the total
      uint4* a4 = reinterpret_cast<uint4*>(a + lane * kPer);
      const uint4 u0 = a4[0], u1 = a4[1];
      uint32_t kq[kPer] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
      uint32_t mine = 0;
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        if (lane * kPer + j >= n_valid) kq[j] = 0;
        mine += kq[j];
      }
      uint32_t x = mine;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(kFull, x, o);
        if (lane >= o) x += y;
      }
      uint32_t e[kPer];
      uint32_t run = x - mine;
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        e[j] = run;
        run += kq[j];
      }
      a4[0] = make_uint4(e[0], e[1], e[2], e[3]);
      a4[1] = make_uint4(e[4], e[5], e[6], e[7]);
      return __shfl_sync(kFull, x, 31);
    };
    n_wqe = prefix8(s_wstart);
    prefix8(s_pstart);
  } else {
    uint32_t kq[kPer], mine = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const uint32_t q = lane * kPer + j;
      kq[j] = q < n_valid ? wqes_of(p, s_put[s_perm[q]]) : 0u;
      mine += kq[j];
    }
    uint32_t x = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(kFull, x, o);
      if (lane >= o) x += y;
    }
    uint32_t run = x - mine;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      s_wstart[lane * kPer + j] = run;
      run += kq[j];
    }
    n_wqe = __shfl_sync(kFull, x, 31);
  }
  if (lane == 0) s_wstart[kTile] = n_wqe;
  __syncwarp();
  for (uint32_t v = lane; v < R; v += 32) {
    s_wrun[v] = s_wstart[s_run[v]];
    if (kPsn) s_prun[v] = s_pstart[s_run[v]];
  }
  __syncwarp();
  // 5. Write-out: lane l writes the tile's WQEs l, l + 32, ... (ring order),
  //    both halves; a WQE's put is the last one whose first WQE is at or
  //    before it.
  const uint64_t C = 1ull << p.cshift;
  const uint64_t slot_mask = p.depth - 1;
  const uint32_t extra = n_wqe - n_valid;
  for (uint32_t wq = lane; wq < n_wqe; wq += 32) {
    // Every put makes at least one WQE, so WQE wq belongs to a put in
    // [wq - extra, wq]: search only there.
    uint32_t lo = wq > extra ? wq - extra : 0u;
    uint32_t hi = (wq + 1 < n_valid ? wq + 1 : n_valid);  // s_wstart[lo] <= wq < s_wstart[hi]
    while (hi - lo > 1) {
      const uint32_t mid = (lo + hi) >> 1;
      if (s_wstart[mid] <= wq) lo = mid;
      else hi = mid;
    }
    const uint32_t o = s_perm[lo];
    const uint32_t frag = wq - s_wstart[lo];
    const ulonglong2 pu = s_put[o];
    const uint32_t pe = (uint32_t)(pu.y >> 32) & 0xFFFFu, qp = (uint32_t)(pu.y >> 48);
    const uint32_t v = pe * p.n_qp + qp;
    const uint64_t slots = s_slots[v];
    if (!slots) continue;
    const uint64_t seq = s_seq0[v] + (wq - s_wrun[v]);
    const uint64_t c = (pu.x >> p.cshift) + frag;  // the fragment's chunk
    const uint64_t start = frag == 0 ? pu.x : (c << p.cshift);
    const uint64_t stop = pu.x + (uint32_t)pu.y;
    const uint64_t end = ((c + 1) << p.cshift) < stop ? ((c + 1) << p.cshift) : stop;
    unsigned char* d = reinterpret_cast<unsigned char*>(slots + ((seq & slot_mask) << 6));
    // one 16-byte read for the chunk's remote address, rkey and lkey
    const ulonglong2 ck = ld_table16(p.chunk_pack + (uint64_t)pe * p.n_chunks + c, pol_last);
    st_stream32(d, ck.x + (start & (C - 1)), p.local_base + start,
                (end - start) | (ck.y & 0xFFFFFFFF00000000ull), ck.y & 0xFFFFFFFFull, pol_first);
    // u32 batch index at byte 40, first PSN at byte 44
    uint64_t w5 = t0 + o;
    if (kPsn)
      w5 |= (uint64_t)(s_psn0[v] + (s_pstart[lo] - s_prun[v]) + psns_before(p, pu.x, frag)) << 32;
    st_stream32(d + 32, seq, w5, 0ull, 0ull, pol_first);
  }
}

// Allow the scatter kernel its largest shared-memory footprint (once per device).
int prepare_scatter() {
  static bool done_for[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (!done_for[dev & 63]) {
    cudaError_t e = cudaFuncSetAttribute(
        wqe_scatter_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMaxSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(wqe_scatter_kernel<true>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMaxSmem);
    if (e != cudaSuccess) return cuda_failure(e);
    e = cudaFuncSetAttribute(wqe_scatter_vmm_kernel<false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMaxSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(wqe_scatter_vmm_kernel<true>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMaxSmem);
    if (e != cudaSuccess) return cuda_failure(e);
    // Two histograms (WQEs and PSNs) of up to 1025 bins per warp.
    const int count_smem = (int)((size_t)kCountWarps * (kMaxRings + 1) * 4 * 2);
    e = cudaFuncSetAttribute(wqe_count_kernel<false, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, count_smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(wqe_count_kernel<true, false>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, count_smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(wqe_count_kernel<true, true>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, count_smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(wqe_count_kernel<false, false, true>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, count_smem);
    if (e != cudaSuccess) return cuda_failure(e);
    done_for[dev & 63] = true;
  }
  return 0;
}

}  // namespace wqe
}  // namespace db

using namespace db;

extern "C" int db_wqe_vmm_workspace_size(uint64_t n, uint32_t world, uint32_t n_qp,
                                         uint64_t heap_size, uint32_t chunk_shift,
                                         size_t* bytes) {
  if (!bytes || world == 0 || n_qp == 0 || (uint64_t)world * n_qp > wqe::kMaxRings) return -EINVAL;
  if (chunk_shift < 4 || chunk_shift > 48 || heap_size == 0 || n >= (1ull << 32)) return -EINVAL;
  const uint64_t n_chunks = ((heap_size - 1) >> chunk_shift) + 1;
  if (n_chunks > (1ull << 32)) return -EINVAL;
  *bytes = wqe::vmm_ws_bytes_for(n, world * n_qp, world, n_chunks);
  return 0;
}

extern "C" int db_wqe_workspace_size(uint64_t n, uint32_t n_rings, size_t* bytes) {
  if (!bytes || n_rings == 0 || n_rings > wqe::kMaxRings || n >= (1ull << 32)) return -EINVAL;
  *bytes = wqe::ws_bytes_for(n, n_rings);
  return 0;
}

namespace {

// Checks shared by both entry points; fills the common Params fields.
// Returns 0, a negative errno, or 1 for an empty batch already handled.
int setup(wqe::Params& p, const db_put_req* req, uint64_t n, uint32_t world, uint32_t n_qp,
          uint64_t local_base, uint64_t heap_size, db_wqe* rings, uint64_t depth,
          uint64_t* head, uint32_t* count, db_counters* ctr, void* ws, size_t ws_bytes,
          cudaStream_t s) {
  if (world == 0 || n_qp == 0 || (uint64_t)world * n_qp > wqe::kMaxRings) return -EINVAL;
  if (depth == 0 || (depth & (depth - 1)) != 0) return -EINVAL;
  if (n >= (1ull << 32)) return -EINVAL;
  const uint32_t R = world * n_qp;
  if (!count || !aligned(count, 4)) return -EINVAL;
  if (ctr && !aligned(ctr, 8)) return -EINVAL;
  if (n == 0) {
    cudaMemsetAsync(count, 0, (size_t)R * 4, s);
    if (ctr) cudaMemsetAsync(ctr, 0, sizeof(db_counters), s);
    const int rc = launch_result();
    return rc ? rc : 1;
  }
  if (!req || !rings || !head || !ws) return -EINVAL;
  if (!aligned(req, 16) || !aligned(rings, 64) || !aligned(head, 8) || !aligned(ws, 256))
    return -EINVAL;
  if (ws_bytes < wqe::ws_bytes_for(n, R)) return -ENOSPC;
  char* w = static_cast<char*>(ws);
  p.req = reinterpret_cast<const ulonglong2*>(req);
  p.n = n;
  p.n_tiles = wqe::tiles_for(n);
  p.stride = wqe::stride_for(n);
  p.world = world;
  p.n_qp = n_qp;
  p.R = R;
  p.V = R + 1;
  p.local_base = local_base;
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
  p.psn_counts = reinterpret_cast<uint32_t*>(w + wqe::kCountsOff + wqe::column_bytes(n, R));
  p.psn_old = reinterpret_cast<uint64_t*>(w + wqe::kPsnOldOff);
  p.psn_tot = reinterpret_cast<uint64_t*>(w + wqe::kPsnTotOff);
  return 0;
}

// Count, scan, scatter.
int run(const wqe::Params& p, cudaStream_t s) {
  int rc = wqe::prepare_scatter();
  if (rc) return rc;
  if (p.vmm) {
    const uint64_t total = (uint64_t)p.world * p.n_chunks;
    uint64_t g = (total + 255) / 256;
    const uint64_t cap = (uint64_t)num_sms() * 8;
    if (g > cap) g = cap;
    wqe::vmm_pack_kernel<<<(unsigned)g, 256, 0, s>>>(p);
    if ((rc = launch_result())) return rc;
  }
  uint64_t count_grid = (uint64_t)num_sms() * 8;
  const uint64_t count_need = (p.n_tiles + wqe::kCountWarps - 1) / wqe::kCountWarps;
  if (count_grid > count_need) count_grid = count_need;
  {
    const size_t count_smem = (size_t)wqe::kCountWarps * p.V * 4 * (p.mtu ? 2 : 1);
    if (!p.vmm && p.transport) {
      wqe::wqe_count_kernel<false, false, true><<<(unsigned)count_grid, wqe::kCountThreads, count_smem, s>>>(p);
      rc = launch_result();
    } else if (!p.vmm) {
      wqe::wqe_count_kernel<false, false><<<(unsigned)count_grid, wqe::kCountThreads, count_smem, s>>>(p);
      rc = launch_result();
    } else {
      void (*count)(const wqe::Params) = p.mtu ? wqe::wqe_count_kernel<true, true>
                                               : wqe::wqe_count_kernel<true, false>;
      if (DB_WQE_PDL) {  // after the pack kernel just launched on `s`
        rc = launch_dependent(count, (unsigned)count_grid, wqe::kCountThreads, count_smem, s, p);
      } else {
        count<<<(unsigned)count_grid, wqe::kCountThreads, count_smem, s>>>(p);
        rc = launch_result();
      }
    }
  }
  if (rc) return rc;
  const unsigned scan_grid = p.V * (p.mtu ? 2 : 1);
  if (DB_WQE_PDL) {
    rc = launch_dependent(wqe::wqe_scan_kernel, scan_grid, wqe::kScanThreads, 0, s, p);
  } else {
    wqe::wqe_scan_kernel<<<scan_grid, wqe::kScanThreads, 0, s>>>(p);
    rc = launch_result();
  }
  if (rc) return rc;
  void (*scatter)(const wqe::Params) =
      p.vmm ? (p.mtu ? wqe::wqe_scatter_vmm_kernel<true> : wqe::wqe_scatter_vmm_kernel<false>)
            : p.transport ? wqe::wqe_scatter_kernel<true>
                          : wqe::wqe_scatter_kernel<false>;
  const int sw = p.vmm ? wqe::vmm_scatter_warps(p.V, p.mtu != 0)
                       : wqe::scatter_warps(p.V);  // kSWarps, fewer when many rings
  const size_t smem = p.vmm ? wqe::vmm_scatter_smem(p.V, p.mtu != 0) : wqe::scatter_smem(p.V);
  const unsigned grid = (unsigned)((p.n_tiles + sw - 1) / sw);
  if (DB_WQE_PDL) return launch_dependent(scatter, grid, sw * 32, smem, s, p);
  scatter<<<grid, sw * 32, smem, s>>>(p);
  return launch_result();
}

}  // namespace

extern "C" int db_wqe_bucket(const db_put_req* req, uint64_t n, const uint64_t* peer_ptrs,
                             const uint32_t* rkeys, uint32_t world, uint32_t n_qp,
                             uint64_t local_base, uint32_t lkey, uint64_t heap_size,
                             db_wqe* rings, uint64_t depth, uint64_t* head, uint32_t* count,
                             db_counters* ctr, void* ws, size_t ws_bytes, void* stream) {
  cudaStream_t s = (cudaStream_t)stream;
  wqe::Params p{};
  const int rc = setup(p, req, n, world, n_qp, local_base, heap_size, rings, depth, head, count,
                       ctr, ws, ws_bytes, s);
  if (rc) return rc < 0 ? rc : 0;
  if (!peer_ptrs || !rkeys || !aligned(peer_ptrs, 8) || !aligned(rkeys, 4)) return -EINVAL;
  p.peer_ptrs = peer_ptrs;
  p.rkeys = rkeys;
  p.lkey = lkey;
  p.vmm = false;
  return run(p, s);
}

extern "C" int db_wqe_bucket_transport(const db_put_req* req, uint64_t n,
                                       const uint64_t* peer_ptrs, const uint32_t* rkeys,
                                       const uint8_t* transport, uint32_t world, uint32_t n_qp,
                                       uint64_t local_base, uint32_t lkey, uint64_t heap_size,
                                       db_wqe* rings, uint64_t depth, uint64_t* head,
                                       uint32_t* count, db_direct* direct, uint64_t* n_direct,
                                       db_counters* ctr, void* ws, size_t ws_bytes,
                                       void* stream) {
  cudaStream_t s = (cudaStream_t)stream;
  if (!n_direct || !aligned(n_direct, 8)) return -EINVAL;
  wqe::Params p{};
  const int rc = setup(p, req, n, world, n_qp, local_base, heap_size, rings, depth, head, count,
                       ctr, ws, ws_bytes, s);
  if (rc == 1) {  // empty batch: counts and counters already zeroed
    cudaMemsetAsync(n_direct, 0, 8, s);
    return launch_result();
  }
  if (rc) return rc;
  if (!peer_ptrs || !rkeys || !transport || !direct) return -EINVAL;
  if (!aligned(peer_ptrs, 8) || !aligned(rkeys, 4) || !aligned(direct, 32)) return -EINVAL;
  p.peer_ptrs = peer_ptrs;
  p.rkeys = rkeys;
  p.lkey = lkey;
  p.vmm = false;
  p.transport = transport;
  p.direct = reinterpret_cast<unsigned char*>(direct);
  p.n_direct = n_direct;
  p.V = p.R + 2;  // rings, invalid, direct
  return run(p, s);
}

extern "C" int db_wqe_bucket_vmm(const db_put_req* req, uint64_t n, const uint64_t* chunk_raddr,
                                 const uint32_t* chunk_rkey, const uint32_t* chunk_lkey,
                                 uint32_t chunk_shift, uint32_t world, uint32_t n_qp,
                                 uint64_t local_base, uint64_t heap_size, db_wqe* rings,
                                 uint64_t depth, uint64_t* head, uint32_t* count, uint32_t mtu,
                                 uint64_t* psn_head, db_counters* ctr, void* ws, size_t ws_bytes,
                                 void* stream) {
  cudaStream_t s = (cudaStream_t)stream;
  if (chunk_shift < 4 || chunk_shift > 48) return -EINVAL;
  if (mtu != 0 && (mtu < 512 || mtu > (1u << 20) || chunk_shift < 12 || !psn_head ||
                   !aligned(psn_head, 8)))
    return -EINVAL;
  if (heap_size == 0) return -EINVAL;
  if (depth > (1ull << 31)) return -EINVAL;
  const uint64_t n_chunks = ((heap_size - 1) >> chunk_shift) + 1;
  if (n_chunks > (1ull << 32)) return -EINVAL;
  wqe::Params p{};
  const int rc = setup(p, req, n, world, n_qp, local_base, heap_size, rings, depth, head, count,
                       ctr, ws, ws_bytes, s);
  if (rc) return rc < 0 ? rc : 0;
  if (!chunk_raddr || !chunk_rkey || !chunk_lkey || !aligned(chunk_raddr, 8) ||
      !aligned(chunk_rkey, 4) || !aligned(chunk_lkey, 4))
    return -EINVAL;
  if (ws_bytes < wqe::vmm_ws_bytes_for(n, world * n_qp, world, n_chunks)) return -ENOSPC;
  p.chunk_pack = reinterpret_cast<ulonglong2*>(static_cast<char*>(ws) +
                                               wqe::vmm_table_off(n, world * n_qp));
  p.vmm = true;
  p.mtu = mtu;
  if (mtu) {
    p.mtu_magic = ~0ull / mtu + 1;
    p.psn_per_chunk = ((1ull << chunk_shift) + mtu - 1) / mtu;
  }
  p.psn_head = psn_head;
  p.cshift = chunk_shift;
  p.n_chunks = n_chunks;
  p.chunk_raddr = chunk_raddr;
  p.chunk_rkey = chunk_rkey;
  p.chunk_lkey = chunk_lkey;
  return run(p, s);
}
