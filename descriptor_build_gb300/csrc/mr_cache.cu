// Registration-cache mutation batches (sm_103a).
//
// Sources: "NCCL expert course 26: GPUDirect RDMA, DMA-BUF, MR and the
// registration cache" -- "IB Backend MR Cache" (a containing MR is reused
// and takes a reference; partial overlap registers anew; deregistration
// drops a reference and removes the MR at zero; an unknown handle is an
// error), "Communicator User Registration Cache" (insert in address order),
// the ncclCommRegister experiment; xNVMe "uPCIe CUDA" backend page
// (xnvme_buf_register: whole 64 KiB device pages, refcounted).
//
// Registration, all on the caller's stream, no host round trip, gives the
// result of the batch's requests made one at a time in batch order:
//   1. the MR lookup (overlap path, 4 KiB or 64 KiB granules) classifies
//      every request against the table before the batch;
//   2. the misses are flagged, one bit each in flag words, and compacted by
//      an exclusive scan of the words' set bits;
//   3. a stable LSD radix sort (8-bit digits, reduce-then-scan over
//      4,096-key tiles, in-tile ranks from __match_any_sync) orders them by
//      widened start ascending, then end descending, so equal ranges are
//      adjacent and in request order: one sort on the start granule and the
//      length in granules packed in one key, or, when a miss's start or
//      length does not fit that key, a sort on the end and then a stable
//      one on the start;
//   4. a distinct range makes a new record unless a range before it in that
//      order that reaches its end (one that holds it) was asked for earlier:
//      a dominance pass (a merge sort on the end carrying prefix minima of
//      the first request) gives each range the earliest request among the
//      ranges that hold it;
//   5. the new records are numbered in table order; a second dominance pass
//      gives every request the lowest-positioned record holding it when it
//      is made (an old one, or a new one made before it);
//   6. each record is written to the merged table by the pass that finds
//      its place there (old records keep their references; new ones start
//      at none); one pass then gives every request its kind and handle and
//      adds its reference to that record.
// Deregistration counts each record's handles; only a record whose last
// reference the batch reaches needs its handles' batch order, found in a
// bucket of its own (no sort); survivors are compacted by a scan.
#include <cerrno>

#include "common.cuh"
#include "mr_internal.h"
#include "mrcache.h"

namespace db {

// Every kernel of a registration or deregistration batch is launched as a
// programmatic dependent of the one before it (launch_dep): it starts by
// waiting for that kernel (and so for the whole stream before it), then lets
// the next kernel's CTAs be scheduled while it runs.
__device__ __forceinline__ void kernel_prologue() {
  wait_for_prerequisites();
  dependents_may_launch();
}
namespace mrc {

constexpr int kScanThreads = 1024;
constexpr int kScanItems = 8;
constexpr uint64_t kScanChunk = (uint64_t)kScanThreads * kScanItems;
constexpr int kSortThreads = 256;
constexpr int kSortItems = 16;
constexpr uint64_t kSortTile = (uint64_t)kSortThreads * kSortItems;
constexpr int kThreads = 256;
constexpr uint64_t kMaxItems = 1ull << 31;

inline size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }
inline uint64_t ceil_div(uint64_t a, uint64_t b) { return (a + b - 1) / b; }
inline unsigned grid_for(uint64_t n) {
  uint64_t g = ceil_div(n, kThreads);
  const uint64_t cap = (uint64_t)num_sms() * 16;
  if (g > cap) g = cap;
  return (unsigned)(g ? g : 1);
}
#define FOR_EACH(i, n) \
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < (n); i += (uint64_t)gridDim.x * blockDim.x)

// ------------------------------------------------------------------ scan
// Exclusive scan of n u32 values: block sums, then each block re-scans with
// its offset, the sum of the earlier blocks' sums -- summed by the block
// itself when there are at most kScanFusedBlocks blocks, else found first by
// a one-CTA scan of the block sums. n is known on the host,
// or (Len::dev) worked out on the device as mul * ceil(*dev / div), at most
// the host's n: the count columns of a sort cover only the tiles that hold
// items, and the blocks past them return at once. With Len::diff given the
// length is 0 unless bits [shift, shift + 8) of *diff are set (the counts of
// a sort pass that does not run are not scanned).
struct Len {
  const uint32_t* dev;
  uint32_t mul, div;
  const unsigned long long* diff = nullptr;
  uint32_t shift = 0;
};
__device__ __forceinline__ uint64_t live_len(uint64_t n, const Len& l) {
  if (!l.dev) return n;
  if (l.diff && ((*l.diff >> l.shift) & 255u) == 0) return 0;
  const uint64_t m = (uint64_t)l.mul * ((*l.dev + (uint64_t)l.div - 1) / l.div);
  return m < n ? m : n;
}
// Within a block's chunk, warp w takes the kScanItems * 32 items at
// w * kScanItems * 32 and its lane l the four at g * 128 + 4 l for each
// group g, so every load and store of a warp covers 512 contiguous bytes.
constexpr int kScanGroups = kScanItems / 4;
static_assert(kScanItems % 4 == 0, "groups of four items");
// Loads the four items at b (those at or past n read as 0).
__device__ __forceinline__ uint4 scan_load4(const uint32_t* in, uint64_t b, uint64_t n) {
  if (b + 4 <= n) return *reinterpret_cast<const uint4*>(in + b);
  uint4 x = make_uint4(0u, 0u, 0u, 0u);
  if (b < n) x.x = in[b];
  if (b + 1 < n) x.y = in[b + 1];
  if (b + 2 < n) x.z = in[b + 2];
  return x;
}
__device__ __forceinline__ uint64_t scan_group_base(uint32_t g) {
  return (uint64_t)blockIdx.x * kScanChunk + (uint64_t)(threadIdx.x >> 5) * (kScanItems * 32) +
         (uint64_t)g * 128 + 4u * (threadIdx.x & 31);
}
// kPopc: the values are the set bits of each word (a scan of flag words).
__device__ __forceinline__ uint4 popc4(uint4 x) {
  return make_uint4(__popc(x.x), __popc(x.y), __popc(x.z), __popc(x.w));
}
template <bool kPopc>
__global__ void __launch_bounds__(kScanThreads) scan_reduce(const uint32_t* in, uint64_t n_max,
                                                            Len len, uint32_t* bsum) {
  kernel_prologue();
  __shared__ uint32_t s_w[32];
  const uint64_t n = live_len(n_max, len);
  if ((uint64_t)blockIdx.x * kScanChunk >= n && blockIdx.x > 0) return;
  uint32_t v = 0;
#pragma unroll
  for (int g = 0; g < kScanGroups; ++g) {
    uint4 x = scan_load4(in, scan_group_base(g), n);
    if (kPopc) x = popc4(x);
    v += x.x + x.y + x.z + x.w;
  }
  uint32_t ex, tot;
  block_excl_scan<32>(v, ex, tot, s_w);
  if (threadIdx.x == 0) bsum[blockIdx.x] = tot;
}
__global__ void __launch_bounds__(kScanThreads) scan_bsums(uint32_t* bsum, uint64_t n_max,
                                                           Len len, uint32_t* total) {
  kernel_prologue();
  __shared__ uint32_t s_w[32];
  const uint64_t n = live_len(n_max, len);
  const uint64_t nb = n ? (n + kScanChunk - 1) / kScanChunk : 1;
  uint32_t carry = 0;
  for (uint64_t b0 = 0; b0 < nb; b0 += kScanThreads) {
    const uint64_t b = b0 + threadIdx.x;
    const uint32_t v = b < nb ? bsum[b] : 0u;
    uint32_t ex, tot;
    block_excl_scan<32>(v, ex, tot, s_w);
    if (b < nb) bsum[b] = carry + ex;
    carry += tot;
    __syncthreads();  // s_w is written again by the next round
  }
  if (threadIdx.x == 0 && total) *total = carry;
}
// in and out may be the same array: a block reads its whole chunk before
// writing any of it.
// prefixed: bsum holds the blocks' exclusive prefixes (scan_bsums wrote the
// total); else their sums, and the block whose chunk holds item n - 1 (block
// 0 when n is 0) writes the total.
constexpr uint64_t kScanFusedBlocks = 4096;
template <bool kPopc>
__global__ void __launch_bounds__(kScanThreads) scan_apply(const uint32_t* in, uint32_t* out,
                                                           uint64_t n_max, Len len,
                                                           const uint32_t* bsum,
                                                           uint32_t* total, bool prefixed) {
  kernel_prologue();
  __shared__ uint32_t s_w[32];
  __shared__ uint32_t s_before;
  const uint64_t n = live_len(n_max, len);
  if ((uint64_t)blockIdx.x * kScanChunk >= n && blockIdx.x > 0) return;
  const uint32_t lane = threadIdx.x & 31;
  uint4 x[kScanGroups];
  uint32_t v = 0;
#pragma unroll
  for (int g = 0; g < kScanGroups; ++g) {
    x[g] = scan_load4(in, scan_group_base(g), n);
    if (kPopc) x[g] = popc4(x[g]);
    v += x[g].x + x[g].y + x[g].z + x[g].w;
  }
  uint32_t before = 0;  // the earlier blocks' sums
  for (uint32_t b = threadIdx.x; b < blockIdx.x && !prefixed; b += kScanThreads) before += bsum[b];
  before = warp_sum32(before);
  if (lane == 0) s_w[threadIdx.x >> 5] = before;
  __syncthreads();
  if (threadIdx.x < 32) {
    const uint32_t y = warp_sum32(s_w[threadIdx.x]);
    if (threadIdx.x == 0) s_before = y;
  }
  __syncthreads();  // s_w is written again by the scan below
  const uint32_t block0 = prefixed ? bsum[blockIdx.x] : s_before;
  // Lane 0's exclusive prefix (lanes in order) is the total of the warps
  // before this one.
  uint32_t ex, tot;
  block_excl_scan<32>(v, ex, tot, s_w);
  if (!prefixed && total && threadIdx.x == 0 && blockIdx.x == (n ? (n - 1) / kScanChunk : 0))
    *total = block0 + tot;
  uint32_t run = block0 + __shfl_sync(kFull, ex, 0);
#pragma unroll
  for (int g = 0; g < kScanGroups; ++g) {
    const uint32_t gs = x[g].x + x[g].y + x[g].z + x[g].w;
    uint32_t incl = gs;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(kFull, incl, o);
      if (lane >= (uint32_t)o) incl += y;
    }
    const uint32_t e0 = run + incl - gs;
    const uint4 r = make_uint4(e0, e0 + x[g].x, e0 + x[g].x + x[g].y, e0 + x[g].x + x[g].y + x[g].z);
    run += __shfl_sync(kFull, incl, 31);
    const uint64_t b = scan_group_base(g);
    if (b + 4 <= n) {
      *reinterpret_cast<uint4*>(out + b) = r;
    } else if (b < n) {
      out[b] = r.x;
      if (b + 1 < n) out[b + 1] = r.y;
      if (b + 2 < n) out[b + 2] = r.z;
    }
  }
}
inline size_t scan_tmp_words(uint64_t n) { return (size_t)ceil_div(n ? n : 1, kScanChunk); }
template <bool kPopc>
int scan_t(const uint32_t* in, uint32_t* out, uint64_t n, uint32_t* total, uint32_t* bsum,
           cudaStream_t s, Len len) {
  if (n == 0) {
    if (total) cudaMemsetAsync(total, 0, 4, s);
    return launch_result();
  }
  const uint64_t nb = ceil_div(n, kScanChunk);
  launch_dep(scan_reduce<kPopc>, (unsigned)nb, kScanThreads, 0, s, in, n, len, bsum);
  const bool prefixed = nb > kScanFusedBlocks;
  if (prefixed) launch_dep(scan_bsums, 1, kScanThreads, 0, s, bsum, n, len, total);
  launch_dep(scan_apply<kPopc>, (unsigned)nb, kScanThreads, 0, s, in, out, n, len,
             (const uint32_t*)bsum, total, prefixed);
  return launch_result();
}
int scan(const uint32_t* in, uint32_t* out, uint64_t n, uint32_t* total, uint32_t* bsum,
         cudaStream_t s, Len len = Len{nullptr, 0, 1}) {
  return scan_t<false>(in, out, n, total, bsum, s, len);
}

// ------------------------------------------------------------ flag words
// A flag pass writes one bit per item, 32 consecutive items per word (a
// warp's ballot). The scan of the words' set bits gives each word the
// number of flags set before it, so a flagged item's place among them is
// wpos[i / 32] + the bits set below it in its word. Against a u32 flag and
// a u32 place per item this moves a 32nd of the bytes.
__device__ __forceinline__ bool flag_at(const uint32_t* bits, uint64_t i) {
  return (bits[i >> 5] >> (i & 31)) & 1u;
}
__device__ __forceinline__ uint32_t flag_pos(const uint32_t* bits, const uint32_t* wpos,
                                             uint64_t i) {
  return wpos[i >> 5] + __popc(bits[i >> 5] & ((1u << (i & 31)) - 1u));
}
// Steps of 32 consecutive items per warp over [0, n): every lane takes part
// in every step (its item i0 + lane may lie past n), so a step can end in a
// ballot. Block sizes are multiples of 32.
#define FOR_EACH_WARP(i0, n)                                                                 \
  for (uint64_t i0 = (uint64_t)blockIdx.x * blockDim.x + (threadIdx.x & ~31u); i0 < (n); \
       i0 += (uint64_t)gridDim.x * blockDim.x)
__device__ __forceinline__ void put_flags(uint32_t* bits, uint64_t i0, bool f) {
  const uint32_t w = __ballot_sync(kFull, f);
  if ((threadIdx.x & 31) == 0) bits[i0 >> 5] = w;
}
// Scan of the flag words of items [0, n_max), or of the first *n_dev items
// when n_dev is given (the words past them are not read); *total = the
// flags set.
int scan_flags(const uint32_t* bits, uint32_t* wpos, uint64_t n_max, uint32_t* total,
               uint32_t* bsum, cudaStream_t s, const uint32_t* n_dev = nullptr) {
  return scan_t<true>(bits, wpos, ceil_div(n_max, 32), total, bsum, s,
                      n_dev ? Len{n_dev, 1u, 32u} : Len{nullptr, 0, 1});
}

// ------------------------------------------------------------- radix sort
// One stable pass on 8 bits of a u64 key (value u32 alongside), over the
// first *n_dev items of arrays that hold up to n_max. counts is
// [256][tiles], digit-major, so its exclusive scan gives each (digit, tile)
// its first output position.
//
// Passes on a digit that every key shares keep the order, so they are
// skipped: `diff` (the OR of key ^ key[0] over the items, worked out on the
// device before the first pass) says which digits vary. The host launches
// every pass; a skipped one returns at once, and the others find their
// input buffer from the number of passes run before them. A last kernel
// moves the result into the buffer the host expects when the two differ.
__device__ __forceinline__ bool pass_runs(uint64_t diff, uint32_t shift) {
  return ((diff >> shift) & 255u) != 0;
}
__device__ __forceinline__ uint32_t passes_run_below(uint64_t diff, uint32_t shift) {
  uint32_t c = 0;
  for (uint32_t t = 0; t < shift; t += 8) c += pass_runs(diff, t) ? 1u : 0u;
  return c;
}
// One atomic per CTA: the warps' ORs meet in shared memory first. With
// only_if given and *only_if zero no digit is marked, so no pass runs.
__global__ void __launch_bounds__(kThreads) radix_diff(const uint64_t* key, const uint32_t* n_dev,
                                                       const uint32_t* only_if,
                                                       unsigned long long* diff) {
  kernel_prologue();
  __shared__ unsigned long long s_or;
  const uint64_t n = *n_dev;
  if (n == 0 || (only_if && *only_if == 0)) return;
  if (threadIdx.x == 0) s_or = 0;
  __syncthreads();
  const uint64_t k0 = key[0];
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  uint64_t d = 0;
  uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n; i += 4 * stride)
    d |= (key[i] ^ k0) | (key[i + stride] ^ k0) | (key[i + 2 * stride] ^ k0) |
         (key[i + 3 * stride] ^ k0);
  for (; i < n; i += stride) d |= key[i] ^ k0;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) d |= __shfl_xor_sync(kFull, d, o);
  if ((threadIdx.x & 31) == 0 && d) atomicOr(&s_or, (unsigned long long)d);
  __syncthreads();
  if (threadIdx.x == 0 && s_or) atomicOr(diff, s_or);
}
__global__ void __launch_bounds__(kSortThreads) radix_count(const uint64_t* key0,
                                                            const uint64_t* key1, uint32_t cur0,
                                                            const unsigned long long* diff,
                                                            const uint32_t* n_dev, uint32_t shift,
                                                            uint32_t* counts, uint32_t tiles) {
  kernel_prologue();
  __shared__ uint32_t hist[256];
  const uint64_t dv = *diff;
  if (!pass_runs(dv, shift)) return;
  const uint64_t* key = ((cur0 + passes_run_below(dv, shift)) & 1u) ? key1 : key0;
  const uint64_t n = *n_dev;
  const uint64_t t0 = (uint64_t)blockIdx.x * kSortTile;
  if (t0 >= n) return;  // past the items: not a column entry
  tiles = (uint32_t)((n + kSortTile - 1) / kSortTile);  // columns over the live tiles only
  hist[threadIdx.x] = 0;
  __syncthreads();
#pragma unroll 4
  for (int j = 0; j < kSortItems; ++j) {
    const uint64_t i = t0 + (uint64_t)j * kSortThreads + threadIdx.x;
    if (i < n) atomicAdd(&hist[(uint32_t)(key[i] >> shift) & 255u], 1u);
  }
  __syncthreads();
  counts[(uint64_t)threadIdx.x * tiles + blockIdx.x] = hist[threadIdx.x];
}
// A tile's items keep their index order: warp w ranks the 512 items
// t0 + 512w .. t0 + 512w + 511 itself (rounds of 32, rank inside the round
// from __match_any_sync, earlier rounds from a warp-private count), then one
// prefix over the warps gives each item its place in the tile sorted by
// digit. The tile is reordered in shared memory and written out run by run,
// so consecutive threads write consecutive addresses.
constexpr int kSortWarps = kSortThreads / 32;
constexpr int kWarpItems = (int)(kSortTile / kSortWarps);  // 512
constexpr size_t kScatterSmem =
    sizeof(uint32_t) * (kSortWarps * 256 + 256 + 256 + 32) + kSortTile * (8 + 4);
__global__ void __launch_bounds__(kSortThreads, 3) radix_scatter(
    uint64_t* key0, uint64_t* key1, uint32_t* val0, uint32_t* val1, uint32_t cur0,
    const unsigned long long* diff, const uint32_t* n_dev, uint32_t shift, const uint32_t* offs,
    uint32_t tiles) {
  kernel_prologue();
  extern __shared__ __align__(16) unsigned char smem[];
  const uint64_t dv = *diff;
  if (!pass_runs(dv, shift)) return;
  const bool from1 = ((cur0 + passes_run_below(dv, shift)) & 1u) != 0;
  const uint64_t* key = from1 ? key1 : key0;
  const uint32_t* val = from1 ? val1 : val0;
  uint64_t* key_out = from1 ? key0 : key1;
  uint32_t* val_out = from1 ? val0 : val1;
  uint64_t* s_key = reinterpret_cast<uint64_t*>(smem);                     // [kSortTile]
  uint32_t* s_val = reinterpret_cast<uint32_t*>(s_key + kSortTile);        // [kSortTile]
  uint32_t* s_hist = s_val + kSortTile;                                    // [warps][256]
  uint32_t* s_tdig = s_hist + kSortWarps * 256;                            // [256]
  uint32_t* s_goff = s_tdig + 256;                                         // [256]
  uint32_t* s_w = s_goff + 256;                                            // [32]
  const uint64_t n = *n_dev;
  const uint64_t t0 = (uint64_t)blockIdx.x * kSortTile;
  if (t0 >= n) return;  // no items in this tile
  tiles = (uint32_t)((n + kSortTile - 1) / kSortTile);  // columns over the live tiles only
  const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int w = 0; w < kSortWarps; ++w) s_hist[w * 256 + threadIdx.x] = 0;
  s_goff[threadIdx.x] = offs[(uint64_t)threadIdx.x * tiles + blockIdx.x];
  __syncthreads();
  // 1. ranks inside each warp's chunk
  constexpr int kRounds = kWarpItems / 32;
  const uint64_t wbase = t0 + (uint64_t)warp * kWarpItems;
  uint64_t k[kRounds];
  uint32_t v[kRounds], r[kRounds];
#pragma unroll
  for (int j = 0; j < kRounds; ++j) {
    const uint64_t i = wbase + (uint64_t)j * 32 + lane;
    const bool ok = i < n;
    k[j] = ok ? key[i] : 0ull;
    v[j] = ok ? val[i] : 0u;
    const uint32_t d = ok ? ((uint32_t)(k[j] >> shift) & 255u) : 256u + lane;
    const uint32_t peers = __match_any_sync(kFull, d);
    const uint32_t rank = __popc(peers & lanemask_lt());
    const uint32_t before = ok ? s_hist[warp * 256 + d] : 0u;
    r[j] = ok ? before + rank : 0xFFFFFFFFu;
    __syncwarp();
    if (ok && rank == 0) s_hist[warp * 256 + d] = before + __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  // 2. per digit: counts of the earlier warps, and where the digit starts in the tile
  uint32_t run = 0;
#pragma unroll
  for (int w = 0; w < kSortWarps; ++w) {
    const uint32_t c = s_hist[w * 256 + threadIdx.x];
    s_hist[w * 256 + threadIdx.x] = run;
    run += c;
  }
  uint32_t ex, tot;
  block_excl_scan<kSortWarps>(run, ex, tot, s_w);
  s_tdig[threadIdx.x] = ex;
  __syncthreads();
  // 3. reorder the tile by digit in shared memory
#pragma unroll
  for (int j = 0; j < kRounds; ++j) {
    if (r[j] == 0xFFFFFFFFu) continue;
    const uint32_t d = (uint32_t)(k[j] >> shift) & 255u;
    const uint32_t lp = s_tdig[d] + s_hist[warp * 256 + d] + r[j];
    s_key[lp] = k[j];
    s_val[lp] = v[j];
  }
  __syncthreads();
  // 4. write the digit runs out
  const uint64_t cnt = n - t0 < kSortTile ? n - t0 : kSortTile;
  for (uint32_t i = threadIdx.x; i < cnt; i += kSortThreads) {
    const uint64_t kk = s_key[i];
    const uint32_t d = (uint32_t)(kk >> shift) & 255u;
    const uint32_t pos = s_goff[d] + (i - s_tdig[d]);
    key_out[pos] = kk;
    val_out[pos] = s_val[i];
  }
}

// After `passes` launched passes the host expects the result in buffer
// cur0 ^ (passes & 1); it is in cur0 ^ (passes run & 1).
__global__ void __launch_bounds__(kThreads) radix_settle(uint64_t* key0, uint64_t* key1,
                                                         uint32_t* val0, uint32_t* val1,
                                                         uint32_t cur0, uint32_t passes,
                                                         const unsigned long long* diff,
                                                         const uint32_t* n_dev) {
  kernel_prologue();
  const uint32_t ran = passes_run_below(*diff, 8u * passes);
  if (((ran ^ passes) & 1u) == 0) return;
  const bool in1 = ((cur0 + ran) & 1u) != 0;
  const uint64_t* ks = in1 ? key1 : key0;
  const uint32_t* vs = in1 ? val1 : val0;
  uint64_t* kd = in1 ? key0 : key1;
  uint32_t* vd = in1 ? val0 : val1;
  const uint64_t n = *n_dev;
  FOR_EACH(i, n) {
    kd[i] = ks[i];
    vd[i] = vs[i];
  }
}

struct SortBufs {
  uint64_t* key[2];
  uint32_t* val[2];
  uint32_t* counts;           // [256][tiles]
  uint32_t* bsum;             // scan scratch
  uint64_t n_max;
  unsigned long long* diff;   // OR of key ^ key[0] over the items
};
inline uint32_t sort_tiles(uint64_t n_max) { return (uint32_t)ceil_div(n_max ? n_max : 1, kSortTile); }
inline size_t sort_count_words(uint64_t n_max) { return (size_t)256 * sort_tiles(n_max); }
// The scatter's shared memory is above the default 48 KiB: opt in once per device.
int prepare_scatter() {
  static bool done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (!done[dev & 63]) {
    if (cudaFuncSetAttribute(radix_scatter, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kScatterSmem) != cudaSuccess)
      return launch_result();
    done[dev & 63] = true;
  }
  return 0;
}
// Sorts by bits [0, bits) of the key; the result is in buffer `cur` on return.
// skip_shared: look for digits every key shares and skip their passes (a
// sort whose key width is already tight runs every pass without looking).
// only_if (with skip_shared): sort only when *only_if is nonzero on the
// device; otherwise every pass returns at once (the result still lands in
// buffer `cur`).
int radix_sort(SortBufs& b, int& cur, const uint32_t* n_dev, int bits, bool skip_shared,
               cudaStream_t s, const uint32_t* only_if = nullptr) {
  if (int rc = prepare_scatter()) return rc;
  const uint32_t tiles = sort_tiles(b.n_max);
  const uint64_t nc = (uint64_t)256 * tiles;
  const uint32_t cur0 = (uint32_t)cur;
  if (cudaMemsetAsync(b.diff, skip_shared ? 0 : 0xFF, sizeof(*b.diff), s) != cudaSuccess)
    return launch_result();
  int rc = 0;
  if (skip_shared) {
    const unsigned dg = grid_for(b.n_max) < (unsigned)num_sms() * 4 ? grid_for(b.n_max)
                                                                      : (unsigned)num_sms() * 4;
    launch_dep(radix_diff, dg, kThreads, 0, s, b.key[cur0], n_dev, only_if, b.diff);
    if ((rc = launch_result())) return rc;
  }
  uint32_t passes = 0;
  for (int shift = 0; shift < bits; shift += 8, ++passes) {
    launch_dep(radix_count, tiles, kSortThreads, 0, s, b.key[0], b.key[1], cur0, b.diff, n_dev,
               (uint32_t)shift, b.counts, tiles);
    if ((rc = launch_result())) return rc;
    if ((rc = scan(b.counts, b.counts, nc, nullptr, b.bsum, s,
                   Len{n_dev, 256u, (uint32_t)kSortTile, b.diff, (uint32_t)shift})))
      return rc;
    launch_dep(radix_scatter, tiles, kSortThreads, kScatterSmem, s,
               b.key[0], b.key[1], b.val[0], b.val[1],
               cur0, b.diff, n_dev, (uint32_t)shift,
               b.counts, tiles);
    if ((rc = launch_result())) return rc;
    cur ^= 1;
  }
  if (!skip_shared) return 0;
  launch_dep(radix_settle, grid_for(b.n_max), kThreads, 0, s,
             b.key[0], b.key[1], b.val[0], b.val[1], cur0,
             passes, b.diff, n_dev);
  return launch_result();
}

// ------------------------------------------------- dominance minimum (CDQ)
// Over a sequence of n items (n read on the device, at most n_max), each
// with an end e, an optional key (kNone: not a point) and an optional query
// id (kNone: not a query): for every query item i, the least key over the
// points j < i whose end is at least e_i, written to ans[query id] (kNone
// if there is none). A merge sort on e, descending, carries the answers:
// when two neighbouring runs merge, every query of the right run takes the
// least key over the points of the left run that reach its end -- a prefix
// of the left run in that order -- so each pair (j < i) is met exactly
// once, at the merge of the two runs that first hold both. Runs of up to
// kCdqTile items merge in shared memory; longer ones output tile by output
// tile along the merge path. The prefix minima of the keys are kept per
// tile (pm) with the minimum of the run's earlier tiles (cpm).
constexpr uint32_t kNone = 0xFFFFFFFFu;
constexpr int kCdqTile = 2048;
constexpr int kCdqThreads = 512;
constexpr int kCdqPer = kCdqTile / kCdqThreads;  // 4
struct CdqBufs {
  uint64_t* e[2];
  uint32_t* key[2];
  uint32_t* qid[2];
  uint32_t* ans[2];
  uint32_t* pm[2];   // [n_max] prefix minimum of the keys within each tile
  uint32_t* cmin;    // [tiles] minimum key of each tile
  uint32_t* cpm[2];  // [tiles] minimum key of the run's tiles before each tile
  uint64_t n_max;
  unsigned int* err;  // DB_ERR_TABLE_ORDER if a merge finds unsorted input
};
__host__ __device__ inline uint64_t cdq_tiles(uint64_t n) {
  return ((n ? n : 1) + kCdqTile - 1) / kCdqTile;
}
// Merge levels after the tile level: runs of kCdqTile << l merge for l = 0, 1, ...
inline uint32_t cdq_levels(uint64_t n) {
  uint32_t l = 0;
  while (((uint64_t)kCdqTile << l) < n) ++l;
  return l;
}
__device__ __forceinline__ uint32_t cdq_levels_dev(uint64_t n) {
  uint32_t l = 0;
  while (((uint64_t)kCdqTile << l) < n) ++l;
  return l;
}

// pm[i] = the least key over positions [run start, i] of runs of `seg`
// items (a power of two) in the order `ord`; a thread owns positions
// 4t .. 4t + 3. Ends with every thread past a barrier after the writes.
__device__ __forceinline__ void seg_prefix_min(const uint32_t* sk, const uint16_t* ord,
                                               uint32_t nt, uint32_t seg, uint32_t* pm,
                                               uint32_t* s_w) {
  const uint32_t base = threadIdx.x * kCdqPer;
  const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t v[kCdqPer];
#pragma unroll
  for (int u = 0; u < kCdqPer; ++u) v[u] = base + u < nt ? sk[ord[base + u]] : kNone;
  if (seg <= (uint32_t)kCdqPer) {  // runs inside the thread
#pragma unroll
    for (int u = 1; u < kCdqPer; ++u)
      if ((u & (seg - 1)) != 0) v[u] = min(v[u], v[u - 1]);
  } else {
#pragma unroll
    for (int u = 1; u < kCdqPer; ++u) v[u] = min(v[u], v[u - 1]);
    const uint32_t tpr = seg / kCdqPer;               // threads per run
    const uint32_t wseg = tpr < 32 ? tpr : 32u;       // its part inside a warp
    uint32_t x = v[kCdqPer - 1];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(kFull, x, o);
      if ((lane & (wseg - 1)) >= (uint32_t)o) x = min(x, y);
    }
    const uint32_t prev = __shfl_up_sync(kFull, x, 1);
    uint32_t before = (lane & (wseg - 1)) ? prev : kNone;
    if (tpr > 32) {  // earlier warps of the same run
      if (lane == 31) s_w[warp] = x;
      __syncthreads();
      const uint32_t wpr = tpr / 32;
      for (uint32_t w = warp & ~(wpr - 1); w < warp; ++w) before = min(before, s_w[w]);
    }
#pragma unroll
    for (int u = 0; u < kCdqPer; ++u) v[u] = min(v[u], before);
  }
#pragma unroll
  for (int u = 0; u < kCdqPer; ++u)
    if (base + u < nt) pm[base + u] = v[u];
  __syncthreads();
}

// Tile level: items [t0, t0 + nt) sorted by end (descending, stable) in
// shared memory, answers from the pairs inside the tile; out to buffer 0.
constexpr size_t kCdqTileSmem = (size_t)kCdqTile * (8 + 4 * 4 + 2 * 2);
__global__ void __launch_bounds__(kCdqThreads) cdq_tile(const uint64_t* e_in,
                                                        const uint32_t* key_in,
                                                        const uint32_t* qid_in,
                                                        const uint32_t* n_dev, CdqBufs b) {
  kernel_prologue();
  extern __shared__ __align__(16) unsigned char cdq_smem[];
  uint64_t* se = reinterpret_cast<uint64_t*>(cdq_smem);
  uint32_t* sk = reinterpret_cast<uint32_t*>(se + kCdqTile);
  uint32_t* sq = sk + kCdqTile;
  uint32_t* sa = sq + kCdqTile;
  uint32_t* pm = sa + kCdqTile;
  uint16_t* const ord0 = reinterpret_cast<uint16_t*>(pm + kCdqTile);
  uint16_t* const ord1 = ord0 + kCdqTile;
  __shared__ uint32_t s_w[kCdqThreads / 32];
  const uint64_t n = *n_dev;
  for (uint64_t t0 = (uint64_t)blockIdx.x * kCdqTile; t0 < n;
       t0 += (uint64_t)gridDim.x * kCdqTile) {
    const uint32_t nt = (uint32_t)(n - t0 < kCdqTile ? n - t0 : kCdqTile);
    for (uint32_t x = threadIdx.x; x < nt; x += kCdqThreads) {
      se[x] = e_in[t0 + x];
      sk[x] = key_in[t0 + x];
      sq[x] = qid_in[t0 + x];
      sa[x] = kNone;
      ord0[x] = (uint16_t)x;
      pm[x] = sk[x];
    }
    __syncthreads();
    int cur = 0;
    for (uint32_t s = 1; s < nt; s <<= 1) {
      // Outputs 4t .. 4t + 3 of the merge of each run with the neighbouring
      // one: where they start on the merge path, then four steps, left first
      // on equal ends. A right item taken after c left items takes the least
      // key of the left run's first c (its prefix minima, pm).
      const uint16_t* oc = cur ? ord1 : ord0;
      uint16_t* on = cur ? ord0 : ord1;
      const uint32_t first = threadIdx.x * kCdqPer;
      if (first < nt) {
        uint32_t pb = first / (2 * s) * (2 * s);
        uint32_t nl = nt - pb < s ? nt - pb : s;
        uint32_t nr = pb + s < nt ? (nt - pb - s < s ? nt - pb - s : s) : 0u;
        const uint32_t d = first - pb;
        uint32_t lo = d > nr ? d - nr : 0u, hi = d < nl ? d : nl;
        while (lo < hi) {
          const uint32_t mid = (lo + hi) >> 1;
          if (se[oc[pb + s + d - mid - 1]] <= se[oc[pb + mid]]) lo = mid + 1;
          else hi = mid;
        }
        uint32_t ia = lo, ib = d - lo;
  #pragma unroll
        for (int u = 0; u < kCdqPer; ++u) {
          const uint32_t o = first + u;
          if (o >= nt) break;
          if (o - pb == 2 * s) {  // runs of one or two: the next pair of runs
            pb = o;
            nl = nt - pb < s ? nt - pb : s;
            nr = pb + s < nt ? (nt - pb - s < s ? nt - pb - s : s) : 0u;
            ia = ib = 0;
          }
          const bool left = ib >= nr || (ia < nl && se[oc[pb + ia]] >= se[oc[pb + s + ib]]);
          const uint32_t x = left ? oc[pb + ia] : oc[pb + s + ib];
          if (!left && ia > 0 && sq[x] != kNone) sa[x] = min(sa[x], pm[pb + ia - 1]);
          on[o] = (uint16_t)x;
          if (left) ++ia;
          else ++ib;
        }
      }
      __syncthreads();
      cur ^= 1;
      seg_prefix_min(sk, cur ? ord1 : ord0, nt, 2 * s, pm, s_w);
    }
    for (uint32_t i = threadIdx.x; i < nt; i += kCdqThreads) {
      const uint32_t x = (cur ? ord1 : ord0)[i];
      b.e[0][t0 + i] = se[x];
      b.key[0][t0 + i] = sk[x];
      b.qid[0][t0 + i] = sq[x];
      b.ans[0][t0 + i] = sa[x];
      b.pm[0][t0 + i] = pm[i];
    }
    if (threadIdx.x == 0) b.cpm[0][t0 / kCdqTile] = kNone;  // a tile is its whole run
    __syncthreads();  // shared memory is reused by the next tile
  }
}

// Merge level l: runs of len = kCdqTile << l, buffers (l & 1) to (l & 1) ^ 1.
// A CTA makes tile c of the output: the merge of the slices of the two runs
// that precede it in the merged order (found by a warp-parallel binary
// search on the merge path), in shared memory, written out whole with the
// tile's prefix minima of the keys. A right-run query takes the least key of
// the left run's prefix reaching its end, from the input's prefix minima.
//
// The merge path: the first d items of the merge are i items of the left
// run and d - i of the right run for the least i at which the right run's
// (d - i)-th item is ahead of the left run's (i + 1)-th, R[d - i - 1] > L[i]
// (a right item is ahead only with a strictly greater end); that test turns
// from false to true as i grows, and with none, i is the largest possible.
__device__ __forceinline__ uint64_t corank_warp(const uint64_t* L, uint64_t nL, const uint64_t* R,
                                                uint64_t nR, uint64_t d) {
  const uint32_t lane = threadIdx.x & 31;
  uint64_t lo = d > nR ? d - nR : 0, hi = d < nL ? d : nL;  // answer in [lo, hi]
  // probe t(i) = R[d - i - 1] <= L[i] (true before the answer)
  while (hi - lo > 32) {
    const uint64_t step = (hi - lo + 31) / 32;
    const uint64_t at = lo + lane * step;
    bool t = false;
    if (at < hi) t = R[d - at - 1] <= L[at];
    const uint32_t k = __popc(__ballot_sync(kFull, t));
    const uint64_t nlo = k ? lo + (k - 1) * step + 1 : lo;
    const uint64_t nhi = lo + k * step < hi ? lo + k * step : hi;
    lo = nlo;
    hi = nhi;
  }
  bool t = false;
  if (lo + lane < hi) t = R[d - (lo + lane) - 1] <= L[lo + lane];
  return lo + __popc(__ballot_sync(kFull, t));
}
// The slices' ends, keys, query ids and answers are staged in shared memory;
// thread t makes outputs 4t .. 4t + 3 of the tile: it finds how many of the
// first 4t come from the left slice (a search on the merge path inside the
// slices) and merges four from there, left first on equal ends. A right item
// taken after c items of the left run (i0 before the slice) is a query over
// the left run's prefix of length c.
constexpr size_t kCdqMergeSmem = (size_t)kCdqTile * (8 + 4 * 3);
// Three CTAs per SM (at most 42 registers a thread) measured faster than two.
__global__ void __launch_bounds__(kCdqThreads, 3) cdq_merge(CdqBufs b, const uint32_t* n_dev,
                                                         uint32_t level) {
  kernel_prologue();
  extern __shared__ __align__(16) unsigned char cdq_smem[];
  uint64_t* seg = reinterpret_cast<uint64_t*>(cdq_smem);  // left slice, then right slice
  uint32_t* sk = reinterpret_cast<uint32_t*>(seg + kCdqTile);
  uint32_t* sq = sk + kCdqTile;
  uint32_t* sa = sq + kCdqTile;
  __shared__ uint64_t s_i0, s_i1;
  __shared__ uint32_t s_w[kCdqThreads / 32];
  const uint64_t n = *n_dev;
  const uint64_t len = (uint64_t)kCdqTile << level;
  if (len >= n) return;  // this level is not needed
  for (uint64_t o0 = (uint64_t)blockIdx.x * kCdqTile; o0 < n;
       o0 += (uint64_t)gridDim.x * kCdqTile) {
    const uint64_t o1 = o0 + kCdqTile < n ? o0 + kCdqTile : n;
    const bool odd = (level & 1u) != 0;  // input buffer 1, output 0
    const uint64_t* E = odd ? b.e[1] : b.e[0];
    const uint32_t* Kin = odd ? b.key[1] : b.key[0];
    const uint32_t* Qin = odd ? b.qid[1] : b.qid[0];
    const uint32_t* Ain = odd ? b.ans[1] : b.ans[0];
    const uint32_t* PMin = odd ? b.pm[1] : b.pm[0];
    const uint32_t* CPMin = odd ? b.cpm[1] : b.cpm[0];
    uint64_t* Eo = odd ? b.e[0] : b.e[1];
    uint32_t* Ko = odd ? b.key[0] : b.key[1];
    uint32_t* Qo = odd ? b.qid[0] : b.qid[1];
    uint32_t* Ao = odd ? b.ans[0] : b.ans[1];
    uint32_t* PMo = odd ? b.pm[0] : b.pm[1];
    const uint64_t pb = o0 / (2 * len) * (2 * len);
    const uint64_t nL = pb + len < n ? len : n - pb;
    const uint64_t rb = pb + nL;
    const uint64_t nR = pb + 2 * len < n ? len : n - rb;
    const uint64_t d0 = o0 - pb, d1 = o1 - pb;
    if (threadIdx.x < 32) {
      const uint64_t i = corank_warp(E + pb, nL, E + rb, nR, d0);
      if (threadIdx.x == 0) s_i0 = i;
    } else if (threadIdx.x < 64) {
      const uint64_t i = corank_warp(E + pb, nL, E + rb, nR, d1);
      if (threadIdx.x == 32) s_i1 = i;
    }
    __syncthreads();
    const uint64_t i0 = s_i0, i1 = s_i1, j0 = d0 - i0, j1 = d1 - i1;
    // A slice pair that is not a split of this tile (impossible for sorted
    // runs) is reported and the tile left unwritten.
    if (i1 < i0 || i1 > nL || j0 > d0 || j1 < j0 || j1 > nR) {
      if (threadIdx.x == 0) atomicOr(b.err, DB_ERR_TABLE_ORDER);
      __syncthreads();
      continue;
    }
    const uint32_t na = (uint32_t)(i1 - i0), nb = (uint32_t)(j1 - j0), nt = na + nb;
    for (uint32_t x = threadIdx.x; x < nt; x += kCdqThreads) {
      const uint64_t gi = x < na ? pb + i0 + x : rb + j0 + (x - na);
      seg[x] = E[gi];
      sk[x] = Kin[gi];
      sq[x] = Qin[gi];
      sa[x] = Ain[gi];
    }
    __syncthreads();
    const uint64_t* sl = seg;
    const uint64_t* sr = seg + na;
    const uint32_t base = threadIdx.x * kCdqPer;
    uint64_t oe[kCdqPer];
    uint32_t ok[kCdqPer], oq[kCdqPer], oa[kCdqPer];
    {
      // left items among the first `base` outputs: the least ia in [lo, hi]
      // with sr[base - ia - 1] > sl[ia] (a right item is ahead only with a
      // strictly greater end), hi when there is none
      uint32_t lo = base > nb ? base - nb : 0u, hi = base < na ? base : na;
      while (lo < hi) {
        const uint32_t mid = (lo + hi) >> 1;
        if (sr[base - mid - 1] <= sl[mid]) lo = mid + 1;
        else hi = mid;
      }
      uint32_t ia = lo, ib = base - lo;
#pragma unroll
      for (int u = 0; u < kCdqPer; ++u) {
        oe[u] = 0;
        ok[u] = oq[u] = oa[u] = kNone;
        if (base + u >= nt) continue;
        const bool left = ib >= nb || (ia < na && sl[ia] >= sr[ib]);
        const uint32_t x = left ? ia : na + ib;
        uint32_t a = sa[x];
        const uint32_t q = sq[x];
        if (!left && q != kNone) {
          const uint64_t c = i0 + ia;  // left-run items with an end at least this one's
          if (c > 0) {
            const uint64_t j = pb + c - 1;
            a = min(a, min(PMin[j], CPMin[j / kCdqTile]));
          }
        }
        oe[u] = seg[x];
        ok[u] = sk[x];
        oq[u] = q;
        oa[u] = a;
        if (left) ++ia;
        else ++ib;
      }
    }
    // prefix minima of the keys over the tile's outputs, and the write-out
    uint32_t v[kCdqPer];
    uint32_t run = kNone;
  #pragma unroll
    for (int u = 0; u < kCdqPer; ++u) {
      run = min(run, ok[u]);
      v[u] = run;
    }
    const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t x = run;
  #pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(kFull, x, o);
      if (lane >= o) x = min(x, y);
    }
    if (lane == 31) s_w[warp] = x;
    const uint32_t up = __shfl_up_sync(kFull, x, 1);
    __syncthreads();
    uint32_t before = lane ? up : kNone;
    for (uint32_t w = 0; w < warp; ++w) before = min(before, s_w[w]);
    if (base + kCdqPer <= nt) {
      uint64_t* ep = Eo + o0 + base;
      reinterpret_cast<ulonglong2*>(ep)[0] = make_ulonglong2(oe[0], oe[1]);
      reinterpret_cast<ulonglong2*>(ep)[1] = make_ulonglong2(oe[2], oe[3]);
      *reinterpret_cast<uint4*>(Ko + o0 + base) = make_uint4(ok[0], ok[1], ok[2], ok[3]);
      *reinterpret_cast<uint4*>(Qo + o0 + base) = make_uint4(oq[0], oq[1], oq[2], oq[3]);
      *reinterpret_cast<uint4*>(Ao + o0 + base) = make_uint4(oa[0], oa[1], oa[2], oa[3]);
      *reinterpret_cast<uint4*>(PMo + o0 + base) =
          make_uint4(min(before, v[0]), min(before, v[1]), min(before, v[2]), min(before, v[3]));
    } else {
  #pragma unroll
      for (int u = 0; u < kCdqPer; ++u) {
        if (base + u >= nt) break;
        Eo[o0 + base + u] = oe[u];
        Ko[o0 + base + u] = ok[u];
        Qo[o0 + base + u] = oq[u];
        Ao[o0 + base + u] = oa[u];
        PMo[o0 + base + u] = min(before, v[u]);
      }
    }
    if (threadIdx.x == kCdqThreads - 1) {
      uint32_t all = kNone;
      for (int w = 0; w < kCdqThreads / 32; ++w) all = min(all, s_w[w]);
      b.cmin[o0 / kCdqTile] = all;
    }
    __syncthreads();  // shared memory is reused by the next tile
  }
}

// cpm[t] = the least cmin over the tiles before t in its merged run (one
// CTA, 1,024 tiles at a time): a segmented scan, a run's first tile a head.
__global__ void __launch_bounds__(1024) cdq_cpm(CdqBufs b, const uint32_t* n_dev, uint32_t level) {
  kernel_prologue();
  __shared__ uint32_t s_v[1024];
  __shared__ uint8_t s_f[1024];
  const uint64_t n = *n_dev;
  const uint64_t len2 = (uint64_t)kCdqTile << (level + 1);  // merged run length
  if ((len2 >> 1) >= n) return;
  const uint64_t tiles = cdq_tiles(n);
  const uint64_t per = len2 / kCdqTile;  // tiles per merged run
  const uint32_t tid = threadIdx.x;
  uint32_t carry = kNone;  // inclusive minimum of the open run up to the last block
  for (uint64_t t0 = 0; t0 < tiles; t0 += 1024) {
    const uint64_t t = t0 + tid;
    const bool head = (t % per) == 0;
    s_v[tid] = t < tiles ? b.cmin[t] : kNone;
    s_f[tid] = head ? 1 : 0;
    __syncthreads();
    for (uint32_t d = 1; d < 1024; d <<= 1) {
      uint32_t v = s_v[tid];
      uint8_t f = s_f[tid];
      if (tid >= d && !f) {
        v = min(v, s_v[tid - d]);
        f = s_f[tid - d];
      }
      __syncthreads();
      s_v[tid] = v;
      s_f[tid] = f;
      __syncthreads();
    }
    // s_v[tid]: minimum from the last head in the block (or its start) to tid
    const uint32_t prev = tid ? (s_f[tid - 1] ? s_v[tid - 1] : min(s_v[tid - 1], carry)) : carry;
    if (t < tiles) ((level & 1u) ? b.cpm[0] : b.cpm[1])[t] = head ? kNone : prev;
    __syncthreads();
    carry = s_f[1023] ? s_v[1023] : min(s_v[1023], carry);
    __syncthreads();
  }
}

// Answers to the queries, from the buffer the last level wrote.
__global__ void cdq_out(CdqBufs b, const uint32_t* n_dev, uint32_t* ans) {
  kernel_prologue();
  const uint64_t n = *n_dev;
  const bool fin1 = (cdq_levels_dev(n) & 1u) != 0;
  const uint32_t* Q = fin1 ? b.qid[1] : b.qid[0];
  const uint32_t* A = fin1 ? b.ans[1] : b.ans[0];
  FOR_EACH(i, n) {
    const uint32_t q = Q[i];
    if (q != kNone) ans[q] = A[i];
  }
}

// The whole computation on items e_in / key_in / qid_in (at most b.n_max,
// *n_dev of them); every launch is a dependent of the one before.
int cdq_dominance_min(const uint64_t* e_in, const uint32_t* key_in, const uint32_t* qid_in,
                      const uint32_t* n_dev, CdqBufs& b, uint32_t* ans, cudaStream_t s) {
  static bool ready[64] = {false};  // the tile kernel's shared memory is above 48 KiB
  int dev = 0;
  cudaGetDevice(&dev);
  if (!ready[dev & 63]) {
    if (cudaFuncSetAttribute(cdq_tile, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kCdqTileSmem) != cudaSuccess ||
        cudaFuncSetAttribute(cdq_merge, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kCdqMergeSmem) != cudaSuccess)
      return launch_result();
    ready[dev & 63] = true;
  }
  // Loops over the tiles of the device-side length: one wave of CTAs.
  uint64_t tiles = cdq_tiles(b.n_max);
  const uint64_t wave = (uint64_t)num_sms() * 3;
  if (tiles > wave) tiles = wave;
  int rc = 0;
  launch_dep(cdq_tile, (unsigned)tiles, kCdqThreads, kCdqTileSmem, s, e_in, key_in, qid_in,
             n_dev, b);
  if ((rc = launch_result())) return rc;
  const uint32_t levels = cdq_levels(b.n_max);
  for (uint32_t l = 0; l < levels; ++l) {
    launch_dep(cdq_merge, (unsigned)tiles, kCdqThreads, kCdqMergeSmem, s, b, n_dev, l);
    if ((rc = launch_result())) return rc;
    if (l + 1 < levels) {  // the last level's tile minima are never read
      launch_dep(cdq_cpm, 1, 1024, 0, s, b, n_dev, l);
      if ((rc = launch_result())) return rc;
    }
  }
  launch_dep(cdq_out, grid_for(b.n_max), kThreads, 0, s, b, n_dev, ans);
  return launch_result();
}

// ------------------------------------------------------------- registration
struct RegHeader {   // 256 bytes at the start of the registration workspace
  uint32_t m;        // requests that missed the table before the batch
  uint32_t u;        // new records (requests no earlier request's range held)
  uint32_t d;        // distinct ranges among the misses
  uint32_t nb;       // items of the second dominance pass (new records and queries)
  unsigned int err;  // an inconsistency the passes found (DB_ERR_TABLE_ORDER)
  uint32_t dk;       // distinct ranges the first dominance pass needs
  uint32_t wide;     // a miss whose start or length does not fit the packed sort key
  uint32_t pad;
  db_counters lookup;  // counters of the lookup pass
};

__device__ __forceinline__ void widen(const db_range* q, uint64_t k, uint32_t gshift,
                                      uint64_t& base, uint64_t& aend) {
  const uint64_t g = 1ull << gshift;
  const uint64_t addr = q[k].addr, size = q[k].size;
  base = addr & ~(g - 1);
  aend = (addr + size + g - 1) & ~(g - 1);  // valid requests only: no wrap
}

// Four kinds a lane (one u32 load; kind0 is 4-byte aligned and padded), so
// a warp step covers 128 requests, four flag words: lanes 8w .. 8w + 7 hold
// word w's 32 bits, four each, gathered by three shuffles.
__global__ void reg_mark(const uint8_t* kind0, uint64_t n_q, uint32_t* bits) {
  kernel_prologue();
  const uint32_t lane = threadIdx.x & 31;
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x * 4;
  for (uint64_t b0 = ((uint64_t)blockIdx.x * blockDim.x + (threadIdx.x & ~31u)) * 4; b0 < n_q;
       b0 += stride) {
    const uint64_t k = b0 + 4 * lane;
    uint32_t nib = 0;
    if (k < n_q) {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(kind0 + k);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (k + j < n_q && ((w >> (8 * j)) & 255u) == DB_MR_MISS) nib |= 1u << j;
    }
    uint32_t x = nib << (4 * (lane & 7));
    x |= __shfl_xor_sync(kFull, x, 1);
    x |= __shfl_xor_sync(kFull, x, 2);
    x |= __shfl_xor_sync(kFull, x, 4);
    if ((lane & 7) == 0 && b0 + 4 * lane < n_q) bits[(b0 >> 5) + (lane >> 3)] = x;
  }
}
// The packed sort key: the start granule above kLenBits bits that hold the
// length in granules complemented, so one ascending sort orders the ranges
// by start ascending, then end descending. It holds starts below
// 2^(64 - kLenBits) granules and lengths below 2^kLenBits granules.
constexpr uint32_t kLenBits = 24;
constexpr uint64_t kLenMask = (1ull << kLenBits) - 1;
// The range a packed key holds.
__device__ __forceinline__ void unpack_key(uint64_t k, uint32_t gshift, uint64_t& b, uint64_t& e) {
  const uint64_t g = k >> kLenBits, len = kLenMask - (k & kLenMask);
  b = g << gshift;
  e = (g + len) << gshift;
}
__global__ void reg_compact(const db_range* q, const uint32_t* bits, const uint32_t* wpos,
                            uint64_t n_q, uint32_t gshift, uint64_t* key, uint32_t* val,
                            RegHeader* h) {
  kernel_prologue();
  bool wide = false;
  FOR_EACH(k, n_q) {
    if (!flag_at(bits, k)) continue;
    uint64_t b, e;
    widen(q, k, gshift, b, e);
    const uint64_t g = b >> gshift, len = (e - b) >> gshift;
    const bool fits = (g >> (64 - kLenBits)) == 0 && len <= kLenMask;
    wide |= !fits;
    const uint32_t at = flag_pos(bits, wpos, k);
    key[at] = (g << kLenBits) | (kLenMask - len);  // rewritten when some miss does not fit
    val[at] = (uint32_t)k;
  }
  if (__syncthreads_or(wide) && threadIdx.x == 0) atomicOr(&h->wide, 1u);
}
// Only when the packed key does not hold every miss: the key of the sort on
// the end (descending) or, after it, of the stable sort on the start.
__global__ void reg_rekey(const db_range* q, const RegHeader* h, uint64_t n_max, uint32_t gshift,
                          const uint32_t* val, uint64_t* key, bool by_end) {
  kernel_prologue();
  if (!h->wide) return;
  const uint64_t m = h->m;
  FOR_EACH(i, n_max) {
    if (i >= m) break;
    uint64_t b, e;
    widen(q, val[i], gshift, b, e);
    key[i] = by_end ? ~e >> gshift : b >> gshift;
  }
}
// Run starts of equal widened ranges over the sorted misses (flags of the
// m first items; their scan reads no further). Packed keys are equal
// exactly when their ranges are; the end and start keys of the two-sort
// path are not, so then the ranges are read again.
__global__ void reg_runs(const db_range* q, const RegHeader* h, uint32_t gshift,
                         const uint32_t* val, const uint64_t* key, uint32_t* bits) {
  kernel_prologue();
  const uint64_t m = h->m;
  const bool packed = !h->wide;
  FOR_EACH_WARP(i0, m) {
    const uint64_t i = i0 + (threadIdx.x & 31);
    bool f = i < m;
    if (f && i > 0) {
      if (packed) {
        f = key[i] != key[i - 1];
      } else {
        uint64_t b0, e0, b1, e1;
        widen(q, val[i - 1], gshift, b0, e0);
        widen(q, val[i], gshift, b1, e1);
        f = (b0 != b1 || e0 != e1);
      }
    }
    put_flags(bits, i0, f);
  }
}
// Count of a[0..n) below x (strict) or at most x.
__device__ __forceinline__ uint64_t count_below(const uint64_t* a, uint64_t n, uint64_t x,
                                                bool or_equal) {
  uint64_t lo = 0, hi = n;
  while (lo < hi) {
    const uint64_t mid = (lo + hi) >> 1;
    const uint64_t v = a[mid];
    if (v < x || (or_equal && v == x)) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}
// The distinct missed ranges, in (start ascending, end descending) order:
// start, end, the request that first asked for it, and whether a later
// request asked for it again.
__global__ void reg_distinct(const db_range* q, const RegHeader* h, uint64_t n_max,
                             uint32_t gshift, const uint32_t* val, const uint64_t* key,
                             const uint32_t* bits, const uint32_t* wpos, uint64_t* db,
                             uint64_t* de, uint32_t* first, uint8_t* again) {
  kernel_prologue();
  const uint64_t m = h->m;
  const bool packed = !h->wide;
  FOR_EACH(i, n_max) {
    if (i >= m) break;
    if (!flag_at(bits, i)) continue;
    const uint32_t p = flag_pos(bits, wpos, i);
    uint64_t b, e;
    if (packed) unpack_key(key[i], gshift, b, e);
    else widen(q, val[i], gshift, b, e);
    db[p] = b;
    de[p] = e;
    first[p] = val[i];
    again[p] = (i + 1 < m && !flag_at(bits, i + 1)) ? 1 : 0;
  }
}
// Items of the first dominance pass: a distinct range is a query for the
// least first request among the ranges before it that reach its end (the
// ranges that hold it) and a point keyed by its own first request. A range
// that nothing before it reaches (prefix maximum of the ends, pm) is held by
// none; one before which the next range starts at or past its end holds
// none: such a range takes no part (held[] = none), and the rest keep their
// order. The others are flagged (flags of the d first items; their scan
// reads no further).
__global__ void reg_keep_a(const RegHeader* h, const uint64_t* db, const uint64_t* de,
                           const uint64_t* pm, uint32_t* held, uint32_t* keep) {
  kernel_prologue();
  const uint64_t d = h->d;
  FOR_EACH_WARP(p0, d) {
    const uint64_t p = p0 + (threadIdx.x & 31);
    bool k = false;
    if (p < d) {
      const bool nested = p > 0 && pm[p - 1] >= de[p];
      const bool holds = p + 1 < d && db[p + 1] < de[p];
      held[p] = kNone;
      k = nested || holds;
    }
    put_flags(keep, p0, k);
  }
}
__global__ void reg_items_a(const RegHeader* h, uint64_t n_max, const uint32_t* keep,
                            const uint32_t* kpos, const uint64_t* de, const uint32_t* first,
                            uint64_t* ce_in, uint32_t* ck_in, uint32_t* cq_in) {
  kernel_prologue();
  const uint64_t d = h->d;
  FOR_EACH(p, n_max) {
    if (p >= d) break;
    if (!flag_at(keep, p)) continue;
    const uint32_t at = flag_pos(keep, kpos, p);
    ce_in[at] = de[p];
    ck_in[at] = first[p];
    cq_in[at] = (uint32_t)p;
  }
}
// A distinct range makes a new record when no range before it that holds it
// was asked for earlier (then its first request finds no record holding it).
// Flags of the d first items; their scan reads no further.
__global__ void reg_creators(const RegHeader* h, const uint32_t* first, const uint32_t* held_by,
                             uint32_t* cflag) {
  kernel_prologue();
  const uint64_t d = h->d;
  FOR_EACH_WARP(p0, d) {
    const uint64_t p = p0 + (threadIdx.x & 31);
    put_flags(cflag, p0, p < d && held_by[p] > first[p]);
  }
}
// New records in (start ascending, end descending) order: c = cpos[p].
__global__ void reg_clist(const RegHeader* h, uint64_t n_max, const uint32_t* cflag,
                          const uint32_t* cpos, const uint64_t* db, uint32_t* cp, uint64_t* cb) {
  kernel_prologue();
  const uint64_t d = h->d;
  FOR_EACH(p, n_max) {
    if (p >= d) break;
    if (!flag_at(cflag, p)) continue;
    const uint32_t c = flag_pos(cflag, cpos, p);
    cp[c] = (uint32_t)p;
    cb[c] = db[p];
  }
}
// Table order of the new records: start ascending, then end ascending (a
// later new record of the same start ends later: it was not held by the
// earlier one). Within a run of equal starts the list above is in the
// opposite order of ends, so record c of a run [gs, ge) goes to gs + ge - 1 - c.
//
// A new record can be the answer of a later request only when its range is
// asked for again, or it holds another missed range (then the next distinct
// range starts before its end), or it may take a hit from an old record that
// starts inside it (an old start lies strictly between its start and end);
// point[j] says so, and the other new records stay out of the second
// dominance pass (a request they could answer has a holder that is in it at
// a position no later, or keeps its old record either way). Its place in
// the merged table is npos[j] = j + the old records starting at or before
// it; when that table fits out_cap the record is written there, with no
// references yet (reg_resolve adds them).
__global__ void reg_cplace(const RegHeader* h, uint64_t n_max, const uint32_t* cp,
                           const uint64_t* cb, const uint64_t* db, const uint64_t* de,
                           const uint32_t* first, const uint8_t* again, const uint64_t* start,
                           uint64_t n_mr, const uint32_t* new_lkey, uint64_t o_cap,
                           uint64_t* nstart, uint64_t* nend, uint32_t* creator_of, uint64_t* cend,
                           uint8_t* point, uint32_t* npos, uint64_t* o_start, uint64_t* o_end,
                           uint32_t* o_lkey, uint32_t* o_refs) {
  kernel_prologue();
  const uint64_t u = h->u, d = h->d;
  const bool fits = n_mr + u <= o_cap;
  FOR_EACH(c, n_max) {
    if (c >= u) break;
    const uint64_t b = cb[c];
    uint64_t gs = c, ge = c + 1;
    if ((c > 0 && cb[c - 1] == b) || (c + 1 < u && cb[c + 1] == b)) {
      uint64_t lo = 0, hi = c;  // first with start b
      while (lo < hi) {
        const uint64_t mid = (lo + hi) >> 1;
        if (cb[mid] < b) lo = mid + 1;
        else hi = mid;
      }
      gs = lo;
      lo = c + 1;
      hi = u;  // first with a greater start
      while (lo < hi) {
        const uint64_t mid = (lo + hi) >> 1;
        if (cb[mid] <= b) lo = mid + 1;
        else hi = mid;
      }
      ge = lo;
    }
    const uint64_t j = gs + ge - 1 - c;
    const uint32_t p = cp[c];
    const uint64_t e = de[p];
    const uint32_t f = first[p];
    nstart[j] = b;
    nend[j] = e;
    creator_of[f] = (uint32_t)j;
    cend[c] = e;
    const uint64_t o = count_below(start, n_mr, b, true);  // first old record starting past b
    const uint64_t w = j + o;
    npos[j] = (uint32_t)w;
    if (fits) {
      o_start[w] = b;
      o_end[w] = e;
      o_lkey[w] = new_lkey[f];
      o_refs[w] = 0;
    }
    const bool pt = again[p] || (p + 1 < d && db[p + 1] < e) || (o < n_mr && start[o] < e);
    point[j] = pt ? 1 : 0;
  }
}
// reach[o] = the largest end of a new record starting before old record o
// (a prefix maximum of cend over the list, which is in start order): a hit
// on o can be taken by a new record only if its end is within that reach.
// Its place in the merged table is remap[o] = o + the new records starting
// before it; when that table fits out_cap the record is written there with
// its references before the batch (reg_resolve adds the batch's).
__global__ void reg_reach(const RegHeader* h, const uint64_t* cb, const uint64_t* pmax,
                          const uint64_t* start, const uint64_t* end, const uint32_t* lkey,
                          const uint32_t* refs, uint64_t n, uint64_t o_cap, uint64_t* reach,
                          int64_t* remap, uint64_t* o_start, uint64_t* o_end, uint32_t* o_lkey,
                          uint32_t* o_refs) {
  kernel_prologue();
  const uint64_t u = h->u;
  const bool fits = n + u <= o_cap;
  FOR_EACH(o, n) {
    const uint64_t s = start[o];
    uint64_t lo = 0, hi = u;  // new records starting before s
    while (lo < hi) {
      const uint64_t mid = (lo + hi) >> 1;
      if (cb[mid] < s) lo = mid + 1;
      else hi = mid;
    }
    reach[o] = lo ? pmax[lo - 1] : 0;
    if (fits) {
      const uint64_t w = o + lo;  // old first on equal starts
      remap[o] = (int64_t)w;
      o_start[w] = s;
      o_end[w] = end[o];
      o_lkey[w] = lkey[o];
      o_refs[w] = refs[o];
    }
  }
}
// Items of the second dominance pass, in request order: the new records
// that may answer a request (key: table position among the new records,
// end) and the requests whose record is still open -- misses that made no
// record, and hits on an old record that a new record may precede (query
// id: the request).
__global__ void reg_roles(const db_range* q, uint64_t n_q, uint32_t gshift, const uint8_t* kind0,
                          const int32_t* idx, const uint64_t* reach, const uint32_t* creator_of,
                          const uint8_t* point, uint32_t* role) {
  kernel_prologue();
  // Two warp steps at a time, so that both steps' dependent loads (the
  // creator or the old record, then its point flag or reach) are in flight
  // together.
  const uint64_t step = (uint64_t)gridDim.x * blockDim.x;
  const uint32_t lane = threadIdx.x & 31;
  for (uint64_t k0 = (uint64_t)blockIdx.x * blockDim.x + (threadIdx.x & ~31u); k0 < n_q;
       k0 += 2 * step) {
    uint64_t k[2] = {k0 + lane, k0 + step + lane};
    uint8_t kd[2];
    uint32_t c[2];
    int32_t o[2];
    uint64_t e[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      kd[u] = k[u] < n_q ? kind0[k[u]] : (uint8_t)DB_MR_INVALID;
      c[u] = kNone;
      o[u] = 0;
      e[u] = 0;
      if (kd[u] == DB_MR_MISS) {
        c[u] = creator_of[k[u]];
      } else if (kd[u] == DB_MR_EXACT || kd[u] == DB_MR_CONTAINED) {
        uint64_t b;
        widen(q, k[u], gshift, b, e[u]);
        o[u] = idx[k[u]];
      }
    }
    bool r[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      r[u] = false;
      if (kd[u] == DB_MR_MISS) r[u] = c[u] == kNone || point[c[u]];
      else if (kd[u] == DB_MR_EXACT || kd[u] == DB_MR_CONTAINED)
        r[u] = reach[o[u]] >= e[u];  // a new record starting before the old one may hold it
    }
    put_flags(role, k0, r[0]);
    if (k0 + step < n_q) put_flags(role, k0 + step, r[1]);
  }
}

// Inclusive prefix maximum of n u64 values (n on the device, at most n_max).
// A thread takes kPmItems consecutive values; block maxima first, then each
// block scans its chunk from the maximum of the blocks before it -- found by
// the block itself when there are at most kScanFusedBlocks blocks, else by a
// one-CTA scan of the block maxima.
constexpr int kMaxScanThreads = 1024;
constexpr int kPmItems = 8;
constexpr uint64_t kPmChunk = (uint64_t)kMaxScanThreads * kPmItems;
__device__ __forceinline__ void pm_load(const uint64_t* in, uint64_t b, uint64_t n,
                                        uint64_t (&x)[kPmItems]) {
  if (b + kPmItems <= n) {
    const ulonglong2* p = reinterpret_cast<const ulonglong2*>(in + b);
#pragma unroll
    for (int j = 0; j < kPmItems / 2; ++j) {
      const ulonglong2 v = p[j];
      x[2 * j] = v.x;
      x[2 * j + 1] = v.y;
    }
  } else {
#pragma unroll
    for (int j = 0; j < kPmItems; ++j) x[j] = b + j < n ? in[b + j] : 0;
  }
}
__device__ __forceinline__ uint64_t max64(uint64_t a, uint64_t b) { return a > b ? a : b; }
// The maximum over the block (every thread gets it).
__device__ __forceinline__ uint64_t block_max(uint64_t v, uint64_t* s_w) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max64(v, __shfl_xor_sync(kFull, v, o));
  if ((threadIdx.x & 31) == 0) s_w[threadIdx.x >> 5] = v;
  __syncthreads();
  v = s_w[threadIdx.x & 31];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max64(v, __shfl_xor_sync(kFull, v, o));
  __syncthreads();  // s_w may be written again
  return v;
}
__global__ void __launch_bounds__(kMaxScanThreads) pmax_reduce(const uint64_t* in,
                                                               const uint32_t* n_dev,
                                                               uint64_t* bmax) {
  kernel_prologue();
  __shared__ uint64_t s_w[32];
  const uint64_t n = *n_dev;
  if ((uint64_t)blockIdx.x * kPmChunk >= n) return;
  uint64_t x[kPmItems];
  pm_load(in, (uint64_t)blockIdx.x * kPmChunk + (uint64_t)threadIdx.x * kPmItems, n, x);
  uint64_t v = 0;
#pragma unroll
  for (int j = 0; j < kPmItems; ++j) v = max64(v, x[j]);
  v = block_max(v, s_w);
  if (threadIdx.x == 0) bmax[blockIdx.x] = v;
}
// More than kScanFusedBlocks blocks: bmax becomes the exclusive prefix maximum.
__global__ void __launch_bounds__(1024) pmax_blocks(uint64_t* bmax, const uint32_t* n_dev) {
  kernel_prologue();
  __shared__ uint64_t s_w[32];
  const uint64_t nb = (*n_dev + kPmChunk - 1) / kPmChunk;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint64_t carry = 0;  // the maximum of the blocks before this round
  for (uint64_t b0 = 0; b0 < nb; b0 += 1024) {
    const uint64_t b = b0 + threadIdx.x;
    const uint64_t v = b < nb ? bmax[b] : 0;
    uint64_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint64_t y = __shfl_up_sync(kFull, x, o);
      if (lane >= o && y > x) x = y;
    }
    if (lane == 31) s_w[warp] = x;
    __syncthreads();
    const uint64_t up = __shfl_up_sync(kFull, x, 1);
    uint64_t ex = lane ? up : 0;  // exclusive within the warp
    for (int w = 0; w < warp; ++w) ex = max64(ex, s_w[w]);
    ex = max64(ex, carry);
    if (b < nb) bmax[b] = ex;
    uint64_t all = carry;
    for (int w = 0; w < 32; ++w) all = max64(all, s_w[w]);
    __syncthreads();  // s_w is written again in the next round
    carry = all;
  }
}
__global__ void __launch_bounds__(kMaxScanThreads) pmax_apply(const uint64_t* in,
                                                              const uint32_t* n_dev,
                                                              const uint64_t* bmax, bool prefixed,
                                                              uint64_t* out) {
  kernel_prologue();
  __shared__ uint64_t s_w[32];
  const uint64_t n = *n_dev;
  if ((uint64_t)blockIdx.x * kPmChunk >= n) return;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint64_t b = (uint64_t)blockIdx.x * kPmChunk + (uint64_t)threadIdx.x * kPmItems;
  uint64_t x[kPmItems];
  pm_load(in, b, n, x);
  uint64_t before = 0;  // the blocks before this one
  if (prefixed) {
    before = bmax[blockIdx.x];
  } else {
    for (uint32_t k = threadIdx.x; k < blockIdx.x; k += kMaxScanThreads)
      before = max64(before, bmax[k]);
    before = block_max(before, s_w);
  }
#pragma unroll
  for (int j = 1; j < kPmItems; ++j) x[j] = max64(x[j], x[j - 1]);
  uint64_t t = x[kPmItems - 1];  // inclusive over the threads up to this one
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint64_t y = __shfl_up_sync(kFull, t, o);
    if (lane >= o) t = max64(t, y);
  }
  if (lane == 31) s_w[warp] = t;
  __syncthreads();
  uint64_t ex = __shfl_up_sync(kFull, t, 1);
  ex = lane ? ex : 0;
  for (int w = 0; w < warp; ++w) ex = max64(ex, s_w[w]);
  ex = max64(ex, before);
  if (b + kPmItems <= n) {
    ulonglong2* p = reinterpret_cast<ulonglong2*>(out + b);
#pragma unroll
    for (int j = 0; j < kPmItems / 2; ++j)
      p[j] = make_ulonglong2(max64(ex, x[2 * j]), max64(ex, x[2 * j + 1]));
  } else {
#pragma unroll
    for (int j = 0; j < kPmItems; ++j)
      if (b + j < n) out[b + j] = max64(ex, x[j]);
  }
}
int prefix_max(const uint64_t* in, const uint32_t* n_dev, uint64_t n_max, uint64_t* bmax,
               uint64_t* out, cudaStream_t s) {
  const uint64_t nb = ceil_div(n_max ? n_max : 1, kPmChunk);
  launch_dep(pmax_reduce, (unsigned)nb, kMaxScanThreads, 0, s, in, n_dev, bmax);
  const bool prefixed = nb > kScanFusedBlocks;
  if (prefixed) launch_dep(pmax_blocks, 1, 1024, 0, s, bmax, n_dev);
  launch_dep(pmax_apply, (unsigned)nb, kMaxScanThreads, 0, s, in, n_dev, (const uint64_t*)bmax,
             prefixed, out);
  return launch_result();
}
__global__ void reg_items(const db_range* q, uint64_t n_q, uint32_t gshift, const uint32_t* role,
                          const uint32_t* rpos, const uint32_t* creator_of, uint64_t* ce_in,
                          uint32_t* ck_in, uint32_t* cq_in) {
  kernel_prologue();
  FOR_EACH(k, n_q) {
    if (!flag_at(role, k)) continue;
    uint64_t b, e;
    widen(q, k, gshift, b, e);
    const uint32_t at = flag_pos(role, rpos, k);
    const uint32_t c = creator_of[k];
    ce_in[at] = e;
    ck_in[at] = c;                       // kNone unless k made a record
    cq_in[at] = c == kNone ? (uint32_t)k : kNone;
  }
}
// Every request's record and kind and, when the merged table fits out_cap,
// its handle (the record's place in that table: npos for a new record, remap
// for an old one; -1 for an invalid request or, on a table that breaks the
// order, an unresolved one) and the reference it adds there.
__global__ void reg_resolve(const db_range* q, uint64_t n_q, uint32_t gshift, const uint8_t* kind0,
                            const int32_t* idx, const uint32_t* role, const uint32_t* creator_of,
                            const uint32_t* held, const uint64_t* nstart, const uint64_t* start,
                            const uint32_t* npos, const int64_t* remap, uint64_t n_mr,
                            uint64_t o_cap, int64_t* handle, uint8_t* kind, uint32_t* o_refs,
                            RegHeader* h) {
  kernel_prologue();
  const bool fits = n_mr + h->u <= o_cap;
  // Two requests a thread at a time, their loads in phases (the request,
  // then its creator or holder, then that record's start and place), so
  // that both requests' dependent loads are in flight together.
  const uint64_t step = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t k0 = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; k0 < n_q; k0 += 2 * step) {
    uint64_t k[2] = {k0, k0 + step};
    uint8_t kd[2];
    uint32_t c[2], w[2];
    int32_t o[2];
    bool rl[2];
    uint64_t b[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      kd[u] = k[u] < n_q ? kind0[k[u]] : (uint8_t)DB_MR_INVALID;
      const bool valid = kd[u] != DB_MR_INVALID;
      const bool hit = kd[u] == DB_MR_EXACT || kd[u] == DB_MR_CONTAINED;
      c[u] = valid ? creator_of[k[u]] : kNone;
      rl[u] = valid && flag_at(role, k[u]);
      o[u] = hit ? idx[k[u]] : 0;
      w[u] = kNone;
      b[u] = 0;
      if (rl[u]) {
        uint64_t e;
        widen(q, k[u], gshift, b[u], e);
        w[u] = held[k[u]];  // the least-positioned new record reaching e, made before k
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if (k[u] >= n_q) continue;
      uint32_t rn = kNone;
      uint8_t k1 = kd[u];
      if (kd[u] != DB_MR_INVALID) {
        if (c[u] != kNone) {
          rn = c[u];
          k1 = DB_MR_NEW;
        } else if (rl[u]) {
          const bool holds = w[u] != kNone && nstart[w[u]] <= b[u];
          if (kd[u] == DB_MR_MISS) {
            if (holds) {
              rn = w[u];
              k1 = DB_MR_NEW_DUP;
            } else {
              atomicOr(&h->err, DB_ERR_TABLE_ORDER);  // cannot happen on a valid table
            }
          } else if (holds && nstart[w[u]] < start[o[u]]) {
            rn = w[u];  // the new record comes before the old one in the table
            k1 = DB_MR_NEW_DUP;
          }
        }
      }
      kind[k[u]] = k1;
      if (fits) {
        const int64_t pw = rn != kNone ? (int64_t)npos[rn]
                           : (kd[u] == DB_MR_EXACT || kd[u] == DB_MR_CONTAINED) ? remap[o[u]] : -1;
        handle[k[u]] = pw;
        if (pw >= 0) atomicAdd(&o_refs[pw], 1u);
      }
    }
  }
}
// No requests: the table is copied through.
__global__ void reg_copy(const uint64_t* start, const uint64_t* end, const uint32_t* lkey,
                         const uint32_t* refs, uint64_t n, uint64_t o_cap, uint64_t* o_start,
                         uint64_t* o_end, uint32_t* o_lkey, uint32_t* o_refs, int64_t* remap) {
  kernel_prologue();
  if (n > o_cap) return;
  FOR_EACH(i, n) {
    o_start[i] = start[i];
    o_end[i] = end[i];
    o_lkey[i] = lkey[i];
    o_refs[i] = refs[i];
    remap[i] = (int64_t)i;
  }
}
__global__ void reg_final(const RegHeader* h, uint64_t n, uint64_t o_cap, db_counters* ctr) {
  kernel_prologue();
  const uint64_t total = n + h->u;
  ctr->total = total;
  ctr->n_invalid = h->lookup.n_invalid;
  ctr->n_overflow = total > o_cap ? 1 : 0;
  ctr->err = h->lookup.err | h->err;
}

struct RegLayout {
  size_t lookup, hdr, idx, lk, kind0, flag, pos, key0, key1, val0, val1, counts, bsum,
      diff, de, nstart, nend, npos, first, cp, cb, creator_of, cend, pmax, bmax, reach,
      ce0, ce1, ck0, ck1, cq0, cq1, ca0, ca1, cpm_tile, cpm_tile1, cmin, cpm, cpm1, held, again,
      point, total;
};
RegLayout reg_layout(uint64_t n_q, uint64_t n_mr) {
  RegLayout L;
  const uint64_t q = n_q ? n_q : 1;
  size_t o = 0;
  auto take = [&](size_t bytes) { const size_t at = o; o += up256(bytes); return at; };
  L.lookup = take(mr::workspace_bytes(n_mr));
  L.hdr = take(sizeof(RegHeader));
  L.idx = take(q * 4);
  L.lk = take(q * 4);
  L.kind0 = take(q);
  L.flag = take(ceil_div(q, 32) * 4);  // flag words
  L.pos = take(ceil_div(q, 32) * 4);   // their exclusive prefix
  L.key0 = take(q * 8);
  L.key1 = take(q * 8);
  L.val0 = take(q * 4);
  L.val1 = take(q * 4);
  L.counts = take(sort_count_words(q) * 4);
  L.bsum = take(scan_tmp_words(sort_count_words(q) > q ? sort_count_words(q) : q) * 4);
  L.diff = take(8);
  L.de = take(q * 8);
  L.nstart = take(q * 8);
  L.nend = take(q * 8);
  L.npos = take(q * 4);
  L.first = take(q * 4);
  L.cp = take(q * 4);
  L.cb = take(q * 8);
  L.creator_of = take(q * 4);
  L.cend = take(q * 8);
  L.pmax = take(q * 8);
  L.bmax = take(ceil_div(q, kPmChunk) * 8);
  L.reach = take((n_mr ? n_mr : 1) * 8);
  L.ce0 = take(q * 8);
  L.ce1 = take(q * 8);
  L.ck0 = take(q * 4);
  L.ck1 = take(q * 4);
  L.cq0 = take(q * 4);
  L.cq1 = take(q * 4);
  L.ca0 = take(q * 4);
  L.ca1 = take(q * 4);
  L.cpm_tile = take(q * 4);
  L.cpm_tile1 = take(q * 4);
  L.cmin = take(cdq_tiles(q) * 4);
  L.cpm = take(cdq_tiles(q) * 4);
  L.cpm1 = take(cdq_tiles(q) * 4);
  L.held = take(q * 4);
  L.again = take(q);
  L.point = take(q);
  L.total = o;
  return L;
}

// ----------------------------------------------------------- deregistration
// A record's handles in batch order drop its references one by one: with c
// handles and R references, all of them drop one when c < R; otherwise the
// first R - 1 drop one, the R-th releases the record and the rest are stale
// ("IB Backend MR Cache": the MR goes at zero; an unknown handle is an
// error). Only a contested record (R >= 1, c >= R, c >= 2) needs its
// handles' order: they go into a bucket of the record's own (slots from an
// exclusive scan of the counts, in any order), and a handle's rank is the
// number of smaller handle indices in the bucket -- counted by the handle
// itself in a bucket of at most kSmallBucket, else compared with the
// record's releasing handle, found by a radix select over the bucket.
struct DeregHeader {
  uint32_t nbig;     // records with more than kSmallBucket handles
  uint32_t kept;     // records after the batch
  unsigned long long stale;
};
constexpr uint32_t kSmallBucket = 16;
constexpr int kSelectThreads = 256;
__device__ __forceinline__ uint64_t dereg_record(const int64_t* handle, uint64_t k, uint64_t n) {
  const int64_t x = handle[k];
  return (x >= 0 && (uint64_t)x < n) ? (uint64_t)x : n;  // n: no such record
}
__device__ __forceinline__ bool contested(uint32_t c, uint32_t R) {
  return R >= 1 && c >= R && c >= 2;
}
// Handles per record; the handle that counts a record's (kSmallBucket + 1)-th
// puts it on the list of large buckets (once per record).
__global__ void dereg_count(const int64_t* handle, uint64_t n_h, uint64_t n, uint32_t* cnt,
                            uint32_t* big, DeregHeader* h) {
  kernel_prologue();
  FOR_EACH(k, n_h) {
    const uint64_t r = dereg_record(handle, k, n);
    if (r < n && atomicAdd(&cnt[r], 1u) == kSmallBucket) big[atomicAdd(&h->nbig, 1u)] = (uint32_t)r;
  }
}
// cur[r] starts as the record's first bucket slot and ends one past its last.
__global__ void dereg_fill(const int64_t* handle, uint64_t n_h, uint64_t n, const uint32_t* cnt,
                           const uint32_t* refs, uint32_t* cur, uint32_t* bucket) {
  kernel_prologue();
  FOR_EACH(k, n_h) {
    const uint64_t r = dereg_record(handle, k, n);
    if (r < n && contested(cnt[r], refs[r])) bucket[atomicAdd(&cur[r], 1u)] = (uint32_t)k;
  }
}
// The releasing handle of each contested large bucket: its R-th smallest
// handle index, 8 bits at a time from the top (a CTA per record).
__global__ void __launch_bounds__(kSelectThreads) dereg_select(
    const DeregHeader* h, const uint32_t* big, const uint32_t* cnt, const uint32_t* refs,
    const uint32_t* cur, const uint32_t* bucket, uint32_t* rel) {
  kernel_prologue();
  __shared__ uint32_t hist[256];
  __shared__ uint32_t s_w[kSelectThreads / 32];
  __shared__ uint32_t s_digit, s_before;
  const uint32_t nbig = h->nbig;
  for (uint32_t b = blockIdx.x; b < nbig; b += gridDim.x) {
    const uint32_t r = big[b];
    const uint32_t c = cnt[r], R = refs[r];
    if (!contested(c, R)) continue;  // the same for the whole CTA
    const uint32_t* L = bucket + (cur[r] - c);
    uint32_t prefix = 0, want = R - 1;  // rank of the releaser among the handles left
    for (int shift = 24; shift >= 0; shift -= 8) {
      const uint32_t hi = shift == 24 ? 0u : (0xFFFFFFFFu << (shift + 8));
      hist[threadIdx.x] = 0;
      __syncthreads();
      for (uint32_t i = threadIdx.x; i < c; i += kSelectThreads) {
        const uint32_t x = L[i];
        if ((x & hi) == prefix) atomicAdd(&hist[(x >> shift) & 255u], 1u);
      }
      __syncthreads();
      const uint32_t v = hist[threadIdx.x];
      uint32_t ex, tot;
      block_excl_scan<kSelectThreads / 32>(v, ex, tot, s_w);
      if (ex <= want && want < ex + v) {  // exactly one digit
        s_digit = threadIdx.x;
        s_before = ex;
      }
      __syncthreads();
      prefix |= s_digit << shift;
      want -= s_before;
      __syncthreads();  // hist, s_w and s_digit are written again
    }
    if (threadIdx.x == 0) rel[r] = prefix;
  }
}
__global__ void dereg_status(const int64_t* handle, uint64_t n_h, uint64_t n, const uint32_t* cnt,
                             const uint32_t* refs, const uint32_t* cur, const uint32_t* bucket,
                             const uint32_t* rel, uint8_t* status, DeregHeader* h) {
  kernel_prologue();
  unsigned long long stale = 0;
  FOR_EACH(k, n_h) {
    const uint64_t r = dereg_record(handle, k, n);
    uint8_t st = DB_DEREG_STALE;
    if (r < n) {
      const uint32_t c = cnt[r], R = refs[r];
      if (c < R) {
        st = DB_DEREG_OK;
      } else if (R >= 1) {
        uint32_t rank = 0;  // handles of the record before this one
        if (c == 1) {
          rank = 0;
        } else if (c <= kSmallBucket) {
          const uint32_t* L = bucket + (cur[r] - c);
          for (uint32_t i = 0; i < c; ++i) rank += L[i] < (uint32_t)k;
        } else {
          const uint32_t x = rel[r];  // rank R - 1
          rank = (uint32_t)k < x ? 0u : (uint32_t)k == x ? R - 1 : R;
        }
        st = rank + 1 < R ? DB_DEREG_OK : rank + 1 == R ? DB_DEREG_RELEASED : DB_DEREG_STALE;
      }
    }
    stale += st == DB_DEREG_STALE;
    status[k] = st;
  }
  stale = warp_sum64(stale);
  if ((threadIdx.x & 31) == 0 && stale) atomicAdd(&h->stale, stale);
}
// A record survives when its handles leave a reference: c < R.
__global__ void dereg_keep(const uint32_t* refs, const uint32_t* cnt, uint64_t n, uint32_t* keep) {
  kernel_prologue();
  FOR_EACH_WARP(i0, n) {
    const uint64_t i = i0 + (threadIdx.x & 31);
    put_flags(keep, i0, i < n && refs[i] > cnt[i]);
  }
}
__global__ void dereg_place(const uint64_t* start, const uint64_t* end, const uint32_t* lkey,
                            const uint32_t* refs, const uint32_t* cnt, const uint32_t* keep,
                            const uint32_t* kpos, uint64_t n, uint64_t* o_start, uint64_t* o_end,
                            uint32_t* o_lkey, uint32_t* o_refs, int64_t* remap) {
  kernel_prologue();
  FOR_EACH(i, n) {
    if (!flag_at(keep, i)) {
      remap[i] = -1;
      continue;
    }
    const uint32_t w = flag_pos(keep, kpos, i);
    o_start[w] = start[i];
    o_end[w] = end[i];
    o_lkey[w] = lkey[i];
    o_refs[w] = refs[i] - cnt[i];
    remap[i] = w;
  }
}
__global__ void dereg_final(const DeregHeader* h, db_counters* ctr) {
  kernel_prologue();
  ctr->total = h->kept;
  ctr->n_invalid = h->stale;
  ctr->n_overflow = 0;
  ctr->err = 0;
}

struct DeregLayout {
  size_t hdr, cnt, cur, bucket, rel, big, bsum, keep, kpos, total;
};
DeregLayout dereg_layout(uint64_t n_h, uint64_t n_mr) {
  DeregLayout L;
  const uint64_t q = n_h ? n_h : 1, n = n_mr ? n_mr : 1;
  size_t o = 0;
  auto take = [&](size_t bytes) { const size_t at = o; o += up256(bytes); return at; };
  L.hdr = take(sizeof(DeregHeader));
  L.cnt = take(n * 4);
  L.cur = take(n * 4);
  L.bucket = take(q * 4);
  L.rel = take(n * 4);
  L.big = take(n * 4);
  L.bsum = take(scan_tmp_words(n) * 4);
  L.keep = take(ceil_div(n, 32) * 4);  // flag words
  L.kpos = take(ceil_div(n, 32) * 4);
  L.total = o;
  return L;
}

}  // namespace mrc
}  // namespace db

using namespace db;

extern "C" uint64_t db_mr_capacity_for(uint64_t n) {
  if (n == 0) return 0;
  uint64_t c = 32;
  while (c < n) c <<= 1;
  return c;
}

extern "C" int db_mr_register_workspace_size(uint64_t n_q, uint64_t n_mr, size_t* bytes) {
  if (!bytes || n_q >= mrc::kMaxItems || n_mr >= mrc::kMaxItems) return -EINVAL;
  *bytes = mrc::reg_layout(n_q, n_mr).total;
  return 0;
}

extern "C" int db_mr_register(const db_range* q, uint64_t n_q, const uint32_t* new_lkey,
                              uint32_t granule_shift, const uint64_t* start, const uint64_t* end,
                              const uint32_t* lkey, const uint32_t* refs, uint64_t n_mr,
                              uint64_t* out_start, uint64_t* out_end, uint32_t* out_lkey,
                              uint32_t* out_refs, uint64_t out_cap, int64_t* handle,
                              uint8_t* kind, int64_t* remap, db_counters* ctr, void* ws,
                              size_t ws_bytes, void* stream) {
  using namespace mrc;
  if (granule_shift != 12 && granule_shift != 16) return -EINVAL;
  if (n_q >= kMaxItems || n_mr >= kMaxItems || out_cap >= kMaxItems) return -EINVAL;
  if (!ws || !aligned(ws, 256) || (ctr && !aligned(ctr, 8))) return -EINVAL;
  if (n_q && (!q || !new_lkey || !handle || !kind || !aligned(q, 16) || !aligned(new_lkey, 4) ||
              !aligned(handle, 8)))
    return -EINVAL;
  if (n_mr && (!start || !end || !lkey || !refs || !remap || !aligned(start, 8) ||
               !aligned(end, 8) || !aligned(lkey, 4) || !aligned(refs, 4) || !aligned(remap, 8)))
    return -EINVAL;
  if (out_cap && (!out_start || !out_end || !out_lkey || !out_refs || !aligned(out_start, 8) ||
                  !aligned(out_end, 8) || !aligned(out_lkey, 4) || !aligned(out_refs, 4)))
    return -EINVAL;
  const RegLayout L = reg_layout(n_q, n_mr);
  if (ws_bytes < L.total) return -ENOSPC;
  cudaStream_t s = (cudaStream_t)stream;
  char* w = static_cast<char*>(ws);
  auto at = [&](size_t off) { return static_cast<void*>(w + off); };
  RegHeader* h = static_cast<RegHeader*>(at(L.hdr));
  int32_t* idx = static_cast<int32_t*>(at(L.idx));
  uint8_t* kind0 = static_cast<uint8_t*>(at(L.kind0));
  uint32_t* flag = static_cast<uint32_t*>(at(L.flag));
  uint32_t* pos = static_cast<uint32_t*>(at(L.pos));
  uint32_t* bsum = static_cast<uint32_t*>(at(L.bsum));
  SortBufs sb{{static_cast<uint64_t*>(at(L.key0)), static_cast<uint64_t*>(at(L.key1))},
              {static_cast<uint32_t*>(at(L.val0)), static_cast<uint32_t*>(at(L.val1))},
              static_cast<uint32_t*>(at(L.counts)), bsum, n_q,
              static_cast<unsigned long long*>(at(L.diff))};
  uint64_t* nstart = static_cast<uint64_t*>(at(L.nstart));
  uint64_t* nend = static_cast<uint64_t*>(at(L.nend));
  uint32_t* npos = static_cast<uint32_t*>(at(L.npos));

  int rc = 0;
  if (cudaMemsetAsync(h, 0, sizeof(RegHeader), s) != cudaSuccess ||
      (n_q && cudaMemsetAsync(at(L.creator_of), 0xFF, n_q * 4, s) != cudaSuccess))
    return launch_result();
  // 1. lookup against the table as it stands
  if (n_q) {
    rc = mr::lookup(q, n_q, start, end, lkey, n_mr, idx, static_cast<uint32_t*>(at(L.lk)), kind0,
                    &h->lookup, at(L.lookup), mr::workspace_bytes(n_mr), s, true,
                    (int)granule_shift);
    if (rc) return rc;
    // 2. the misses, compacted in request order
    launch_dep(reg_mark, grid_for(n_q), kThreads, 0, s, kind0, n_q, flag);
    if ((rc = launch_result())) return rc;
    if ((rc = scan_flags(flag, pos, n_q, &h->m, bsum, s))) return rc;
    launch_dep(reg_compact, grid_for(n_q), kThreads, 0, s, q, (const uint32_t*)flag,
               (const uint32_t*)pos, n_q, granule_shift, sb.key[0], sb.val[0], h);
    if ((rc = launch_result())) return rc;
    // 3. sort the misses by (start ascending, end descending), stable in
    //    request order: on the packed key, or on the end and then the start
    int cur = 0;
    launch_dep(reg_rekey, grid_for(n_q), kThreads, 0, s, q, (const RegHeader*)h, n_q,
               granule_shift, (const uint32_t*)sb.val[cur], sb.key[cur], true);
    if ((rc = launch_result())) return rc;
    if ((rc = radix_sort(sb, cur, &h->m, 64, true, s))) return rc;
    launch_dep(reg_rekey, grid_for(n_q), kThreads, 0, s, q, (const RegHeader*)h, n_q,
               granule_shift, (const uint32_t*)sb.val[cur], sb.key[cur], false);
    if ((rc = launch_result())) return rc;
    // 64 bits: an even number of passes, so a sort that does not run leaves
    // the items where the host expects them (no move back)
    if ((rc = radix_sort(sb, cur, &h->m, 64, true, s, &h->wide))) return rc;
    // 4. distinct ranges; a range makes a record when no range that holds it
    //    (one before it in this order reaching its end) was asked for earlier
    const uint32_t* sval = sb.val[cur];
    const uint64_t* skey = sb.key[cur];
    uint64_t* db = sb.key[cur ^ 1];  // free once sorted
    uint64_t* de = static_cast<uint64_t*>(at(L.de));
    uint32_t* first = static_cast<uint32_t*>(at(L.first));
    uint32_t* held = static_cast<uint32_t*>(at(L.held));
    CdqBufs cb_{{static_cast<uint64_t*>(at(L.ce0)), static_cast<uint64_t*>(at(L.ce1))},
                {static_cast<uint32_t*>(at(L.ck0)), static_cast<uint32_t*>(at(L.ck1))},
                {static_cast<uint32_t*>(at(L.cq0)), static_cast<uint32_t*>(at(L.cq1))},
                {static_cast<uint32_t*>(at(L.ca0)), static_cast<uint32_t*>(at(L.ca1))},
                {static_cast<uint32_t*>(at(L.cpm_tile)), static_cast<uint32_t*>(at(L.cpm_tile1))},
                static_cast<uint32_t*>(at(L.cmin)),
                {static_cast<uint32_t*>(at(L.cpm)), static_cast<uint32_t*>(at(L.cpm1))}, n_q,
                &h->err};
    launch_dep(reg_runs, grid_for(n_q), kThreads, 0, s, q, (const RegHeader*)h, granule_shift,
               sval, skey, flag);
    if ((rc = launch_result())) return rc;
    if ((rc = scan_flags(flag, pos, n_q, &h->d, bsum, s, &h->m))) return rc;
    uint8_t* again = static_cast<uint8_t*>(at(L.again));
    uint8_t* point = static_cast<uint8_t*>(at(L.point));
    launch_dep(reg_distinct, grid_for(n_q), kThreads, 0, s, q, (const RegHeader*)h, n_q,
               granule_shift, sval, skey, (const uint32_t*)flag, (const uint32_t*)pos, db, de,
               first, again);
    if ((rc = launch_result())) return rc;
    uint64_t* pmax = static_cast<uint64_t*>(at(L.pmax));
    uint64_t* bmax = static_cast<uint64_t*>(at(L.bmax));
    if ((rc = prefix_max(de, &h->d, n_q, bmax, pmax, s))) return rc;
    launch_dep(reg_keep_a, grid_for(n_q), kThreads, 0, s, (const RegHeader*)h,
               (const uint64_t*)db, (const uint64_t*)de, (const uint64_t*)pmax, held, flag);
    if ((rc = launch_result())) return rc;
    if ((rc = scan_flags(flag, pos, n_q, &h->dk, bsum, s, &h->d))) return rc;
    launch_dep(reg_items_a, grid_for(n_q), kThreads, 0, s, (const RegHeader*)h, n_q,
               (const uint32_t*)flag, (const uint32_t*)pos, (const uint64_t*)de,
               (const uint32_t*)first, cb_.e[1], cb_.key[1], cb_.qid[1]);
    if ((rc = launch_result())) return rc;
    if ((rc = cdq_dominance_min(cb_.e[1], cb_.key[1], cb_.qid[1], &h->dk, cb_, held, s)))
      return rc;
    launch_dep(reg_creators, grid_for(n_q), kThreads, 0, s, (const RegHeader*)h,
               (const uint32_t*)first, (const uint32_t*)held, flag);
    if ((rc = launch_result())) return rc;
    if ((rc = scan_flags(flag, pos, n_q, &h->u, bsum, s, &h->d))) return rc;
    uint32_t* cp = static_cast<uint32_t*>(at(L.cp));
    uint64_t* cbs = static_cast<uint64_t*>(at(L.cb));
    uint32_t* creator_of = static_cast<uint32_t*>(at(L.creator_of));
    uint64_t* cend = static_cast<uint64_t*>(at(L.cend));
    uint64_t* reach = static_cast<uint64_t*>(at(L.reach));
    launch_dep(reg_clist, grid_for(n_q), kThreads, 0, s, h, n_q, flag, pos, db, cp, cbs);
    if ((rc = launch_result())) return rc;
    // 5. the new records in table order, and both kinds of record in the
    //    merged table; old records a new one may precede
    launch_dep(reg_cplace, grid_for(n_q), kThreads, 0, s, h, n_q, cp, cbs, db, de, first,
               (const uint8_t*)again, start, n_mr, new_lkey, out_cap, nstart, nend, creator_of,
               cend, point, npos, out_start, out_end, out_lkey, out_refs);
    if ((rc = launch_result())) return rc;
    if ((rc = prefix_max(cend, &h->u, n_q, bmax, pmax, s))) return rc;
    if (n_mr) {
      launch_dep(reg_reach, grid_for(n_mr), kThreads, 0, s, (const RegHeader*)h,
                 (const uint64_t*)cbs, (const uint64_t*)pmax, start, end, lkey, refs, n_mr,
                 out_cap, reach, remap, out_start, out_end, out_lkey, out_refs);
      if ((rc = launch_result())) return rc;
    }
    // 6. every request's record: the lowest-positioned one holding it when
    //    it is made (an old one, or a new one made before it)
    launch_dep(reg_roles, grid_for(n_q), kThreads, 0, s, q, n_q, granule_shift, kind0, idx,
               (const uint64_t*)reach, (const uint32_t*)creator_of, (const uint8_t*)point, flag);
    if ((rc = launch_result())) return rc;
    if ((rc = scan_flags(flag, pos, n_q, &h->nb, bsum, s))) return rc;
    launch_dep(reg_items, grid_for(n_q), kThreads, 0, s, q, n_q, granule_shift, flag, pos,
               creator_of, cb_.e[1], cb_.key[1], cb_.qid[1]);
    if ((rc = launch_result())) return rc;
    if ((rc = cdq_dominance_min(cb_.e[1], cb_.key[1], cb_.qid[1], &h->nb, cb_, held, s)))
      return rc;
    // 7. every request's kind, handle and reference
    launch_dep(reg_resolve, grid_for(n_q), kThreads, 0, s, q, n_q, granule_shift, kind0, idx,
               flag, creator_of, held, nstart, start, (const uint32_t*)npos,
               (const int64_t*)remap, n_mr, out_cap, handle, kind, out_refs, h);
    if ((rc = launch_result())) return rc;
  } else if (n_mr) {
    // no requests: the table is copied through (and checked like a lookup would)
    rc = mr::lookup(nullptr, 0, start, end, lkey, n_mr, nullptr, nullptr, nullptr, &h->lookup,
                    at(L.lookup), mr::workspace_bytes(n_mr), s, true, (int)granule_shift);
    if (rc) return rc;
    launch_dep(reg_copy, grid_for(n_mr), kThreads, 0, s, start, end, lkey, refs, n_mr, out_cap,
               out_start, out_end, out_lkey, out_refs, remap);
    if ((rc = launch_result())) return rc;
  }
  if (ctr) {
    launch_dep(reg_final, 1, 1, 0, s, h, n_mr, out_cap, ctr);
    return launch_result();
  }
  return 0;
}

extern "C" int db_mr_deregister_workspace_size(uint64_t n_h, uint64_t n_mr, size_t* bytes) {
  if (!bytes || n_h >= mrc::kMaxItems || n_mr >= mrc::kMaxItems) return -EINVAL;
  *bytes = mrc::dereg_layout(n_h, n_mr).total;
  return 0;
}

extern "C" int db_mr_deregister(const int64_t* handle, uint64_t n_h, const uint64_t* start,
                                const uint64_t* end, const uint32_t* lkey, const uint32_t* refs,
                                uint64_t n_mr, uint64_t* out_start, uint64_t* out_end,
                                uint32_t* out_lkey, uint32_t* out_refs, int64_t* remap,
                                uint8_t* status, db_counters* ctr, void* ws, size_t ws_bytes,
                                void* stream) {
  using namespace mrc;
  if (n_h >= kMaxItems || n_mr >= kMaxItems) return -EINVAL;
  if (!ws || !aligned(ws, 256) || (ctr && !aligned(ctr, 8))) return -EINVAL;
  if (n_h && (!handle || !status || !aligned(handle, 8))) return -EINVAL;
  if (n_mr && (!start || !end || !lkey || !refs || !remap || !out_start || !out_end ||
               !out_lkey || !out_refs || !aligned(start, 8) || !aligned(end, 8) ||
               !aligned(lkey, 4) || !aligned(refs, 4) || !aligned(remap, 8) ||
               !aligned(out_start, 8) || !aligned(out_end, 8) || !aligned(out_lkey, 4) ||
               !aligned(out_refs, 4)))
    return -EINVAL;
  const DeregLayout L = dereg_layout(n_h, n_mr);
  if (ws_bytes < L.total) return -ENOSPC;
  cudaStream_t s = (cudaStream_t)stream;
  char* w = static_cast<char*>(ws);
  auto at = [&](size_t off) { return static_cast<void*>(w + off); };
  DeregHeader* h = static_cast<DeregHeader*>(at(L.hdr));
  uint32_t* bsum = static_cast<uint32_t*>(at(L.bsum));
  uint32_t* cnt = static_cast<uint32_t*>(at(L.cnt));
  uint32_t* cur = static_cast<uint32_t*>(at(L.cur));
  uint32_t* bucket = static_cast<uint32_t*>(at(L.bucket));
  uint32_t* rel = static_cast<uint32_t*>(at(L.rel));
  uint32_t* big = static_cast<uint32_t*>(at(L.big));
  uint32_t* keep = static_cast<uint32_t*>(at(L.keep));
  uint32_t* kpos = static_cast<uint32_t*>(at(L.kpos));
  if (cudaMemsetAsync(h, 0, sizeof(DeregHeader), s) != cudaSuccess ||
      (n_mr && cudaMemsetAsync(cnt, 0, n_mr * 4, s) != cudaSuccess))
    return launch_result();
  int rc = 0;
  if (n_h) {
    launch_dep(dereg_count, grid_for(n_h), kThreads, 0, s, handle, n_h, n_mr, cnt, big, h);
    if ((rc = launch_result())) return rc;
    if (n_mr) {
      if ((rc = scan(cnt, cur, n_mr, nullptr, bsum, s))) return rc;
      launch_dep(dereg_fill, grid_for(n_h), kThreads, 0, s, handle, n_h, n_mr,
                 (const uint32_t*)cnt, refs, cur, bucket);
      if ((rc = launch_result())) return rc;
      uint64_t sel = n_h / (kSmallBucket + 1);  // at most this many large buckets
      const uint64_t cap = (uint64_t)num_sms() * 4;
      sel = sel < 1 ? 1 : sel > cap ? cap : sel;
      launch_dep(dereg_select, (unsigned)sel, kSelectThreads, 0, s, (const DeregHeader*)h,
                 (const uint32_t*)big, (const uint32_t*)cnt, refs, (const uint32_t*)cur,
                 (const uint32_t*)bucket, rel);
      if ((rc = launch_result())) return rc;
    }
    launch_dep(dereg_status, grid_for(n_h), kThreads, 0, s, handle, n_h, n_mr,
               (const uint32_t*)cnt, refs, (const uint32_t*)cur, (const uint32_t*)bucket,
               (const uint32_t*)rel, status, h);
    if ((rc = launch_result())) return rc;
  }
  if (n_mr) {
    launch_dep(dereg_keep, grid_for(n_mr), kThreads, 0, s, refs, (const uint32_t*)cnt, n_mr, keep);
    if ((rc = launch_result())) return rc;
    if ((rc = scan_flags(keep, kpos, n_mr, &h->kept, bsum, s))) return rc;
    launch_dep(dereg_place, grid_for(n_mr), kThreads, 0, s,
               start, end, lkey, refs, (const uint32_t*)cnt, keep, kpos, n_mr,
               out_start, out_end, out_lkey, out_refs, remap);
    if ((rc = launch_result())) return rc;
  }
  if (ctr) {
    launch_dep(dereg_final, 1, 1, 0, s, h, ctr);
    return launch_result();
  }
  return 0;
}
