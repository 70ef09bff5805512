// Device helpers shared by the descriptor-building kernels (sm_103a).
//
// - 16-byte vector loads/stores with L2 eviction hints (inline PTX)
// - status words for single-pass decoupled-lookback scans, tagged by a
//   ticket "lap" so that the status ring never needs clearing
// - a bounded wait: every spin gives up after kWaitLimitNs of %globaltimer,
//   sets DB_ERR_TIMEOUT and lets the kernel finish
// - the "last CTA" hand-off that returns a workspace header to its
//   between-calls state
#pragma once

#include <cerrno>
#include <cstdint>
#include <cuda_runtime.h>

#include "descbuild.h"

namespace db {

constexpr unsigned kFull = 0xFFFFFFFFu;

// ----------------------------------------------------------------- memory ops
// L2 eviction-priority policies (createpolicy has no inputs, so the compiler
// may hoist it out of loops).
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t pol;
  asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t pol;
  asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Streaming 16-byte load of data read once: no L1 allocation, L2 hint `pol`.
__device__ __forceinline__ ulonglong2 ld_stream16(const void* p, uint64_t pol) {
  ulonglong2 v;
  asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v2.u64 {%0, %1}, [%2], %3;"
      : "=l"(v.x), "=l"(v.y)
      : "l"(p), "l"(pol));
  return v;
}

// Read-only loads of tables reused across CTAs (L1 allowed, L2 hint `pol`).
__device__ __forceinline__ uint64_t ld_table8(const uint64_t* p, uint64_t pol) {
  uint64_t v;
  asm("ld.global.nc.L2::cache_hint.u64 %0, [%1], %2;" : "=l"(v) : "l"(p), "l"(pol));
  return v;
}
__device__ __forceinline__ ulonglong2 ld_table16(const void* p, uint64_t pol) {
  ulonglong2 v;
  asm("ld.global.nc.L2::cache_hint.v2.u64 {%0, %1}, [%2], %3;"
      : "=l"(v.x), "=l"(v.y)
      : "l"(p), "l"(pol));
  return v;
}
__device__ __forceinline__ uint32_t ld_table4(const uint32_t* p, uint64_t pol) {
  uint32_t v;
  asm("ld.global.nc.L2::cache_hint.u32 %0, [%1], %2;" : "=r"(v) : "l"(p), "l"(pol));
  return v;
}

// Output stores this kernel never reads back. DB_STORE_HINT 1: no L1
// allocation and the L2 policy `pol`; 0: plain stores (`pol` unused).
#ifndef DB_STORE_HINT
#define DB_STORE_HINT 1
#endif
__device__ __forceinline__ void st_stream16(void* p, uint64_t a, uint64_t b, uint64_t pol) {
  if (DB_STORE_HINT)
    asm volatile("st.global.L1::no_allocate.L2::cache_hint.v2.u64 [%0], {%1, %2}, %3;" ::"l"(p),
                 "l"(a), "l"(b), "l"(pol)
                 : "memory");
  else
    asm volatile("st.global.v2.u64 [%0], {%1, %2};" ::"l"(p), "l"(a), "l"(b) : "memory");
}
// 32-byte store (sm_100+): p must be 32-byte aligned.
__device__ __forceinline__ void st_stream32(void* p, uint64_t a, uint64_t b, uint64_t c, uint64_t d,
                                            uint64_t pol) {
  if (DB_STORE_HINT)
    asm volatile("st.global.L1::no_allocate.L2::cache_hint.v4.u64 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p),
                 "l"(a), "l"(b), "l"(c), "l"(d), "l"(pol)
                 : "memory");
  else
    asm volatile("st.global.v4.u64 [%0], {%1, %2, %3, %4};" ::"l"(p), "l"(a), "l"(b), "l"(c),
                 "l"(d)
                 : "memory");
}
// 32-byte read-only load (sm_100+): p must be 32-byte aligned.
__device__ __forceinline__ void ld_table32(const void* p, uint64_t pol, uint64_t& a, uint64_t& b,
                                           uint64_t& c, uint64_t& d) {
  asm("ld.global.nc.L2::cache_hint.v4.u64 {%0, %1, %2, %3}, [%4], %5;"
      : "=l"(a), "=l"(b), "=l"(c), "=l"(d)
      : "l"(p), "l"(pol));
}
__device__ __forceinline__ void st_stream8(void* p, uint64_t a, uint64_t pol) {
  if (DB_STORE_HINT)
    asm volatile("st.global.L1::no_allocate.L2::cache_hint.u64 [%0], %1, %2;" ::"l"(p), "l"(a),
                 "l"(pol)
                 : "memory");
  else
    asm volatile("st.global.u64 [%0], %1;" ::"l"(p), "l"(a) : "memory");
}

// Tile status words. The flag and the value travel in one aligned 64-bit
// word, so a reader that sees the flag sees its value, and no other memory
// is published through the word: relaxed (not acquire / release) ordering is
// enough, and it lets a lane's four lookback loads be in flight together.
__device__ __forceinline__ uint64_t ld_relaxed(const unsigned long long* p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_relaxed(unsigned long long* p, uint64_t v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// ------------------------------------------------------------ lookback status
// Status word of one tile and one value: [63:62] flag, [61:40] epoch tag,
// [39:0] value. Tile t of a call owns word t (times the values per tile) of
// the workspace's status array; the tag is the call's epoch (a counter in the
// workspace header that the last CTA of every call advances), so words left
// over from earlier calls read as "not yet published" and the array never
// needs clearing -- except when the 22-bit tag wraps, where the last CTA
// clears the words used so far before the tag can repeat.
enum : uint32_t { kEmpty = 0, kAggregate = 1, kPrefix = 2, kFailed = 3 };

constexpr uint64_t kValueMask = (1ull << 40) - 1;
constexpr uint32_t kEpochMask = (1u << 22) - 1;
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s: a wait this long means no progress

__device__ __forceinline__ uint64_t status_word(uint32_t flag, uint32_t epoch, uint64_t value) {
  return ((uint64_t)flag << 62) | ((uint64_t)(epoch & kEpochMask) << 40) | (value & kValueMask);
}

__device__ __forceinline__ uint32_t status_flag(uint64_t w, uint32_t epoch) {
  if ((uint32_t)((w >> 40) & kEpochMask) != (epoch & kEpochMask)) return kEmpty;
  return (uint32_t)(w >> 62);
}

// Header shared by the workspaces of the scanning kernels (first 256 bytes).
// The status words live in their own region of the workspace, at a fixed
// offset, and nothing else is ever written there.
struct ScanHeader {
  unsigned long long ticket;    // next tile of the current call (0 between calls)
  unsigned int done;            // CTAs finished in the current call
  unsigned int err;             // DB_ERR_* seen in the current call
  unsigned int epoch;           // tag of the current call's status words
  unsigned int aux;             // kAuxFailed / kAuxClearPending
  unsigned long long hw_words;  // most status words any call has used
  unsigned long long acc[5];    // per-kernel accumulators, zero between calls (the PRP
                                // build keeps in acc[4] the epoch of the last call its
                                // pair kernel completed)
};
constexpr size_t kScanHeaderBytes = 256;
constexpr unsigned int kAuxFailed = 1u;        // the first pass of a call failed
constexpr unsigned int kAuxClearPending = 2u;  // status words still to clear (tag wrapped)

// Clear the status words used so far (every thread of one CTA).
__device__ __forceinline__ void clear_status(ScanHeader* h, unsigned long long* status,
                                             uint64_t cap_words) {
  const uint64_t words = h->hw_words < cap_words ? h->hw_words : cap_words;
  for (uint64_t x = threadIdx.x; x < words; x += blockDim.x) status[x] = 0;
}

// Run by every thread of the last CTA to finish, after all other CTAs of the
// call are done: advance the epoch and return the ticket to 0. When the
// epoch tag wraps, the status words used so far are cleared now, or -- when
// a later kernel of the same call still reads them (clear_now false) -- the
// clear is left pending for that kernel.
__device__ __forceinline__ void end_of_call(ScanHeader* h, unsigned long long* status,
                                            uint64_t used_words, uint64_t cap_words,
                                            bool clear_now) {
  __shared__ unsigned int s_wrap;
  if (threadIdx.x == 0) {
    const unsigned long long hw = h->hw_words > used_words ? h->hw_words : used_words;
    const unsigned int next = h->epoch + 1;
    s_wrap = (next & kEpochMask) == 0;
    h->hw_words = hw;
    h->epoch = next;
    h->ticket = 0;
    h->done = 0;
    if (s_wrap && !clear_now) h->aux |= kAuxClearPending;
  }
  __syncthreads();
  if (s_wrap && clear_now) clear_status(h, status, cap_words);
  __threadfence();
}

// Backoff for a bounded spin: sleeps doubling from 32 ns up to
// DB_BACKOFF_MAX_NS. Returns false once the wait has lasted kWaitLimitNs.
#ifndef DB_BACKOFF_MAX_NS
#define DB_BACKOFF_MAX_NS 2048
#endif
struct Backoff {
  uint64_t t0;
  uint32_t ns;
  __device__ __forceinline__ Backoff() : t0(globaltimer_ns()), ns(32) {}
  __device__ __forceinline__ bool wait() {
    if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
    __nanosleep(ns);
    if (ns < DB_BACKOFF_MAX_NS) ns <<= 1;
    return true;
  }
};

// ------------------------------------------------------------------ reductions
__device__ __forceinline__ uint64_t warp_sum64(uint64_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

__device__ __forceinline__ uint32_t warp_sum32(uint32_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

// Block-wide exclusive scan of one u32 per thread. `s_warp` holds kWarps u32.
// Ends with every thread past a barrier that follows the last write of s_warp.
template <int kWarps>
__device__ __forceinline__ void block_excl_scan(uint32_t v, uint32_t& excl, uint32_t& total,
                                                uint32_t* s_warp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t y = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = lane < kWarps ? s_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      uint32_t y = __shfl_up_sync(kFull, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kWarps) s_warp[lane] = w;
  }
  __syncthreads();
  excl = (warp ? s_warp[warp - 1] : 0u) + x - v;
  total = s_warp[kWarps - 1];
}

// The same scan on 64-bit values.
template <int kWarps>
__device__ __forceinline__ void block_excl_scan64(uint64_t v, uint64_t& excl, uint64_t& total,
                                                  uint64_t* s_warp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint64_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint64_t y = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint64_t w = lane < kWarps ? s_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      uint64_t y = __shfl_up_sync(kFull, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kWarps) s_warp[lane] = w;
  }
  __syncthreads();
  excl = (warp ? s_warp[warp - 1] : 0ull) + x - v;
  total = s_warp[kWarps - 1];
}

// ----------------------------------------------------------- host-side checks
inline bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

// Record and map a CUDA error from the most recent launch.
int launch_result();
// Record a failed CUDA runtime call and return -EIO.
int cuda_failure(cudaError_t e);
int num_sms();

// Programmatic dependent launch: the kernel may start once every CTA of the
// kernel before it on `s` has started (or that kernel has ended), and must
// execute `griddepcontrol.wait` before it reads what that kernel writes.
// Every kernel launched this way waits before it exits, so the kernels after
// it still see the whole stream before them complete.
template <typename P>
inline int launch_dependent(void (*kernel)(P), unsigned grid, unsigned block, size_t smem,
                            cudaStream_t s, const P& params) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, params);
  if (e != cudaSuccess) return cuda_failure(e);
  return launch_result();
}
// The same for kernels of any signature, as a statement: a failed launch is
// left for launch_result() like one made with <<< >>>.
template <typename... K, typename... A>
inline void launch_dep(void (*kernel)(K...), unsigned grid, unsigned block, size_t smem,
                       cudaStream_t s, A&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  (void)cudaLaunchKernelEx(&cfg, kernel, static_cast<A&&>(args)...);
}
__device__ __forceinline__ void dependents_may_launch() {
  asm volatile("griddepcontrol.launch_dependents;");
}
__device__ __forceinline__ void wait_for_prerequisites() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace db
