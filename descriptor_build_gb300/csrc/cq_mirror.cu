// Completion-queue mirror (sm_103a).
//
// Source: xNVMe "uPCIe CUDA" backend page, "Completions in device memory"
// (completion queues kept in device memory, forwarded to the host CQ by a
// GPU kernel). Here: one warp per queue forwards each entry whose phase tag
// has turned; a per-queue slot holds the two CQ addresses, the depth, a
// generation (odd while attached) and an acknowledgement.
//
// One CTA of one warp per slot. Each pass of a warp's loop:
//   1. every kCheckNs: the stop flag, the time limit (the launch never
//      outlives limit_ns) and the slot's generation (acquire, system
//      scope), all in host memory. A generation change ends the current
//      queue (acknowledge the odd value worked under) and takes up the new
//      one; with no queue taken up, an even value g > 0 gets ack = g - 1. Between
//      checks a pass touches only device memory, except for its copies;
//   2. lane l reads the phase dword of entry head + l (a window of up to 32
//      entries); the run of leading lanes whose tag is the expected one is
//      copied: after a fence each of those lanes reads its whole entry,
//      writes dwords 0..2 to the host CQ and then dword 3 with a
//      system-scope release store, so the host sees the body before the tag;
//   3. head and phase advance and are published in the slot, so a later
//      launch resumes from them.
// An idle warp sleeps with a growing backoff (32 .. 256 ns); a warp with no
// queue sleeps 1 us.
#include <cerrno>
#include <ctime>

#include "common.cuh"
#include "cqmirror.h"

namespace db {
namespace cq {

static_assert(sizeof(db_cq_slot) == 64, "a slot is 64 bytes");

constexpr uint32_t kPhaseBit = 1u << 16;
constexpr uint64_t kCheckNs = 8000;  // host-memory flags read at most this often
constexpr uint32_t kIdleMaxNs = 256;

__device__ __forceinline__ uint32_t ld_acquire_sys(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.sys.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t ld_volatile32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.volatile.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint64_t ld_volatile64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.volatile.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint4 ld_volatile128(const uint32_t* p) {
  uint4 v;
  asm volatile("ld.volatile.global.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}
__device__ __forceinline__ void st_volatile32(uint32_t* p, uint32_t v) {
  asm volatile("st.volatile.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void st_volatile64(uint64_t* p, uint64_t v) {
  asm volatile("st.volatile.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void st_body(uint32_t* p, uint32_t a, uint32_t b, uint32_t c) {
  asm volatile("st.volatile.global.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(a), "r"(b) : "memory");
  asm volatile("st.volatile.global.u32 [%0], %1;" ::"l"(p + 2), "r"(c) : "memory");
}
__device__ __forceinline__ void st_release_sys(uint32_t* p, uint32_t v) {
  asm volatile("st.release.sys.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

struct Params {
  db_cq_slot* slots;
  const uint32_t* stop;
  uint64_t limit_ns;
  db_counters* ctr;
};

// A queue's fields as the kernel takes them up; `ok` is false for a slot
// that db_cq_attach would have refused.
struct Queue {
  const uint32_t* dev;
  uint32_t* host;
  uint32_t depth;
  bool ok;
  bool timed;
};

__device__ __forceinline__ Queue read_queue(db_cq_slot* s) {
  Queue q;
  const uint64_t d = ld_volatile64(&s->dev_cq), h = ld_volatile64(&s->host_cq);
  q.depth = ld_volatile32(&s->depth);
  q.timed = (ld_volatile32(&s->flags) & DB_CQ_TIMED) != 0;
  q.ok = d && h && !(d & 15) && !(h & 15) && q.depth >= 2 && q.depth <= DB_CQ_MAX_DEPTH;
  q.dev = reinterpret_cast<const uint32_t*>(d);
  q.host = reinterpret_cast<uint32_t*>(h);
  return q;
}

__global__ void __launch_bounds__(32) cq_mirror_kernel(const Params p) {
  db_cq_slot* s = p.slots + blockIdx.x;
  const uint32_t lane = threadIdx.x;
  const uint64_t deadline = __shfl_sync(kFull, globaltimer_ns(), 0) + p.limit_ns;

  uint32_t cur = 0;          // the generation last taken up (0: none yet)
  bool active = false;       // cur is odd and its queue is being served
  Queue q{nullptr, nullptr, 0, false, false};
  uint32_t head = 0, phase = 1;
  uint64_t copied_gen = 0, copied_launch = 0;
  uint32_t last_ack = lane == 0 ? ld_volatile32(&s->ack) : 0;
  bool timed_out = false, bad = false;
  uint32_t idle_ns = 32;
  uint64_t next_check = 0;  // lane 0's clock

  for (;;) {
    // 1. stop, limit and generation, every kCheckNs
    uint32_t go = 0, g = cur;
    if (lane == 0) {
      const uint64_t now = globaltimer_ns();
      if (now >= next_check) {
        next_check = now + kCheckNs;
        if (ld_volatile32(p.stop) != 0) go = 1;
        else if (now >= deadline) go = 2;
        else g = ld_acquire_sys(&s->generation);
      }
    }
    go = __shfl_sync(kFull, go, 0);
    if (go) {
      timed_out = go == 2;
      break;
    }
    g = __shfl_sync(kFull, g, 0);
    if (g != cur) {
      if (lane == 0) {
        uint32_t ack = last_ack;
        if ((cur & 1u) && g != cur) ack = cur;            // done with the one worked under
        else if (!(g & 1u) && g > 0) ack = g - 1;         // detached before it was taken up
        if (ack != last_ack) {
          __threadfence_system();  // host CQ writes and progress before the acknowledgement
          st_release_sys(&s->ack, ack);
          last_ack = ack;
        }
      }
      cur = g;
      active = false;
      if (g & 1u) {
        uint32_t ok = 0, h = 0, ph = 1;
        uint64_t c = 0;
        if (lane == 0) {
          q = read_queue(s);
          ok = q.ok;
          if (q.ok) {
            if (ld_volatile32(&s->seen) == g) {  // resume where a previous launch stopped
              h = ld_volatile32(&s->head);
              ph = ld_volatile32(&s->phase) & 1u;
              c = ld_volatile64(&s->copied);
              if (h >= q.depth) h = 0;
            } else {
              st_volatile32(&s->head, 0);
              st_volatile32(&s->phase, 1);
              st_volatile64(&s->copied, 0);
              __threadfence_system();
              st_volatile32(&s->seen, g);
            }
          }
        }
        ok = __shfl_sync(kFull, ok, 0);
        if (ok) {
          q.dev = reinterpret_cast<const uint32_t*>(
              __shfl_sync(kFull, reinterpret_cast<uintptr_t>(q.dev), 0));
          q.host = reinterpret_cast<uint32_t*>(
              __shfl_sync(kFull, reinterpret_cast<uintptr_t>(q.host), 0));
          q.depth = __shfl_sync(kFull, q.depth, 0);
          q.timed = __shfl_sync(kFull, q.timed ? 1 : 0, 0) != 0;
          head = __shfl_sync(kFull, h, 0);
          phase = __shfl_sync(kFull, ph, 0);
          copied_gen = __shfl_sync(kFull, c, 0);
          active = true;
          idle_ns = 32;
        } else {
          bad = true;
        }
      }
      continue;
    }
    if (!active) {
      __nanosleep(1000);
      continue;
    }
    // 2. the window of entries after head
    const uint32_t win = q.depth < 32 ? q.depth : 32;
    uint32_t pos = head + lane, expect = phase;
    if (pos >= q.depth) {
      pos -= q.depth;
      expect ^= 1u;
    }
    bool fresh = false;
    if (lane < win) fresh = ((ld_volatile32(q.dev + 4ull * pos + 3) & kPhaseBit) != 0) == (expect != 0);
    const uint32_t mask = __ballot_sync(kFull, fresh);
    const uint32_t run = (~mask == 0) ? 32u : (uint32_t)(__ffs(~mask) - 1);
    if (run == 0) {
      __nanosleep(idle_ns);
      idle_ns = idle_ns < kIdleMaxNs ? idle_ns * 2 : kIdleMaxNs;
      continue;
    }
    idle_ns = 32;
    const uint64_t t_seen = q.timed ? globaltimer_ns() : 0;  // the batch's tags are in
    __threadfence();  // the tags seen above before the bodies read below
    if (lane < run) {
      const uint4 e = ld_volatile128(q.dev + 4ull * pos);
      uint32_t* dst = q.host + 4ull * pos;
      st_body(dst, e.x, e.y, e.z);
      st_release_sys(dst + 3, e.w);
      if (q.timed) asm volatile("fence.sc.sys;" ::: "memory");  // this lane's writes performed
    }
    // 3. advance and publish
    head += run;
    if (head >= q.depth) {
      head -= q.depth;
      phase ^= 1u;
    }
    copied_gen += run;
    copied_launch += run;
    __syncwarp();
    if (lane == 0) {
      if (q.timed) {
        const uint64_t dt = globaltimer_ns() - t_seen;
        st_volatile32(&s->lat_ns, dt < 0xFFFFFFFFull ? (uint32_t)dt : 0xFFFFFFFFu);
        asm volatile("st.release.sys.global.u64 [%0], %1;" ::"l"(&s->lat_seq), "l"(copied_gen)
                     : "memory");
      }
      st_volatile32(&s->head, head);
      st_volatile32(&s->phase, phase);
      st_volatile64(&s->copied, copied_gen);
    }
  }
  if (lane == 0 && p.ctr) {
    if (copied_launch) atomicAdd(reinterpret_cast<unsigned long long*>(&p.ctr->total),
                                 (unsigned long long)copied_launch);
    if (bad) atomicAdd(reinterpret_cast<unsigned long long*>(&p.ctr->n_invalid), 1ull);
    if (timed_out) atomicOr(reinterpret_cast<unsigned long long*>(&p.ctr->err),
                            (unsigned long long)DB_ERR_TIMEOUT);
  }
  __threadfence_system();
}

// Host-side pointer kinds: pinned host memory, or device memory.
int pointer_kind(const void* p, cudaMemoryType* kind) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return -ENODEV;
  }
  *kind = a.type;
  return 0;
}
int require(const void* p, cudaMemoryType want) {
  cudaMemoryType k;
  const int rc = pointer_kind(p, &k);
  if (rc) return rc;
  if (k == want || k == cudaMemoryTypeManaged) return 0;
  return -ENODEV;
}

}  // namespace cq
}  // namespace db

using namespace db;

extern "C" int db_cq_mirror(db_cq_slot* slots, uint32_t n_slots, const uint32_t* stop,
                            uint64_t limit_ns, db_counters* ctr, void* stream) {
  if (!slots || !stop || n_slots == 0 || n_slots > DB_CQ_MAX_SLOTS) return -EINVAL;
  if (limit_ns == 0 || limit_ns > DB_CQ_MAX_LIMIT_NS) return -EINVAL;
  if (!aligned(slots, 64) || !aligned(stop, 4) || (ctr && !aligned(ctr, 8))) return -EINVAL;
  int rc = cq::require(slots, cudaMemoryTypeHost);
  if (!rc) rc = cq::require(stop, cudaMemoryTypeHost);
  if (!rc && ctr) rc = cq::require(ctr, cudaMemoryTypeDevice);
  if (rc) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  if (ctr && cudaMemsetAsync(ctr, 0, sizeof(db_counters), s) != cudaSuccess) return launch_result();
  cq::Params p{slots, stop, limit_ns, ctr};
  cq::cq_mirror_kernel<<<n_slots, 32, 0, s>>>(p);
  return launch_result();
}

extern "C" int db_cq_attach(db_cq_slot* slot, uint64_t dev_cq, uint64_t host_cq, uint32_t depth,
                            uint32_t* generation) {
  if (!slot || !generation || !aligned(slot, 64)) return -EINVAL;
  if (depth < 2 || depth > DB_CQ_MAX_DEPTH) return -EINVAL;
  if (!dev_cq || !host_cq || (dev_cq & 15) || (host_cq & 15)) return -EINVAL;
  int rc = cq::require(reinterpret_cast<const void*>(dev_cq), cudaMemoryTypeDevice);
  if (!rc) rc = cq::require(reinterpret_cast<const void*>(host_cq), cudaMemoryTypeHost);
  if (rc) return rc;
  const uint32_t g = __atomic_load_n(&slot->generation, __ATOMIC_ACQUIRE);
  if (g & 1u) return -EBUSY;
  if (g > 0 && __atomic_load_n(&slot->ack, __ATOMIC_ACQUIRE) != g - 1) return -EBUSY;
  if (g >= 0xFFFFFFFDu) return -EINVAL;  // generations exhausted
  __atomic_store_n(&slot->dev_cq, dev_cq, __ATOMIC_RELAXED);
  __atomic_store_n(&slot->host_cq, host_cq, __ATOMIC_RELAXED);
  __atomic_store_n(&slot->depth, depth, __ATOMIC_RELAXED);
  __atomic_store_n(&slot->generation, g + 1, __ATOMIC_RELEASE);
  *generation = g + 1;
  return 0;
}

extern "C" int db_cq_detach(db_cq_slot* slot, uint32_t* generation) {
  if (!slot || !generation) return -EINVAL;
  const uint32_t g = __atomic_load_n(&slot->generation, __ATOMIC_ACQUIRE);
  if (!(g & 1u)) return -EINVAL;
  __atomic_store_n(&slot->generation, g + 1, __ATOMIC_RELEASE);
  *generation = g;
  return 0;
}

extern "C" int db_cq_wait_ack(const db_cq_slot* slot, uint32_t generation, uint64_t timeout_ns) {
  if (!slot) return -EINVAL;
  timespec t0, t;
  clock_gettime(CLOCK_MONOTONIC, &t0);
  for (;;) {
    if (__atomic_load_n(&slot->ack, __ATOMIC_ACQUIRE) == generation) return 0;
    clock_gettime(CLOCK_MONOTONIC, &t);
    const uint64_t el = (uint64_t)(t.tv_sec - t0.tv_sec) * 1000000000ull + t.tv_nsec - t0.tv_nsec;
    if (el >= timeout_ns) return -ETIMEDOUT;
    const timespec nap{0, 1000};
    nanosleep(&nap, nullptr);
  }
}

extern "C" int db_cq_host_reap(const void* host_cq, uint32_t depth, uint32_t* head,
                               uint32_t* phase, void* out, uint32_t max) {
  if (!host_cq || !head || !phase || (!out && max) || depth < 2 || *head >= depth) return -EINVAL;
  const uint32_t* cq = static_cast<const uint32_t*>(host_cq);
  uint32_t* o = static_cast<uint32_t*>(out);
  uint32_t h = *head, ph = *phase & 1u, n = 0;
  while (n < max) {
    const uint32_t* e = cq + 4ull * h;
    const uint32_t w3 = __atomic_load_n(e + 3, __ATOMIC_ACQUIRE);
    if (((w3 >> 16) & 1u) != ph) break;
    for (int k = 0; k < 3; ++k) o[4ull * n + k] = __atomic_load_n(e + k, __ATOMIC_RELAXED);
    o[4ull * n + 3] = w3;
    ++n;
    if (++h == depth) {
      h = 0;
      ph ^= 1u;
    }
  }
  *head = h;
  *phase = ph;
  return (int)n;
}

extern "C" void db_cq_request_stop(uint32_t* stop) {
  if (stop) __atomic_store_n(stop, 1u, __ATOMIC_RELEASE);
}
