// Host-side helpers of the C ABI: error strings, launch-error capture, SM count.
#include <cstring>

#include "common.cuh"

namespace db {

static thread_local int g_last_cuda_error = 0;

int launch_result() {
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) return 0;
  g_last_cuda_error = (int)e;
  return -EIO;
}

int cuda_failure(cudaError_t e) {
  cudaGetLastError();  // clear it: the code is returned through db_last_cuda_error
  g_last_cuda_error = (int)e;
  return -EIO;
}

int num_sms() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  int& c = cached[dev & 63];
  if (c == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v < 1)
      v = 1;
    c = v;
  }
  return c;
}

}  // namespace db

extern "C" const char* db_strerror(int code) {
  switch (code) {
    case 0:
      return "success";
    case -EINVAL:
      return "invalid argument (null or misaligned pointer, or value out of range)";
    case -ENOSPC:
      return "workspace too small";
    case -EIO:
      return "CUDA launch failed (see db_last_cuda_error)";
    case -E2BIG:
      return "batch larger than the built-in workspace allows (DB_PRP_STATIC_MAX_REQUESTS)";
    case -EBUSY:
      return "slot busy (attached, or its previous generation not yet acknowledged)";
    case -ETIMEDOUT:
      return "timed out";
    case -ENODEV:
      return "no CUDA device, or memory of the wrong kind (pinned host or device memory expected)";
    default:
      return "unknown error";
  }
}

extern "C" int db_last_cuda_error(void) { return db::g_last_cuda_error; }
