// status.cu -- error reporting and small host utilities shared by the C ABI.
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <vector>

#include "common.cuh"

namespace w4 {

static thread_local char g_last_error[512] = "";

int set_error(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return code;
}

int check_launch(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(W4A16_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return W4A16_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int device_index() {
  int d = 0;
  cudaGetDevice(&d);
  return d;
}

int num_sms() {
  static std::mutex mu;
  static std::vector<int> cache;
  const int d = device_index();
  std::lock_guard<std::mutex> lk(mu);
  if ((int)cache.size() <= d) cache.resize(d + 1, 0);
  if (cache[d] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d) != cudaSuccess || n <= 0) n = 1;
    cache[d] = n;
  }
  return cache[d];
}

}  // namespace w4

extern "C" const char* w4a16_last_error(void) { return w4::g_last_error; }

extern "C" int w4a16_version(void) { return 100; }
