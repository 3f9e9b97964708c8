// The device-side error word of libtf and its host accessors.
//
// Kernels that wait on shared-memory barriers give up after a bounded time
// instead of hanging; they then record a nonzero code here.  One word per
// device, defined in this translation unit only; other units receive its
// device address as a kernel argument.
#include <cuda_runtime.h>

#include <atomic>

#include "../../include/tf.h"
#include "tf_abi.h"

namespace tf {

__device__ unsigned g_tf_error;

unsigned* device_error_ptr() {
  static std::atomic<unsigned*> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return nullptr;
  if (dev < 64) {
    unsigned* p = cache[dev].load(std::memory_order_acquire);
    if (p) return p;
  }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_tf_error) != cudaSuccess) return nullptr;
  if (dev < 64) cache[dev].store(static_cast<unsigned*>(p), std::memory_order_release);
  return static_cast<unsigned*>(p);
}

namespace {
std::atomic<int> g_stall{0};
std::atomic<unsigned long long> g_wait_ns{0};
}  // namespace

TestHook test_hook() {
  const unsigned long long w = g_wait_ns.load(std::memory_order_acquire);
  return TestHook{g_stall.load(std::memory_order_acquire), w ? (uint64_t)w : 4000000000ull};
}

}  // namespace tf

extern "C" int tf_test_stall_copies(int stall, unsigned int timeout_us) {
  if (stall && timeout_us == 0) return TF_ERR_INVALID_ARG;
  tf::g_wait_ns.store(stall ? (unsigned long long)timeout_us * 1000ull : 0ull, std::memory_order_release);
  tf::g_stall.store(stall ? 1 : 0, std::memory_order_release);
  return TF_OK;
}

extern "C" int tf_device_error(unsigned int* code) {
  if (!code) return TF_ERR_INVALID_ARG;
  unsigned v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, tf::g_tf_error, sizeof v) != cudaSuccess) return TF_ERR_CUDA;
  if (cudaMemcpyToSymbol(tf::g_tf_error, &zero, sizeof zero) != cudaSuccess) return TF_ERR_CUDA;
  // a call cut short may have left tf_gemv_noalloc's arrival counters dirty
  if (v != 0 && tf::clear_noalloc_scratch() != TF_OK) return TF_ERR_CUDA;
  *code = v;
  return TF_OK;
}
