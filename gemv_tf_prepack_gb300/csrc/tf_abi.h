// Argument checks and device queries shared by the ABI entry points.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/tf.h"
#include "tf_format.h"

namespace tf {

// Device address of the current device's error word (cached per device).
unsigned* device_error_ptr();

// Zero the current device's tf_gemv_noalloc scratch array (synchronous).
int clear_noalloc_scratch();

// The failure-detection test hook (tf_test_stall_copies): while `stall` is
// set, kernels issue no weight or activation copies, and every bounded wait
// gives up after wait_ns (4 s when the hook is off).
struct TestHook {
  int stall;
  uint64_t wait_ns;
};
TestHook test_hook();

// TMA maps over the activations x [M, K] (BF16, row-major); columns past K
// and rows past M read as zero.  encode_x_map: box of 128 columns x M rows,
// no swizzle (one GEMV tile's slice).  encode_x_map_sw128: box of 64
// columns x `rows` rows with the 128-byte swizzle (one GEMM operand slab).
int encode_x_map(const uint16_t* x, int M, int K, CUtensorMap* map);
int encode_x_map_sw128(const uint16_t* x, int M, int K, int rows, CUtensorMap* map);
// encode_y_map: the output y [M, N] BF16 (N a multiple of 8) as a 2-D map
// with a box of 128 columns (N) x 16 rows (M), for tile stores.
int encode_y_map(const uint16_t* y, int M, int N, CUtensorMap* map);

// TMA map over the S x KT units of a blob (8-byte elements): one box is the
// eight units of a 128-row tile at one kt, written densely (unit after unit)
// to shared memory.  INT4 units: dims {unit/8, KT, S}, box {unit/8, 1, 8};
// INT8 units (more than 256 elements): dims {unit/16, 2, KT, S}, box
// {unit/16, 2, 1, 8}.
int encode_units_map(const uint8_t* units, int S, int KT, int unit_bytes, CUtensorMap* map);

// Output epilogues: fused steps after the product (the pages' kernels end
// at the product).
enum EpiMode : int {
  kEpiPlain = 0,     // y[m, n]
  kEpiSiluGate = 1,  // gate/up rows interleaved in blocks of 8: h[m, j] = silu(gate_j) * up_j
  kEpiSplit3 = 2,    // rows [0, n1) -> y, [n1, n1 + n2) -> y1, the rest -> y2 (fused QKV)
};

// Where and how a kernel writes its FP32 sums.  The bias (BF16 [N], or
// null) is added to each sum before anything else.
struct Epi {
  uint16_t* y;   // plain: [M, N]; silu gate: [M, N / 2]; split: [M, n1]
  uint16_t* y1;  // split: [M, n2]
  uint16_t* y2;  // split: [M, N - n1 - n2] (null when that is 0)
  const uint16_t* bias;
  int mode, N, M, n1, n2;
};

// Host checks of an epilogue (after the layer's): outputs present, 2-byte
// aligned, and the mode's own rules (silu gate: N a multiple of 16; split:
// n1 >= 1, n2 >= 0, n1 + n2 <= N).
inline int check_epi(const Epi& e) {
  auto odd = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 1u) != 0; };
  if (!e.y) return TF_ERR_INVALID_ARG;
  if (odd(e.y) || odd(e.bias)) return TF_ERR_ALIGNMENT;
  if (e.mode == kEpiSiluGate && e.N % 16 != 0) return TF_ERR_INVALID_ARG;
  if (e.mode == kEpiSplit3) {
    if (e.n1 < 1 || e.n2 < 0 || e.n1 > e.N - e.n2) return TF_ERR_INVALID_ARG;
    if ((e.n2 > 0 && !e.y1) || (e.N - e.n1 - e.n2 > 0 && !e.y2)) return TF_ERR_INVALID_ARG;
    if (odd(e.y1) || odd(e.y2)) return TF_ERR_ALIGNMENT;
  }
  return TF_OK;
}

// The stream GEMV (gemv_stream.cu): M <= 8, groups of 64, any multiple of
// 128 or per channel, activations that fit in shared memory; no workspace.
// stream_plan returns 1 and fills *P when it takes the layer.
struct StreamPlan {
  int G, Mp, NS, npre, off_x, off_xs, off_red, off_ctl, max_slabs, half, compact;
  size_t smem;
};
int stream_plan(const Geometry& G, int M, StreamPlan* P);
int run_stream(const Geometry& G, const StreamPlan& P, const void* blob, const uint16_t* x, const Epi& epi, int M,
               cudaStream_t stream);

// Split-K workspaces (tf_gemv, tf_gemm, the no-alloc scratch) keep their
// arrival counters in this many bytes at the start and the partial sums
// after them, so that no layer's partial sums ever land on another layer's
// counters: one workspace can serve layers of any shape.
constexpr size_t kWorkspaceCounterBytes = 16384;

// tf_gemm for 1 <= M <= 8 on the slab or tile GEMV of gemv.cu, which keep
// tf_gemm's per-weight BF16 rounding.  small_m_workspace gives the
// workspace bytes (0 for the slab GEMV), or UNSUPPORTED when the layer is
// not theirs (K % 8 != 0, M > 8).
int small_m_workspace(const Geometry& G, int M, size_t* bytes);
int run_small_m(const Geometry& G, const void* blob, const uint16_t* x, const Epi& epi, int M, void* workspace,
                size_t workspace_bytes, cudaStream_t stream);

inline bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Streaming multiprocessors of the current device (cached per device).
inline int sm_count() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return -1;
  if (dev < 64) {
    int v = cache[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return -1;
  if (dev < 64) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

// Common validation of a device blob against the layer description.
inline int check_blob(const void* blob, size_t blob_bytes, int N, int K, int bits, int group,
                      Geometry* G) {
  int rc = make_geometry(N, K, bits, group, G);
  if (rc) return rc;
  if (!blob) return TF_ERR_INVALID_ARG;
  if (!aligned16(blob)) return TF_ERR_ALIGNMENT;
  if (blob_bytes != G->total_bytes) return TF_ERR_BAD_BLOB;
  return TF_OK;
}

// Status of the launch just made; peeks so that unrelated sticky errors of
// other libraries are neither reported as ours nor cleared.
inline int launch_status() {
  cudaError_t e = cudaPeekAtLastError();
  if (e == cudaSuccess) return TF_OK;
  cudaGetLastError();  // a launch error of ours is not sticky; clear it
  return TF_ERR_CUDA;
}

// Launch with programmatic dependent launch; opts the kernel in, once per
// device, to the largest ring a plan can ask for.
template <class Kern, class... Args>
int launch_pdl(Kern kfn, std::atomic<unsigned long long>& opted, int grid, int threads, int smem_max, size_t smem,
               cudaStream_t s, Args... args) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return TF_ERR_CUDA;
  if (!(opted.load(std::memory_order_acquire) & (1ull << dev))) {
    if (cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max) != cudaSuccess ||
        cudaFuncSetAttribute(kfn, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess)
      return TF_ERR_CUDA;
    opted.fetch_or(1ull << dev, std::memory_order_acq_rel);
  }
  if (smem > (size_t)smem_max) return TF_ERR_UNSUPPORTED;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kfn, args...) != cudaSuccess) {
    cudaGetLastError();
    return TF_ERR_CUDA;
  }
  return launch_status();
}

}  // namespace tf
