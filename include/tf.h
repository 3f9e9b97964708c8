/*
 * tf.h — C ABI of libtf: a GB300 (sm_103a) fused mixed-precision linear layer.
 *
 * The operation is the one the TileFuse pages describe ("TileFuse: A Fused
 * Mixed-Precision Kernel Library for Efficient Quantized LLM Inference on
 * AMD NPUs", section "Methodology", item 1 "Fused mixed-precision
 * microkernels"): AWQ-style packed INT4/INT8 weights are unpacked,
 * dequantised per group or per channel to BF16 as (q - zero) * scale, and
 * consumed in the same kernel by a GEMV (token generation, batch 1) or a
 * GEMM (prefill):
 *
 *     y[m, n] = sum_k x[m, k] * bf16_rne((q[n, k] - z[n, k/g]) * s[n, k/g])
 *
 * with x BF16 [M, K], y BF16 [M, N], FP32 accumulation and one final
 * round-to-nearest-even to BF16.  W is N (out) x K (in).
 *
 * Conventions shared by every call:
 *  - bits is 4 or 8.  group is 32, 64, any multiple of 128 that divides K,
 *    or 0 for per output channel (one group spanning all of K).  K must be
 *    a multiple of the group, and of 8 unless per channel.  1 <= N, K <= 32768 (Contributions 2:
 *    the layout stays valid for dimensions up to 32K).
 *  - BF16 values are passed as their uint16 bit patterns.
 *  - Natural-order inputs (host memory): INT4 qweight is uint32
 *    [N, ceil(K/8)], eight codes per word, low nibble first along K (a last,
 *    partial word keeps its unused nibbles zero); INT8 qweight is uint8
 *    [N, K]; scales uint16 [N, K/g]; zeros uint8 [N, K/g] (0..2^bits-1).
 *  - The caller allocates and owns every buffer.  The library allocates no
 *    memory; its only global state is cached device attributes, one
 *    device-side error word per device and the fixed scratch array of
 *    tf_gemv_noalloc.
 *  - Every call returns TF_OK (0) or a negative TF_ERR_* code and never
 *    aborts.  Device calls only enqueue work on the given stream (NULL means
 *    the legacy default stream) and return without synchronising; a
 *    TF_ERR_CUDA return means the launch itself failed.
 *  - Calls are thread-safe.  Two device calls that share a workspace must
 *    not run concurrently.
 *  - Workspaces (tf_gemv, tf_gemm) keep their arrival counters in the first
 *    16384 bytes and everything else after them, and every call that
 *    completes leaves those counters at zero.  So one workspace, zero-filled
 *    once and at least as large as the largest size asked for, can serve
 *    calls of any layer and any M, tf_gemv and tf_gemm alike, in turn on one
 *    stream.  After a call that reported a device error (tf_device_error
 *    nonzero), zero it again.
 *  - The GEMV kernels start early under programmatic dependent launch: they
 *    read the blob and the bias before waiting for the kernel launched just
 *    before them on the stream (x, y and the workspace only after it).  The
 *    weights and the bias must therefore not be written by that kernel.
 *  - Device state (the error word, the scratch array of tf_gemv_noalloc,
 *    cached device attributes) is looked up once per device, in the context
 *    current at the first call: the device's primary context, which the
 *    CUDA runtime uses.  Calls under another driver context, or after
 *    cudaDeviceReset while the library stays loaded, are not supported.
 *  - The host checks blob_bytes against (N, K, bits, group); the kernels also
 *    read the device blob's 64-byte header and, when it describes another
 *    layer (for instance a blob of the same size with N and K swapped), write
 *    nothing and record 0x800 in the device error word (tf_device_error).
 */
#ifndef TF_H_
#define TF_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TF_VERSION 6  /* 3: tf_prepack_awq, tf_gemv_bias, tf_gemm_bias; 4: tf_gemv_noalloc,
                         TF_ERR_SCRATCH_LIMIT, device-side check of the blob header;
                         5: tf_prepack_gate_up, tf_gemv_silu_gate, tf_gemm_silu_gate,
                         tf_gemv_qkv, tf_gemm_qkv; 6: workspaces with a fixed leading
                         counter region (one workspace serves every layer), tf_gemm
                         at M <= 8 on the GEMV kernels */

#define TF_OK 0
#define TF_ERR_INVALID_ARG (-1) /* null pointer, bad size or bad combination */
#define TF_ERR_UNSUPPORTED (-2) /* dims > 32768, bits/group not supported, M too large for the call */
#define TF_ERR_ALIGNMENT (-3)   /* a device pointer is not 16-byte aligned */
#define TF_ERR_WORKSPACE (-4)   /* workspace missing or smaller than required */
#define TF_ERR_BAD_BLOB (-5)    /* header magic/version/fields do not match */
#define TF_ERR_CUDA (-6)        /* a CUDA runtime call or a launch failed */
#define TF_ERR_DEVICE (-7)      /* a kernel reported an error (see tf_device_error) */
#define TF_ERR_SCRATCH_LIMIT (-8) /* tf_gemv_noalloc: the layer needs more than its fixed scratch */

/* Library version (TF_VERSION). */
int tf_version(void);

/* Static, human-readable name of a status code. */
const char* tf_status_string(int status);

/*
 * Pre-tiled blob format ("interleaved pre-tiling", Methodology 2: metadata is
 * packed into the weight tiles and the matrix is reordered so that each
 * consumer's tiles are contiguous, valid up to 32K).
 *
 * Blob = 64-byte header + S*KT units (S = 8*ceil(N/128) slabs of 16 rows,
 * KT = ceil(K/128)).  Unit (s, kt) covers rows 16s..16s+15 and columns
 * 128kt..128kt+127 of W and sits at byte 64 + (s*KT + kt) * unit_bytes:
 * slab-major, so the units of any run of whole slabs are one contiguous
 * range, and the eight slabs 8nb..8nb+7 at one kt form a 128 x 128 tile.
 * A unit holds its 16 x 128 codes in mma.sync fragment order, then its BF16
 * scales, then its zeros, then zero padding to a multiple of 16 (INT4) or 32
 * (INT8) bytes, so one
 * contiguous read brings everything the unit needs.  The header is
 * little-endian: u32 magic 0x4B504654, u32 version 2, i32 N, K, bits, group,
 * unit_n (16), unit_k (128), S, KT, unit_bytes, groups_per_unit,
 * u64 total_bytes, 8 zero bytes.  Padding rows (n >= N) and columns (k >= K)
 * dequantise to exactly zero.
 */

/* Size in bytes of the blob for this layer; writes *bytes. */
int tf_prepack_size(int N, int K, int bits, int group, size_t* bytes);

/*
 * Offline pre-tiling (host, synchronous, pure).  qweight / scales / zeros are
 * host arrays in natural order (see above); out is a host buffer of at least
 * tf_prepack_size bytes.  Codes or zeros above 2^bits - 1 give
 * TF_ERR_INVALID_ARG.  The caller uploads the blob to the device.
 */
int tf_prepack(const void* qweight, const uint16_t* scales, const uint8_t* zeros,
               int N, int K, int bits, int group, void* out, size_t out_bytes);

/*
 * Offline pre-tiling of an INT4 layer as AWQ checkpoints store it (TileFuse,
 * Contributions 1: the fused kernels take AWQ-style weights as published,
 * with no re-quantisation of the model); host, synchronous, pure.
 * Input layout (AWQ's GEMM format):
 *   qweight     int32 [K, N/8]: word (k, c) holds the codes of W[8c + j, k],
 *               j = 0..7, with the code of column 8c + j in nibble
 *               (0, 4, 1, 5, 2, 6, 3, 7)[j] (bits 4*nibble .. 4*nibble+3);
 *               equivalently nibble i holds column 8c + (0, 2, 4, 6, 1, 3, 5, 7)[i];
 *   qzeros      int32 [K/g, N/8]: the zero points, packed the same way;
 *   scales_f16  IEEE binary16 bits [K/g, N].
 * g = group, or K for group = 0 (one group per row); group as for tf_prepack.
 * Each scale is rounded to BF16 (round to nearest even), since the blob and
 * the kernels dequantise to BF16 as bf16_rne((q - z) * s); the result is the
 * blob tf_prepack makes from the same codes, zeros and those BF16 scales.
 * N must be a multiple of 8 (TF_ERR_INVALID_ARG otherwise); out is a host
 * buffer of at least tf_prepack_size(N, K, 4, group) bytes.
 */
int tf_prepack_awq(const int32_t* qweight, const int32_t* qzeros, const uint16_t* scales_f16,
                   int N, int K, int group, void* out, size_t out_bytes);

/*
 * Offline pre-tiling of the gate and up projections of a gated MLP into the
 * one layer tf_gemv_silu_gate / tf_gemm_silu_gate take (host, synchronous,
 * pure; an addition of this library, the pages fuse no epilogue).  Each
 * projection is F x K in natural order (arrays as for tf_prepack, same bits
 * and group); the blob is the layer of N = 2F rows whose rows 16j .. 16j + 7
 * are gate rows 8j .. 8j + 7 and rows 16j + 8 .. 16j + 15 the up rows
 * 8j .. 8j + 7 (its natural-order row r is gate row 8 (r / 16) + r mod 8
 * when r mod 16 < 8, else that up row).  F must be a multiple of 8; out is
 * a host buffer of at least tf_prepack_size(2F, K, bits, group) bytes.
 */
int tf_prepack_gate_up(const void* gate_qweight, const uint16_t* gate_scales, const uint8_t* gate_zeros,
                       const void* up_qweight, const uint16_t* up_scales, const uint8_t* up_zeros,
                       int F, int K, int bits, int group, void* out, size_t out_bytes);

/*
 * Exact inverse of tf_prepack (host).  Reads N, K, bits, group from the
 * header and writes natural-order qweight, scales and zeros (sizes as for
 * tf_prepack).  TF_ERR_BAD_BLOB if the header is inconsistent with bytes.
 */
int tf_unprepack(const void* blob, size_t bytes, void* qweight, uint16_t* scales,
                 uint8_t* zeros);

/* Parse a host copy of the 64-byte header; any output pointer may be NULL. */
int tf_blob_info(const void* header, size_t bytes, int* N, int* K, int* bits, int* group);

/*
 * Debug / parity path: dequantise the whole device-resident blob to dense
 * BF16 w[N, K] (row-major, device memory) with exactly the unpack and
 * dequant arithmetic the GEMV and GEMM kernels use
 * (bf16_rne((q - z) * s), Methodology 1).  blob and w must be 16-byte
 * aligned; blob_bytes is the blob's size (checked against N, K, bits, group).
 */
int tf_dequant(const void* blob, size_t blob_bytes, int N, int K, int bits, int group,
               uint16_t* w, cudaStream_t stream);

/*
 * Workspace bytes tf_gemv needs on the current device for this layer and M
 * (16384 bytes of per-block arrival counters, then the split-K partial
 * sums; 0 for the layers whose blocks each stream whole slabs).  The
 * workspace must be zero-filled before its first use; every tf_gemv that
 * completes leaves the arrival counters at zero again (the partial sums are
 * always written before they are read), so one workspace can be reused by
 * calls ordered on one stream, for any layer (see the workspace rule
 * above).  After a call that reported a device error (tf_device_error
 * nonzero) zero the workspace again before reusing it.
 */
int tf_gemv_workspace_size(int N, int K, int bits, int group, int M, size_t* bytes);

/*
 * Fused GEMV for token generation ("GEMV dataflow co-design", Methodology 3;
 * batch 1, and up to 8 rows at no extra cost): y[M, N] = x[M, K] * W^T.
 * Each weight code is read from HBM once, unpacked in registers and fed
 * straight to the tensor cores (mma.sync, FP32 accumulation), with the whole
 * chip streaming weights.
 *  - Groups of 64, multiples of 128 or per channel, with x small enough to
 *    stay resident in shared memory (M * K up to about 64K elements): every
 *    block (one per SM, or one per 16-row slab on smaller layers) owns whole
 *    slabs, each warp streams a contiguous run of them.  The codes enter the
 *    tensor cores exactly (as FP16), x is converted to FP16 with a
 *    power-of-two scale per 128-column block (exact), and (q - z) * s is
 *    applied per group in FP32 to the sums: the result is
 *    sum_k x * (q - z) * s without rounding each dequantised weight to BF16
 *    (tf_dequant and tf_gemm keep that rounding).
 *  - The others (groups of 32, or x too large for the above) with K >= 1024
 *    and x resident: whole slabs per block (one block per slab on small
 *    layers), K split over the block's warps, each weight dequantised to
 *    BF16 in registers (as tf_dequant and tf_gemm do).
 *  - The rest (K < 1024, or x too large even for that): K split across all
 *    blocks, the last-arriving block of each row block adding the partial
 *    sums.
 * Every addition happens in a fixed order, so results are deterministic run
 * to run.
 * Device pointers: blob (16-byte aligned), x [M, K] BF16 (16-byte aligned),
 * y [M, N] BF16, workspace (16-byte aligned, >= tf_gemv_workspace_size; may
 * be NULL when that is 0).  1 <= M <= 8, else TF_ERR_UNSUPPORTED.  With
 * K % 8 != 0 (per channel) only the stream GEMV takes the layer, reading x
 * element by element: its activations must fit in shared memory next to
 * the weight ring (M * K up to about 64K elements), else
 * TF_ERR_UNSUPPORTED.
 */
int tf_gemv(const void* blob, size_t blob_bytes, int N, int K, int bits, int group,
            const uint16_t* x, uint16_t* y, int M, void* workspace, size_t workspace_bytes,
            cudaStream_t stream);

/*
 * tf_gemv with a bias in the epilogue: y[m, n] = bf16_rne(sum_k x[m, k] *
 * w[n, k] + bias[n]), the BF16 bias added to the FP32 sum before its one
 * rounding (a fused epilogue; the pages' kernels end at the product).  bias
 * is a device array of N BF16 values, or NULL for none (exactly tf_gemv);
 * an odd address gives TF_ERR_ALIGNMENT.  Everything else as for tf_gemv.
 */
int tf_gemv_bias(const void* blob, size_t blob_bytes, int N, int K, int bits, int group,
                 const uint16_t* x, const uint16_t* bias, uint16_t* y, int M, void* workspace,
                 size_t workspace_bytes, cudaStream_t stream);

/*
 * Workspace bytes tf_gemm needs on the current device for this layer and M.
 * M <= 8 (K % 8 == 0): what the slab or tile GEMV behind it needs (0 for
 * the slab GEMV: K >= 1024 with x resident in shared memory).  Else, to
 * split the K dimension of its last, partial wave of output tiles across
 * all SMs (stream-K): 16384 bytes of per-tile arrival counters, then FP32
 * partial sums, 0 when the tiles fill whole waves; plus, when K % 8 != 0
 * (per channel), a copy of x with rows padded to a multiple of 8 elements
 * (a TMA tensor's rows must be multiples of 16 bytes) after the counters
 * and partial sums, rewritten by every call.  Like the GEMV workspace it
 * must be zero-filled before its first use, and every tf_gemm that
 * completes leaves its counters at zero.  After a call that reported a
 * device error (tf_device_error nonzero) zero it again before reusing it.
 */
int tf_gemm_workspace_size(int N, int K, int bits, int group, int M, size_t* bytes);

/*
 * Fused GEMM for prefill (Methodology 1: each weight tile is unpacked and
 * dequantised once into on-chip memory and reused for the tile's MMAs):
 * y[M, N] = x[M, K] * W^T for any M >= 1, with tcgen05 tensor-core MMAs
 * accumulating in tensor memory.  Device pointers: blob, x and y 16-byte
 * aligned.  With a workspace (16-byte aligned, >= tf_gemm_workspace_size)
 * the output tiles of the last, partial wave are split along K across all
 * SMs and their partial sums added in a fixed order (same result every run);
 * with workspace NULL (workspace_bytes ignored) every tile is computed whole
 * by one SM.  A workspace smaller than required gives TF_ERR_WORKSPACE.
 * With K % 8 != 0 (per channel) the workspace is required (it holds the
 * padded copy of x, made by a small kernel on the stream before the GEMM);
 * NULL gives TF_ERR_WORKSPACE.
 * M <= 8 with K % 8 == 0 is a weight stream, not a contraction: it runs on
 * the slab or tile GEMV of tf_gemv (every weight dequantised to BF16 in
 * registers, exactly as here, and fed to mma.sync), given the workspace
 * that tf_gemm_workspace_size asks for, or with none when that is 0; with
 * workspace NULL on a layer that needs one, the tensor-core pipeline runs
 * with every tile whole.
 */
int tf_gemm(const void* blob, size_t blob_bytes, int N, int K, int bits, int group,
            const uint16_t* x, uint16_t* y, int M, void* workspace, size_t workspace_bytes,
            cudaStream_t stream);

/*
 * tf_gemm with a bias in the epilogue: y[m, n] = bf16_rne(sum_k x[m, k] *
 * w[n, k] + bias[n]) (bias: device, N BF16 values, or NULL for none, which
 * is exactly tf_gemm; an odd address gives TF_ERR_ALIGNMENT).  Everything
 * else as for tf_gemm.
 */
int tf_gemm_bias(const void* blob, size_t blob_bytes, int N, int K, int bits, int group,
                 const uint16_t* x, const uint16_t* bias, uint16_t* y, int M, void* workspace,
                 size_t workspace_bytes, cudaStream_t stream);

/*
 * Fused epilogues (additions of this library; the pages' kernels end at the
 * product).  Each runs the GEMV or GEMM of the layer exactly as tf_gemv_bias
 * / tf_gemm_bias do (same limits on M, same workspace, same sums) and
 * changes only where the biased FP32 sums s[m, n] = sum_k x[m, k] w[n, k]
 * (+ bias[n], bias in the layer's row order, or NULL) go.
 *
 * SiLU gate, for the gate/up projection of a gated MLP packed by
 * tf_prepack_gate_up (N = 2F, a multiple of 16, else TF_ERR_INVALID_ARG):
 *     h[m, 8j + i] = bf16_rne(silu(s[m, 16j + i]) * s[m, 16j + 8 + i]),
 *     i = 0..7, silu(a) = a / (1 + e^-a), computed in FP32;
 * h is device memory, BF16 [M, N/2], 2-byte aligned.  The N x M
 * intermediate never reaches memory.
 */
int tf_gemv_silu_gate(const void* blob, size_t blob_bytes, int N, int K, int bits, int group,
                      const uint16_t* x, const uint16_t* bias, uint16_t* h, int M, void* workspace,
                      size_t workspace_bytes, cudaStream_t stream);
int tf_gemm_silu_gate(const void* blob, size_t blob_bytes, int N, int K, int bits, int group,
                      const uint16_t* x, const uint16_t* bias, uint16_t* h, int M, void* workspace,
                      size_t workspace_bytes, cudaStream_t stream);

/*
 * Split, for a fused QKV projection (the three weight matrices stacked
 * along N into one layer): rows [0, nq) go to q [M, nq], rows
 * [nq, nq + nk) to k [M, nk] and rows [nq + nk, N) to v [M, N - nq - nk],
 * each BF16 row-major device memory, 2-byte aligned, rounded once as by
 * tf_gemv_bias.  nq >= 1, nk >= 0, nq + nk <= N, else TF_ERR_INVALID_ARG; k
 * (v) may be NULL only when it gets no rows.
 */
int tf_gemv_qkv(const void* blob, size_t blob_bytes, int N, int K, int bits, int group,
                const uint16_t* x, const uint16_t* bias, uint16_t* q, uint16_t* k, uint16_t* v,
                int nq, int nk, int M, void* workspace, size_t workspace_bytes, cudaStream_t stream);
int tf_gemm_qkv(const void* blob, size_t blob_bytes, int N, int K, int bits, int group,
                const uint16_t* x, const uint16_t* bias, uint16_t* q, uint16_t* k, uint16_t* v,
                int nq, int nk, int M, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * tf_gemv without a caller-provided workspace, for callers that cannot
 * allocate device memory where they run the layer (code living inside
 * another framework's memory pool, plugins that are handed only their input
 * and output pointers, latency-critical paths where an allocation may block
 * or fail).  The paper has no counterpart: it is an addition of this
 * library.  Arguments and results are those of tf_gemv; the split-K scratch
 * is a fixed device array of TF_GEMV_NOALLOC_SCRATCH_BYTES inside libtf that
 * every GPU which loads the library keeps until the process exits.  No
 * cudaMalloc/cudaFree or allocating library routine is called.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current); make that first call
 *    before capturing a stream into a CUDA graph.
 *  - Every call on a device shares the one array.  Its arrival counters are
 *    zero when the library is loaded, and every call that completes leaves
 *    them at zero, so no call clears them first.  A call cut short by a
 *    device error may leave them dirty: tf_device_error, when it reports an
 *    error, also clears the array.  Calls that overlap on the GPU (other
 *    streams, other host threads) race on the array: order them on one
 *    stream or use tf_gemv.
 *  - A layer whose scratch would exceed TF_GEMV_NOALLOC_SCRATCH_BYTES is
 *    rejected with TF_ERR_SCRATCH_LIMIT (every N, K <= 32768 fits on GPUs
 *    with up to ~200 SMs).
 */
#define TF_GEMV_NOALLOC_SCRATCH_BYTES (4u << 20)
int tf_gemv_noalloc(const void* blob, size_t blob_bytes, int N, int K, int bits, int group,
                    const uint16_t* x, uint16_t* y, int M, cudaStream_t stream);

/*
 * Failure-detection test hook (the paper has no counterpart; off by
 * default, process-wide, not for production use).  While stall is nonzero,
 * every later device call issues no weight or activation copies, so its
 * first bounded wait runs out after timeout_us microseconds (> 0): the
 * kernel records its wait code in the device error word (see
 * tf_device_error), writes no output and exits with no copy in flight, and
 * the device stays usable.  tf_test_stall_copies(0, 0) turns it off and
 * restores the 4-second limit.  TF_ERR_INVALID_ARG for stall with
 * timeout_us == 0.
 */
int tf_test_stall_copies(int stall, unsigned int timeout_us);

/*
 * Read and clear the current device's error word (synchronous).  Kernels
 * that wait on on-chip barriers give up after a bounded time instead of
 * hanging, set a nonzero code here and exit; *code receives 0 if nothing
 * went wrong since the last read.  Codes: 0x100-0x500 a GEMM wait ran out
 * (producer, dequant, MMA, epilogue, drain), 0x600 a tile or slab GEMV wait,
 * 0x700 a stream GEMV wait, 0x800 the device blob's header does not match
 * the call (nothing written).  The first code since the last read is kept.
 * When the code is nonzero it also zeroes the tf_gemv_noalloc scratch array
 * of the device (a call cut short may have left its counters dirty).
 */
int tf_device_error(unsigned int* code);

#ifdef __cplusplus
}
#endif

#endif /* TF_H_ */
