// Stream GEMV of libtf: token generation (M <= 8) for layers with INT4 or
// INT8 codes, groups of 64, any multiple of 128, or per channel, whose
// activations fit in shared memory next to the weight ring.
//
// TileFuse, Methodology 3 ("GEMV dataflow co-design"): at batch 1 a
// quantised linear layer stops being bound by memory once unpacking and
// dequantisation are added, and the weight stream has to be spread over the
// whole array.  On GB300 the stream itself is cheap (1-D bulk copies of
// contiguous ranges of the pre-tiled blob into shared memory); what costs is
// the per-weight arithmetic.  This kernel keeps it to one logical operation
// per two weights:
//
//  * A code q placed in the low bits of an FP16 with a zero exponent field
//    IS the subnormal q * 2^-24, exactly.  So `word & 0x000F000F` turns two
//    INT4 codes into an FP16x2 tensor-core operand, and `word & 0x00F000F0`
//    the next two, as 16 q * 2^-24 (INT8: byte masks and byte permutes).
//  * The activations are converted once per CTA to FP16, each 128-column
//    block of each token with its own power-of-two scale (exact: BF16 has 8
//    significant bits, FP16 11; the scale keeps the block's largest |x| just
//    below 2^15).  Each product x * q is then exact, and the tensor cores
//    (mma.sync m16n8k16, FP32 accumulation) sum them per group; the block's
//    scale is undone in the group's FP32 epilogue.
//  * Dequantisation (q - z) * s is applied per group, in FP32, to that sum:
//        sum_k x_k (q_k - z) s = s * (sum_k x_k q_k - z * sum_k x_k),
//    with sum_k x_k per group and token computed once per CTA.  The result
//    is the dequantised product without the per-weight BF16 rounding of
//    (q - z) * s (the parity path tf_dequant keeps that rounding bit for
//    bit); the pages' "dequantise to BF16" becomes "codes exact in FP16, scale
//    and zero in FP32".
//
// Work split.  Each CTA (one per SM, or one per slab on layers with fewer
// 16-row slabs than SMs) owns whole slabs, the slab count shared out as
// evenly as whole slabs allow (the CTAs that start first take the extra
// ones); a slab split between two CTAs would need a cross-SM reduction
// whose L2 round trip at the end of the layer costs more than the
// up-to-one-slab imbalance.  Even a layer of a few slabs runs faster this
// way than with K split across all SMs (the tile GEMV of gemv.cu: 2 to 5
// times slower on 256 to 2304-row layers).  The CTA's slabs are
// one contiguous byte range of the blob (units are slab-major), shared out
// evenly over its sixteen warps: a warp's share is a contiguous run of
// units, which it streams through its own small ring of shared-memory stages
// (one bulk copy and one mbarrier per stage), so warps never wait for one
// another.  A warp keeps one running sum per slab and parks it in shared
// memory when its run crosses into the next slab; after the stream the CTA
// adds the sixteen warps' sums of each slab in warp order (a fixed order:
// the same result every run) and writes y.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>

#include "../../include/tf.h"
#include "tf_abi.h"
#include "tf_device.cuh"
#include "tf_format.h"
#include "tf_sm100.cuh"

#ifndef TF_STREAM_NS_MAX
#define TF_STREAM_NS_MAX 2  // deepest per-warp ring of the plan (stages)
#endif
#ifndef TF_STREAM_WARPS
#define TF_STREAM_WARPS 16  // warps per CTA (one CTA per SM)
#endif
#ifndef TF_STREAM_NPRE
#define TF_STREAM_NPRE 1    // stages per warp requested before the previous kernel on the stream has finished
#endif

namespace tf {
namespace {

constexpr int kSW = TF_STREAM_WARPS;  // warps per CTA
constexpr int kSThreads = 32 * kSW;
constexpr int kSmemMax = 227 * 1024;  // one CTA per SM
constexpr uint64_t kDrainNs = 200000000ull;
constexpr unsigned kErrStreamWait = 0x700;

// Units per stage of a warp's ring (one bulk copy): 4 INT4 or 2 INT8 units,
// about 4 KB, or half that when large activations leave less room.
__host__ __device__ constexpr int warp_stage_units(int bits, bool half) { return (bits == 4 ? 4 : 2) / (half ? 2 : 1); }

struct StreamArgs {
  const uint8_t* units;  // the blob's units (after the header)
  const uint16_t* x;     // [M, K] BF16
  Epi epi;               // where y goes (plain, SiLU gate or split) and the bias
  unsigned* err;
  int nslab;             // slabs holding real rows
  int N, K, M, Mp, KT, G, group;
  int NS, npre;          // per-warp ring: stages, stages requested before the grid dependency resolves
  int off_x, off_xs, off_red, off_ctl;  // byte offsets in the 128-aligned dynamic shared memory
  int max_slabs;         // slabs of the busiest CTA
  int compact;           // parked sums: 1 = two slots per warp, 0 = one slot per (slab, warp)
  int stall;             // failure-detection test: issue no copies, so that the first wait runs out
  uint64_t wait_ns;      // limit of every wait
};

// The run of units of warp w of a CTA whose units are [u0, u1).
__device__ __forceinline__ void warp_run(int u0, int u1, int w, int& g0, int& nu) {
  g0 = u0 + (u1 - u0) * w / kSW;
  nu = u0 + (u1 - u0) * (w + 1) / kSW - g0;
}

// One bulk copy: units [g, g + n) (global, memory order) into a ring stage.
// The arrive carries no memory ordering: the stage's earlier readers have
// already used the values they loaded.
template <int BITS, int GPT>
__device__ __forceinline__ void warp_fill(const StreamArgs& a, uint32_t dst, uint32_t bar, int g, int n) {
  constexpr int UB = unit_bytes_gpu(BITS, GPT);
  if (a.stall) return;
  mbar_arrive_expect_tx_relaxed(bar, (uint32_t)(n * UB));
  // the weights are read once per call: they should not push the
  // activations and other live data out of L2
  bulk_load_hint(dst, a.units + (size_t)g * UB, (uint32_t)(n * UB), bar, l2_evict_first_policy());
}

// ---------------------------------------------------------------------------
// per-unit arithmetic

// D += A * B with FP16 operands, FP32 accumulation.
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// D = A * B (no accumulator input).
__device__ __forceinline__ void mma_f16_first(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  const float z = 0.f;
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};\n"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(z));
}

// The four A-fragment registers of one MMA from its packed codes.
//  INT4, one word w (codes i = 0..7, register r holding codes r and r + 4):
//    r = 0: w & 0x000F000F          -> q * 2^-24        (row gr)
//    r = 1: w & 0x00F000F0          -> 16 q * 2^-24     (row gr + 8)
//    r = 2, 3: the same on w >> 8.
//  INT8, two words u0, u1 (code i in byte i of u0 for i < 4, byte i - 4 of
//  u1 otherwise): the byte masks give registers of codes (0, 2), (1, 3),
//  (4, 6), (5, 7), i.e. columns (c, c + 2) and (c + 1, c + 3) of a
//  4-column group; the activations are stored with the same permutation.
__device__ __forceinline__ void codes_w4(uint32_t w, uint32_t (&a)[4]) {
  const uint32_t w8 = w >> 8;
  a[0] = w & 0x000F000Fu;
  a[1] = w & 0x00F000F0u;
  a[2] = w8 & 0x000F000Fu;
  a[3] = w8 & 0x00F000F0u;
}

__device__ __forceinline__ void codes_w8(uint32_t u0, uint32_t u1, uint32_t (&a)[4]) {
  a[0] = u0 & 0x00FF00FFu;
  a[1] = __byte_perm(u0, 0u, 0x7371);  // bytes 1, 3 of u0 with zero high bytes
  a[2] = u1 & 0x00FF00FFu;
  a[3] = __byte_perm(u1, 0u, 0x7371);
}

// A unit's codes and metadata for one lane.
template <int BITS, int GPT>
struct Unit {
  uint4 w[2][BITS == 4 ? 1 : 2];
  uint32_t sp[GPT], zp[GPT];
};

struct Lane {
  int w, s[2], z[2], x;  // byte offsets: codes in the unit, scale pair / zero entry per group, x fragment
};

template <int BITS, int GPT>
__device__ __forceinline__ Lane lane_offsets(int lane, int M) {
  constexpr int SB = BITS == 4 ? 16 : 32;
  const int gr = lane >> 2, t = lane & 3;
  Lane o;
  o.w = lane * SB;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int gi = GPT == 1 ? 0 : h;
    o.s[h] = unit_scale_offset(BITS, gi, gr);
    o.z[h] = unit_zero_offset(BITS, GPT, gi, gr);
  }
  // B-fragment column gr is token gr; lanes past the last token read token 0
  // (their columns of D are never stored).
  o.x = (gr < M ? gr : 0) * 256 + 32 * t;
  return o;
}

template <int BITS, int GPT>
__device__ __forceinline__ void load_unit(Unit<BITS, GPT>& R, const uint8_t* ub, const Lane& o) {
  constexpr int SB = BITS == 4 ? 16 : 32;
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int v = 0; v < SB / 16; ++v) R.w[h][v] = *reinterpret_cast<const uint4*>(ub + o.w + h * 32 * SB + v * 16);
#pragma unroll
  for (int g = 0; g < GPT; ++g) {
    R.sp[g] = *reinterpret_cast<const uint32_t*>(ub + o.s[g]);
    R.zp[g] = BITS == 4 ? (uint32_t)ub[o.z[g]] : (uint32_t)*reinterpret_cast<const uint16_t*>(ub + o.z[g]);
  }
}

// Per-group dequantisation of a group's sums: y += f s (acc - z X), rows gr
// (acc[0..1]) and gr + 8 (acc[2..3]), tokens 2t, 2t + 1.  XF holds per token
// {X, f}: X = 2^-24 * sum_k x_k over the group in the block's scaled units
// (the codes carry 2^-24) and f = 2^(24 - e) undoes the block's scale 2^e.
// INT4 rows gr + 8 carry 16 q, so their zero is taken as 16 z (the 1/16 is
// applied at the end).
template <int BITS, bool ONE>
__device__ __forceinline__ void dequant_group(uint32_t sp, uint32_t zp, const float* XF, const float (&acc)[4],
                                              float (&yacc)[4]) {
  const float s_lo = __uint_as_float(sp << 16), s_hi = __uint_as_float(sp & 0xFFFF0000u);
  // -z as float: 2^23 - (2^23 + z), exact
  float nz_lo, nz_hi;
  if (BITS == 4) {
    nz_lo = 8388608.f - __uint_as_float(and_or(zp, 0x0Fu, 0x4B000000u));
    nz_hi = 8388608.f - __uint_as_float(and_or(zp, 0xF0u, 0x4B000000u));
  } else {
    nz_lo = 8388608.f - __uint_as_float(and_or(zp, 0xFFu, 0x4B000000u));
    nz_hi = 8388608.f - __uint_as_float(__byte_perm(zp, 0x4B000000u, 0x7441));
  }
  if (ONE) {
    const float2 xf = *reinterpret_cast<const float2*>(XF);
    yacc[0] = fmaf(s_lo * xf.y, fmaf(nz_lo, xf.x, acc[0]), yacc[0]);
    yacc[2] = fmaf(s_hi * xf.y, fmaf(nz_hi, xf.x, acc[2]), yacc[2]);
  } else {
    const float4 xf = *reinterpret_cast<const float4*>(XF);  // tokens 2t, 2t + 1
    yacc[0] = fmaf(s_lo * xf.y, fmaf(nz_lo, xf.x, acc[0]), yacc[0]);
    yacc[1] = fmaf(s_lo * xf.w, fmaf(nz_lo, xf.z, acc[1]), yacc[1]);
    yacc[2] = fmaf(s_hi * xf.y, fmaf(nz_hi, xf.x, acc[2]), yacc[2]);
    yacc[3] = fmaf(s_hi * xf.w, fmaf(nz_hi, xf.z, acc[3]), yacc[3]);
  }
}

// Component j of a 16-byte register group.
__device__ __forceinline__ uint32_t comp(const uint4& v, int j) {
  return j == 0 ? v.x : (j == 1 ? v.y : (j == 2 ? v.z : v.w));
}

// NU units at once: xu[u] = unit u's activations (fp16 [M][128]) plus this
// lane's fragment offset, xsu[u] = its group sums (plus this lane's token
// pair).  The MMAs of all units and both K halves are interleaved, one
// accumulator per (unit, half), so that 2 NU independent chains hide the
// tensor pipe's latency.
template <int BITS, int GPT, bool ONE, int NU>
__device__ __forceinline__ void units_step(const Unit<BITS, GPT>* W, const uint8_t* const* xu,
                                           const float* const* xsu, int xs_half, float (&yacc)[4]) {
  float acc[NU][2][4];
  uint32_t xs[NU][2][8];
#pragma unroll
  for (int u = 0; u < NU; ++u)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint4 xa = *reinterpret_cast<const uint4*>(xu[u] + h * 128);
      const uint4 xb = *reinterpret_cast<const uint4*>(xu[u] + h * 128 + 16);
      xs[u][h][0] = xa.x; xs[u][h][1] = xa.y; xs[u][h][2] = xa.z; xs[u][h][3] = xa.w;
      xs[u][h][4] = xb.x; xs[u][h][5] = xb.y; xs[u][h][6] = xb.z; xs[u][h][7] = xb.w;
    }
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int u = 0; u < NU; ++u) {
        uint32_t af[4];
        if (BITS == 4) {
          codes_w4(comp(W[u].w[h][0], j), af);
        } else {
          const uint4& v = W[u].w[h][BITS == 4 ? 0 : (j >> 1)];
          codes_w8(comp(v, (2 * j) & 3), comp(v, (2 * j + 1) & 3), af);
        }
        if (j == 0) mma_f16_first(acc[u][h], af, xs[u][h][2 * j], xs[u][h][2 * j + 1]);
        else mma_f16(acc[u][h], af, xs[u][h][2 * j], xs[u][h][2 * j + 1]);
      }
#pragma unroll
  for (int u = 0; u < NU; ++u) {
    if (GPT == 1) {
      float sum[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) sum[e] = acc[u][0][e] + acc[u][1][e];
      dequant_group<BITS, ONE>(W[u].sp[0], W[u].zp[0], xsu[u], sum, yacc);
    } else {
#pragma unroll
      for (int h = 0; h < 2; ++h)
        dequant_group<BITS, ONE>(W[u].sp[GPT == 1 ? 0 : h], W[u].zp[GPT == 1 ? 0 : h], xsu[u] + h * xs_half,
                                 acc[u][h], yacc);
    }
  }
}

// ---------------------------------------------------------------------------
// activations: BF16 [M, K] -> FP16 [kt][token][128] in shared memory, scaled
// per token by a power of two, plus per-group sums

// The exponent fields of the eight BF16 values of a chunk, reduced to the
// largest per 16-bit lane (two lanes per word, each holding its field << 7);
// the sign and mantissa bits are masked off, so unsigned 16-bit maxima
// order the fields.
__device__ __forceinline__ uint32_t chunk_max_exponent2(const uint4 v) {
  constexpr uint32_t kExp = 0x7F807F80u;
  return __vmaxu2(__vmaxu2(v.x & kExp, v.y & kExp), __vmaxu2(v.z & kExp, v.w & kExp));
}

// Power-of-two exponent e that maps the largest |x| of a token (BF16
// exponent field E) below 2^15, clamped so that 2^e and 2^(24 - e) are normal
// floats.
// Eight BF16 activations from p, of which the first n (>= 1) exist (the
// rest read as zero), element by element: rows of K % 8 != 0 values are
// not 16-byte aligned.
__device__ __forceinline__ uint4 load_x8(const uint16_t* p, int n) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t lo = 2 * i < n ? __ldcg(p + 2 * i) : 0u, hi = 2 * i + 1 < n ? __ldcg(p + 2 * i + 1) : 0u;
    w[i] = lo | hi << 16;
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ int token_shift(uint32_t E) {
  const int e = 141 - (int)E;
  return e < -103 ? -103 : (e > 127 ? 127 : e);
}

__device__ __forceinline__ float pow2f(int e) { return __uint_as_float((uint32_t)(127 + e) << 23); }

__device__ __forceinline__ uint32_t h2_bits(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// ---------------------------------------------------------------------------
// slab reductions


// ---------------------------------------------------------------------------
// the kernel

template <int BITS, int GPT, bool ONE, bool HALF>
__global__ void __launch_bounds__(kSThreads, 1) gemv_stream_kernel(const StreamArgs a) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  // 128-byte alignment by offsetting the array itself (not through an integer
  // cast), so that every access below stays a shared-memory access
  uint8_t* smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
  constexpr int UB = unit_bytes_gpu(BITS, GPT);
  constexpr int S = warp_stage_units(BITS, HALF);
  constexpr int SB = S * UB;  // bytes of a stage
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gr = lane >> 2, t = lane & 3;
  const int c = blockIdx.x;
  const int NS = a.NS;
  const int Mp = a.Mp;
  const int KT = a.KT;
  const int x_unit = ONE ? 256 : a.M * 256;  // bytes of one unit's activations
  const int xs_row = ONE ? 1 : 8;             // group sums per group: tokens (padded to 8)
  const int xs_half = ONE ? 2 : 16;           // floats between the two halves' {X, f} entries (GPT 2)

  const uint32_t sbase = smem_u32(smem);
  uint8_t* xres = smem + a.off_x;
  float* xsum = reinterpret_cast<float*>(smem + a.off_xs);  // {X, f} per (group of a unit, token)
  // parked sums: [max_slabs][16 warps][16 rows][Mp], or (compact) [16 warps][2][16 rows][Mp]
  float* red = reinterpret_cast<float*>(smem + a.off_red);
  const uint32_t full = sbase + (uint32_t)a.off_ctl;      // [16 warps][NS] mbarriers
  int* flags = reinterpret_cast<int*>(smem + a.off_ctl + 8 * kSW * NS);  // [0] a wait ran out, [1] bad header
  float* bias_s = reinterpret_cast<float*>(smem + a.off_ctl + 8 * kSW * NS + 8);  // this CTA's rows' bias

  // This CTA's whole slabs [s0, s0 + nslabs), i.e. units [u0, u1), and this
  // warp's run [g0, g0 + nu) of them (memory order).
  // The first nslab mod G CTAs take one slab more than the others.  Blocks
  // are placed on SMs in index order as the previous kernel's blocks leave
  // them, so the low indices start first: the extra slabs go where the
  // stream starts earliest, and the last blocks to start have the least to
  // do.
  const int q_all = a.nslab / a.G, r_all = a.nslab - q_all * a.G;
  const int s0 = c * q_all + (c < r_all ? c : r_all);
  const int nslabs = q_all + (c < r_all ? 1 : 0);
  const int u0 = s0 * KT, u1 = (s0 + nslabs) * KT;
  int g0, nu;
  warp_run(u0, u1, warp, g0, nu);
  const int nst = (nu + S - 1) / S;  // stages of this warp
  const uint32_t ring = sbase + (uint32_t)(warp * NS * SB);
  const uint32_t wbar = full + 8u * (uint32_t)(warp * NS);

  uint4 h0 = make_uint4(0, 0, 0, 0), h1 = h0;
  if (threadIdx.x == 0) {
    // the header of the blob, compared with the call's arguments before
    // anything is written (see below)
    load_header(a.units, h0, h1);
    for (int i = 0; i < kSW * NS; ++i) mbar_init(full + 8 * i, 1);
    flags[0] = 0;
    flags[1] = 0;
    mbar_init_fence();
  }
  // Parked sums start at zero: a warp writes only the slabs its run touches.
  // Compact form: a warp's run touches at most two slabs (it is shorter than
  // a slab: a CTA never holds more than 16 slabs), so each warp has two
  // slots, for the slab of its first unit and the next.
  for (int i = threadIdx.x; i < (a.compact ? 2 * kSW : nslabs * kSW) * 16 * Mp; i += kSThreads) red[i] = 0.f;
  __syncthreads();
  // The static weights start streaming before the previous kernel on the
  // stream has finished; x, y and the workspace wait for it.
  const int npre = nst < a.npre ? nst : a.npre;
  const int nring = nst < NS ? nst : NS;
  if (threadIdx.x == 0) griddep_launch_dependents();
  if (lane == 0)  // every warp requests its own stages
    for (int i = 0; i < npre; ++i)
      warp_fill<BITS, GPT>(a, ring + (uint32_t)(i * SB), wbar + 8u * i, g0 + i * S, nu - i * S < S ? nu - i * S : S);
  // the bias, static like the weights, is read before the dependency too
  if (a.epi.bias)
    for (int i = threadIdx.x; i < nslabs * kSlabN; i += kSThreads) {
      const int nn = s0 * kSlabN + i;
      bias_s[i] = nn < a.N ? bf16_bits_to_float(a.epi.bias[nn]) : 0.f;
    }
  griddep_wait();
  // Activations: each half warp takes one 128-column block of one token at
  // a time (lane l: columns 8l .. 8l + 7), straight into registers: its
  // largest exponent, the power-of-two scale, the FP16 conversion and the
  // group sums all come from shuffles inside the half warp, so one barrier
  // publishes everything.
  {
    const int hw = lane >> 4, r = lane & 15;
    const int hid = warp * 2 + hw;  // half warp of the CTA
    const int nblk = KT * a.M;
    constexpr int kBatch = 4;  // blocks per half warp whose loads are in flight together
    // blocks hid, hid + 32, hid + 64, ... (every half warp busy, loads batched)
    for (int base = 0; base < nblk; base += 2 * kSW * kBatch) {  // uniform over the warp
      uint4 v[kBatch];
#pragma unroll
      for (int q = 0; q < kBatch; ++q) {
        const int b = base + q * 2 * kSW + hid;
        const int kt = ONE ? b : b / a.M, m = ONE ? 0 : b - kt * a.M;
        const int col = kt * kTileK + 8 * r;
        v[q] = make_uint4(0, 0, 0, 0);
        if (b < nblk && col < a.K) {
          const uint16_t* src = a.x + (size_t)m * a.K + col;
          v[q] = a.K % 8 == 0 ? __ldcg(reinterpret_cast<const uint4*>(src)) : load_x8(src, a.K - col);
        }
      }
#pragma unroll
      for (int q = 0; q < kBatch; ++q) {
        const int b = base + q * 2 * kSW + hid;  // uniform over the half warp
        if (base + q * 2 * kSW >= nblk) break;   // uniform over the warp
        uint32_t E2 = chunk_max_exponent2(v[q]);
#pragma unroll
        for (int d = 1; d < 16; d <<= 1) E2 = __vmaxu2(E2, __shfl_xor_sync(0xFFFFFFFFu, E2, d));
        const uint32_t E = max(E2 & 0xFFFFu, E2 >> 16) >> 7;  // largest exponent field of the block
        const int e = token_shift(E);
        const float sc = pow2f(e);
        const uint32_t w[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
        float f[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          f[2 * i] = __uint_as_float(w[i] << 16) * sc;
          f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u) * sc;
        }
        float sum = ((f[0] + f[1]) + (f[2] + f[3])) + ((f[4] + f[5]) + (f[6] + f[7]));
        sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 1);
        sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 2);
        sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 4);
        if (GPT == 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 8);
        if (b < nblk) {
          const int kt = ONE ? b : b / a.M, m = ONE ? 0 : b - kt * a.M;
          uint4* p = reinterpret_cast<uint4*>(xres + (kt * a.M + m) * 256 + r * 16);
          if (BITS == 4)
            *p = make_uint4(h2_bits(f[0], f[1]), h2_bits(f[2], f[3]), h2_bits(f[4], f[5]), h2_bits(f[6], f[7]));
          else  // columns (c, c + 2), (c + 1, c + 3) of each 4-column group, as the INT8 codes
            *p = make_uint4(h2_bits(f[0], f[2]), h2_bits(f[1], f[3]), h2_bits(f[4], f[6]), h2_bits(f[5], f[7]));
          if ((r & (GPT == 1 ? 15 : 7)) == 0) {
            const int h = r >> 3;
            *reinterpret_cast<float2*>(xsum + ((kt * GPT + (GPT == 1 ? 0 : h)) * xs_row + m) * 2) =
                make_float2(sum * 5.9604644775390625e-8f, pow2f(24 - e));  // 2^-24, 2^(24 - e)
          }
        }
      }
    }
  }
  if (threadIdx.x == 0) {
    flags[1] = header_matches(h0, h1, a.N, a.K, BITS, a.group) ? 0 : 1;
  }
  __syncthreads();
  bool dead = flags[1] != 0;  // a header that does not match: write nothing
  if (dead && threadIdx.x == 0) atomicCAS(a.err, 0u, kErrBlobHeader);
  // x is in: the rest of the rings follows (requested earlier, these stages
  // would have reached the SM ahead of the activations)
  int issued = a.stall ? 0 : npre;  // stages of this warp requested so far
  if (!dead && !a.stall) {
    if (lane == 0)
      for (int i = npre; i < nring; ++i)
        warp_fill<BITS, GPT>(a, ring + (uint32_t)(i * SB), wbar + 8u * i, g0 + i * S, nu - i * S < S ? nu - i * S : S);
    issued = nring;
  }

  // ---- the stream: this warp's units, S per stage
  const Lane o = lane_offsets<BITS, GPT>(lane, a.M);
  float yacc[4] = {0.f, 0.f, 0.f, 0.f};
  int cur = g0 / KT;  // slab of the running sums
  // park this warp's sums of slab `cur` and go on with the next slab
  auto flush = [&]() {
    float* rb = red + (size_t)(a.compact ? warp * 2 + (cur - g0 / KT) : (cur - s0) * kSW + warp) * 16 * Mp;
    if (ONE) {
      if (t == 0) {
        rb[gr] = yacc[0];
        rb[gr + 8] = yacc[2];
      }
    } else if (2 * t < Mp) {
      *reinterpret_cast<float2*>(rb + gr * Mp + 2 * t) = make_float2(yacc[0], yacc[1]);
      *reinterpret_cast<float2*>(rb + (gr + 8) * Mp + 2 * t) = make_float2(yacc[2], yacc[3]);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) yacc[e] = 0.f;
    ++cur;
  };
  int slot = 0;
  uint32_t par = 0;
  Unit<BITS, GPT> W[S];
  int i = 0;
  for (; i < nst && !dead; ++i) {
    const int lo = g0 + i * S, n = nu - i * S < S ? nu - i * S : S;  // units [lo, lo + n)
    // one lane waits (suspended in hardware between polls), the warp follows
    unsigned ok = 1;
    if (lane == 0) ok = mbar_wait_sleep(wbar + 8u * slot, par, a.err, kErrStreamWait, a.wait_ns) ? 1u : 0u;
    if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) {
      dead = true;
      break;
    }
    const uint8_t* stp = smem + (warp * NS + slot) * SB;
    if (lo == (cur + 1) * KT) flush();
    if (n == S && lo + S <= (cur + 1) * KT) {
      // every unit of the stage belongs to the current slab
      const int kt = lo - cur * KT;
      const uint8_t* xu[S];
      const float* xsu[S];
#pragma unroll
      for (int j = 0; j < S; ++j) {
        load_unit<BITS, GPT>(W[j], stp + j * UB, o);
        xu[j] = xres + (kt + j) * x_unit + o.x;
        xsu[j] = xsum + ((kt + j) * GPT * xs_row + (ONE ? 0 : 2 * t)) * 2;
      }
      if (S % 2 == 0) {  // two units at a time: four independent accumulator chains
#pragma unroll
        for (int j = 0; j < S; j += 2) units_step<BITS, GPT, ONE, 2>(W + j, xu + j, xsu + j, xs_half, yacc);
      } else {
        units_step<BITS, GPT, ONE, S>(W, xu, xsu, xs_half, yacc);
      }
    } else {
#pragma unroll
      for (int j = 0; j < S; ++j) {
        if (j < n) {
          if (lo + j == (cur + 1) * KT) flush();
          const int kt = lo + j - cur * KT;
          load_unit<BITS, GPT>(W[0], stp + j * UB, o);
          const uint8_t* xu = xres + kt * x_unit + o.x;
          const float* xsu = xsum + (kt * GPT * xs_row + (ONE ? 0 : 2 * t)) * 2;
          units_step<BITS, GPT, ONE, 1>(W, &xu, &xsu, xs_half, yacc);
        }
      }
    }
    // The stage's codes have been used (so its reads are complete): refill it.
    __syncwarp();
    if (i + NS < nst) {
      if (lane == 0) {
        const int f = i + NS;
        warp_fill<BITS, GPT>(a, ring + (uint32_t)(slot * SB), wbar + 8u * slot, g0 + f * S,
                             nu - f * S < S ? nu - f * S : S);
      }
      ++issued;
    }
    if (++slot == NS) {
      slot = 0;
      par ^= 1u;
    }
  }
  if (nu > 0 && !dead) flush();
  if (dead && lane == 0) {
    atomicOr(flags, 1);
    // let this warp's copies still in flight land before shared memory goes away
    for (int k = i; k < issued; ++k)
      mbar_wait(wbar + 8u * (k % NS), (uint32_t)(k / NS) & 1u, a.err, kErrStreamWait, kDrainNs);
  }
  __syncthreads();
  if (flags[0] || flags[1]) return;

  // Add the sixteen warps' parked sums of every slab in warp order; write y.
  // (The INT4 rows gr + 8 carry 16 q: their sums are divided by 16 here.)
  const int per = ONE ? 16 : 16 * Mp;
  auto parked = [&](int sl, int idx) {
    float v = 0.f;
    if (!a.compact) {
#pragma unroll
      for (int w = 0; w < kSW; ++w) v += red[(size_t)(sl * kSW + w) * per + idx];
    } else {
      // the warps whose runs touch slab s0 + sl, in warp order
#pragma unroll 4
      for (int w = 0; w < kSW; ++w) {
        int wg0, wnu;
        warp_run(u0, u1, w, wg0, wnu);
        const int d = s0 + sl - wg0 / KT;  // slot of this slab in warp w
        if (wnu > 0 && (d == 0 || d == 1)) v += red[(size_t)(w * 2 + d) * per + idx];
      }
    }
    return v;
  };
  const bool gate = a.epi.mode == kEpiSiluGate;
  for (int q = threadIdx.x; q < nslabs * per; q += kSThreads) {
    const int sl = q / per, idx = q - sl * per;
    const int row = ONE ? idx : idx / Mp, tok = ONE ? 0 : idx - row * Mp;
    const int nn = (s0 + sl) * kSlabN + row;
    if (tok >= a.M || nn >= a.N || (gate && row >= 8)) continue;
    const float v = parked(sl, idx);
    if (gate) {  // gate row nn (row < 8) with its up row nn + 8
      const float u = parked(sl, idx + 8 * Mp);
      const float ub = BITS == 4 ? u * 0.0625f : u;
      const float* b = bias_s + sl * kSlabN + row;
      epi_put_gate(a.epi, tok, nn, a.epi.bias ? v + b[0] : v, a.epi.bias ? ub + b[8] : ub);
    } else {
      const float vb = BITS == 4 && row >= 8 ? v * 0.0625f : v;
      epi_put(a.epi, tok, nn, a.epi.bias ? vb + bias_s[sl * kSlabN + row] : vb);
    }
  }
}

}  // namespace

// ---------------------------------------------------------------------------
// host side

int stream_plan(const Geometry& G, int M, StreamPlan* P) {
  if (G.gpt > 2 || M < 1 || M > 8) return 0;
  const int sms = sm_count();
  if (sms <= 0) return 0;
  const int nslab = (G.N + kSlabN - 1) / kSlabN;
  // one CTA per slab on layers with fewer slabs than SMs
  StreamPlan S{};
  S.G = nslab < sms ? nslab : sms;
  S.Mp = M == 1 ? 1 : (M + 1) / 2 * 2;
  S.max_slabs = (nslab + S.G - 1) / S.G;
  const int xres = (G.KT * M * 256 + 127) / 128 * 128;
  const int xs = (G.KT * G.gpt * (M == 1 ? 1 : 8) * 8 + 127) / 128 * 128;
  // full-size stages and one parked slot per (slab, warp) first; then
  // half-size stages; then two parked slots per warp
  for (int cfg = 0; cfg < 4; ++cfg) {
    const int half = cfg & 1, compact = cfg >> 1;
    if (compact && S.max_slabs > kSW) break;  // two slots need runs shorter than a slab
    const int red = (compact ? 2 : S.max_slabs) * kSW * 16 * S.Mp * 4;
    const int stage = warp_stage_units(G.bits, half != 0) * G.unit_bytes;
    for (int ns = TF_STREAM_NS_MAX; ns >= 2; --ns) {
      const int ring = (kSW * ns * stage + 127) / 128 * 128;
      const int ctl = 8 * kSW * ns + 8 + S.max_slabs * kSlabN * 4;  // mbarriers, flags, the rows' bias
      const size_t smem = 128 + (size_t)ring + xres + xs + red + ctl;
      if (smem <= (size_t)kSmemMax) {
        S.half = half;
        S.compact = compact;
        S.NS = ns;
        S.npre = TF_STREAM_NPRE < ns ? TF_STREAM_NPRE : ns;
        S.off_x = ring;
        S.off_xs = S.off_x + xres;
        S.off_red = S.off_xs + xs;
        S.off_ctl = S.off_red + red;
        S.smem = smem;
        *P = S;
        return 1;
      }
    }
  }
  return 0;
}

template <int BITS, int GPT, bool ONE>
static int launch_stream(const StreamArgs& a, bool half, size_t smem, cudaStream_t s) {
  static std::atomic<unsigned long long> opted{0}, opted_half{0};
  if (half) return launch_pdl(gemv_stream_kernel<BITS, GPT, ONE, true>, opted_half, a.G, kSThreads, kSmemMax, smem, s, a);
  return launch_pdl(gemv_stream_kernel<BITS, GPT, ONE, false>, opted, a.G, kSThreads, kSmemMax, smem, s, a);
}

int run_stream(const Geometry& G, const StreamPlan& P, const void* blob, const uint16_t* x, const Epi& epi, int M,
               cudaStream_t stream) {
  StreamArgs a;
  a.units = static_cast<const uint8_t*>(blob) + kHeaderBytes;
  a.x = x; a.epi = epi;
  a.err = device_error_ptr();
  if (!a.err) return TF_ERR_CUDA;
  a.nslab = (G.N + kSlabN - 1) / kSlabN;
  a.N = G.N; a.K = G.K; a.M = M; a.Mp = P.Mp; a.KT = G.KT; a.G = P.G; a.group = G.group;
  a.NS = P.NS; a.npre = P.npre;
  a.off_x = P.off_x; a.off_xs = P.off_xs; a.off_red = P.off_red; a.off_ctl = P.off_ctl;
  a.max_slabs = P.max_slabs;
  a.compact = P.compact;
  const TestHook hook = test_hook();
  a.stall = hook.stall;
  a.wait_ns = hook.wait_ns;
  const bool one = M == 1, h = P.half != 0;
  if (G.bits == 4) {
    if (G.gpt == 1)
      return one ? launch_stream<4, 1, true>(a, h, P.smem, stream) : launch_stream<4, 1, false>(a, h, P.smem, stream);
    return one ? launch_stream<4, 2, true>(a, h, P.smem, stream) : launch_stream<4, 2, false>(a, h, P.smem, stream);
  }
  if (G.gpt == 1)
    return one ? launch_stream<8, 1, true>(a, h, P.smem, stream) : launch_stream<8, 1, false>(a, h, P.smem, stream);
  return one ? launch_stream<8, 2, true>(a, h, P.smem, stream) : launch_stream<8, 2, false>(a, h, P.smem, stream);
}

}  // namespace tf
