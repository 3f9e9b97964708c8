// Dequant (parity path) and fused GEMV kernels of libtf, with their C ABI.
//
// GEMV = token generation at batch 1 (TileFuse, Methodology 3 "GEMV dataflow
// co-design").  The pages' point is that a quantised GEMV, memory-bound at
// full precision, turns compute-bound once unpack and dequant are added, and
// that the weight stream must be spread over the whole array.  The GB300
// version: every SM streams contiguous runs of pre-tiled units, each lane
// unpacks and dequantises its codes in registers, and the dequantised BF16
// fragments go straight into mma.sync so that the tensor cores do the
// multiply-accumulate instead of CUDA-core FMAs.
//
// The layers with groups of 64, any multiple of 128 or per channel whose
// activations fit in shared memory (every decode projection of a
// Llama-class model) go to the stream GEMV of gemv_stream.cu, which skips
// the per-weight BF16 rounding.  This file holds the entry points, the
// routing, and the two GEMVs for the other layers (groups of 32, or
// activations too large), and for tf_gemm at M <= 8, which dequantise each
// weight to BF16 in registers (bit-exact, as tf_dequant) and share one inner
// step (one 16-row x 128-column unit per warp):
//  * slab GEMV, for layers with K >= 1024 whose activations fit in shared
//    memory: each CTA owns whole slabs over all of K (one CTA per slab on
//    layers with fewer slabs than SMs), its eight (or sixteen) warps split K,
//    and a slab's partial sums meet in shared memory.  No CTA waits on
//    another, so a layer ends as soon as its last slab is done.
//  * tile GEMV, for the rest (K < 1024, or activations too large to stay
//    resident): K is split across CTAs too; a 128-row block shared by
//    several CTAs is summed by the last of them, in a fixed order, from FP32
//    partials in a workspace.
#include <cuda_runtime.h>

#include <atomic>

#include "../../include/tf.h"
#include "tf_abi.h"
#include "tf_device.cuh"
#include "tf_format.h"
#include "tf_sm100.cuh"

namespace tf {
namespace {

// ===========================================================================
// tf_dequant: one CTA per 128 x 128 tile, one thread per (slab, K half, slot).

template <int BITS, int GPT>
__global__ void __launch_bounds__(512) dequant_kernel(const uint8_t* __restrict__ units, int N, int K,
                                                      int KT, int g, int group, unsigned* err,
                                                      uint16_t* __restrict__ w) {
  constexpr int UB = unit_bytes_gpu(BITS, GPT);
  constexpr int SB = BITS == 4 ? 16 : 32;
  const int tile = blockIdx.x;
  const int nb = tile / KT, kt = tile - nb * KT;
  const int mb = threadIdx.x >> 6;
  const int h = (threadIdx.x >> 5) & 1;
  const int p = threadIdx.x & 31;
  const int gr = p >> 2, t = p & 3;
  const uint8_t* ub = units + ((size_t)(nb * kSlabsPerTile + mb) * KT + kt) * UB;
  const int gi = GPT == 1 ? 0 : (h * 64 + 16 * t) / g;
  const uint32_t sp = *reinterpret_cast<const uint32_t*>(ub + unit_scale_offset(BITS, gi, gr));
  const uint8_t* slot = ub + (h * 32 + p) * SB;
  const uint8_t* zp = ub + unit_zero_offset(BITS, GPT, gi, gr);

  uint32_t lo[8], hi[8];  // rows gr and gr + 8 of this slab, 16 columns each
  if (BITS == 4) {
    const MetaW4 m = meta_w4(sp, *zp);
    const uint4 v = *reinterpret_cast<const uint4*>(slot);
    const uint32_t words[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t a[4];
      dequant_w4(words[j], m, a);
      lo[2 * j] = a[0]; lo[2 * j + 1] = a[2];
      hi[2 * j] = a[1]; hi[2 * j + 1] = a[3];
    }
  } else {
    const MetaW8 m = meta_w8(sp, *reinterpret_cast<const uint16_t*>(zp));
    const uint4 v0 = reinterpret_cast<const uint4*>(slot)[0];
    const uint4 v1 = reinterpret_cast<const uint4*>(slot)[1];
    const uint32_t words[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t a[4];
      dequant_w8(words[2 * j], words[2 * j + 1], m, a);
      lo[2 * j] = a[0]; lo[2 * j + 1] = a[2];
      hi[2 * j] = a[1]; hi[2 * j + 1] = a[3];
    }
  }
  // a blob whose header describes another layer: write nothing
  uint4 h0, h1;
  load_header(units, h0, h1);
  if (!header_matches(h0, h1, N, K, BITS, group)) {
    if (threadIdx.x == 0 && tile == 0) atomicCAS(err, 0u, kErrBlobHeader);
    return;
  }
  const int n0 = nb * kTileN + mb * kSlabN + gr;
  const int k0 = kt * kTileK + h * 64 + 16 * t;
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int n = n0 + 8 * e;
    if (n >= N) continue;
    const uint32_t* src = e ? hi : lo;
    uint16_t* dst = w + (size_t)n * K + k0;
    if (K % 8 == 0) {  // rows of whole 16-byte pieces
      if (k0 < K) *reinterpret_cast<uint4*>(dst) = make_uint4(src[0], src[1], src[2], src[3]);
      if (k0 + 8 < K) *reinterpret_cast<uint4*>(dst + 8) = make_uint4(src[4], src[5], src[6], src[7]);
    } else {  // per channel with K % 8 != 0: element by element
#pragma unroll
      for (int c = 0; c < 16; ++c)
        if (k0 + c < K) dst[c] = (uint16_t)(src[c >> 1] >> (16 * (c & 1)));
    }
  }
}

// ===========================================================================
// GEMV: the per-warp unit step shared by both kernels.

constexpr int kGemvWarps = 8;
constexpr int kGemvThreads = 32 * kGemvWarps;
constexpr uint64_t kGemvDrainNs = 200000000ull;  // bounded wait for copies still in flight after an error
constexpr unsigned kErrGemvWait = 0x600;

// Registers of one unit's weights for one lane: its slot in both K halves
// and the unit's scale / zero words.
template <int BITS, int GPT>
struct WRegs {
  uint4 w[2][BITS == 4 ? 1 : 2];
  uint32_t sp[GPT == 1 ? 1 : 2], zp[GPT == 1 ? 1 : 2];
};

// Unit-relative byte offsets of one lane's operands.
struct LaneOffsets {
  int w, s0, s1, z0, z1, x;
};

template <int BITS, int GPT>
__device__ __forceinline__ LaneOffsets lane_offsets(int lane, int g, int M) {
  constexpr int SB = BITS == 4 ? 16 : 32;
  const int gr = lane >> 2, t = lane & 3;
  const int gi0 = GPT == 1 ? 0 : (16 * t) / g;         // group of this lane's columns in K half 0
  const int gi1 = GPT == 1 ? 0 : (64 + 16 * t) / g;    // ... and in K half 1
  LaneOffsets o;
  o.w = lane * SB;  // slot p = 4 gr + t = lane
  o.s0 = unit_scale_offset(BITS, gi0, gr);
  o.s1 = unit_scale_offset(BITS, gi1, gr);
  o.z0 = unit_zero_offset(BITS, GPT, gi0, gr);
  o.z1 = unit_zero_offset(BITS, GPT, gi1, gr);
  // B-fragment column gr is token gr; lanes past the last token read token
  // 0 instead (their columns of D are computed but never stored).
  o.x = (gr < M ? gr : 0) * 256 + 32 * t;
  return o;
}

// ub: the unit in shared memory.
template <int BITS, int GPT>
__device__ __forceinline__ void load_w(WRegs<BITS, GPT>& R, const uint8_t* ub, const LaneOffsets& o) {
  constexpr int SB = BITS == 4 ? 16 : 32;
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int v = 0; v < SB / 16; ++v) R.w[h][v] = *reinterpret_cast<const uint4*>(ub + o.w + h * 32 * SB + v * 16);
  R.sp[0] = *reinterpret_cast<const uint32_t*>(ub + o.s0);
  R.zp[0] = BITS == 4 ? (uint32_t)ub[o.z0] : (uint32_t)*reinterpret_cast<const uint16_t*>(ub + o.z0);
  if (GPT > 1) {
    R.sp[GPT == 1 ? 0 : 1] = *reinterpret_cast<const uint32_t*>(ub + o.s1);
    R.zp[GPT == 1 ? 0 : 1] = BITS == 4 ? (uint32_t)ub[o.z1] : (uint32_t)*reinterpret_cast<const uint16_t*>(ub + o.z1);
  }
}

// B fragments of K half h: x[token][h*64 + 16t .. +16] from the unit's
// activation slice xb = x[0..M)[128 columns] in shared memory.
__device__ __forceinline__ void load_x(uint32_t (&xs)[8], const uint8_t* xb, const LaneOffsets& o, int h) {
  const uint4 a = *reinterpret_cast<const uint4*>(xb + o.x + h * 128);
  const uint4 b = *reinterpret_cast<const uint4*>(xb + o.x + h * 128 + 16);
  xs[0] = a.x; xs[1] = a.y; xs[2] = a.z; xs[3] = a.w;
  xs[4] = b.x; xs[5] = b.y; xs[6] = b.z; xs[7] = b.w;
}

// Unpack, dequantise (bit-exact BF16) and multiply-accumulate K half h of a unit.
template <int BITS, int GPT>
__device__ __forceinline__ void mma_half(const WRegs<BITS, GPT>& R, int h, const uint32_t (&xs)[8],
                                         float (&acc)[4]) {
  const int mi = GPT == 1 ? 0 : h;
  if (BITS == 4) {
    const MetaW4 m = meta_w4(R.sp[mi], R.zp[mi]);
    const uint32_t words[4] = {R.w[h][0].x, R.w[h][0].y, R.w[h][0].z, R.w[h][0].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t af[4];
      dequant_w4(words[j], m, af);
      mma_16816(acc, af, xs[2 * j], xs[2 * j + 1]);
    }
  } else {
    const MetaW8 m = meta_w8(R.sp[mi], R.zp[mi]);
    const uint4 v0 = R.w[h][0], v1 = R.w[h][BITS == 4 ? 0 : 1];
    const uint32_t words[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t af[4];
      dequant_w8(words[2 * j], words[2 * j + 1], m, af);
      mma_16816(acc, af, xs[2 * j], xs[2 * j + 1]);
    }
  }
}

// A whole unit with its activations already in registers (xs[h]).
template <int BITS, int GPT>
__device__ __forceinline__ void mma_unit(const WRegs<BITS, GPT>& R, const uint32_t (&xs)[2][8], float (&acc)[2][4]) {
  mma_half(R, 0, xs[0], acc[0]);
  mma_half(R, 1, xs[1], acc[1]);
}

// v = this lane's sums for rows n0, n0 + 8 and tokens 2t, 2t + 1, written
// through the epilogue (which adds the bias before the one rounding to BF16).
// In the SiLU-gate epilogue n0 is a gate row and n0 + 8 its up row.
__device__ __forceinline__ void store_y(const Epi& e, int n0, int t, const float (&v)[4]) {
  const int m0 = 2 * t, m1 = 2 * t + 1, n1 = n0 + 8;
  if (n0 >= e.N) return;
  if (e.mode == kEpiSiluGate) {
    if (m0 < e.M) epi_put_gate(e, m0, n0, epi_biased(e, n0, v[0]), epi_biased(e, n1, v[2]));
    if (m1 < e.M) epi_put_gate(e, m1, n0, epi_biased(e, n0, v[1]), epi_biased(e, n1, v[3]));
    return;
  }
  if (m0 < e.M) epi_put(e, m0, n0, epi_biased(e, n0, v[0]));
  if (m1 < e.M) epi_put(e, m1, n0, epi_biased(e, n0, v[1]));
  if (n1 < e.N) {
    if (m0 < e.M) epi_put(e, m0, n1, epi_biased(e, n1, v[2]));
    if (m1 < e.M) epi_put(e, m1, n1, epi_biased(e, n1, v[3]));
  }
}

__device__ __forceinline__ uint8_t* align128(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 127) & ~uintptr_t(127));
}

// Wait on a ring barrier with every lane; the result is the same for the
// whole warp (a lane that gave up makes the warp give up).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, unsigned* err, uint64_t wait_ns) {
  return mbar_wait_warp(bar, parity, err, kErrGemvWait, wait_ns);
}

// ===========================================================================
// tile GEMV (split-K across CTAs)
//
// Work split: the T = NB * KT tiles (eight units: the eight slabs of a
// 128-row block at one kt) are numbered n-block major and CTA c streams tiles
// [c*T/G, (c+1)*T/G).  A shared-memory ring holds four INT4 or two INT8 tiles
// per stage (one bulk copy per unit, issued by the lanes of one warp); the
// tiles' activation slices x[:, kt*128 : kt*128+128] arrive alongside by 2-D
// TMA (zero-filled past K).  The warp that hands a stage back last refills
// it, so no warp is dedicated to (or delayed by) producing.  Warp w of the
// CTA owns slab w of every tile, so no intra-CTA reduction is needed.  A
// CTA's range covers whole or partial 128-row blocks ("segments"); a whole
// block is written straight to y, a partial one is stored as FP32 fragments
// in the workspace and the last of the block's contributors (arrival counter
// per slab) adds them in CTA order — a fixed order, so the result does not
// depend on arrival order.
//
// Both GEMV kernels use programmatic dependent launch: the weight stream
// (static data) starts before the previous kernel on the stream has
// finished; activations, y and the workspace are touched only after it has.

// tiles per ring stage of the tile GEMV
__host__ __device__ constexpr int tiles_per_stage(int bits) { return bits == 4 ? 4 : 2; }
static_assert(tiles_per_stage(4) * kSlabsPerTile <= 32 && tiles_per_stage(8) * kSlabsPerTile <= 32,
              "one lane issues the bulk copy of one unit of a stage");

struct GemvArgs {
  const uint8_t* units;
  Epi epi;  // where y goes (plain, SiLU gate or split) and the bias
  float4* partials;    // [G][S_max][8 warps][32 lanes]
  unsigned* counters;  // [NB][8 warps], zero on entry and on exit
  unsigned* err;
  long long T;
  uint64_t wait_ns;  // limit of every wait
  int stall;         // failure-detection test: issue no copies
  int N, K, M, KT, g, G, S_max, group;
  int NS, stage_bytes, x_off;  // shared-memory ring: stages, bytes per stage, x slice offset
};

__device__ __forceinline__ long long tile_begin(long long c, long long T, int G) { return c * T / G; }

// CTA whose range holds tile x.
__device__ __forceinline__ int cta_of_tile(long long x, long long T, int G) {
  return (int)(((x + 1) * G - 1) / T);
}

// End of a segment of row block nb.  A whole block is written to y at once.
// A partial one is only stored in the workspace here; it is published (one
// fence for all of them) and counted at the end of the CTA's range, when no
// bulk copy of this CTA is in flight any more — a fence issued mid-stream
// waits behind the stream and delays the whole grid.  Returns true when the
// segment is pending.
__device__ __forceinline__ bool end_segment(const GemvArgs& a, int c, long long t0, int nb, bool whole, int warp,
                                            int lane, const float (&v)[4]) {
  const int gr = lane >> 2, t = lane & 3;
  if (whole) {
    store_y(a.epi, nb * kTileN + warp * kSlabN + gr, t, v);
    return false;
  }
  const int seg = nb - (int)(t0 / a.KT);
  __stcg(a.partials + ((size_t)(c * a.S_max + seg) * 8 + warp) * 32 + lane, make_float4(v[0], v[1], v[2], v[3]));
  return true;
}

// Count this CTA's contribution to row block nb (after the fence); the last
// contributor adds all partials in CTA order, writes y and resets the counter.
__device__ __forceinline__ void publish_segment(const GemvArgs& a, int nb, int warp, int lane) {
  const int gr = lane >> 2, t = lane & 3;
  unsigned old = 0;
  if (lane == 0) old = atomicAdd(a.counters + nb * 8 + warp, 1u);
  old = __shfl_sync(0xFFFFFFFFu, old, 0);
  const long long first_tile = (long long)nb * a.KT;
  const int c_first = cta_of_tile(first_tile, a.T, a.G);
  const int c_last = cta_of_tile(first_tile + a.KT - 1, a.T, a.G);
  if (old != (unsigned)(c_last - c_first)) return;
  fence_acq_rel_gpu();  // acquire: every contributor's partials are visible
  // Issue the loads of up to sixteen contributors at once, then add them in
  // CTA order: one L2 round trip per sixteen contributors, same sum every run.
  float s[4] = {0.f, 0.f, 0.f, 0.f};
  for (int c0 = c_first; c0 <= c_last; c0 += 16) {
    float4 u[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int cc = c0 + j;
      if (cc <= c_last) {
        const int sg = nb - (int)(tile_begin(cc, a.T, a.G) / a.KT);
        u[j] = __ldcg(a.partials + ((size_t)(cc * a.S_max + sg) * 8 + warp) * 32 + lane);
      }
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      if (c0 + j <= c_last) {
        s[0] += u[j].x; s[1] += u[j].y; s[2] += u[j].z; s[3] += u[j].w;
      }
    }
  }
  store_y(a.epi, nb * kTileN + warp * kSlabN + gr, t, s);
  if (lane == 0) a.counters[nb * 8 + warp] = 0u;
}

// Segment bookkeeping of one warp: local index of the segment's last tile,
// whether the segment covers its whole row block, and the block.
struct Segment {
  int end, nb;
  bool whole;
};

__device__ __forceinline__ Segment first_segment(long long t0, int ntile, int KT) {
  Segment g;
  g.nb = (int)(t0 / KT);
  const int kt0 = (int)(t0 - (long long)g.nb * KT);
  const int len = KT - kt0;
  g.end = (len < ntile ? len : ntile) - 1;
  g.whole = kt0 == 0 && len <= ntile;
  return g;
}

__device__ __forceinline__ void next_segment(Segment& g, int ntile, int KT) {
  const int start = g.end + 1;
  const int left = ntile - start;
  g.end = start + (KT < left ? KT : left) - 1;
  g.whole = KT <= left;
  ++g.nb;
}

// Issue fill f of this CTA's ring (tiles TPS*f .. of its range and their
// activation slices) into stage s.  Called by all lanes of one warp: lane i
// copies unit i % 8 of tile i / 8; lane 0 arms the barrier and loads the
// activations.  The activations are read only once the grid dependency has
// resolved (x).  `issued` counts the fills whose copies were started (for
// the drain after a wait that ran out).
template <int BITS, int GPT, int TPS>
__device__ __forceinline__ void issue_fill(const GemvArgs& a, const CUtensorMap* tmx, uint32_t sbase, uint32_t full,
                                           long long t0, int ntile, int f, int s, bool weights, bool x, int lane,
                                           int* issued) {
  constexpr int UB = unit_bytes_gpu(BITS, GPT);
  const int i = f * TPS;
  const int n = ntile - i < TPS ? ntile - i : TPS;
  if (a.stall) return;
  const uint32_t x_bytes = (uint32_t)a.M * 256u;
  const uint32_t bar = full + 8u * s;
  const uint32_t dst = sbase + (uint32_t)(s * a.stage_bytes);
  if (weights) {
    if (lane == 0) {
      mbar_arrive_expect_tx(bar, (uint32_t)n * ((uint32_t)(kSlabsPerTile * UB) + x_bytes));
      atomicMax(issued, f + 1);
    }
    __syncwarp();
    if (lane < n * kSlabsPerTile) {
      const int j = lane / kSlabsPerTile, mb = lane % kSlabsPerTile;
      const long long tt = t0 + i + j;
      const int nb = (int)(tt / a.KT), kt = (int)(tt - (long long)nb * a.KT);
      bulk_load_hint(dst + (uint32_t)(lane * UB), a.units + ((size_t)(nb * kSlabsPerTile + mb) * a.KT + kt) * UB,
                     (uint32_t)UB, bar, l2_evict_first_policy());  // weights are read once per call
    }
  }
  if (x && lane == 0) {
    for (int q = 0; q < n; ++q) {
      const int kt = (int)((t0 + i + q) % a.KT);
      tma_load_2d(dst + (uint32_t)a.x_off + (uint32_t)q * x_bytes, tmx, kt * kTileK, 0, bar);
    }
  }
}

template <int BITS, int GPT>
__global__ void __launch_bounds__(kGemvThreads, 2) gemv_kernel(const __grid_constant__ CUtensorMap tmx,
                                                               const GemvArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align128(smem_raw);
  constexpr int UB = unit_bytes_gpu(BITS, GPT);
  constexpr int kTilesPerStage = tiles_per_stage(BITS);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x;
  const long long t0 = tile_begin(c, a.T, a.G), t1 = tile_begin(c + 1, a.T, a.G);
  const int ntile = (int)(t1 - t0);
  const int nfill = (ntile + kTilesPerStage - 1) / kTilesPerStage;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t full = sbase + (uint32_t)(a.NS * a.stage_bytes);
  const uint32_t empty = full + 8u * a.NS;
  // per-stage release counters: the last warp to hand a stage back refills it
  unsigned* released = reinterpret_cast<unsigned*>(smem + a.NS * a.stage_bytes + 16 * a.NS);
  int* bad = reinterpret_cast<int*>(released + a.NS);  // the blob's header does not match the call
  int* issued = bad + 1;                               // fills whose copies were started
  int* dead = bad + 2;                                 // a wait ran out
  const int npre = nfill < a.NS ? nfill : a.NS;
  uint4 h0 = make_uint4(0, 0, 0, 0), h1 = h0;
  if (threadIdx.x == 0) {
    load_header(a.units, h0, h1);  // compared below, once the grid dependency has resolved
    for (int i = 0; i < a.NS; ++i) {
      mbar_init(full + 8 * i, 1);
      mbar_init(empty + 8 * i, kGemvWarps);
      released[i] = 0;
    }
    *issued = 0;
    *dead = 0;
    mbar_init_fence();
  }
  __syncthreads();
  if (ntile <= 0) return;
  if (warp == 0) {
    if (lane == 0) {
      griddep_launch_dependents();
      prefetch_tensormap(&tmx);
    }
    // static weights first, before the grid dependency resolves
    for (int f = 0; f < npre; ++f)
      issue_fill<BITS, GPT, kTilesPerStage>(a, &tmx, sbase, full, t0, ntile, f, f, true, false, lane, issued);
  }
  // y, x and the workspace may still be in use by the previous grid
  griddep_wait();
  if (threadIdx.x == 0) {
    *bad = header_matches(h0, h1, a.N, a.K, BITS, a.group) ? 0 : 1;
    if (*bad) atomicCAS(a.err, 0u, kErrBlobHeader);
  }
  if (warp == 0)
    for (int f = 0; f < npre; ++f)
      issue_fill<BITS, GPT, kTilesPerStage>(a, &tmx, sbase, full, t0, ntile, f, f, false, true, lane, issued);
  __syncthreads();
  // With a header that does not match, the stream still runs to the end (so
  // that every copy lands) but nothing is written.
  const bool write = *bad == 0;

  const int gr = lane >> 2, t = lane & 3;  // mma.sync fragment coordinates
  (void)gr;
  const LaneOffsets o = lane_offsets<BITS, GPT>(lane, a.g, a.M);
  const int x_stride = a.M * 256;

  float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  WRegs<BITS, GPT> R;
  uint32_t xs[2][8];
  Segment seg = first_segment(t0, ntile, a.KT);
  // at most two segments of a contiguous range are partial: its first and its last
  int pending0 = 0, pending1 = 0, npending = 0;
  int s = 0;
  uint32_t lap = 0;
  for (int f = 0; f < nfill; ++f) {
    if (!warp_wait(full + 8 * s, lap & 1u, a.err, a.wait_ns)) {
      if (lane == 0) atomicExch(dead, 1);
      break;
    }
    const int i0 = f * kTilesPerStage;
    const int n = ntile - i0 < kTilesPerStage ? ntile - i0 : kTilesPerStage;
    const uint8_t* st = smem + s * a.stage_bytes;
    const uint8_t* xst = st + a.x_off;
#pragma unroll
    for (int j = 0; j < kTilesPerStage; ++j) {
      if (j < n) {
        load_w(R, st + (j * kSlabsPerTile + warp) * UB, o);
        load_x(xs[0], xst + j * x_stride, o, 0);
        load_x(xs[1], xst + j * x_stride, o, 1);
        if (j == n - 1) {
          // the whole stage has been read: hand it back; the last warp to do
          // so refills it
          __syncwarp();
          unsigned refill = 0;
          if (lane == 0) {
            mbar_arrive(empty + 8 * s);
            if (atomicAdd(released + s, 1u) == kGemvWarps - 1) {
              released[s] = 0;
              refill = f + a.NS < nfill && mbar_wait(empty + 8 * s, lap & 1u, a.err, kErrGemvWait, a.wait_ns);
            }
          }
          if (__shfl_sync(0xFFFFFFFFu, refill, 0))
            issue_fill<BITS, GPT, kTilesPerStage>(a, &tmx, sbase, full, t0, ntile, f + a.NS, s, true, true, lane,
                                                  issued);
        }
        mma_unit(R, xs, acc);
        if (i0 + j == seg.end) {
          const float v[4] = {acc[0][0] + acc[1][0], acc[0][1] + acc[1][1], acc[0][2] + acc[1][2],
                              acc[0][3] + acc[1][3]};
          if (write && end_segment(a, c, t0, seg.nb, seg.whole, warp, lane, v)) {
            if (npending == 0) pending0 = seg.nb; else pending1 = seg.nb;
            ++npending;
          }
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[h][q] = 0.f;
          next_segment(seg, ntile, a.KT);
        }
      }
    }
    if (++s == a.NS) { s = 0; ++lap; }
  }
  (void)t;
  if (npending > 0) {
    fence_acq_rel_gpu();  // release: this lane's partials before any count below
    __syncwarp();
    publish_segment(a, pending0, warp, lane);
    if (npending > 1) publish_segment(a, pending1, warp, lane);
  }
  __syncthreads();
  if (threadIdx.x == 0 && *dead) {
    // A wait ran out: let the copies still in flight land before the CTA's
    // shared memory goes away.  A fill is started only after every warp has
    // handed back the fill NS before it, so only the last NS started fills
    // can be outstanding.
    const int n_iss = *issued;
    for (int f = n_iss > a.NS ? n_iss - a.NS : 0; f < n_iss; ++f)
      mbar_wait(full + 8 * (f % a.NS), (uint32_t)(f / a.NS) & 1u, a.err, kErrGemvWait, kGemvDrainNs);
  }
}

// ===========================================================================
// slab GEMV (whole slabs per CTA, K split across the CTA's warps)
//
// CTA c owns slabs [c*spc, min((c+1)*spc, nslab)) — one contiguous byte
// range of the blob — over all of K.  Its ring stage holds U = NW*UPW
// consecutive units of one slab (one bulk copy).  All of x is copied once,
// into a resident buffer, with 16-byte cp.async (load/store path, so it does
// not queue behind weight copies already issued to the TMA unit).  A CTA has
// eight warps (two CTAs per SM) or, when x is too large to stay resident
// next to a ring at two CTAs per SM, sixteen (one per SM).  Layers whose x
// does not fit even then take the tile GEMV.
// Warp w takes units w, w + NW, ... of every stage.  At the end of a slab
// each warp parks its partial sums in its own shared-memory slot and goes
// on; after the last slab the eight warps add the CTA's slabs in parallel
// (each slab's eight partials in warp order) and write y, so no warp waits
// for another inside the stream.

// Units per warp per ring stage (the eight-warp configuration's stages are
// twice as large: fewer handovers per unit).
__host__ __device__ constexpr int slab_units_per_warp(int bits, int nw) {
  return (bits == 4 ? 2 : 1) * (nw == 8 ? 2 : 1);
}

struct SlabArgs {
  const uint8_t* units;
  const uint16_t* x;
  Epi epi;  // where y goes (plain, SiLU gate or split) and the bias
  unsigned* err;
  uint64_t wait_ns;  // limit of every wait
  int stall;         // failure-detection test: issue no copies
  int N, K, M, KT, g, group;
  int nslab, spc, QPS;  // slabs holding real rows, slabs per CTA, ring fills per slab
  int NS, stage_bytes, xres_off, red_off, ctl_off;  // offsets in the 128-aligned shared memory
};

// 16-byte chunks r = r0, r0 + step, ... of the activations x[M, K], into
// [unit][token][128] at dst; columns past K are zero-filled.
__device__ __forceinline__ void copy_x(const SlabArgs& a, uint32_t dst, int r0, int step) {
  const int per_m = a.KT * 16;
  for (int m = 0; m < a.M; ++m) {
    const uint16_t* xm = a.x + (size_t)m * a.K;
    for (int r = r0; r < per_m; r += step) {
      const int col = 8 * r;
      const bool in = col < a.K;
      cp_async_16(dst + (uint32_t)((r >> 4) * a.M * 256 + m * 256 + (r & 15) * 16), xm + (in ? col : 0),
                  in ? 16u : 0u);
    }
  }
}

// Fill f of the CTA whose first slab is s0: units [U*q, U*q + n) of slab
// s0 + f / QPS (q = f % QPS) into stage st, as one bulk copy issued by lane 0.
template <int BITS, int GPT, int NW>
__device__ __forceinline__ void slab_fill(const SlabArgs& a, uint32_t sbase, uint32_t full, int s0, int f, int st,
                                          int lane) {
  constexpr int UB = unit_bytes_gpu(BITS, GPT);
  constexpr int U = NW * slab_units_per_warp(BITS, NW);
  const int qs = f / a.QPS;
  const int sl = s0 + qs, k0 = (f - qs * a.QPS) * U;
  const int n = a.KT - k0 < U ? a.KT - k0 : U;
  const uint32_t bar = full + 8u * st;
  const uint32_t dst = sbase + (uint32_t)(st * a.stage_bytes);
  if (lane == 0 && !a.stall) {
    mbar_arrive_expect_tx(bar, (uint32_t)(n * UB));
    bulk_load_hint(dst, a.units + ((size_t)sl * a.KT + k0) * UB, (uint32_t)(n * UB), bar,
                   l2_evict_first_policy());  // weights are read once per call
  }
}

// Hand stage st (fill f) back; the last warp to do so refills it with fill
// f + NS.  The release counter's acquire-release atomic orders every warp's
// reads of the stage before the refill that overwrites it.
template <int BITS, int GPT, int NW>
__device__ __forceinline__ void hand_back_stage(const SlabArgs& a, uint32_t sbase, uint32_t full, unsigned* released,
                                                int* ctl, int s0, int f, int st, int nfill, bool dead, int lane) {
  __syncwarp();
  unsigned refill = 0;
  if (lane == 0 && atom_add_acq_rel_cta(released + st, 1u) == NW - 1) {
    released[st] = 0;
    refill = !dead && f + a.NS < nfill;
    if (refill && !a.stall) atomicAdd(ctl, 1);
  }
  if (__shfl_sync(0xFFFFFFFFu, refill, 0)) slab_fill<BITS, GPT, NW>(a, sbase, full, s0, f + a.NS, st, lane);
}

template <int BITS, int GPT, int NW>
__global__ void __launch_bounds__(NW * 32, NW == 8 ? 2 : 1) gemv_slab_kernel(const SlabArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align128(smem_raw);
  constexpr int UB = unit_bytes_gpu(BITS, GPT);
  constexpr int UPW = slab_units_per_warp(BITS, NW);
  constexpr int U = NW * UPW;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gr = lane >> 2, t = lane & 3;
  const int s0 = blockIdx.x * a.spc;
  const int ns = a.nslab - s0 < a.spc ? a.nslab - s0 : a.spc;  // >= 1 for every CTA of the grid
  const int nfill = ns * a.QPS;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t full = sbase + (uint32_t)a.ctl_off;
  unsigned* released = reinterpret_cast<unsigned*>(smem + a.ctl_off + 8 * a.NS);  // [NS] warps done with a stage
  int* ctl = reinterpret_cast<int*>(released + a.NS);  // [0] fills issued, [1] some wait ran out
  float4* red = reinterpret_cast<float4*>(smem + a.red_off);  // [spc slabs][8 warps][8 rows][tq lanes]
  float2* red2 = reinterpret_cast<float2*>(red);               // M = 1: [spc slabs][8 warps][8 rows]
  const int tq = (a.M + 1) >> 1;  // lanes per row group holding real tokens (2t, 2t + 1)
  const int npre = nfill < a.NS ? nfill : a.NS;
  uint4 h0 = make_uint4(0, 0, 0, 0), h1 = h0;
  if (threadIdx.x == 0) {
    load_header(a.units, h0, h1);  // compared below, before anything is written
    for (int i = 0; i < a.NS; ++i) {
      mbar_init(full + 8 * i, 1);
      released[i] = 0;
    }
    ctl[0] = a.stall ? 0 : npre;  // fills issued
    ctl[1] = 0;
    mbar_init_fence();
  }
  __syncthreads();
  // Static weights start streaming before the grid dependency resolves, but
  // only the first stage: the activation copies issued at the dependency
  // would otherwise reach the SM behind every prefetched stage; the other
  // stages follow them.
  if (warp == 0) {
    if (lane == 0) griddep_launch_dependents();
    if (npre > 0) slab_fill<BITS, GPT, NW>(a, sbase, full, s0, 0, 0, lane);
  }
  // y and x may still be in use by the previous grid
  griddep_wait();
  copy_x(a, sbase + (uint32_t)a.xres_off, threadIdx.x, NW * 32);
  if (warp == 0)
    for (int f = 1; f < npre; ++f) slab_fill<BITS, GPT, NW>(a, sbase, full, s0, f, f, lane);
  cp_async_wait_all();
  if (threadIdx.x == 0 && !header_matches(h0, h1, a.N, a.K, BITS, a.group)) {
    ctl[1] = 1;  // write nothing; the stream still runs, so that every copy lands
    atomicCAS(a.err, 0u, kErrBlobHeader);
  }
  __syncthreads();

  const LaneOffsets o = lane_offsets<BITS, GPT>(lane, a.g, a.M);
  const int x_unit = a.M * 256;
  // This warp's units of a stage are w, w + NW, ...: their offsets in the
  // stage and in the resident activations (from the stage's first unit).
  int woff[UPW], xoff[UPW];
#pragma unroll
  for (int j = 0; j < UPW; ++j) {
    woff[j] = (j * NW + warp) * UB;
    xoff[j] = (j * NW + warp) * x_unit;
  }
  const int last_n = a.KT - (a.QPS - 1) * U;  // units in the last stage of a slab (1..U)
  float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  WRegs<BITS, GPT> R[UPW];
  bool dead = ctl[1] != 0;  // a wait ran out (or a bad header): stop computing, keep the bookkeeping going
  int st = 0, q = 0, si = 0;
  uint32_t lap = 0;
  const uint8_t* stp = smem;                         // stage st
  const uint8_t* const xres = smem + a.xres_off;     // resident activations
  const uint8_t* xq = xres;                          // ... of this stage's first unit
  for (int f = 0; f < nfill; ++f) {
    const bool whole = q < a.QPS - 1 || last_n == U;  // every warp has UPW units in this stage
    const int n = whole ? U : last_n;
    if (!dead && !warp_wait(full + 8 * st, lap & 1u, a.err, a.wait_ns)) dead = true;
    const uint8_t* xp = xq;
    if (!dead) {
#pragma unroll
      for (int j = 0; j < UPW; ++j)
        if (whole || j * NW + warp < n) load_w(R[j], stp + woff[j], o);
    }
    // The stage goes back as soon as its weights are in registers.
    hand_back_stage<BITS, GPT, NW>(a, sbase, full, released, ctl, s0, f, st, nfill, dead, lane);
    if (!dead) {
#pragma unroll
      for (int j = 0; j < UPW; ++j) {
        if (whole || j * NW + warp < n) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t xs[8];
            load_x(xs, xp + xoff[j], o, h);
            mma_half(R[j], h, xs, acc[h]);
          }
        }
      }
    }
    if (++q == a.QPS) {
      // Slab s0 + si is done for this warp: park its partial sums (only
      // lanes t < tq hold real tokens); the slabs are reduced after the loop.
      if (a.M == 1) {  // one token: only (row gr, token 0) and (row gr + 8, token 0) are real
        if (t == 0)
          red2[(si * NW + warp) * 8 + gr] = make_float2(acc[0][0] + acc[1][0], acc[0][2] + acc[1][2]);
      } else if (t < tq) {
        red[((si * NW + warp) * 8 + gr) * tq + t] =
            make_float4(acc[0][0] + acc[1][0], acc[0][1] + acc[1][1], acc[0][2] + acc[1][2], acc[0][3] + acc[1][3]);
      }
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[h][e] = 0.f;
      q = 0;
      ++si;
      xq = xres;
    } else {
      xq += U * x_unit;
    }
    if (++st == a.NS) {
      st = 0;
      ++lap;
      stp = smem;
    } else {
      stp += a.stage_bytes;
    }
  }
  if (dead && lane == 0) atomicOr(ctl + 1, 1);
  __syncthreads();
  // Every warp's partial sums of every slab are parked: warp w adds the eight
  // partials of slabs w, w + 8, ... in warp order and writes their 16 rows.
  if (!ctl[1] && t < tq) {
    for (int i = warp; i < ns; i += NW) {
      float v[4] = {0.f, 0.f, 0.f, 0.f};
      if (a.M == 1) {
        const float2* rb = red2 + i * NW * 8 + gr;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
          const float2 u = rb[w * 8];
          v[0] += u.x; v[2] += u.y;
        }
      } else {
        const float4* rb = red + (i * NW * 8 + gr) * tq + t;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
          const float4 u = rb[w * 8 * tq];
          v[0] += u.x; v[1] += u.y; v[2] += u.z; v[3] += u.w;
        }
      }
      store_y(a.epi, (s0 + i) * kSlabN + gr, t, v);
    }
  }
  if (threadIdx.x == 0 && ctl[1]) {
    // A wait ran out: let the copies still in flight land before the CTA's
    // shared memory goes away.  Only the last NS fills can be outstanding.
    const int issued = ctl[0];
    for (int f = issued > a.NS ? issued - a.NS : 0; f < issued; ++f)
      mbar_wait(full + 8 * (f % a.NS), (uint32_t)(f / a.NS) & 1u, a.err, kErrGemvWait, kGemvDrainNs);
  }
}

// ===========================================================================
// host side

// Two CTAs per SM: 2 x (113 KB + 1 KB the runtime reserves per CTA) = 228 KB.
// One CTA per SM (the 16-warp slab configuration): 227 KB.
constexpr int kGemvSmemMax = 113 * 1024;
constexpr int kGemvSmemMax1 = 227 * 1024;
constexpr int kGemvSmemBudget = kGemvSmemMax - 128;  // ring + control bytes (128 for the alignment slack)

struct GemvPlan {
  bool slab;  // slab GEMV (else tile GEMV)
  int G;      // CTAs
  int NS, stage_bytes, x_off;
  // tile GEMV
  long long T;
  int S_max;
  size_t partial_bytes, counter_bytes;
  // slab GEMV
  int nw;  // warps per CTA: 8 (two CTAs per SM) or 16 (one CTA per SM)
  int nslab, spc, QPS, xres_off, red_off, ctl_off;
  size_t smem;
};

inline int clampi(int v, int lo, int hi) { return v < lo ? lo : (v > hi ? hi : v); }

// Deepest slab-GEMV ring (<= max_ns stages) that fits the budget next to
// the resident x (xres bytes, 0 if none), the parked partial sums (spc slabs
// x nw warps x 8 rows x ceil(M/2) lanes of four floats; two floats at M = 1)
// and the control words; 0 if not even two stages fit.
inline int slab_ring(GemvPlan* P, int M, int stage, int xres, int max_ns, int budget) {
  const int red = P->spc * P->nw * 8 * (M == 1 ? 8 : ((M + 1) / 2) * 16);
  for (int ns = max_ns; ns >= 2; --ns) {
    const int ctl = 8 * ns + 4 * ns + 8;
    if (ns * stage + xres + red + ctl <= budget) {
      P->NS = ns;
      P->stage_bytes = stage;
      P->xres_off = ns * stage;
      P->red_off = P->xres_off + xres;
      P->ctl_off = P->red_off + red;
      P->smem = 128 + (size_t)P->ctl_off + ctl;
      return ns;
    }
  }
  return 0;
}

inline int gemv_plan(const Geometry& Gm, int M, GemvPlan* P) {
  const int sms = sm_count();
  if (sms <= 0) return TF_ERR_CUDA;
  *P = GemvPlan{};
  // these kernels move x rows as 16-byte pieces (the stream GEMV takes
  // per-channel layers with K % 8 != 0 whenever their activations fit)
  if (Gm.K % 8 != 0) return TF_ERR_UNSUPPORTED;
  const int nslab = (Gm.N + kSlabN - 1) / kSlabN;
  if (Gm.KT >= kGemvWarps) {
    // Whole slabs per CTA, one CTA per slab on layers with fewer slabs than
    // SMs: 2.3 to 3.7 times faster there than splitting K across all SMs
    // (the tile GEMV), e.g. 1024 x 11008 W4 g32 at M = 1 in 8.1 us, not 18.8.
    P->slab = true;
    P->nslab = nslab;
    const int xres = (Gm.KT * M * 256 + 127) / 128 * 128;
    // (1) Eight warps, two CTAs per SM, x resident next to a ring of two
    // 32-unit stages: a deeper prefetch makes the flood at the start of each
    // layer larger, and the activation load every warp waits for queues
    // behind it (three stages cost the four-layer decode step about 1 us).
    P->nw = 8;
    P->spc = (nslab + 2 * sms - 1) / (2 * sms);
    P->G = (nslab + P->spc - 1) / P->spc;
    const int U8 = 8 * slab_units_per_warp(Gm.bits, 8);
    P->QPS = (Gm.KT + U8 - 1) / U8;
    if (slab_ring(P, M, (U8 * Gm.unit_bytes + 127) / 128 * 128, xres, 2, kGemvSmemBudget) >= 2) return TF_OK;
    // (2) x too large for that: sixteen warps, one CTA per SM, x resident
    // next to a ring of two to four stages.
    P->nw = 16;
    P->spc = (nslab + sms - 1) / sms;
    P->G = (nslab + P->spc - 1) / P->spc;
    const int U16 = 16 * slab_units_per_warp(Gm.bits, 16);
    P->QPS = (Gm.KT + U16 - 1) / U16;
    if (slab_ring(P, M, (U16 * Gm.unit_bytes + 127) / 128 * 128, xres, 4, kGemvSmemMax1 - 128) >= 2) return TF_OK;
    // x does not fit even then: the tile GEMV takes the layer, reading each
    // activation slice once per tile.  (Slices travelling with every slab
    // stage, which each CTA re-reads from L2 for every slab, were slower:
    // 232 against 212 us for 32768 x 32768 at M = 4.)
    *P = GemvPlan{};
  }
  const int TPS = tiles_per_stage(Gm.bits);
  P->slab = false;
  P->T = (long long)Gm.NB * Gm.KT;
  P->G = (int)(P->T < 2LL * sms ? P->T : 2LL * sms);
  const long long per_cta = (P->T + P->G - 1) / P->G;
  P->S_max = (int)((per_cta + Gm.KT - 1) / Gm.KT + 1);
  P->partial_bytes = (size_t)P->G * P->S_max * 8 * 32 * sizeof(float4);
  P->counter_bytes = ((size_t)Gm.NB * 8 * sizeof(unsigned) + 255) / 256 * 256;
  P->x_off = (TPS * kSlabsPerTile * Gm.unit_bytes + 127) / 128 * 128;
  P->stage_bytes = P->x_off + TPS * M * 256;
  // ring + control words (barriers, release counters, header / issued / dead)
  P->NS = clampi((kGemvSmemBudget - 12) / (P->stage_bytes + 20), 2, 6);
  P->smem = 128 + (size_t)P->NS * P->stage_bytes + 16 * P->NS + 4 * P->NS + 12;
  return TF_OK;
}

// Workspace of the tile GEMV: the arrival counters in the first
// kWorkspaceCounterBytes, the partial sums after them.
inline size_t gemv_scratch_bytes(const GemvPlan& P) {
  return P.slab ? 0 : kWorkspaceCounterBytes + P.partial_bytes;
}

template <int BITS, int GPT>
int launch_tile(const CUtensorMap& map, const GemvArgs& a, size_t smem, cudaStream_t s) {
  static std::atomic<unsigned long long> opted{0};
  return launch_pdl(gemv_kernel<BITS, GPT>, opted, a.G, kGemvThreads, kGemvSmemMax, smem, s, map, a);
}

template <int BITS, int GPT>
int launch_slab(const SlabArgs& a, int nw, int grid, size_t smem, cudaStream_t s) {
  static std::atomic<unsigned long long> opted8{0}, opted16{0};
  if (nw == 16) return launch_pdl(gemv_slab_kernel<BITS, GPT, 16>, opted16, grid, 512, kGemvSmemMax1, smem, s, a);
  return launch_pdl(gemv_slab_kernel<BITS, GPT, 8>, opted8, grid, 256, kGemvSmemMax, smem, s, a);
}

// The GEMV of a checked layer with a plan; partials / counters are the
// tile GEMV's scratch (unused by the slab GEMV).
int run_gemv(const Geometry& G, const GemvPlan& P, const void* blob, const uint16_t* x, const Epi& epi, int M,
             float4* partials, unsigned* counters, cudaStream_t stream) {
  unsigned* err = device_error_ptr();
  if (!err) return TF_ERR_CUDA;
  const TestHook hook = test_hook();
  const uint8_t* units = static_cast<const uint8_t*>(blob) + kHeaderBytes;
  if (P.slab) {
    SlabArgs a;
    a.units = units; a.x = x; a.epi = epi; a.err = err;
    a.wait_ns = hook.wait_ns; a.stall = hook.stall;
    a.N = G.N; a.K = G.K; a.M = M; a.KT = G.KT; a.g = G.g; a.group = G.group;
    a.nslab = P.nslab; a.spc = P.spc; a.QPS = P.QPS;
    a.NS = P.NS; a.stage_bytes = P.stage_bytes; a.xres_off = P.xres_off;
    a.red_off = P.red_off; a.ctl_off = P.ctl_off;
    if (G.bits == 4) {
      if (G.gpt == 1) return launch_slab<4, 1>(a, P.nw, P.G, P.smem, stream);
      if (G.gpt == 2) return launch_slab<4, 2>(a, P.nw, P.G, P.smem, stream);
      return launch_slab<4, 4>(a, P.nw, P.G, P.smem, stream);
    }
    if (G.gpt == 1) return launch_slab<8, 1>(a, P.nw, P.G, P.smem, stream);
    if (G.gpt == 2) return launch_slab<8, 2>(a, P.nw, P.G, P.smem, stream);
    return launch_slab<8, 4>(a, P.nw, P.G, P.smem, stream);
  }
  CUtensorMap map;
  int rc = encode_x_map(x, M, G.K, &map);
  if (rc) return rc;
  GemvArgs a;
  a.units = units; a.epi = epi; a.partials = partials; a.counters = counters; a.err = err;
  a.wait_ns = hook.wait_ns; a.stall = hook.stall;
  a.T = P.T;
  a.N = G.N; a.K = G.K; a.M = M; a.KT = G.KT; a.g = G.g; a.group = G.group;
  a.G = P.G; a.S_max = P.S_max;
  a.NS = P.NS; a.stage_bytes = P.stage_bytes; a.x_off = P.x_off;
  if (G.bits == 4) {
    if (G.gpt == 1) return launch_tile<4, 1>(map, a, P.smem, stream);
    if (G.gpt == 2) return launch_tile<4, 2>(map, a, P.smem, stream);
    return launch_tile<4, 4>(map, a, P.smem, stream);
  }
  if (G.gpt == 1) return launch_tile<8, 1>(map, a, P.smem, stream);
  if (G.gpt == 2) return launch_tile<8, 2>(map, a, P.smem, stream);
  return launch_tile<8, 4>(map, a, P.smem, stream);
}

template <int BITS, int GPT>
void launch_dequant(const uint8_t* units, const Geometry& G, unsigned* err, uint16_t* w, cudaStream_t s) {
  dequant_kernel<BITS, GPT><<<G.NB * G.KT, 512, 0, s>>>(units, G.N, G.K, G.KT, G.g, G.group, err, w);
}

// The GEMV of one call, y written through epi.
int gemv_epi(const void* blob, size_t blob_bytes, int N, int K, int bits, int group, const uint16_t* x,
             const Epi& epi, int M, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  Geometry G;
  int rc = check_blob(blob, blob_bytes, N, K, bits, group, &G);
  if (rc) return rc;
  if (!x || M < 1) return TF_ERR_INVALID_ARG;
  if (M > 8) return TF_ERR_UNSUPPORTED;
  rc = check_epi(epi);
  if (rc) return rc;
  if (!aligned16(x) || !aligned16(workspace)) return TF_ERR_ALIGNMENT;
  StreamPlan SP;
  if (stream_plan(G, M, &SP)) return run_stream(G, SP, blob, x, epi, M, stream);
  GemvPlan P;
  rc = gemv_plan(G, M, &P);
  if (rc) return rc;
  const size_t need = gemv_scratch_bytes(P);
  if (need > 0 && (!workspace || workspace_bytes < need)) return TF_ERR_WORKSPACE;
  return run_gemv(G, P, blob, x, epi, M,
                  need ? reinterpret_cast<float4*>(static_cast<char*>(workspace) + kWorkspaceCounterBytes) : nullptr,
                  static_cast<unsigned*>(workspace), stream);
}

}  // namespace

// tf_gemm for M <= 8: the slab or tile GEMV (never the stream GEMV, whose
// sums skip the per-weight rounding that tf_gemm keeps).
int small_m_workspace(const Geometry& G, int M, size_t* bytes) {
  if (M > 8) return TF_ERR_UNSUPPORTED;
  GemvPlan P;
  const int rc = gemv_plan(G, M, &P);
  if (rc) return rc;
  *bytes = gemv_scratch_bytes(P);
  return TF_OK;
}

int run_small_m(const Geometry& G, const void* blob, const uint16_t* x, const Epi& epi, int M, void* workspace,
                size_t workspace_bytes, cudaStream_t stream) {
  if (M > 8) return TF_ERR_UNSUPPORTED;
  GemvPlan P;
  const int rc = gemv_plan(G, M, &P);
  if (rc) return rc;
  const size_t need = gemv_scratch_bytes(P);
  if (need > 0 && (!workspace || workspace_bytes < need)) return TF_ERR_WORKSPACE;
  return run_gemv(G, P, blob, x, epi, M,
                  need ? reinterpret_cast<float4*>(static_cast<char*>(workspace) + kWorkspaceCounterBytes) : nullptr,
                  static_cast<unsigned*>(workspace), stream);
}

}  // namespace tf

using namespace tf;

extern "C" {

int tf_dequant(const void* blob, size_t blob_bytes, int N, int K, int bits, int group, uint16_t* w,
               cudaStream_t stream) {
  Geometry G;
  int rc = check_blob(blob, blob_bytes, N, K, bits, group, &G);
  if (rc) return rc;
  if (!w) return TF_ERR_INVALID_ARG;
  if (!aligned16(w)) return TF_ERR_ALIGNMENT;
  const uint8_t* units = static_cast<const uint8_t*>(blob) + kHeaderBytes;
  unsigned* err = device_error_ptr();
  if (!err) return TF_ERR_CUDA;
  if (bits == 4) {
    if (G.gpt == 1) launch_dequant<4, 1>(units, G, err, w, stream);
    else if (G.gpt == 2) launch_dequant<4, 2>(units, G, err, w, stream);
    else launch_dequant<4, 4>(units, G, err, w, stream);
  } else {
    if (G.gpt == 1) launch_dequant<8, 1>(units, G, err, w, stream);
    else if (G.gpt == 2) launch_dequant<8, 2>(units, G, err, w, stream);
    else launch_dequant<8, 4>(units, G, err, w, stream);
  }
  return launch_status();
}

int tf_gemv_workspace_size(int N, int K, int bits, int group, int M, size_t* bytes) {
  if (!bytes) return TF_ERR_INVALID_ARG;
  Geometry G;
  int rc = make_geometry(N, K, bits, group, &G);
  if (rc) return rc;
  if (M < 1) return TF_ERR_INVALID_ARG;
  if (M > 8) return TF_ERR_UNSUPPORTED;
  StreamPlan SP;
  if (stream_plan(G, M, &SP)) {
    *bytes = 0;
    return TF_OK;
  }
  GemvPlan P;
  rc = gemv_plan(G, M, &P);
  if (rc) return rc;
  *bytes = gemv_scratch_bytes(P);
  return TF_OK;
}

int tf_gemv(const void* blob, size_t blob_bytes, int N, int K, int bits, int group, const uint16_t* x,
            uint16_t* y, int M, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return tf_gemv_bias(blob, blob_bytes, N, K, bits, group, x, nullptr, y, M, workspace, workspace_bytes, stream);
}

int tf_gemv_bias(const void* blob, size_t blob_bytes, int N, int K, int bits, int group, const uint16_t* x,
                 const uint16_t* bias, uint16_t* y, int M, void* workspace, size_t workspace_bytes,
                 cudaStream_t stream) {
  Epi e{y, nullptr, nullptr, bias, kEpiPlain, N, M, 0, 0};
  return gemv_epi(blob, blob_bytes, N, K, bits, group, x, e, M, workspace, workspace_bytes, stream);
}

int tf_gemv_silu_gate(const void* blob, size_t blob_bytes, int N, int K, int bits, int group, const uint16_t* x,
                      const uint16_t* bias, uint16_t* h, int M, void* workspace, size_t workspace_bytes,
                      cudaStream_t stream) {
  Epi e{h, nullptr, nullptr, bias, kEpiSiluGate, N, M, 0, 0};
  return gemv_epi(blob, blob_bytes, N, K, bits, group, x, e, M, workspace, workspace_bytes, stream);
}

int tf_gemv_qkv(const void* blob, size_t blob_bytes, int N, int K, int bits, int group, const uint16_t* x,
                const uint16_t* bias, uint16_t* q, uint16_t* k, uint16_t* v, int nq, int nk, int M, void* workspace,
                size_t workspace_bytes, cudaStream_t stream) {
  Epi e{q, k, v, bias, kEpiSplit3, N, M, nq, nk};
  return gemv_epi(blob, blob_bytes, N, K, bits, group, x, e, M, workspace, workspace_bytes, stream);
}

// ===========================================================================
// tf_gemv_noalloc: tf_gemv with its scratch in a fixed device array.
//
// Some callers cannot allocate device memory at the point where they run a
// layer: code that runs inside another framework's memory pool, plugins
// handed only input and output pointers, or real-time paths where an
// allocation may block or fail.  For them the split-K scratch of the tile
// GEMV (FP32 partial sums + arrival counters) lives in this file-scope
// array, which every GPU that loads the library holds until the process
// exits; the slab GEMV needs none.  Host code must not pass the array's name
// to a kernel (on the host it is only a stand-in): its device address is
// looked up once per device with cudaGetSymbolAddress, with that device
// current.

}  // extern "C"

static __device__ __align__(256) unsigned char tf_gemv_scratch[TF_GEMV_NOALLOC_SCRATCH_BYTES];

// Bytes at the start of tf_gemv_scratch kept for the arrival counters (one
// per 128-row block and warp, at most 256 x 8 for N <= 32768), as in a
// caller's workspace.
constexpr size_t kNoallocCounterBytes = kWorkspaceCounterBytes;

namespace {

// Device address of tf_gemv_scratch on the current device (cached per device).
unsigned char* gemv_scratch_address() {
  static std::atomic<unsigned char*> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  unsigned char* p = cache[dev].load(std::memory_order_acquire);
  if (p) return p;
  void* addr = nullptr;
  if (cudaGetSymbolAddress(&addr, tf_gemv_scratch) != cudaSuccess || !addr) return nullptr;
  cache[dev].store(static_cast<unsigned char*>(addr), std::memory_order_release);
  return static_cast<unsigned char*>(addr);
}

}  // namespace

namespace tf {

int clear_noalloc_scratch() {
  unsigned char* scratch = gemv_scratch_address();
  if (!scratch) return TF_ERR_CUDA;
  return cudaMemset(scratch, 0, TF_GEMV_NOALLOC_SCRATCH_BYTES) == cudaSuccess ? TF_OK : TF_ERR_CUDA;
}

}  // namespace tf

extern "C" {

int tf_gemv_noalloc(const void* blob, size_t blob_bytes, int N, int K, int bits, int group, const uint16_t* x,
                    uint16_t* y, int M, cudaStream_t stream) {
  Geometry G;
  int rc = check_blob(blob, blob_bytes, N, K, bits, group, &G);
  if (rc) return rc;
  if (!x || !y || M < 1) return TF_ERR_INVALID_ARG;
  if (M > 8) return TF_ERR_UNSUPPORTED;
  if (!aligned16(x)) return TF_ERR_ALIGNMENT;
  const Epi e{y, nullptr, nullptr, nullptr, kEpiPlain, N, M, 0, 0};
  StreamPlan SP;
  if (stream_plan(G, M, &SP)) return run_stream(G, SP, blob, x, e, M, stream);
  GemvPlan P;
  rc = gemv_plan(G, M, &P);
  if (rc) return rc;
  // The arrival counters have a fixed region at the start of the array, the
  // partial sums the rest: the counters are zero when the library is loaded,
  // no layer's partial sums ever land on them, and every call that completes
  // leaves the counters it used at zero (the last arriver of each row block
  // resets its own), so no call has to clear them first.  A call cut short
  // by a device error may leave them dirty: tf_device_error, which reports
  // that error, zeroes the array.
  if (P.counter_bytes > kNoallocCounterBytes ||
      P.partial_bytes > (size_t)TF_GEMV_NOALLOC_SCRATCH_BYTES - kNoallocCounterBytes)
    return TF_ERR_SCRATCH_LIMIT;
  if (P.slab) return run_gemv(G, P, blob, x, e, M, nullptr, nullptr, stream);
  unsigned char* scratch = gemv_scratch_address();
  if (!scratch) return TF_ERR_CUDA;
  return run_gemv(G, P, blob, x, e, M, reinterpret_cast<float4*>(scratch + kNoallocCounterBytes),
                  reinterpret_cast<unsigned*>(scratch), stream);
}

}  // extern "C"
