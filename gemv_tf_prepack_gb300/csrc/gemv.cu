// Dequant (parity path) and fused GEMV kernels of libtf, with their C ABI.
//
// GEMV = token generation at batch 1 (TileFuse, Methodology 3 "GEMV dataflow
// co-design").  The pages' point is that a quantised GEMV, memory-bound at
// full precision, turns compute-bound once unpack and dequant are added, and
// that the weight stream must be spread over the whole array.  The GB300
// version: every SM streams one contiguous run of pre-tiled bytes (the
// blob's tile order makes each CTA's share a single address range), each
// lane unpacks and dequantises its codes in registers, and the dequantised
// BF16 fragments go straight into mma.sync so that the tensor cores do the
// multiply-accumulate instead of CUDA-core FMAs.
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
// tf_dequant: one CTA per tile, one thread per (row block, quad, slot).

template <int BITS, int GPT>
__global__ void __launch_bounds__(512) dequant_kernel(const uint8_t* __restrict__ tiles, int N, int K,
                                                      int KT, int g, int tile_bytes,
                                                      uint16_t* __restrict__ w) {
  const int tile = blockIdx.x;
  const int nb = tile / KT, kt = tile - nb * KT;
  const int mb = threadIdx.x >> 6;
  const int h = (threadIdx.x >> 5) & 1;
  const int p = threadIdx.x & 31;
  const int gr = p >> 2, t = p & 3;
  constexpr int WB = kTileN * kTileK * BITS / 8;
  constexpr int SB = BITS == 4 ? 16 : 32;
  constexpr int ZB = BITS == 4 ? 64 : 128;
  const uint8_t* tb = tiles + (size_t)tile * tile_bytes;
  const int gi = GPT == 1 ? 0 : (h * 64 + 16 * t) / g;
  const uint32_t sp = *reinterpret_cast<const uint32_t*>(tb + WB + gi * 256 + (mb * 8 + gr) * 4);
  const uint8_t* slot = tb + ((mb * 2 + h) * 32 + p) * SB;

  uint32_t lo[8], hi[8];  // rows gr and gr + 8 of this block, 16 columns each
  if (BITS == 4) {
    const MetaW4 m = meta_w4(sp, tb[WB + GPT * 256 + gi * ZB + mb * 8 + gr]);
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
    const uint32_t zp = *reinterpret_cast<const uint16_t*>(tb + WB + GPT * 256 + gi * ZB + (mb * 8 + gr) * 2);
    const MetaW8 m = meta_w8(sp, zp);
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
  const int n0 = nb * kTileN + mb * 16 + gr;
  const int k0 = kt * kTileK + h * 64 + 16 * t;
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int n = n0 + 8 * e;
    if (n >= N) continue;
    const uint32_t* src = e ? hi : lo;
    uint16_t* dst = w + (size_t)n * K + k0;
    if (k0 < K) *reinterpret_cast<uint4*>(dst) = make_uint4(src[0], src[1], src[2], src[3]);
    if (k0 + 8 < K) *reinterpret_cast<uint4*>(dst + 8) = make_uint4(src[4], src[5], src[6], src[7]);
  }
}

// ===========================================================================
// tf_gemv
//
// Work split: the T = NB * KT tiles are numbered in blob order and CTA c
// streams tiles [c*T/G, (c+1)*T/G) — one contiguous byte range, which a
// shared-memory ring fetches with 1-D bulk copies (four INT4 or two INT8 tiles per stage), the
// tiles' activation slices x[:, kt*128 : kt*128+128] arriving alongside by
// 2-D TMA (zero-filled past K).  The warp that hands a stage back last
// refills it, so no warp is dedicated to (or delayed by) producing.  Warp w
// of the CTA owns row block w (16 rows) of every tile, so no intra-CTA
// reduction is needed.  A
// CTA's range covers whole or partial 128-row blocks ("segments"); a whole
// block is written straight to y, a partial one is stored as FP32 fragments
// in the workspace and the last of the block's contributors (arrival counter
// per row block) adds them in CTA order — a fixed order, so the result does
// not depend on arrival order.
//
// The kernel is launched with programmatic dependent launch: the weight
// stream (static data) starts before the previous kernel on the stream has
// finished; activations, y and the workspace are touched only after it has.

constexpr int kGemvConsumers = 8;                  // one warp per 16-row block
// tiles per ring stage (one bulk copy)
__host__ __device__ constexpr int tiles_per_stage(int bits) { return bits == 4 ? 4 : 2; }
constexpr int kGemvThreads = 32 * kGemvConsumers;
constexpr uint64_t kGemvTimeoutNs = 4000000000ull;
constexpr unsigned kErrGemvWait = 0x600;

struct GemvArgs {
  const uint8_t* tiles;
  uint16_t* y;
  float4* partials;    // [G][S_max][8 warps][32 lanes]
  unsigned* counters;  // [NB][8 warps], zero on entry and on exit
  unsigned* err;
  long long T;
  int N, K, M, KT, g, tile_bytes, G, S_max;
  int NS, stage_bytes, x_off;  // shared-memory ring: stages, bytes per stage, x slice offset
};

__device__ __forceinline__ long long tile_begin(long long c, long long T, int G) { return c * T / G; }

// CTA whose range holds tile x.
__device__ __forceinline__ int cta_of_tile(long long x, long long T, int G) {
  return (int)(((x + 1) * G - 1) / T);
}

__device__ __forceinline__ void store_y(const GemvArgs& a, int n0, int t, const float (&v)[4]) {
  const int m0 = 2 * t, m1 = 2 * t + 1, n1 = n0 + 8;
  if (n0 < a.N) {
    if (m0 < a.M) a.y[(size_t)m0 * a.N + n0] = __bfloat16_as_ushort(__float2bfloat16_rn(v[0]));
    if (m1 < a.M) a.y[(size_t)m1 * a.N + n0] = __bfloat16_as_ushort(__float2bfloat16_rn(v[1]));
  }
  if (n1 < a.N) {
    if (m0 < a.M) a.y[(size_t)m0 * a.N + n1] = __bfloat16_as_ushort(__float2bfloat16_rn(v[2]));
    if (m1 < a.M) a.y[(size_t)m1 * a.N + n1] = __bfloat16_as_ushort(__float2bfloat16_rn(v[3]));
  }
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
    store_y(a, nb * kTileN + warp * 16 + gr, t, v);
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
  store_y(a, nb * kTileN + warp * 16 + gr, t, s);
  if (lane == 0) a.counters[nb * 8 + warp] = 0u;
}

// Registers of one tile for one consumer lane: its weight slot in both K
// quads, the activation fragments and the tile's scale / zero words.
template <int BITS, int GPT>
struct TileRegs {
  uint4 w[2][BITS == 4 ? 1 : 2];
  uint4 x[2][2];
  uint32_t sp[GPT == 1 ? 1 : 2], zp[GPT == 1 ? 1 : 2];
};

struct LaneOffsets {
  int w, s, z, x, gi0, gi1;
  bool x_on;  // this lane's B-fragment column is a real token (gr < M)
};

template <int BITS, int GPT>
__device__ __forceinline__ void load_tile(TileRegs<BITS, GPT>& R, const uint8_t* tb, const uint8_t* xb,
                                          const LaneOffsets& o) {
  constexpr int SB = BITS == 4 ? 16 : 32;
  constexpr int ZB = BITS == 4 ? 64 : 128;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
#pragma unroll
    for (int v = 0; v < SB / 16; ++v) R.w[h][v] = *reinterpret_cast<const uint4*>(tb + o.w + h * 32 * SB + v * 16);
    // Columns of B past M only feed columns of D that are never stored: those
    // lanes keep whatever their registers hold and skip the shared-memory read.
    if (o.x_on) {
      R.x[h][0] = *reinterpret_cast<const uint4*>(xb + o.x + h * 128);
      R.x[h][1] = *reinterpret_cast<const uint4*>(xb + o.x + h * 128 + 16);
    }
  }
  R.sp[0] = *reinterpret_cast<const uint32_t*>(tb + o.s + o.gi0 * 256);
  R.zp[0] = BITS == 4 ? (uint32_t)tb[o.z + o.gi0 * ZB] : (uint32_t)*reinterpret_cast<const uint16_t*>(tb + o.z + o.gi0 * ZB);
  if (GPT > 1) {
    R.sp[GPT == 1 ? 0 : 1] = *reinterpret_cast<const uint32_t*>(tb + o.s + o.gi1 * 256);
    R.zp[GPT == 1 ? 0 : 1] = BITS == 4 ? (uint32_t)tb[o.z + o.gi1 * ZB]
                                        : (uint32_t)*reinterpret_cast<const uint16_t*>(tb + o.z + o.gi1 * ZB);
  }
}

// Unpack, dequantise (bit-exact BF16) and multiply-accumulate one tile.
template <int BITS, int GPT>
__device__ __forceinline__ void mma_tile(const TileRegs<BITS, GPT>& R, float (&acc)[2][4]) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int mi = GPT == 1 ? 0 : h;
    const uint32_t xs[8] = {R.x[h][0].x, R.x[h][0].y, R.x[h][0].z, R.x[h][0].w,
                            R.x[h][1].x, R.x[h][1].y, R.x[h][1].z, R.x[h][1].w};
    if (BITS == 4) {
      const MetaW4 m = meta_w4(R.sp[mi], R.zp[mi]);
      const uint32_t words[4] = {R.w[h][0].x, R.w[h][0].y, R.w[h][0].z, R.w[h][0].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t af[4];
        dequant_w4(words[j], m, af);
        mma_16816(acc[h], af, xs[2 * j], xs[2 * j + 1]);
      }
    } else {
      const MetaW8 m = meta_w8(R.sp[mi], R.zp[mi]);
      const uint4 v0 = R.w[h][0], v1 = R.w[h][BITS == 4 ? 0 : 1];
      const uint32_t words[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t af[4];
        dequant_w8(words[2 * j], words[2 * j + 1], m, af);
        mma_16816(acc[h], af, xs[2 * j], xs[2 * j + 1]);
      }
    }
  }
}

// Segment bookkeeping of one consumer warp: local index of the segment's
// last tile, whether the segment covers its whole row block, and the block.
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

// Issue fill f of this CTA's ring (tiles 2f, 2f+1 of its range and their
// activation slices) into slot s.  The activations are read only once the
// grid dependency has resolved (x_ok).
template <int TPS>
__device__ __forceinline__ void issue_fill(const GemvArgs& a, const CUtensorMap* tmx, uint32_t sbase, uint32_t full,
                                           long long t0, int ntile, int f, int s, bool weights, bool x) {
  const int i = f * TPS;
  const int n = ntile - i < TPS ? ntile - i : TPS;
  const uint32_t x_bytes = (uint32_t)a.M * 256u;
  const uint32_t bar = full + 8u * s;
  const uint32_t dst = sbase + (uint32_t)(s * a.stage_bytes);
  if (weights) {
    mbar_arrive_expect_tx(bar, (uint32_t)n * ((uint32_t)a.tile_bytes + x_bytes));
    bulk_load(dst, a.tiles + (t0 + i) * a.tile_bytes, (uint32_t)(n * a.tile_bytes), bar);
  }
  if (x) {
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
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x;
  const long long t0 = tile_begin(c, a.T, a.G), t1 = tile_begin(c + 1, a.T, a.G);
  const int ntile = (int)(t1 - t0);
  constexpr int kTilesPerStage = tiles_per_stage(BITS);
  const int nfill = (ntile + kTilesPerStage - 1) / kTilesPerStage;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t full = sbase + (uint32_t)(a.NS * a.stage_bytes);
  const uint32_t empty = full + 8u * a.NS;
  // per-slot release counters: the last warp to hand a slot back refills it
  unsigned* released = reinterpret_cast<unsigned*>(smem + a.NS * a.stage_bytes + 16 * a.NS);
  const int npre = nfill < a.NS ? nfill : a.NS;
  if (threadIdx.x == 0) {
    for (int i = 0; i < a.NS; ++i) {
      mbar_init(full + 8 * i, 1);
      mbar_init(empty + 8 * i, kGemvConsumers);
      released[i] = 0;
    }
    mbar_init_fence();
    if (ntile > 0) {
      griddep_launch_dependents();
      prefetch_tensormap(&tmx);
      // static weights first, before the grid dependency resolves
      for (int f = 0; f < npre; ++f) issue_fill<kTilesPerStage>(a, &tmx, sbase, full, t0, ntile, f, f, true, false);
    }
  }
  __syncthreads();
  if (ntile <= 0) return;
  // y, x and the workspace may still be in use by the previous grid
  griddep_wait();
  if (threadIdx.x == 0)
    for (int f = 0; f < npre; ++f) issue_fill<kTilesPerStage>(a, &tmx, sbase, full, t0, ntile, f, f, false, true);

  const int gr = lane >> 2, t = lane & 3;  // mma.sync fragment coordinates
  constexpr int SB = BITS == 4 ? 16 : 32;
  constexpr int WB = kTileN * kTileK * BITS / 8;
  LaneOffsets o;
  o.w = warp * 2 * 32 * SB + lane * SB;  // slot p = 4 gr + t = lane
  o.s = WB + (warp * 8 + gr) * 4;
  o.z = WB + GPT * 256 + (BITS == 4 ? (warp * 8 + gr) : (warp * 8 + gr) * 2);
  o.gi0 = GPT == 1 ? 0 : (16 * t) / a.g;
  o.gi1 = GPT == 1 ? 0 : (64 + 16 * t) / a.g;
  o.x_on = gr < a.M;
  o.x = (o.x_on ? gr : 0) * 256 + 32 * t;
  const int x_stride = a.M * 256;

  float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  TileRegs<BITS, GPT> R;
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int v = 0; v < 2; ++v) R.x[h][v] = make_uint4(0, 0, 0, 0);
  Segment seg = first_segment(t0, ntile, a.KT);
  // at most two segments of a contiguous range are partial: its first and its last
  int pending0 = 0, pending1 = 0, npending = 0;
  int s = 0;
  uint32_t lap = 0;
  for (int f = 0; f < nfill; ++f) {
    if (!mbar_wait(full + 8 * s, lap & 1u, a.err, kErrGemvWait, kGemvTimeoutNs)) break;
    const int i0 = f * kTilesPerStage;
    const int n = ntile - i0 < kTilesPerStage ? ntile - i0 : kTilesPerStage;
    const uint8_t* st = smem + s * a.stage_bytes;
    const uint8_t* xs = st + a.x_off;
#pragma unroll
    for (int j = 0; j < kTilesPerStage; ++j) {
      if (j < n) {
        load_tile(R, st + j * a.tile_bytes, xs + j * x_stride, o);
        if (j == n - 1) {
          // the whole stage has been read: hand it back; the last warp to do
          // so refills it
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(empty + 8 * s);
            if (atomicAdd(released + s, 1u) == kGemvConsumers - 1) {
              released[s] = 0;
              if (f + a.NS < nfill && mbar_wait(empty + 8 * s, lap & 1u, a.err, kErrGemvWait, kGemvTimeoutNs))
                issue_fill<kTilesPerStage>(a, &tmx, sbase, full, t0, ntile, f + a.NS, s, true, true);
            }
          }
          __syncwarp();
        }
        mma_tile(R, acc);
        if (i0 + j == seg.end) {
          const float v[4] = {acc[0][0] + acc[1][0], acc[0][1] + acc[1][1], acc[0][2] + acc[1][2],
                              acc[0][3] + acc[1][3]};
          if (end_segment(a, c, t0, seg.nb, seg.whole, warp, lane, v)) {
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
  if (npending > 0) {
    fence_acq_rel_gpu();  // release: this lane's partials before any count below
    __syncwarp();
    publish_segment(a, pending0, warp, lane);
    if (npending > 1) publish_segment(a, pending1, warp, lane);
  }
}

// Grid of the GEMV: two CTAs per SM, never more CTAs than tiles.
struct GemvPlan {
  long long T;
  int G, S_max;
  int NS, stage_bytes, x_off;
  size_t smem, partial_bytes, counter_bytes;
};

constexpr int kGemvSmemBudget = 110 * 1024;  // ring bytes per CTA; two CTAs share an SM
constexpr int kGemvSmemMax = 113 * 1024;

inline int gemv_plan(const Geometry& Gm, int M, GemvPlan* P) {
  const int kTilesPerStage = tiles_per_stage(Gm.bits);
  const int sms = sm_count();
  if (sms <= 0) return TF_ERR_CUDA;
  P->T = (long long)Gm.NB * Gm.KT;
  P->G = (int)(P->T < 2LL * sms ? P->T : 2LL * sms);
  const long long per_cta = (P->T + P->G - 1) / P->G;
  P->S_max = (int)((per_cta + Gm.KT - 1) / Gm.KT + 1);
  P->partial_bytes = (size_t)P->G * P->S_max * 8 * 32 * sizeof(float4);
  P->counter_bytes = ((size_t)Gm.NB * 8 * sizeof(unsigned) + 255) / 256 * 256;
  P->x_off = (kTilesPerStage * Gm.tile_bytes + 127) / 128 * 128;
  P->stage_bytes = P->x_off + kTilesPerStage * M * 256;
  int ns = kGemvSmemBudget / P->stage_bytes;
  P->NS = ns < 2 ? 2 : (ns > 6 ? 6 : ns);
  P->smem = 128 + (size_t)P->NS * P->stage_bytes + 16 * P->NS + 4 * P->NS;
  return TF_OK;
}

template <int BITS, int GPT>
int launch_gemv(const CUtensorMap& map, const GemvArgs& a, size_t smem, cudaStream_t s) {
  auto kfn = gemv_kernel<BITS, GPT>;
  // Opt in once per device to the largest ring gemv_plan can ask for.
  static std::atomic<unsigned long long> opted{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return TF_ERR_CUDA;
  if (!(opted.load(std::memory_order_acquire) & (1ull << dev))) {
    if (cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemvSmemMax) != cudaSuccess ||
        cudaFuncSetAttribute(kfn, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess)
      return TF_ERR_CUDA;
    opted.fetch_or(1ull << dev, std::memory_order_acq_rel);
  }
  if (smem > (size_t)kGemvSmemMax) return TF_ERR_UNSUPPORTED;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.G);
  cfg.blockDim = dim3(kGemvThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kfn, map, a) != cudaSuccess) {
    cudaGetLastError();
    return TF_ERR_CUDA;
  }
  return launch_status();
}

template <int BITS, int GPT>
void launch_dequant(const uint8_t* tiles, const Geometry& G, uint16_t* w, cudaStream_t s) {
  dequant_kernel<BITS, GPT><<<G.NB * G.KT, 512, 0, s>>>(tiles, G.N, G.K, G.KT, G.g, G.tile_bytes, w);
}

}  // namespace
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
  const uint8_t* tiles = static_cast<const uint8_t*>(blob) + kHeaderBytes;
  if (bits == 4) {
    if (G.gpt == 1) launch_dequant<4, 1>(tiles, G, w, stream);
    else if (G.gpt == 2) launch_dequant<4, 2>(tiles, G, w, stream);
    else launch_dequant<4, 4>(tiles, G, w, stream);
  } else {
    if (G.gpt == 1) launch_dequant<8, 1>(tiles, G, w, stream);
    else if (G.gpt == 2) launch_dequant<8, 2>(tiles, G, w, stream);
    else launch_dequant<8, 4>(tiles, G, w, stream);
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
  GemvPlan P;
  rc = gemv_plan(G, M, &P);
  if (rc) return rc;
  *bytes = P.partial_bytes + P.counter_bytes;
  return TF_OK;
}

int tf_gemv(const void* blob, size_t blob_bytes, int N, int K, int bits, int group, const uint16_t* x,
            uint16_t* y, int M, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  Geometry G;
  int rc = check_blob(blob, blob_bytes, N, K, bits, group, &G);
  if (rc) return rc;
  if (!x || !y || M < 1) return TF_ERR_INVALID_ARG;
  if (M > 8) return TF_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(workspace)) return TF_ERR_ALIGNMENT;
  GemvPlan P;
  rc = gemv_plan(G, M, &P);
  if (rc) return rc;
  if (!workspace || workspace_bytes < P.partial_bytes + P.counter_bytes) return TF_ERR_WORKSPACE;
  CUtensorMap map;
  rc = encode_x_map(x, M, K, &map);
  if (rc) return rc;
  GemvArgs a;
  a.tiles = static_cast<const uint8_t*>(blob) + kHeaderBytes;
  a.y = y;
  a.partials = static_cast<float4*>(workspace);
  a.counters = reinterpret_cast<unsigned*>(static_cast<char*>(workspace) + P.partial_bytes);
  a.err = device_error_ptr();
  if (!a.err) return TF_ERR_CUDA;
  a.T = P.T;
  a.N = N; a.K = K; a.M = M; a.KT = G.KT; a.g = G.g; a.tile_bytes = G.tile_bytes;
  a.G = P.G; a.S_max = P.S_max;
  a.NS = P.NS; a.stage_bytes = P.stage_bytes; a.x_off = P.x_off;
  if (bits == 4) {
    if (G.gpt == 1) return launch_gemv<4, 1>(map, a, P.smem, stream);
    if (G.gpt == 2) return launch_gemv<4, 2>(map, a, P.smem, stream);
    return launch_gemv<4, 4>(map, a, P.smem, stream);
  }
  if (G.gpt == 1) return launch_gemv<8, 1>(map, a, P.smem, stream);
  if (G.gpt == 2) return launch_gemv<8, 2>(map, a, P.smem, stream);
  return launch_gemv<8, 4>(map, a, P.smem, stream);
}


// ===========================================================================
// tf_gemv_noalloc: tf_gemv with its scratch in a fixed device array.
//
// Some callers cannot allocate device memory at the point where they run a
// layer: code that runs inside another framework's memory pool, plugins
// handed only input and output pointers, or real-time paths where an
// allocation may block or fail.  For them the split-K scratch of the GEMV
// (FP32 partial sums + arrival counters) lives in this file-scope array,
// which every GPU that loads the library holds until the process exits.
// Host code must not pass the array's name to a kernel (on the host it is
// only a stand-in): its device address is looked up once per device with
// cudaGetSymbolAddress, with that device current.

}  // extern "C"

static __device__ __align__(256) unsigned char tf_gemv_scratch[TF_GEMV_NOALLOC_SCRATCH_BYTES];

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

extern "C" {

int tf_gemv_noalloc(const void* blob, size_t blob_bytes, int N, int K, int bits, int group, const uint16_t* x,
                    uint16_t* y, int M, cudaStream_t stream) {
  Geometry G;
  int rc = check_blob(blob, blob_bytes, N, K, bits, group, &G);
  if (rc) return rc;
  if (!x || !y || M < 1) return TF_ERR_INVALID_ARG;
  if (M > 8) return TF_ERR_UNSUPPORTED;
  if (!aligned16(x)) return TF_ERR_ALIGNMENT;
  GemvPlan P;
  rc = gemv_plan(G, M, &P);
  if (rc) return rc;
  if (P.partial_bytes + P.counter_bytes > (size_t)TF_GEMV_NOALLOC_SCRATCH_BYTES) return TF_ERR_SCRATCH_LIMIT;
  unsigned char* scratch = gemv_scratch_address();
  if (!scratch) return TF_ERR_CUDA;
  // The arrival counters must start at zero; a call cut short (device error)
  // could have left them dirty, so clear them on the stream first.
  unsigned char* counters = scratch + P.partial_bytes;
  if (cudaMemsetAsync(counters, 0, P.counter_bytes, stream) != cudaSuccess) return TF_ERR_CUDA;
  CUtensorMap map;
  rc = encode_x_map(x, M, K, &map);
  if (rc) return rc;
  GemvArgs a;
  a.tiles = static_cast<const uint8_t*>(blob) + kHeaderBytes;
  a.y = y;
  a.partials = reinterpret_cast<float4*>(scratch);
  a.counters = reinterpret_cast<unsigned*>(counters);
  a.err = device_error_ptr();
  if (!a.err) return TF_ERR_CUDA;
  a.T = P.T;
  a.N = N; a.K = K; a.M = M; a.KT = G.KT; a.g = G.g; a.tile_bytes = G.tile_bytes;
  a.G = P.G; a.S_max = P.S_max;
  a.NS = P.NS; a.stage_bytes = P.stage_bytes; a.x_off = P.x_off;
  if (bits == 4) {
    if (G.gpt == 1) return launch_gemv<4, 1>(map, a, P.smem, stream);
    if (G.gpt == 2) return launch_gemv<4, 2>(map, a, P.smem, stream);
    return launch_gemv<4, 4>(map, a, P.smem, stream);
  }
  if (G.gpt == 1) return launch_gemv<8, 1>(map, a, P.smem, stream);
  if (G.gpt == 2) return launch_gemv<8, 2>(map, a, P.smem, stream);
  return launch_gemv<8, 4>(map, a, P.smem, stream);
}

}  // extern "C"
