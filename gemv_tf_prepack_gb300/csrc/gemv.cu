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

#include "../../include/tf.h"
#include "tf_abi.h"
#include "tf_device.cuh"
#include "tf_format.h"

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
  const int gr = p & 7, t = p >> 3;
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
// streams tiles [c*T/G, (c+1)*T/G): one contiguous byte range.  Warp w of a
// CTA owns row block w (16 rows) of every tile in that range, so no
// intra-CTA reduction is needed.  A CTA's range covers whole or partial
// 128-row blocks ("segments"); a whole block is written straight to y, a
// partial one is stored as FP32 fragments in the workspace and the last of
// the block's contributors (arrival counter per row block) adds them in CTA
// order — a fixed order, so the result does not depend on arrival order.

struct GemvArgs {
  const uint8_t* tiles;
  const uint16_t* x;
  uint16_t* y;
  float4* partials;    // [G][S_max][8 warps][32 lanes]
  unsigned* counters;  // [NB][8 warps], zero on entry and on exit
  long long T;
  int N, K, M, KT, g, tile_bytes, G, S_max;
};

__device__ __forceinline__ long long tile_begin(long long c, long long T, int G) { return c * T / G; }

// CTA whose range holds tile x.
__device__ __forceinline__ int cta_of_tile(long long x, long long T, int G) {
  return (int)(((x + 1) * G - 1) / T);
}

template <int BITS, int GPT>
struct Stage {
  uint4 w[2][BITS == 4 ? 1 : 2];  // this lane's slot in quad 0 and quad 1
  uint32_t s[GPT == 1 ? 1 : 2];   // scale pair per quad
  uint32_t z[GPT == 1 ? 1 : 2];   // zero byte(s) per quad
};

template <int BITS, int GPT>
__device__ __forceinline__ void load_stage(Stage<BITS, GPT>& S, const uint8_t* tb, int woff, int soff,
                                           int zoff, int gi0, int gi1) {
  constexpr int SB = BITS == 4 ? 16 : 32;
  constexpr int ZB = BITS == 4 ? 64 : 128;
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int v = 0; v < SB / 16; ++v) S.w[h][v] = ld_stream_v4(tb + woff + h * 32 * SB + v * 16);
  S.s[0] = ld_stream_u32(tb + soff + gi0 * 256);
  S.z[0] = BITS == 4 ? ld_stream_u8(tb + zoff + gi0 * ZB) : ld_stream_u16(tb + zoff + gi0 * ZB);
  if (GPT > 1) {
    S.s[GPT == 1 ? 0 : 1] = ld_stream_u32(tb + soff + gi1 * 256);
    S.z[GPT == 1 ? 0 : 1] = BITS == 4 ? ld_stream_u8(tb + zoff + gi1 * ZB) : ld_stream_u16(tb + zoff + gi1 * ZB);
  }
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

// End of a segment of row block nb: write y directly or go through the
// workspace and let the last contributor reduce.
__device__ __forceinline__ void flush_segment(const GemvArgs& a, int c, long long t0, int nb, bool whole,
                                              int warp, int lane, const float (&v)[4]) {
  const int gr = lane >> 2, t = lane & 3;
  const int n0 = nb * kTileN + warp * 16 + gr;
  if (whole) {
    store_y(a, n0, t, v);
    return;
  }
  const int seg = nb - (int)(t0 / a.KT);
  __stcg(a.partials + ((size_t)(c * a.S_max + seg) * 8 + warp) * 32 + lane, make_float4(v[0], v[1], v[2], v[3]));
  __threadfence();
  __syncwarp();
  unsigned old = 0;
  if (lane == 0) old = atomicAdd(a.counters + nb * 8 + warp, 1u);
  old = __shfl_sync(0xFFFFFFFFu, old, 0);
  const long long first_tile = (long long)nb * a.KT;
  const int c_first = cta_of_tile(first_tile, a.T, a.G);
  const int c_last = cta_of_tile(first_tile + a.KT - 1, a.T, a.G);
  if (old != (unsigned)(c_last - c_first)) return;
  __threadfence();
  float s[4] = {0.f, 0.f, 0.f, 0.f};
  for (int cc = c_first; cc <= c_last; ++cc) {
    const int sg = nb - (int)(tile_begin(cc, a.T, a.G) / a.KT);
    const float4 u = __ldcg(a.partials + ((size_t)(cc * a.S_max + sg) * 8 + warp) * 32 + lane);
    s[0] += u.x; s[1] += u.y; s[2] += u.z; s[3] += u.w;
  }
  store_y(a, n0, t, s);
  if (lane == 0) a.counters[nb * 8 + warp] = 0u;
}

template <int BITS, int GPT, int D>
__global__ void __launch_bounds__(256, 2) gemv_kernel(const GemvArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gr = lane >> 2, t = lane & 3;  // mma.sync fragment coordinates
  const int p = 8 * t + gr;                // this lane's slot in a (row block, quad)
  const int c = blockIdx.x;
  const long long t0 = tile_begin(c, a.T, a.G), t1 = tile_begin(c + 1, a.T, a.G);
  if (t0 >= t1) return;

  constexpr int SB = BITS == 4 ? 16 : 32;
  constexpr int WB = kTileN * kTileK * BITS / 8;
  const int woff = warp * 2 * 32 * SB + p * SB;
  const int soff = WB + (warp * 8 + gr) * 4;
  const int zoff = WB + GPT * 256 + (BITS == 4 ? (warp * 8 + gr) : (warp * 8 + gr) * 2);
  const int gi0 = GPT == 1 ? 0 : (16 * t) / a.g;
  const int gi1 = GPT == 1 ? 0 : (64 + 16 * t) / a.g;

  Stage<BITS, GPT> st[D];
#pragma unroll
  for (int s = 0; s < D; ++s)
    if (t0 + s < t1) load_stage(st[s], a.tiles + (t0 + s) * a.tile_bytes, woff, soff, zoff, gi0, gi1);

  const bool x_active = gr < a.M;
  const uint16_t* xrow = a.x + (size_t)(x_active ? gr : 0) * a.K;

  float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  int nb = (int)(t0 / a.KT);
  int kt = (int)(t0 - (long long)nb * a.KT);
  bool seg_whole = kt == 0;

  for (long long base = t0; base < t1; base += D) {
#pragma unroll
    for (int s = 0; s < D; ++s) {
      const long long tau = base + s;
      if (tau < t1) {
        // activations for this tile: x[gr, k0 .. k0+15] per quad
        uint32_t xs[2][8];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int k0 = kt * kTileK + h * 64 + 16 * t;
          uint4 v0 = make_uint4(0, 0, 0, 0), v1 = make_uint4(0, 0, 0, 0);
          if (x_active && k0 < a.K) v0 = ld_keep_v4(xrow + k0);
          if (x_active && k0 + 8 < a.K) v1 = ld_keep_v4(xrow + k0 + 8);
          xs[h][0] = v0.x; xs[h][1] = v0.y; xs[h][2] = v0.z; xs[h][3] = v0.w;
          xs[h][4] = v1.x; xs[h][5] = v1.y; xs[h][6] = v1.z; xs[h][7] = v1.w;
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int mi = GPT == 1 ? 0 : h;
          if (BITS == 4) {
            const MetaW4 m = meta_w4(st[s].s[mi], st[s].z[mi]);
            const uint4 v = st[s].w[h][0];
            const uint32_t words[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              uint32_t af[4];
              dequant_w4(words[j], m, af);
              mma_16816(acc[h], af, xs[h][2 * j], xs[h][2 * j + 1]);
            }
          } else {
            const MetaW8 m = meta_w8(st[s].s[mi], st[s].z[mi]);
            const uint4 v0 = st[s].w[h][0], v1 = st[s].w[h][BITS == 4 ? 0 : 1];
            const uint32_t words[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              uint32_t af[4];
              dequant_w8(words[2 * j], words[2 * j + 1], m, af);
              mma_16816(acc[h], af, xs[h][2 * j], xs[h][2 * j + 1]);
            }
          }
        }
        if (tau + D < t1) load_stage(st[s], a.tiles + (tau + D) * a.tile_bytes, woff, soff, zoff, gi0, gi1);

        if (kt == a.KT - 1 || tau == t1 - 1) {
          const float v[4] = {acc[0][0] + acc[1][0], acc[0][1] + acc[1][1], acc[0][2] + acc[1][2],
                              acc[0][3] + acc[1][3]};
          flush_segment(a, c, t0, nb, seg_whole && kt == a.KT - 1, warp, lane, v);
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[h][i] = 0.f;
          seg_whole = true;
          kt = 0;
          ++nb;
        } else {
          ++kt;
        }
      }
    }
  }
}

// Grid of the GEMV: two 256-thread CTAs per SM, never more CTAs than tiles.
struct GemvPlan {
  long long T;
  int G, S_max;
  size_t partial_bytes, counter_bytes;
};

inline int gemv_plan(const Geometry& Gm, int M, GemvPlan* P) {
  const int sms = sm_count();
  if (sms <= 0) return TF_ERR_CUDA;
  P->T = (long long)Gm.NB * Gm.KT;
  P->G = (int)(P->T < 2LL * sms ? P->T : 2LL * sms);
  const long long per_cta = (P->T + P->G - 1) / P->G;
  P->S_max = (int)((per_cta + Gm.KT - 1) / Gm.KT + 1);
  P->partial_bytes = (size_t)P->G * P->S_max * 8 * 32 * sizeof(float4);
  P->counter_bytes = ((size_t)Gm.NB * 8 * sizeof(unsigned) + 255) / 256 * 256;
  (void)M;
  return TF_OK;
}

template <int BITS, int GPT>
void launch_gemv(const GemvArgs& a, cudaStream_t s) {
  constexpr int D = BITS == 4 ? 4 : 2;
  gemv_kernel<BITS, GPT, D><<<a.G, 256, 0, s>>>(a);
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
  GemvArgs a;
  a.tiles = static_cast<const uint8_t*>(blob) + kHeaderBytes;
  a.x = x;
  a.y = y;
  a.partials = static_cast<float4*>(workspace);
  a.counters = reinterpret_cast<unsigned*>(static_cast<char*>(workspace) + P.partial_bytes);
  a.T = P.T;
  a.N = N; a.K = K; a.M = M; a.KT = G.KT; a.g = G.g; a.tile_bytes = G.tile_bytes;
  a.G = P.G; a.S_max = P.S_max;
  if (bits == 4) {
    if (G.gpt == 1) launch_gemv<4, 1>(a, stream);
    else if (G.gpt == 2) launch_gemv<4, 2>(a, stream);
    else launch_gemv<4, 4>(a, stream);
  } else {
    if (G.gpt == 1) launch_gemv<8, 1>(a, stream);
    else if (G.gpt == 2) launch_gemv<8, 2>(a, stream);
    else launch_gemv<8, 4>(a, stream);
  }
  return launch_status();
}

}  // extern "C"
