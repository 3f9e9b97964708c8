// Fused prefill GEMM of libtf on the 5th-generation tensor cores.
//
// TileFuse, Methodology 1: each weight tile is unpacked and dequantised
// *once* into on-chip memory and the BF16 result is reused for the tile's
// matrix operations.  Here, per CTA output tile of 128 weight rows x BN
// tokens (BN <= 256):
//   warp 0       streams pre-tiled weight tiles (one 3-D TMA box: the eight
//                16-row units of the tile, each carrying its own scales and
//                zeros) into a shared-memory ring;
//   warp 22      streams the matching activation slabs (2-D TMA, 128-byte
//                swizzle) into the operand ring, next to where the dequant
//                warps put the weights;
//   warps 6..21  unpack + dequantise one (16-row block, 64-column slab) of
//                each tile into the UMMA K-major 128-byte-swizzled layout
//                (bit-exact bf16_rne((q - z) * s));
//   warp 1       issues tcgen05.mma (M = 128 weight rows, N = BN tokens,
//                K = 16) from one thread, accumulating in tensor memory;
//                two accumulators let the epilogue of one tile overlap the
//                MMAs of the next;
//   warps 2..5   read the accumulator with tcgen05.ld, add the bias, round
//                to BF16 and store y through the epilogue (plain y by TMA
//                tile stores; the SiLU gate and the QKV split, or N % 8 != 0,
//                element by element).
// Each dequantised 128 x 64 weight slab feeds BN/16 * 4 MMAs, i.e. it is
// reused across all BN tokens of the tile.  CTAs are persistent (one per
// SM) and walk output tiles with the token index fastest, so CTAs that run
// together share weight tiles in L2.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstring>

#include "../../include/tf.h"
#include "tf_abi.h"
#include "tf_device.cuh"
#include "tf_format.h"
#include "tf_sm100.cuh"

namespace tf {

namespace {

constexpr int kThreads = 736;        // 23 warps
constexpr int kXProducerWarp = 22;   // the activation slabs' producer
constexpr int kDequantWarp0 = 6;     // warps 6..21: (row block, slab) pairs
constexpr int kEpilogueWarp0 = 2;    // warps 2..5
constexpr int kEpilogueThreads = 128;
constexpr int kSlabBytesW = 128 * 128;  // 128 rows x 64 BF16
constexpr int kTmemCols = 512;       // two accumulators of up to 256 columns
// Epilogue staging: two buffers of 16 tokens x 128 rows of BF16 (one TMA box each).
constexpr int kEpiChunk = 16;
constexpr int kEpiStageBytes = 2 * kEpiChunk * kTileN * 2;

enum : unsigned {
  kErrProducerWait = 0x100,
  kErrDequantWait = 0x200,
  kErrMmaWait = 0x300,
  kErrEpilogueWait = 0x400,
  kErrDrain = 0x500,
};

struct GemmArgs {
  const uint8_t* units;
  Epi epi;                    // where y goes (plain, SiLU gate or split) and the bias
  unsigned* err;              // device error word
  float* ws;                  // stream-K partial sums: [CTA][2][BN / 16][128 rows][16]
  unsigned* cnt;              // stream-K arrivals per tile (zero on entry and on exit)
  int N, K, M, KT, g, group, tile_bytes;  // tile_bytes: one packed tile (eight units) in shared memory
  int MT, BN, ntiles;
  int dp_tiles;               // tiles [0, dp_tiles) whole per CTA; the rest split along K
  int sk_ctas;                // CTAs [0, sk_ctas) share the split tiles' k-iterations (at least one each)
  int P, OPS;                 // stages of the packed ring and of the operand ring
  uint64_t wait_ns;           // limit of every wait
  int stall;                  // failure-detection test: the producers issue no copies
  int y_tma;                  // 1: whole tiles of a plain y leave through shared-memory staging and TMA stores
  int off_p, off_op, off_epi, off_bar;  // byte offsets in the 1024-aligned dynamic smem
};

// Token m's biased sum v of this thread's row n, through the epilogue.  All
// 32 lanes of the warp (32 consecutive rows from a multiple of 32) call it
// together: the SiLU gate takes the up row's sum from lane + 8.
__device__ __forceinline__ void put_y(const Epi& e, int m, int n, float v) {
  if (e.mode == kEpiSiluGate) {
    const float u = __shfl_down_sync(0xFFFFFFFFu, v, 8);
    if ((n & 8) == 0 && n < e.N) epi_put_gate(e, m, n, v, u);
  } else if (n < e.N) {
    epi_put(e, m, n, v);
  }
}

struct Bars {
  uint32_t full_p, empty_p, full_op, empty_op, tfull, tempty, drain, tmem_slot, flag;
};

// ---------------------------------------------------------------------------
// Schedule.  The output tiles (128 weight rows x BN tokens, token index
// fastest) that do not fill a whole wave of CTAs (all tiles, when there are
// fewer tiles than CTAs and splitting pays) are split along K ("stream-K"):
// the k-iterations of tiles [dp_tiles, ntiles) are divided evenly over CTAs
// [0, sk_ctas) in order (a few CTAs per split tile, at most all of them, and
// at most the number of those k-iterations, so that no range is empty).  The
// other tiles are processed whole, CTA c taking tiles c, c + G, ...  Every
// role of a CTA walks the same sequence: its stream-K segments first, then
// its whole tiles.

struct Work {
  int tile, kb, ke;  // k-tiles [kb, ke) of output tile `tile`
};

struct Sched {
  long long pos, end;  // this CTA's stream-K k-iterations still to hand out
  int dp_next;
};

__device__ __forceinline__ long long sk_begin(const GemmArgs& a, long long c) {
  return (long long)(a.ntiles - a.dp_tiles) * a.KT * (c < a.sk_ctas ? c : a.sk_ctas) / a.sk_ctas;
}

__device__ __forceinline__ Sched sched_begin(const GemmArgs& a) {
  Sched s;
  s.pos = sk_begin(a, blockIdx.x);
  s.end = sk_begin(a, blockIdx.x + 1);
  s.dp_next = blockIdx.x;
  return s;
}

__device__ __forceinline__ bool sched_next(const GemmArgs& a, Sched& s, Work& w) {
  if (s.pos < s.end) {
    const int ti = (int)(s.pos / a.KT);
    const long long t_end = (long long)(ti + 1) * a.KT;
    w.tile = a.dp_tiles + ti;
    w.kb = (int)(s.pos - (long long)ti * a.KT);
    w.ke = (int)((s.end < t_end ? s.end : t_end) - (long long)ti * a.KT);
    s.pos = (long long)ti * a.KT + w.ke;
    return true;
  }
  if (s.dp_next < a.dp_tiles) {
    w.tile = s.dp_next;
    w.kb = 0;
    w.ke = a.KT;
    s.dp_next += gridDim.x;
    return true;
  }
  return false;
}

// CTA whose stream-K range holds k-iteration x.
__device__ __forceinline__ int sk_cta_of(const GemmArgs& a, long long x) {
  const long long total = (long long)(a.ntiles - a.dp_tiles) * a.KT;
  return (int)(((x + 1) * a.sk_ctas - 1) / total);
}

// Partial-sum slot of CTA c's segment of stream-K tile ti: 0 for the tile its
// range starts in, 1 for the tile its range ends in.
__device__ __forceinline__ float* sk_slot(const GemmArgs& a, int c, int ti) {
  const int first = (int)(sk_begin(a, c) / a.KT);
  return a.ws + ((size_t)c * 2 + (ti == first ? 0 : 1)) * ((size_t)128 * a.BN);
}

__device__ __forceinline__ Bars bars_at(uint32_t base, int P, int OPS) {
  Bars b;
  b.full_p = base;
  b.empty_p = b.full_p + 8 * P;
  b.full_op = b.empty_p + 8 * P;
  b.empty_op = b.full_op + 8 * OPS;
  b.tfull = b.empty_op + 8 * OPS;
  b.tempty = b.tfull + 16;
  b.drain = b.tempty + 16;
  b.tmem_slot = b.drain + 8;
  b.flag = b.tmem_slot + 8;
  return b;
}

template <int BITS, int GPT>
__global__ void __launch_bounds__(kThreads, 1) gemm_kernel(const __grid_constant__ CUtensorMap tmx,
                                                           const __grid_constant__ CUtensorMap tmw,
                                                           const __grid_constant__ CUtensorMap tmy,
                                                           const GemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Bars B = bars_at(sbase + a.off_bar, a.P, a.OPS);
  const uint32_t x_slab_bytes = (uint32_t)a.BN * 128;
  const uint32_t op_stage_bytes = kSlabBytesW + x_slab_bytes;
  unsigned* err = a.err;

  if (threadIdx.x == 0) {
    for (int i = 0; i < a.P; ++i) {
      mbar_init(B.full_p + 8 * i, 1);
      mbar_init(B.empty_p + 8 * i, 16);  // every dequant warp reads the tile
    }
    for (int i = 0; i < a.OPS; ++i) {
      mbar_init(B.full_op + 8 * i, 1 + 8);  // producer (with tx) + 8 dequant warps
      mbar_init(B.empty_op + 8 * i, 1);     // tcgen05.commit
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(B.tfull + 8 * i, 1);
      mbar_init(B.tempty + 8 * i, 4);
    }
    mbar_init(B.drain, 1);
    mbar_init_fence();
    prefetch_tensormap(&tmx);
    prefetch_tensormap(&tmw);
    if (a.y_tma) prefetch_tensormap(&tmy);
  }
  if (warp == 1) {
    tmem_alloc(B.tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(smem + (B.tmem_slot - sbase));

  if (warp == 0) {
    // ---------------------------------------------------------- weight producer
    if (lane == 0) {
      int ps = 0;
      uint32_t pph = 0;
      bool ok = true;
      Sched sc = sched_begin(a);
      Work wk;
      while (ok && sched_next(a, sc, wk)) {
        const int nb = wk.tile / a.MT;
        for (int kt = wk.kb; kt < wk.ke && ok; ++kt) {
          ok = mbar_wait(B.empty_p + 8 * ps, pph ^ 1, err, kErrProducerWait, a.wait_ns);
          if (!ok) break;
          const uint32_t dst = sbase + (uint32_t)(a.off_p + ps * a.tile_bytes);
          if (!a.stall) {
            mbar_arrive_expect_tx(B.full_p + 8 * ps, (uint32_t)a.tile_bytes);
            if (BITS == 4)
              tma_load_3d(dst, &tmw, 0, kt, nb * kSlabsPerTile, B.full_p + 8 * ps);
            else
              tma_load_4d(dst, &tmw, 0, 0, kt, nb * kSlabsPerTile, B.full_p + 8 * ps);
          }
          if (++ps == a.P) { ps = 0; pph ^= 1; }
        }
      }
    }
  } else if (warp == kXProducerWarp) {
    // ------------------------------------------------------- activation producer
    // The x slabs have their own producer, so that the packed weight tiles
    // are requested as far ahead as the packed ring allows rather than only
    // as far as the operand ring.
    if (lane == 0) {
      int os = 0;
      uint32_t oph = 0;
      bool ok = true;
      Sched sc = sched_begin(a);
      Work wk;
      while (ok && sched_next(a, sc, wk)) {
        const int mt = wk.tile % a.MT;
        for (int kt = wk.kb; kt < wk.ke && ok; ++kt) {
          for (int h = 0; h < 2; ++h) {
            ok = mbar_wait(B.empty_op + 8 * os, oph ^ 1, err, kErrProducerWait, a.wait_ns);
            if (!ok) break;
            if (!a.stall) {
              mbar_arrive_expect_tx(B.full_op + 8 * os, x_slab_bytes);
              tma_load_2d(sbase + a.off_op + (uint32_t)os * op_stage_bytes + kSlabBytesW, &tmx,
                          kt * kTileK + h * 64, mt * a.BN, B.full_op + 8 * os);
            }
            if (++os == a.OPS) { os = 0; oph ^= 1; }
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, a.BN);
      int os = 0, acc = 0;
      uint32_t oph = 0, aph = 0;
      bool ok = true;
      bool issued = false;
      Sched sc = sched_begin(a);
      Work wk;
      while (ok && sched_next(a, sc, wk)) {
        ok = mbar_wait(B.tempty + 8 * acc, aph ^ 1, err, kErrMmaWait, a.wait_ns);
        if (!ok) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)acc * 256;
        const int nslabs = 2 * (wk.ke - wk.kb);
        for (int sl = 0; sl < nslabs; ++sl) {
          ok = mbar_wait(B.full_op + 8 * os, oph, err, kErrMmaWait, a.wait_ns);
          if (!ok) break;
          tc_fence_after();
          const uint32_t wsl = sbase + a.off_op + (uint32_t)os * op_stage_bytes;
          const uint64_t ad = smem_desc_kmajor_sw128(wsl);
          const uint64_t bd = smem_desc_kmajor_sw128(wsl + kSlabBytesW);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // K = 16 per MMA: +32 bytes inside the swizzle atom
            umma_bf16(d_tmem, ad + 2 * kk, bd + 2 * kk, idesc, (sl | kk) ? 1u : 0u);
          umma_commit(B.empty_op + 8 * os);
          issued = true;
          if (++os == a.OPS) { os = 0; oph ^= 1; }
        }
        if (!ok) break;
        umma_commit(B.tfull + 8 * acc);
        if (++acc == 2) { acc = 0; aph ^= 1; }
      }
      if (issued) {
        // wait for every MMA of this CTA before tensor memory is released
        umma_commit(B.drain);
        mbar_wait(B.drain, 0, err, kErrDrain, a.wait_ns);
      }
    }
  } else if (warp >= kEpilogueWarp0 && warp < kDequantWarp0) {
    // ---------------------------------------------------------------- epilogue
    // Thread (q, lane) owns accumulator row q*32 + lane.  A whole tile goes
    // straight to y.  A stream-K segment is stored as FP32 partial sums
    // ([BN/16][128 rows][16]: 64 contiguous bytes per thread per step); the
    // last of the tile's contributors adds all of them in CTA order (a fixed
    // order: the same result every run) and writes y.
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    const int row = q * 32 + lane;
    volatile unsigned* flag = reinterpret_cast<volatile unsigned*>(smem + (B.flag - sbase));
    // The only writers check the blob's header: with one that does not
    // describe this layer they drain every accumulator but write nothing
    // (no y, no partial sums, no arrival counts).
    uint4 h0, h1;
    load_header(a.units, h0, h1);
    const bool write = header_matches(h0, h1, a.N, a.K, BITS, a.group);
    if (!write && row == 0 && blockIdx.x == 0) atomicCAS(err, 0u, kErrBlobHeader);
    int acc = 0;
    uint32_t aph = 0;
    bool ok = true;
    Sched sc = sched_begin(a);
    Work wk;
    while (ok && sched_next(a, sc, wk)) {
      const int nb = wk.tile / a.MT, mt = wk.tile - nb * a.MT;
      ok = mbar_wait(B.tfull + 8 * acc, aph, err, kErrEpilogueWait, a.wait_ns);
      // the four epilogue warps meet at named barriers below: they must all
      // go on, or all stop
      ok = named_barrier_and(kEpilogueThreads, ok);
      if (!ok) break;
      tc_fence_after();
      const int n = nb * kTileN + row;
      const bool has_bias = a.epi.bias != nullptr;
      const float bv = has_bias && n < a.N ? bf16_bits_to_float(a.epi.bias[n]) : 0.f;
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)acc * 256;
      const bool whole = wk.kb == 0 && wk.ke == a.KT;
      const int ti = wk.tile - a.dp_tiles;
      float* mine = whole ? nullptr : sk_slot(a, blockIdx.x, ti);
      for (int c0 = 0; c0 < a.BN && write; c0 += 16) {
        uint32_t r[16];
        tmem_ld_16(taddr + (uint32_t)c0, r);
        tmem_ld_wait();
        if (whole && a.y_tma) {
          // Stage the chunk (16 tokens x 128 rows, BF16, [token][row]) and
          // write it with one TMA box; rows past N and tokens past M are
          // left out by the tensor map.  Two buffers: before one is
          // overwritten, the store that read it two chunks ago has finished
          // reading.
          if (mt * a.BN + c0 < a.M) {
            const int buf = (c0 / kEpiChunk) & 1;
            if (row == 0) bulk_wait_group_read<1>();
            named_barrier_sync(kEpilogueThreads);
            uint16_t* stg = reinterpret_cast<uint16_t*>(smem + a.off_epi) + buf * (kEpiChunk * kTileN);
#pragma unroll
            for (int j = 0; j < kEpiChunk; ++j)
              stg[j * kTileN + row] = __bfloat16_as_ushort(
                  __float2bfloat16_rn(has_bias ? __uint_as_float(r[j]) + bv : __uint_as_float(r[j])));
            fence_async_shared();
            named_barrier_sync(kEpilogueThreads);
            if (row == 0) {
              tma_store_2d(&tmy, smem_u32(stg), nb * kTileN, mt * a.BN + c0);
              bulk_commit_group();
            }
          }
        } else if (whole) {
          const int m0 = mt * a.BN + c0;
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (m0 + j < a.M) put_y(a.epi, m0 + j, n, has_bias ? __uint_as_float(r[j]) + bv : __uint_as_float(r[j]));
        } else {
          float4* dst = reinterpret_cast<float4*>(mine + ((size_t)(c0 / 16) * 128 + row) * 16);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            __stcg(dst + j, make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                        __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3])));
        }
      }
      // the accumulator has been read: the MMAs of the next segment may start
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(B.tempty + 8 * acc);
      if (++acc == 2) { acc = 0; aph ^= 1; }
      if (whole || !write) continue;
      // stream-K segment: publish the partial sums, count this contribution
      fence_acq_rel_gpu();
      named_barrier_sync(kEpilogueThreads);
      const long long t0 = (long long)ti * a.KT;
      const int c_first = sk_cta_of(a, t0), c_last = sk_cta_of(a, t0 + a.KT - 1);
      if (row == 0) *flag = atomicAdd(a.cnt + ti, 1u) == (unsigned)(c_last - c_first) ? 1u : 0u;
      named_barrier_sync(kEpilogueThreads);
      if (*flag) {
        fence_acq_rel_gpu();  // acquire: every contributor's partial sums are visible
        // CTAs after c_first start their range inside this tile (slot 0);
        // c_first uses slot 0 only if its range starts at the tile's start
        const size_t slot = (size_t)128 * a.BN;
        const float* p0 = a.ws + ((size_t)c_first * 2 + (sk_begin(a, c_first) == t0 ? 0 : 1)) * slot;
        const float* p1 = a.ws + (size_t)(c_first + 1) * 2 * slot;
        const int others = c_last - c_first;
#pragma unroll 1
        for (int c0 = 0; c0 < a.BN; c0 += 16) {
          const size_t off = ((size_t)(c0 / 16) * 128 + row) * 16;
          // one 64-byte run per contributor: all its loads are issued together
          float4 v[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) v[j] = __ldcg(reinterpret_cast<const float4*>(p0 + off) + j);
#pragma unroll 1
          for (int cc = 0; cc < others; ++cc) {
            const float4* src = reinterpret_cast<const float4*>(p1 + (size_t)cc * 2 * slot + off);
            float4 u[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) u[j] = __ldcg(src + j);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              v[j].x += u[j].x; v[j].y += u[j].y; v[j].z += u[j].z; v[j].w += u[j].w;
            }
          }
          const int m0 = mt * a.BN + c0;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float vv[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (m0 + 4 * j + e < a.M) put_y(a.epi, m0 + 4 * j + e, n, has_bias ? vv[e] + bv : vv[e]);
          }
        }
        if (row == 0) a.cnt[ti] = 0u;
      }
      // every epilogue thread has read the flag before the next segment sets it
      named_barrier_sync(kEpilogueThreads);
    }
    // the staged tiles' stores must be done reading shared memory (and
    // writing y) before the CTA ends
    if (row == 0) bulk_wait_group_all();
  } else {
    // ---------------------------------------------------------------- dequant
    // Warp (mb, h): unit mb (rows 16 mb .. 16 mb + 15) and 64-column slab h
    // of every tile, so the two slabs of a tile are dequantised in parallel.
    const int dw = warp - kDequantWarp0;
    const int mb = dw & 7, h = dw >> 3;
    const int gr = lane >> 2, t = lane & 3;  // lane reads slot p = lane (conflict-free)
    constexpr int UB = unit_bytes_gpu(BITS, GPT);
    constexpr int SB = BITS == 4 ? 16 : 32;
    const int r0 = mb * 16 + gr;  // rows r0 and r0 + 8 of the 128-row slab
    // byte offsets of this lane's two 16-byte chunks in rows r0, r0 + 8
    uint32_t dst[2][2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int r = r0 + 8 * e;
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int chunk = 2 * t + cc;
        dst[e][cc] = (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((chunk ^ (r & 7)) << 4));
      }
    }
    const int gi = GPT == 1 ? 0 : (h * 64 + 16 * t) / a.g;
    const int s_off = mb * UB + unit_scale_offset(BITS, gi, gr);
    const int z_off = mb * UB + unit_zero_offset(BITS, GPT, gi, gr);
    const int w_off = mb * UB + (h * 32 + lane) * SB;
    int ps = 0;
    uint32_t pph = 0;
    unsigned slab = (unsigned)h;  // this warp's slabs are h, h + 2, h + 4, ... of the CTA's stream
    // With more than 64 tokens, a stage's proxy fence and full-barrier
    // arrive are deferred until the next k-step's tile has been unpacked and
    // dequantised, so that the fence's wait for the stores overlaps that
    // work.
    int pend = -1;
    bool ok = true;
    Sched sc = sched_begin(a);
    Work wk;
    while (ok && sched_next(a, sc, wk)) {
      for (int kt = wk.kb; kt < wk.ke && ok; ++kt) {
        ok = mbar_wait(B.full_p + 8 * ps, pph, err, kErrDequantWait, a.wait_ns);
        if (!ok) break;
        const uint8_t* pk = smem + a.off_p + (size_t)ps * a.tile_bytes;
        const uint32_t sp = *reinterpret_cast<const uint32_t*>(pk + s_off);
        uint32_t lo[8], hi[8];
        if (BITS == 4) {
          const MetaW4 m = meta_w4(sp, pk[z_off]);
          const uint4 v = *reinterpret_cast<const uint4*>(pk + w_off);
          const uint32_t words[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint32_t f[4];
            dequant_w4(words[j], m, f);
            lo[2 * j] = f[0]; lo[2 * j + 1] = f[2];
            hi[2 * j] = f[1]; hi[2 * j + 1] = f[3];
          }
        } else {
          const MetaW8 m = meta_w8(sp, *reinterpret_cast<const uint16_t*>(pk + z_off));
          const uint4 v0 = reinterpret_cast<const uint4*>(pk + w_off)[0];
          const uint4 v1 = reinterpret_cast<const uint4*>(pk + w_off)[1];
          const uint32_t words[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint32_t f[4];
            dequant_w8(words[2 * j], words[2 * j + 1], m, f);
            lo[2 * j] = f[0]; lo[2 * j + 1] = f[2];
            hi[2 * j] = f[1]; hi[2 * j + 1] = f[3];
          }
        }
        // the packed tile is in registers: hand it back
        __syncwarp();
        if (lane == 0) mbar_arrive(B.empty_p + 8 * ps);
        if (++ps == a.P) { ps = 0; pph ^= 1; }
        if (pend >= 0) {
          fence_async_shared();
          __syncwarp();
          if (lane == 0) mbar_arrive(B.full_op + 8 * pend);
          pend = -1;
        }
        const unsigned os = slab % (unsigned)a.OPS;
        const uint32_t oph = (slab / (unsigned)a.OPS) & 1u;
        ok = mbar_wait(B.empty_op + 8 * os, oph ^ 1, err, kErrDequantWait, a.wait_ns);
        if (!ok) break;
        uint8_t* wsl = smem + a.off_op + (size_t)os * op_stage_bytes;
        *reinterpret_cast<uint4*>(wsl + dst[0][0]) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        *reinterpret_cast<uint4*>(wsl + dst[0][1]) = make_uint4(lo[4], lo[5], lo[6], lo[7]);
        *reinterpret_cast<uint4*>(wsl + dst[1][0]) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(wsl + dst[1][1]) = make_uint4(hi[4], hi[5], hi[6], hi[7]);
        if (a.BN <= 64) {
          // few tokens: the MMAs are waiting for this stage, publish it now
          // (2-3 % faster at M = 16-64; the deferral below pays only at large M)
          fence_async_shared();
          __syncwarp();
          if (lane == 0) mbar_arrive(B.full_op + 8 * os);
        } else {
          pend = (int)os;
        }
        slab += 2;
      }
    }
    if (pend >= 0) {
      fence_async_shared();
      __syncwarp();
      if (lane == 0) mbar_arrive(B.full_op + 8 * pend);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

// ---------------------------------------------------------------------------
// host side

constexpr int kMaxSmem = 227 * 1024;

struct GemmPlan {
  GemmArgs a;
  size_t smem;
  int grid;
  size_t ws_bytes;  // stream-K partial sums (0 without stream-K)
};

// Stream-K bytes of the workspace: the arrival counters in the first
// kWorkspaceCounterBytes (as in every split-K workspace of the library), the
// partial sums after them.
inline size_t sk_scratch_bytes(const GemmPlan& P) { return P.ws_bytes ? kWorkspaceCounterBytes + P.ws_bytes : 0; }

// stream_k: split the tiles of the last, partial wave (plus one whole wave)
// along K; needs sk_scratch_bytes of workspace.
int gemm_plan(const Geometry& G, int M, bool stream_k, int epi_mode, GemmPlan* P) {
  GemmArgs& a = P->a;
  a.N = G.N; a.K = G.K; a.M = M; a.KT = G.KT; a.g = G.g; a.group = G.group;
  a.tile_bytes = kSlabsPerTile * G.unit_bytes;
  if (a.tile_bytes % 128 != 0) return TF_ERR_UNSUPPORTED;  // each packed stage starts 128-byte aligned
  a.BN = M >= 256 ? 256 : (M + 15) / 16 * 16;
  a.MT = (M + a.BN - 1) / a.BN;
  a.ntiles = G.NB * a.MT;
  const int op_stage = kSlabBytesW + a.BN * 128;
  // y as a TMA tensor needs rows of a multiple of 16 bytes (and a plain y)
  a.y_tma = G.N % 8 == 0 && epi_mode == kEpiPlain ? 1 : 0;
  const int epi = a.y_tma ? kEpiStageBytes : 0;
  // The operand ring (1024-byte aligned stages for the 128-byte swizzle)
  // comes first at the aligned base, the packed ring (128-byte aligned tiles)
  // right after it: at BN = 256 that leaves room for a third packed tile,
  // which the weights' latency needs (+3-4 % at M = 2048 against two).
  a.OPS = 0;
  for (int ops = 4; ops >= 2 && a.OPS == 0; --ops)
    for (int p = 4; p >= 2; --p) {
      const int off_op = 0;
      const int off_p = ops * op_stage;
      const int off_epi = (off_p + p * a.tile_bytes + 127) / 128 * 128;
      const int off_bar = off_epi + epi;
      const size_t smem = 1024 + off_bar + 256;
      if (smem <= (size_t)kMaxSmem) {
        a.P = p; a.OPS = ops; a.off_p = off_p; a.off_op = off_op; a.off_epi = off_epi; a.off_bar = off_bar;
        P->smem = smem;
        break;
      }
    }
  if (a.OPS == 0) return TF_ERR_UNSUPPORTED;
  const int sms = sm_count();
  if (sms <= 0) return TF_ERR_CUDA;
  const int rem = a.ntiles % sms;
  // The last contributor to a split tile adds the others' partial sums one
  // contributor after another, one L2 round trip (about 1 us) per 16 columns
  // and contributor, so a split tile is shared by at most 2 CTAs (4 when
  // BN <= 64).
  const int split = a.BN <= 64 ? 4 : 2;
  int sk = 0, sk_ctas = 1;
  if (stream_k && rem != 0) {
    if (a.ntiles > sms) {
      // split the tiles of the partial wave only: every CTA still ends with
      // whole tiles, behind whose MMAs the partial-sum additions are hidden
      sk = rem;
      sk_ctas = split * sk < sms ? split * sk : sms;
    } else {
      // every tile split: worth it when the k-iterations saved (about 1 us
      // each, whatever BN is) exceed the addition left exposed at the end
      const int ctas = split * a.ntiles < sms ? split * a.ntiles : sms;
      const double c = (double)ctas / a.ntiles;
      const double saved = a.KT * (1.0 - 1.0 / c);
      if (saved >= a.BN / 16.0 * (c + 1.0) + 2.0) {
        sk = a.ntiles;
        sk_ctas = ctas;
      }
    }
  }
  if (sk > 0 && ((size_t)sk * sizeof(unsigned) > kWorkspaceCounterBytes)) sk = 0;  // not reached: sk <= SMs
  if (sk > 0) {
    a.dp_tiles = a.ntiles - sk;
    // with fewer k-iterations than CTAs, one k-iteration each for the first ones
    const long long iters = (long long)sk * a.KT;
    a.sk_ctas = iters < sk_ctas ? (int)iters : sk_ctas;
    P->grid = sms;
    P->ws_bytes = (size_t)a.sk_ctas * 2 * 128 * a.BN * sizeof(float);
  } else {
    a.dp_tiles = a.ntiles;
    a.sk_ctas = 1;
    P->grid = a.ntiles < sms ? a.ntiles : sms;
    P->ws_bytes = 0;
  }
  return TF_OK;
}

template <int BITS, int GPT>
int launch_gemm(const CUtensorMap& map, const CUtensorMap& wmap, const CUtensorMap& ymap, const GemmPlan& P,
                cudaStream_t s) {
  auto kfn = gemm_kernel<BITS, GPT>;
  // Opt in once per device to the largest shared-memory carve-out.
  static std::atomic<unsigned long long> opted{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return TF_ERR_CUDA;
  if (!(opted.load(std::memory_order_acquire) & (1ull << dev))) {
    if (cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem) != cudaSuccess)
      return TF_ERR_CUDA;
    opted.fetch_or(1ull << dev, std::memory_order_acq_rel);
  }
  kfn<<<P.grid, kThreads, P.smem, s>>>(map, wmap, ymap, P.a);
  return launch_status();
}

// Bytes of the activations copied to rows of a multiple of 8 elements
// (K % 8 != 0, per channel only: a TMA tensor's rows must be multiples of
// 16 bytes), kept in the caller's workspace after the counter region and
// the stream-K partial sums.
size_t padded_x_bytes(const Geometry& G, int M) {
  if (G.K % 8 == 0) return 0;
  const size_t k8 = (size_t)(G.K + 7) / 8 * 8;
  return ((size_t)M * k8 * sizeof(uint16_t) + 255) / 256 * 256;
}

// xp[m, k] = x[m, k] for k < K, 0 for K <= k < K8.
__global__ void __launch_bounds__(256) pad_x_kernel(const uint16_t* __restrict__ x, uint16_t* __restrict__ xp, int M,
                                                    int K, int K8) {
  const size_t total = (size_t)M * K8;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
    const size_t m = i / K8;
    const int k = (int)(i - m * K8);
    xp[i] = k < K ? x[m * K + k] : (uint16_t)0;
  }
}

// The GEMM of one call, y written through epi.
int gemm_epi(const void* blob, size_t blob_bytes, int N, int K, int bits, int group, const uint16_t* x,
             const Epi& epi, int M, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  Geometry G;
  int rc = check_blob(blob, blob_bytes, N, K, bits, group, &G);
  if (rc) return rc;
  if (!x || M < 1) return TF_ERR_INVALID_ARG;
  rc = check_epi(epi);
  if (rc) return rc;
  if (!aligned16(x) || !aligned16(workspace) || (epi.mode == kEpiPlain && !aligned16(epi.y))) return TF_ERR_ALIGNMENT;
  // Up to 8 tokens the slab or tile GEMV takes the product (one 8-token
  // MMA column per weight fragment, every weight read once) when the
  // workspace it needs is given, or it needs none: the tensor-memory
  // pipeline below spends about a microsecond per k-step whatever M is.
  size_t small_need = 0;
  if (M <= 8 && small_m_workspace(G, M, &small_need) == TF_OK && (workspace || small_need == 0))
    return run_small_m(G, blob, x, epi, M, workspace, workspace_bytes, stream);
  GemmPlan P;
  rc = gemm_plan(G, M, workspace != nullptr, epi.mode, &P);
  if (rc) return rc;
  const size_t pad_bytes = padded_x_bytes(G, M);
  const size_t pad_off = kWorkspaceCounterBytes + P.ws_bytes;
  if (pad_bytes && !workspace) return TF_ERR_WORKSPACE;  // the padded activations live there
  if (workspace && workspace_bytes < (pad_bytes ? pad_off + pad_bytes : sk_scratch_bytes(P))) return TF_ERR_WORKSPACE;
  P.a.cnt = P.ws_bytes ? static_cast<unsigned*>(workspace) : nullptr;
  P.a.ws = P.ws_bytes ? reinterpret_cast<float*>(static_cast<char*>(workspace) + kWorkspaceCounterBytes) : nullptr;
  P.a.units = static_cast<const uint8_t*>(blob) + kHeaderBytes;
  P.a.epi = epi;
  P.a.err = device_error_ptr();
  if (!P.a.err) return TF_ERR_CUDA;
  const TestHook hook = test_hook();
  P.a.wait_ns = hook.wait_ns;
  P.a.stall = hook.stall;
  CUtensorMap map, wmap, ymap;
  const uint16_t* xa = x;
  int ka = K;
  if (pad_bytes) {
    uint16_t* xp = reinterpret_cast<uint16_t*>(static_cast<char*>(workspace) + pad_off);
    ka = (K + 7) / 8 * 8;
    const size_t total = (size_t)M * ka;
    const int blocks = (int)((total + 255) / 256 < 4096 ? (total + 255) / 256 : 4096);
    pad_x_kernel<<<blocks, 256, 0, stream>>>(x, xp, M, K, ka);
    rc = launch_status();
    if (rc) return rc;
    xa = xp;
  }
  rc = encode_x_map_sw128(xa, M, ka, P.a.BN, &map);
  if (rc) return rc;
  rc = encode_units_map(P.a.units, G.S, G.KT, G.unit_bytes, &wmap);
  if (rc) return rc;
  if (P.a.y_tma) {
    rc = encode_y_map(epi.y, M, N, &ymap);
    if (rc) return rc;
  } else {
    memset(&ymap, 0, sizeof(ymap));  // not read by the kernel
  }
  if (bits == 4) {
    if (G.gpt == 1) return launch_gemm<4, 1>(map, wmap, ymap, P, stream);
    if (G.gpt == 2) return launch_gemm<4, 2>(map, wmap, ymap, P, stream);
    return launch_gemm<4, 4>(map, wmap, ymap, P, stream);
  }
  if (G.gpt == 1) return launch_gemm<8, 1>(map, wmap, ymap, P, stream);
  if (G.gpt == 2) return launch_gemm<8, 2>(map, wmap, ymap, P, stream);
  return launch_gemm<8, 4>(map, wmap, ymap, P, stream);
}

}  // namespace
}  // namespace tf

using namespace tf;

extern "C" {

int tf_gemm_workspace_size(int N, int K, int bits, int group, int M, size_t* bytes) {
  if (!bytes) return TF_ERR_INVALID_ARG;
  Geometry G;
  int rc = make_geometry(N, K, bits, group, &G);
  if (rc) return rc;
  if (M < 1) return TF_ERR_INVALID_ARG;
  GemmPlan P;
  rc = gemm_plan(G, M, true, kEpiPlain, &P);
  if (rc) return rc;
  const size_t pad = padded_x_bytes(G, M);
  *bytes = pad ? kWorkspaceCounterBytes + P.ws_bytes + pad : sk_scratch_bytes(P);
  size_t small = 0;
  if (M <= 8 && small_m_workspace(G, M, &small) == TF_OK) *bytes = small;  // the slab or tile GEMV takes these
  return TF_OK;
}

int tf_gemm(const void* blob, size_t blob_bytes, int N, int K, int bits, int group, const uint16_t* x, uint16_t* y,
            int M, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return tf_gemm_bias(blob, blob_bytes, N, K, bits, group, x, nullptr, y, M, workspace, workspace_bytes, stream);
}

int tf_gemm_bias(const void* blob, size_t blob_bytes, int N, int K, int bits, int group, const uint16_t* x,
                 const uint16_t* bias, uint16_t* y, int M, void* workspace, size_t workspace_bytes,
                 cudaStream_t stream) {
  Epi e{y, nullptr, nullptr, bias, kEpiPlain, N, M, 0, 0};
  return gemm_epi(blob, blob_bytes, N, K, bits, group, x, e, M, workspace, workspace_bytes, stream);
}

int tf_gemm_silu_gate(const void* blob, size_t blob_bytes, int N, int K, int bits, int group, const uint16_t* x,
                      const uint16_t* bias, uint16_t* h, int M, void* workspace, size_t workspace_bytes,
                      cudaStream_t stream) {
  Epi e{h, nullptr, nullptr, bias, kEpiSiluGate, N, M, 0, 0};
  return gemm_epi(blob, blob_bytes, N, K, bits, group, x, e, M, workspace, workspace_bytes, stream);
}

int tf_gemm_qkv(const void* blob, size_t blob_bytes, int N, int K, int bits, int group, const uint16_t* x,
                const uint16_t* bias, uint16_t* q, uint16_t* k, uint16_t* v, int nq, int nk, int M, void* workspace,
                size_t workspace_bytes, cudaStream_t stream) {
  Epi e{q, k, v, bias, kEpiSplit3, N, M, nq, nk};
  return gemm_epi(blob, blob_bytes, N, K, bits, group, x, e, M, workspace, workspace_bytes, stream);
}

}  // extern "C"
