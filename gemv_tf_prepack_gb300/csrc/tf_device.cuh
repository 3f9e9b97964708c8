// Device building blocks shared by the dequant, GEMV and GEMM kernels:
// unpack of packed codes and their dequantisation to BF16,
//     w = bf16_rne((q - z) * s)            (TileFuse, Methodology 1)
// done bit-exactly, plus the mma.sync tensor-core step of the GEMV.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "tf_abi.h"
#include "tf_format.h"

namespace tf {

// A BF16 bit pattern as the float it denotes (exact: BF16 is the top half of binary32).
__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// ---------------------------------------------------------------------------
// packed BF16x2 arithmetic (native on sm_90 and later; round to nearest even)

__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// (a & mask) | bits in one LOP3.
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t mask, uint32_t bits) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(mask), "r"(bits));
  return d;
}

// ---------------------------------------------------------------------------
// Per-row dequantisation constants for one lane (rows gr and gr + 8 of a
// 16-row block).  INT4 keeps them as BF16x2 pairs, INT8 as floats.

struct MetaW4 {
  uint32_t z_lo, z_hi;  // bf16x2 (128 + z, 128 + z) for row gr / gr + 8
  uint32_t s_lo, s_hi;  // bf16x2 (s, s)
};

struct MetaW8 {
  float z_lo, z_hi;     // 2^23 + z
  float s_lo, s_hi;     // scale as float
};

// scale_pair: uint32 holding (s[gr], s[gr + 8]) as BF16 (low, high);
// zero_byte: low nibble z[gr], high nibble z[gr + 8].
__device__ __forceinline__ MetaW4 meta_w4(uint32_t scale_pair, uint32_t zero_byte) {
  MetaW4 m;
  m.s_lo = __byte_perm(scale_pair, 0, 0x1010);
  m.s_hi = __byte_perm(scale_pair, 0, 0x3232);
  const uint32_t zz = __byte_perm(zero_byte, 0, 0x4040);  // the zero byte in bytes 0 and 2
  m.z_lo = and_or(zz, 0x000F000Fu, 0x43004300u);
  m.z_hi = and_or(zz >> 4, 0x000F000Fu, 0x43004300u);
  return m;
}

// zero_pair: low byte z[gr], next byte z[gr + 8].
__device__ __forceinline__ MetaW8 meta_w8(uint32_t scale_pair, uint32_t zero_pair) {
  MetaW8 m;
  m.s_lo = __uint_as_float(scale_pair << 16);
  m.s_hi = __uint_as_float(scale_pair & 0xFFFF0000u);
  m.z_lo = 8388608.0f + (float)(zero_pair & 0xFFu);
  m.z_hi = 8388608.0f + (float)((zero_pair >> 8) & 0xFFu);
  return m;
}

// One INT4 word (eight codes) -> the four BF16x2 A-fragment registers.
// Register r takes codes r (low half) and r + 4 (high half); even r belong
// to row gr, odd r to row gr + 8.  OR-ing a code into the mantissa of the
// BF16 0x4300 (= 128) gives 128 + q exactly; subtracting 128 + z is exact
// ((q - z) is a small integer) and the multiply by s rounds once, to
// nearest even: bf16_rne((q - z) * s), bit for bit.
__device__ __forceinline__ void dequant_w4(uint32_t w, const MetaW4& m, uint32_t (&a)[4]) {
  const uint32_t mask = 0x000F000Fu, magic = 0x43004300u;
  a[0] = bf16x2_mul(bf16x2_sub(and_or(w, mask, magic), m.z_lo), m.s_lo);
  a[1] = bf16x2_mul(bf16x2_sub(and_or(w >> 4, mask, magic), m.z_hi), m.s_hi);
  a[2] = bf16x2_mul(bf16x2_sub(and_or(w >> 8, mask, magic), m.z_lo), m.s_lo);
  a[3] = bf16x2_mul(bf16x2_sub(and_or(w >> 12, mask, magic), m.z_hi), m.s_hi);
}

// Eight INT8 codes (bytes of u0 then u1) -> four BF16x2 registers with the
// same register/row convention.  BF16 cannot hold 128 + q for q >= 128, so
// the codes go through float32: placing q in the low byte of 0x4B000000
// gives 2^23 + q exactly, subtracting 2^23 + z is exact, the product with s
// is exact in float32 (8-bit x 8-bit significands) and the conversion to
// BF16 rounds once, to nearest even.
__device__ __forceinline__ void dequant_w8(uint32_t u0, uint32_t u1, const MetaW8& m, uint32_t (&a)[4]) {
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const uint32_t sel = 0x7440u | (uint32_t)r;
    const float lo = __uint_as_float(__byte_perm(u0, 0x4B000000u, sel));
    const float hi = __uint_as_float(__byte_perm(u1, 0x4B000000u, sel));
    const float zz = (r & 1) ? m.z_hi : m.z_lo;
    const float ss = (r & 1) ? m.s_hi : m.s_lo;
    const __nv_bfloat162 v = __floats2bfloat162_rn((lo - zz) * ss, (hi - zz) * ss);
    a[r] = *reinterpret_cast<const uint32_t*>(&v);
  }
}

// ---------------------------------------------------------------------------
// D[16x8] += A[16x16] * B[16x8], BF16 inputs, FP32 accumulation.

__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------------------
// output epilogues (fused steps after the product; the pages' kernels end at
// the product)

// (EpiMode and Epi are declared with the host checks.)

__device__ __forceinline__ uint16_t to_bf16_bits(float v) { return __bfloat16_as_ushort(__float2bfloat16_rn(v)); }

// v + bias[n] (v itself, -0 included, without a bias).
__device__ __forceinline__ float epi_biased(const Epi& e, int n, float v) {
  return e.bias ? v + bf16_bits_to_float(e.bias[n]) : v;
}

// Row n of token m with its biased sum v, rounded once to BF16 (plain or
// split; the caller checks n < N and m < M).
__device__ __forceinline__ void epi_put(const Epi& e, int m, int n, float v) {
  const uint16_t b = to_bf16_bits(v);
  if (e.mode != kEpiSplit3) {
    e.y[(size_t)m * e.N + n] = b;
  } else if (n < e.n1) {
    e.y[(size_t)m * e.n1 + n] = b;
  } else if (n < e.n1 + e.n2) {
    e.y1[(size_t)m * e.n2 + (n - e.n1)] = b;
  } else {
    const int n3 = e.N - e.n1 - e.n2;
    e.y2[(size_t)m * n3 + (n - e.n1 - e.n2)] = b;
  }
}

// SiLU gate of gate row n (n mod 16 < 8, biased sum g) and its up row n + 8
// (biased sum u): h[m, 8 (n / 16) + n mod 8] = bf16_rne(silu(g) * u) with
// silu(a) = a / (1 + e^-a), all in FP32.
__device__ __forceinline__ void epi_put_gate(const Epi& e, int m, int n, float g, float u) {
  const float h = g / (1.f + __expf(-g)) * u;
  e.y[(size_t)m * (e.N >> 1) + ((n >> 4) << 3) + (n & 7)] = to_bf16_bits(h);
}

// ---------------------------------------------------------------------------
// blob header check

// Device error code of a call whose blob header does not describe the layer
// the call names (another layer's blob of the same size, a stale blob).
constexpr unsigned kErrBlobHeader = 0x800;

// True when the 64-byte header in front of `units` carries the magic, the
// format version and (N, K, bits, group) of the call.
__device__ __forceinline__ bool header_matches(const uint4 h0, const uint4 h1, int N, int K, int bits, int group) {
  return h0.x == kMagic && h0.y == kVersion && (int)h0.z == N && (int)h0.w == K && (int)h1.x == bits &&
         (int)h1.y == group;
}

__device__ __forceinline__ void load_header(const uint8_t* units, uint4& h0, uint4& h1) {
  const uint4* hp = reinterpret_cast<const uint4*>(units - kHeaderBytes);
  h0 = __ldg(hp);
  h1 = __ldg(hp + 1);
}

// ---------------------------------------------------------------------------
// loads

// Streamed once: no L1 allocation.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t ld_stream_u32(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t ld_stream_u16(const void* p) {
  unsigned short v;
  asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t ld_stream_u8(const void* p) {
  unsigned short v;
  asm volatile("ld.global.nc.L1::no_allocate.u8 %0, [%1];" : "=h"(v) : "l"(p));
  return v & 0xFFu;
}

// Reused by many warps (activations): keep in L1.
__device__ __forceinline__ uint4 ld_keep_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::evict_last.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

}  // namespace tf
