// Internal description of the pre-tiled blob, shared by the host prepack and
// the device kernels.  The format is documented in include/tf.h; this header
// only gives it names.
//
// The blob is a sequence of units: a unit holds the codes of one 16-row slab
// of W over 128 columns of K, followed by that slab's scales and zeros for
// those columns, so everything one consumer needs for a unit is one
// contiguous run of bytes.  Units are ordered slab-major (all K units of
// slab 0, then slab 1, ...), so the units of any run of whole slabs — what
// one GEMV block streams — are contiguous too.  A GEMM tile is the eight
// slabs of one 128-row block at one K unit.
#pragma once

#include <stddef.h>
#include <stdint.h>

#ifdef __CUDACC__
#define TF_HD __host__ __device__ __forceinline__
#define TF_HDC __host__ __device__ constexpr
#else
#define TF_HD inline
#define TF_HDC constexpr
#endif

namespace tf {

constexpr uint32_t kMagic = 0x4B504654u;  // "TFPK"
constexpr uint32_t kVersion = 2;
constexpr int kHeaderBytes = 64;
constexpr int kSlabN = 16;              // rows of W per unit (one mma row block)
constexpr int kTileK = 128;             // columns of W (K) per unit
constexpr int kTileN = 128;             // rows of a GEMM tile
constexpr int kSlabsPerTile = kTileN / kSlabN;
constexpr int kMaxDim = 32768;          // "dimensions up to 32K"

// Header as stored (little-endian, 64 bytes).
struct BlobHeader {
  uint32_t magic, version;
  int32_t N, K, bits, group, unit_n, unit_k, S, KT, unit_bytes, groups_per_unit;
  uint64_t total_bytes;
  uint64_t reserved;
};
static_assert(sizeof(BlobHeader) == kHeaderBytes, "header is 64 bytes");

// Groups that start inside one unit: 128 / g for g in {32, 64}, else 1.
TF_HD int groups_per_unit(int group) { return (group == 32 || group == 64) ? kTileK / group : 1; }

// Bytes of the codes of a unit (16 x 128 codes).
TF_HD int unit_code_bytes(int bits) { return kSlabN * kTileK * bits / 8; }

// Per group of a unit: 16 BF16 scales, and 16 zeros as nibble pairs (INT4)
// or bytes (INT8).
constexpr int kUnitScaleBytes = 2 * kSlabN;
TF_HD int unit_zero_bytes(int bits) { return bits == 4 ? kSlabN / 2 : kSlabN; }

// Unit size for a given number of groups per unit (a compile-time constant
// of every kernel instantiation): padded to a multiple of 16 bytes (INT4) or
// 32 bytes (INT8, so that each half of a unit is a multiple of 16 bytes and
// a TMA box of one half fits the 256-element limit of 8-byte elements).
TF_HDC int unit_bytes_gpu(int bits, int gpu) {
  return (kSlabN * kTileK * bits / 8 + (kUnitScaleBytes + (bits == 4 ? kSlabN / 2 : kSlabN)) * gpu +
          (bits == 4 ? 15 : 31)) / (bits == 4 ? 16 : 32) * (bits == 4 ? 16 : 32);
}

TF_HD int unit_bytes(int bits, int group) { return unit_bytes_gpu(bits, groups_per_unit(group)); }

// Slot size: bytes of codes one lane owns in a (slab, K half) block.
TF_HD int slot_bytes(int bits) { return bits == 4 ? 16 : 32; }

// Byte offsets inside a unit of the scale pair (rows gr, gr + 8) and of the
// zero entry of row pair gr (INT4: one byte; INT8: two bytes) of group gi.
TF_HD int unit_scale_offset(int bits, int gi, int gr) { return unit_code_bytes(bits) + gi * kUnitScaleBytes + gr * 4; }
TF_HD int unit_zero_offset(int bits, int gpu, int gi, int gr) {
  return unit_code_bytes(bits) + kUnitScaleBytes * gpu + gi * unit_zero_bytes(bits) + gr * (bits == 4 ? 1 : 2);
}

struct Geometry {
  int N, K, bits, group, g;  // g = effective group size (K when per channel)
  int NB, S, KT, unit_bytes, gpt;  // S = 8 * NB slabs (rows padded to 128)
  size_t total_bytes;
};

// Byte offset of unit (s, kt) from the start of the blob.
TF_HD size_t unit_offset(const Geometry& G, int s, int kt) {
  return (size_t)kHeaderBytes + ((size_t)s * G.KT + kt) * G.unit_bytes;
}

// Validates a layer description; returns 0 or a TF_ERR_* code.
inline int make_geometry(int N, int K, int bits, int group, Geometry* out) {
  if (N <= 0 || K <= 0) return -1;
  if (N > kMaxDim || K > kMaxDim) return -2;
  if (bits != 4 && bits != 8) return -2;
  // K % 8 != 0 only per channel (every group size is a multiple of 8)
  if (K % 8 != 0 && group != 0) return -1;
  if (group < 0) return -1;
  int g = group == 0 ? K : group;
  if (group != 0 && !(group == 32 || group == 64 || group % kTileK == 0)) return -2;
  if (K % g != 0) return -1;
  Geometry G;
  G.N = N; G.K = K; G.bits = bits; G.group = group; G.g = g;
  G.NB = (N + kTileN - 1) / kTileN;
  G.S = G.NB * kSlabsPerTile;
  G.KT = (K + kTileK - 1) / kTileK;
  G.unit_bytes = unit_bytes(bits, group);
  G.gpt = groups_per_unit(group);
  G.total_bytes = (size_t)kHeaderBytes + (size_t)G.S * G.KT * G.unit_bytes;
  *out = G;
  return 0;
}

}  // namespace tf
