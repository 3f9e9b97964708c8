// Internal description of the pre-tiled blob, shared by the host prepack and
// the device kernels.  The format is documented in include/tf.h; this header
// only gives it names.
#pragma once

#include <stddef.h>
#include <stdint.h>

#ifdef __CUDACC__
#define TF_HD __host__ __device__ __forceinline__
#else
#define TF_HD inline
#endif

namespace tf {

constexpr uint32_t kMagic = 0x4B504654u;  // "TFPK"
constexpr uint32_t kVersion = 1;
constexpr int kHeaderBytes = 64;
constexpr int kTileN = 128;             // rows of W per tile
constexpr int kTileK = 128;             // columns of W (K) per tile
constexpr int kMaxDim = 32768;          // "dimensions up to 32K"

// Header as stored (little-endian, 64 bytes).
struct BlobHeader {
  uint32_t magic, version;
  int32_t N, K, bits, group, tile_n, tile_k, NB, KT, tile_bytes, groups_per_tile;
  uint64_t total_bytes;
  uint64_t reserved;
};
static_assert(sizeof(BlobHeader) == kHeaderBytes, "header is 64 bytes");

// Groups that start inside one tile: 128 / g for g in {32, 64}, else 1.
TF_HD int groups_per_tile(int group) { return (group == 32 || group == 64) ? kTileK / group : 1; }

// Bytes of the code region of a tile (128 x 128 codes).
TF_HD int tile_weight_bytes(int bits) { return kTileN * kTileK * bits / 8; }

// Bytes of one group's zeros within a tile: nibble pairs (INT4) or bytes (INT8).
TF_HD int tile_zero_bytes(int bits) { return bits == 4 ? kTileN / 2 : kTileN; }

TF_HD int tile_bytes(int bits, int group) {
  const int gpt = groups_per_tile(group);
  const int b = tile_weight_bytes(bits) + 2 * kTileN * gpt + tile_zero_bytes(bits) * gpt;
  return (b + 15) / 16 * 16;
}

// Slot size: bytes of codes one lane owns in a (row block, K quad) block.
TF_HD int slot_bytes(int bits) { return bits == 4 ? 16 : 32; }

struct Geometry {
  int N, K, bits, group, g;  // g = effective group size (K when per channel)
  int NB, KT, tile_bytes, gpt;
  size_t total_bytes;
};

// Validates a layer description; returns 0 or a TF_ERR_* code.
inline int make_geometry(int N, int K, int bits, int group, Geometry* out) {
  if (N <= 0 || K <= 0) return -1;
  if (N > kMaxDim || K > kMaxDim) return -2;
  if (bits != 4 && bits != 8) return -2;
  if (K % 8 != 0) return -1;
  if (group < 0) return -1;
  int g = group == 0 ? K : group;
  if (group != 0 && !(group == 32 || group == 64 || group % kTileK == 0)) return -2;
  if (K % g != 0) return -1;
  Geometry G;
  G.N = N; G.K = K; G.bits = bits; G.group = group; G.g = g;
  G.NB = (N + kTileN - 1) / kTileN;
  G.KT = (K + kTileK - 1) / kTileK;
  G.tile_bytes = tile_bytes(bits, group);
  G.gpt = groups_per_tile(group);
  G.total_bytes = (size_t)kHeaderBytes + (size_t)G.NB * G.KT * G.tile_bytes;
  *out = G;
  return 0;
}

}  // namespace tf
