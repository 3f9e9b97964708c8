// Host side of libtf: the offline interleaved pre-tiling (TileFuse,
// Methodology 2 "Interleaved pre-tiling": quantisation metadata packed into
// the weight tiles, matrix reordered so that each consumer's tiles are
// contiguous, valid up to 32K), its exact inverse, the import of AWQ
// checkpoints as published (Contributions 1: AWQ-style weights consumed
// without re-quantising the model), and the small status API.
#include <algorithm>
#include <cstring>
#include <thread>
#include <vector>

#include "../../include/tf.h"
#include "tf_format.h"

using tf::Geometry;

namespace {

// AWQ checkpoints keep INT4 layers in the layout of AWQ's GEMM kernels:
// qweight int32 [K, N/8] and qzeros int32 [K/g, N/8] each hold the 4-bit
// values of eight consecutive output columns 8c..8c+7 per word, nibble i
// (bits 4i..4i+3) holding column 8c + kAwqOrder[i]; scales are FP16
// [K/g, N].  kAwqNibble is the inverse map: the nibble of column 8c + j.
constexpr int kAwqOrder[8] = {0, 2, 4, 6, 1, 3, 5, 7};
struct AwqNibbles {
  int of[8];
  constexpr AwqNibbles() : of() {
    for (int i = 0; i < 8; ++i) of[kAwqOrder[i]] = i;
  }
};
constexpr AwqNibbles kAwqNibble;

inline int awq_nibble(uint32_t word, int j) { return (word >> (4 * kAwqNibble.of[j])) & 0xF; }

// IEEE binary16 -> BF16, round to nearest even (every binary16 value is in
// BF16's range; only the 10-bit fraction is rounded to 7 bits).
uint16_t f16_to_bf16(uint16_t h) {
  const uint32_t sign = (uint32_t)(h & 0x8000u) << 16;
  const uint32_t e = (h >> 10) & 0x1Fu;
  uint32_t m = h & 0x3FFu, f;  // f: the value as binary32 bits (exact)
  if (e == 0x1Fu) {
    f = sign | 0x7F800000u | (m << 13);
  } else if (e != 0) {
    f = sign | ((e + 112u) << 23) | (m << 13);  // exponent bias 15 -> 127
  } else if (m == 0) {
    f = sign;
  } else {  // subnormal m * 2^-24: normalise the fraction
    uint32_t ex = 113;
    while (!(m & 0x400u)) { m <<= 1; --ex; }
    f = sign | (ex << 23) | ((m & 0x3FFu) << 13);
  }
  if ((f & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((f >> 16) | 0x40u);  // NaN stays NaN
  return (uint16_t)((f + 0x7FFFu + ((f >> 16) & 1u)) >> 16);
}

struct AwqArrays {
  const uint32_t* qweight;  // [K, N/8]
  const uint32_t* qzeros;   // [K/g, N/8]
  const uint16_t* scales;   // FP16 bits [K/g, N]
};

// Natural-order accessors (or an AWQ checkpoint's, when awq is set) with the
// padding rules of the blob format.
struct Source {
  const Geometry& G;
  const uint8_t* q8;     // INT8 codes [N, K]
  const uint32_t* q4;    // INT4 words [N, K/8]
  const uint16_t* s;     // [N, K/g]
  const uint8_t* z;      // [N, K/g]
  int n_groups;
  const AwqArrays* awq;

  int code(int n, int k) const {
    if (awq) return awq_nibble(awq->qweight[(size_t)k * (G.N / 8) + n / 8], n & 7);
    if (G.bits == 4) return (q4[(size_t)n * ((G.K + 7) / 8) + (k >> 3)] >> (4 * (k & 7))) & 0xF;
    return q8[(size_t)n * G.K + k];
  }
  // Group of padded column k (k may lie in the K padding of the last tile).
  int group_of(int k) const {
    return G.gpt > 1 ? k / G.g : (k / tf::kTileK * tf::kTileK) / G.g;
  }
  int padded_code(int n, int k) const {
    if (n >= G.N) return 0;
    if (k < G.K) return code(n, k);
    return zero(n, group_of(k));
  }
  uint16_t scale(int n, int grp) const {
    if (n >= G.N || grp >= n_groups) return 0;
    if (awq) return f16_to_bf16(awq->scales[(size_t)grp * G.N + n]);
    return s[(size_t)n * n_groups + grp];
  }
  uint8_t zero(int n, int grp) const {
    if (n >= G.N || grp >= n_groups) return 0;
    if (awq) return (uint8_t)awq_nibble(awq->qzeros[(size_t)grp * (G.N / 8) + n / 8], n & 7);
    return z[(size_t)n * n_groups + grp];
  }
};

// Header and units of the blob of G from src.
void write_blob(const Geometry& G, const Source& src, uint8_t* o);

// Unit row / column of code i of word j in slot p of K half h.
inline void code_position(int h, int p, int j, int i, int* row, int* col) {
  const int gr = p >> 2, t = p & 3, r = i & 3, e = i >> 2;
  *row = gr + 8 * (r & 1);
  *col = h * 64 + 16 * t + 4 * j + 2 * (r >> 1) + e;
}

void pack_unit(const Source& src, int s, int kt, uint8_t* unit) {
  const Geometry& G = src.G;
  const int sb = tf::slot_bytes(G.bits);
  for (int h = 0; h < 2; ++h)
    for (int p = 0; p < 32; ++p) {
      uint8_t* slot = unit + (h * 32 + p) * sb;
      for (int j = 0; j < 4; ++j) {
        uint32_t word = 0;
        for (int i = 0; i < 8; ++i) {
          int row, col;
          code_position(h, p, j, i, &row, &col);
          const int c = src.padded_code(s * tf::kSlabN + row, kt * tf::kTileK + col);
          if (G.bits == 4)
            word |= (uint32_t)c << (4 * i);
          else
            slot[8 * j + i] = (uint8_t)c;
        }
        if (G.bits == 4) {
          for (int b = 0; b < 4; ++b) slot[4 * j + b] = (uint8_t)(word >> (8 * b));
        }
      }
    }
  for (int gi = 0; gi < G.gpt; ++gi) {
    const int grp = src.group_of(kt * tf::kTileK + (G.gpt > 1 ? gi * G.g : 0));
    for (int gr = 0; gr < 8; ++gr)
      for (int e = 0; e < 2; ++e) {
        const int n = s * tf::kSlabN + gr + 8 * e;
        const uint16_t sc = src.scale(n, grp);
        uint8_t* d = unit + tf::unit_scale_offset(G.bits, gi, gr) + 2 * e;
        d[0] = (uint8_t)(sc & 0xFF);
        d[1] = (uint8_t)(sc >> 8);
        const uint8_t z = src.zero(n, grp);
        uint8_t* zp = unit + tf::unit_zero_offset(G.bits, G.gpt, gi, gr);
        if (G.bits == 4) {
          if (e == 0) *zp = (uint8_t)((*zp & 0xF0) | z);
          else *zp = (uint8_t)((*zp & 0x0F) | (z << 4));
        } else {
          zp[e] = z;
        }
      }
  }
}

void write_header(const Geometry& G, uint8_t* out) {
  tf::BlobHeader h;
  std::memset(&h, 0, sizeof h);
  h.magic = tf::kMagic;
  h.version = tf::kVersion;
  h.N = G.N; h.K = G.K; h.bits = G.bits; h.group = G.group;
  h.unit_n = tf::kSlabN; h.unit_k = tf::kTileK;
  h.S = G.S; h.KT = G.KT; h.unit_bytes = G.unit_bytes; h.groups_per_unit = G.gpt;
  h.total_bytes = G.total_bytes;
  std::memcpy(out, &h, sizeof h);  // the ABI is little-endian
}

// f(s) for every slab s, on up to 32 host threads.
template <class F>
void parallel_slabs(int S, F&& f) {
  unsigned nt = std::max(1u, std::min(std::thread::hardware_concurrency(), 32u));
  nt = std::min<unsigned>(nt, (unsigned)S);
  if (nt <= 1) {
    for (int s = 0; s < S; ++s) f(s);
    return;
  }
  std::vector<std::thread> th;
  for (unsigned w = 0; w < nt; ++w)
    th.emplace_back([&, w] {
      for (int s = (int)w; s < S; s += (int)nt) f(s);
    });
  for (auto& t : th) t.join();
}

void write_blob(const Geometry& G, const Source& src, uint8_t* o) {
  write_header(G, o);
  parallel_slabs(G.S, [&](int s) {
    for (int kt = 0; kt < G.KT; ++kt) {
      uint8_t* unit = o + tf::unit_offset(G, s, kt);
      std::memset(unit, 0, G.unit_bytes);
      pack_unit(src, s, kt, unit);
    }
  });
}

}  // namespace

extern "C" {

int tf_version(void) { return TF_VERSION; }

const char* tf_status_string(int status) {
  switch (status) {
    case TF_OK: return "TF_OK";
    case TF_ERR_INVALID_ARG: return "TF_ERR_INVALID_ARG: null pointer, bad size or bad combination";
    case TF_ERR_UNSUPPORTED: return "TF_ERR_UNSUPPORTED: dimension, bits/group or M not supported";
    case TF_ERR_ALIGNMENT: return "TF_ERR_ALIGNMENT: device pointer not 16-byte aligned";
    case TF_ERR_WORKSPACE: return "TF_ERR_WORKSPACE: workspace missing or too small";
    case TF_ERR_BAD_BLOB: return "TF_ERR_BAD_BLOB: blob header or size mismatch";
    case TF_ERR_CUDA: return "TF_ERR_CUDA: CUDA runtime call or launch failed";
    case TF_ERR_DEVICE: return "TF_ERR_DEVICE: a kernel reported an error";
    case TF_ERR_SCRATCH_LIMIT:
      return "TF_ERR_SCRATCH_LIMIT: the layer needs more scratch than tf_gemv_noalloc's fixed buffer";
    default: return "unknown tf status";
  }
}

int tf_prepack_size(int N, int K, int bits, int group, size_t* bytes) {
  if (!bytes) return TF_ERR_INVALID_ARG;
  Geometry G;
  int rc = tf::make_geometry(N, K, bits, group, &G);
  if (rc) return rc;
  *bytes = G.total_bytes;
  return TF_OK;
}

int tf_prepack(const void* qweight, const uint16_t* scales, const uint8_t* zeros, int N, int K,
               int bits, int group, void* out, size_t out_bytes) {
  if (!qweight || !scales || !zeros || !out) return TF_ERR_INVALID_ARG;
  Geometry G;
  int rc = tf::make_geometry(N, K, bits, group, &G);
  if (rc) return rc;
  if (out_bytes < G.total_bytes) return TF_ERR_INVALID_ARG;
  const int n_groups = K / G.g;
  const int qmax = (1 << bits) - 1;
  for (size_t i = 0; i < (size_t)N * n_groups; ++i)
    if (zeros[i] > qmax) return TF_ERR_INVALID_ARG;
  Source src{G, (const uint8_t*)qweight, (const uint32_t*)qweight, scales, zeros, n_groups, nullptr};
  write_blob(G, src, (uint8_t*)out);
  return TF_OK;
}

int tf_prepack_awq(const int32_t* qweight, const int32_t* qzeros, const uint16_t* scales_f16, int N,
                   int K, int group, void* out, size_t out_bytes) {
  if (!qweight || !qzeros || !scales_f16 || !out) return TF_ERR_INVALID_ARG;
  if (N % 8 != 0) return TF_ERR_INVALID_ARG;
  Geometry G;
  int rc = tf::make_geometry(N, K, 4, group, &G);
  if (rc) return rc;
  if (out_bytes < G.total_bytes) return TF_ERR_INVALID_ARG;
  const AwqArrays awq{(const uint32_t*)qweight, (const uint32_t*)qzeros, scales_f16};
  Source src{G, nullptr, nullptr, nullptr, nullptr, K / G.g, &awq};
  write_blob(G, src, (uint8_t*)out);
  return TF_OK;
}

int tf_prepack_gate_up(const void* gate_qweight, const uint16_t* gate_scales, const uint8_t* gate_zeros,
                       const void* up_qweight, const uint16_t* up_scales, const uint8_t* up_zeros, int F, int K,
                       int bits, int group, void* out, size_t out_bytes) {
  if (!gate_qweight || !gate_scales || !gate_zeros || !up_qweight || !up_scales || !up_zeros || !out)
    return TF_ERR_INVALID_ARG;
  if (F < 8 || F % 8 != 0 || F > 16384) return TF_ERR_INVALID_ARG;
  const int N = 2 * F;
  Geometry G;
  int rc = tf::make_geometry(N, K, bits, group, &G);
  if (rc) return rc;
  if (out_bytes < G.total_bytes) return TF_ERR_INVALID_ARG;
  // Interleave the rows in blocks of 8 (gate, up, gate, up, ...) into one
  // natural-order layer and pack that.
  const int n_groups = K / G.g;
  const size_t row_bytes = bits == 4 ? (size_t)K / 2 : (size_t)K;
  std::vector<uint8_t> q((size_t)N * row_bytes);
  std::vector<uint16_t> s((size_t)N * n_groups);
  std::vector<uint8_t> z((size_t)N * n_groups);
  for (int r = 0; r < N; ++r) {
    const bool up = (r & 15) >= 8;
    const int f = (r >> 4) * 8 + (r & 7);
    const uint8_t* qs = static_cast<const uint8_t*>(up ? up_qweight : gate_qweight);
    memcpy(&q[(size_t)r * row_bytes], qs + (size_t)f * row_bytes, row_bytes);
    memcpy(&s[(size_t)r * n_groups], (up ? up_scales : gate_scales) + (size_t)f * n_groups,
           n_groups * sizeof(uint16_t));
    memcpy(&z[(size_t)r * n_groups], (up ? up_zeros : gate_zeros) + (size_t)f * n_groups, n_groups);
  }
  return tf_prepack(q.data(), s.data(), z.data(), N, K, bits, group, out, out_bytes);
}

int tf_blob_info(const void* header, size_t bytes, int* N, int* K, int* bits, int* group) {
  if (!header || bytes < (size_t)tf::kHeaderBytes) return TF_ERR_INVALID_ARG;
  tf::BlobHeader h;
  std::memcpy(&h, header, sizeof h);
  if (h.magic != tf::kMagic || h.version != tf::kVersion) return TF_ERR_BAD_BLOB;
  Geometry G;
  if (tf::make_geometry(h.N, h.K, h.bits, h.group, &G)) return TF_ERR_BAD_BLOB;
  if (h.unit_n != tf::kSlabN || h.unit_k != tf::kTileK || h.S != G.S || h.KT != G.KT ||
      h.unit_bytes != G.unit_bytes || h.groups_per_unit != G.gpt || h.total_bytes != G.total_bytes)
    return TF_ERR_BAD_BLOB;
  if (N) *N = h.N;
  if (K) *K = h.K;
  if (bits) *bits = h.bits;
  if (group) *group = h.group;
  return TF_OK;
}

int tf_unprepack(const void* blob, size_t bytes, void* qweight, uint16_t* scales, uint8_t* zeros) {
  if (!blob || !qweight || !scales || !zeros) return TF_ERR_INVALID_ARG;
  int N, K, bits, group;
  int rc = tf_blob_info(blob, bytes, &N, &K, &bits, &group);
  if (rc) return rc;
  Geometry G;
  tf::make_geometry(N, K, bits, group, &G);
  if (bytes < G.total_bytes) return TF_ERR_BAD_BLOB;
  const uint8_t* b = (const uint8_t*)blob;
  const int n_groups = K / G.g;
  const int sb = tf::slot_bytes(bits);
  if (bits == 4) std::memset(qweight, 0, (size_t)N * ((K + 7) / 8) * 4);
  // Slab s only holds rows s*16 .. s*16+15: no two slabs write the same word.
  parallel_slabs(G.S, [&](int s) {
    if (s * tf::kSlabN >= N) return;
    for (int kt = 0; kt < G.KT; ++kt) {
      const uint8_t* unit = b + tf::unit_offset(G, s, kt);
      for (int h = 0; h < 2; ++h)
        for (int p = 0; p < 32; ++p) {
          const uint8_t* slot = unit + (h * 32 + p) * sb;
          for (int j = 0; j < 4; ++j)
            for (int i = 0; i < 8; ++i) {
              int row, col;
              code_position(h, p, j, i, &row, &col);
              const int n = s * tf::kSlabN + row, k = kt * tf::kTileK + col;
              if (n >= N || k >= K) continue;
              if (bits == 4) {
                const uint32_t w = (uint32_t)slot[4 * j] | ((uint32_t)slot[4 * j + 1] << 8) |
                                   ((uint32_t)slot[4 * j + 2] << 16) | ((uint32_t)slot[4 * j + 3] << 24);
                const int c = (w >> (4 * i)) & 0xF;
                ((uint32_t*)qweight)[(size_t)n * ((K + 7) / 8) + (k >> 3)] |= (uint32_t)c << (4 * (k & 7));
              } else {
                ((uint8_t*)qweight)[(size_t)n * K + k] = slot[8 * j + i];
              }
            }
        }
      for (int gi = 0; gi < G.gpt; ++gi) {
        const int c0 = kt * tf::kTileK + (G.gpt > 1 ? gi * G.g : 0);
        if (c0 >= K) continue;
        const int grp = c0 / G.g;
        for (int gr = 0; gr < 8; ++gr)
          for (int e = 0; e < 2; ++e) {
            const int n = s * tf::kSlabN + gr + 8 * e;
            if (n >= N) continue;
            const uint8_t* d = unit + tf::unit_scale_offset(bits, gi, gr) + 2 * e;
            scales[(size_t)n * n_groups + grp] = (uint16_t)(d[0] | (d[1] << 8));
            const uint8_t* zp = unit + tf::unit_zero_offset(bits, G.gpt, gi, gr);
            zeros[(size_t)n * n_groups + grp] = bits == 4 ? (uint8_t)((*zp >> (4 * e)) & 0xF) : zp[e];
          }
      }
    }
  });
  return TF_OK;
}

}  // extern "C"
