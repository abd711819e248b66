// Storage of the FP8 operands of the expert GEMMs: E4M3 bytes plus one UE8M0
// (power-of-two) scale per 128-element block along the GEMM's reduction
// dimension K, laid out the way the block-scaled tensor-core MMA reads them.
//
// Values: row-major E4M3 bytes, the same shape as the bf16 tensor they come
// from. Scales: "atoms" of 512 bytes, one per 128 rows (the M or N index of
// the GEMM) and 4 consecutive 128-wide K blocks. Inside an atom the scale of
// (row r, K block kb) is the byte
//     (r % 32) * 16 + ((r % 128) / 32) * 4 + kb % 4,
// so the atom is 32 lines of 16 bytes; tcgen05.cp .32x128b.warpx4 copies line
// i into tensor-memory lane i (and its three replicas), columns c .. c+3, and
// the MMA then finds the scale of row r in column c + (r % 128) / 32, lane
// r % 32, byte kb % 4 (the byte picked by the instruction's scale-factor id).
// Atoms are stored [row block][atom along K]; a UE8M0 byte e means 2^(e-127).
//
// MX layout (the MXFP8 configuration: one scale per 32 consecutive K
// elements): one atom per 128 rows and ONE 128-wide K block; byte
// atom_byte(r, j) holds the scale of the j-th 32-wide piece of that K block,
// and the MMA of K slice j (scale_vec::1X, K = 32) selects it with its
// scale-factor id j.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {
namespace f8 {

constexpr int kBlock = 128;        // quantisation block along K = one GEMM k-block
constexpr int kAtomBytes = 512;    // 128 rows x 4 K blocks, one byte each
constexpr int kAtomKBlocks = 4;

__host__ __device__ constexpr int atom_byte(int r, int kb) {
  return (r & 31) * 16 + ((r & 127) >> 5) * 4 + (kb & 3);
}
// atoms along K for a reduction length K (a multiple of 128)
__host__ __device__ constexpr int64_t atoms_k(int64_t K) {
  return (K / kBlock + kAtomKBlocks - 1) / kAtomKBlocks;
}
// byte offset of the atom holding (row block rb, K block kb); kg = atoms_k(K)
__host__ __device__ constexpr int64_t atom_offset(int64_t rb, int64_t kb, int64_t kg) {
  return (rb * kg + kb / kAtomKBlocks) * kAtomBytes;
}
// bytes of the scale atoms of a rows x K operand (rows a multiple of 128)
__host__ __device__ constexpr int64_t sf_bytes(int64_t rows, int64_t K) {
  return rows / 128 * atoms_k(K) * kAtomBytes;
}

// MX layout: atom of (row block rb, K block kb), KB = K / 128
__host__ __device__ constexpr int64_t mx_atom_offset(int64_t rb, int64_t kb, int64_t KB) {
  return (rb * KB + kb) * kAtomBytes;
}
__host__ __device__ constexpr int64_t mx_sf_bytes(int64_t rows, int64_t K) {
  return rows / 128 * (K / kBlock) * kAtomBytes;
}
// atoms per 128-row block along K, and the scale bytes of a rows x K operand,
// in either layout
__host__ __device__ constexpr int64_t sf_stride(int64_t K, bool mx) {
  return mx ? K / kBlock : atoms_k(K);
}
__host__ __device__ constexpr int64_t sf_bytes_of(int64_t rows, int64_t K, bool mx) {
  return mx ? mx_sf_bytes(rows, K) : sf_bytes(rows, K);
}
// Scale byte of row r's piece holding its 8-element vector c in a row form
// (1 x 128 pieces: one per 16 vectors, atoms_k layout; MX 1 x 32 pieces: one
// per 4 vectors, MX layout); kg = sf_stride(row length, mx).
__host__ __device__ constexpr int64_t row_sf_index(int64_t r, int c, int64_t kg, bool mx) {
  return mx ? mx_atom_offset(r >> 7, c >> 4, kg) + atom_byte((int)r, (c >> 2) & 3)
            : atom_offset(r >> 7, c >> 4, kg) + atom_byte((int)r, c >> 4);
}

}  // namespace f8

// ------------------------------------------- producing the 1-byte form (device)
// UE8M0 code (2^(code-127)) of the block scale 2^ceil(log2(amax/448)) of the
// 1-byte form, from the bits of amax = 2^E * M (1 <= M < 2): amax/448 =
// 2^(E-8) * M/1.75, so ceil(log2(amax/448)) = E - 8 when M <= 1.75 and E - 7
// when M > 1.75 (the quotient of a bf16 amax and 448 never lies just below a
// power of two, so this is the exact ceiling). amax = 0 gives scale 1 (code
// 127). Scales below 2^-127, the smallest UE8M0 value (amax < 448 * 2^-128),
// are raised to 2^-127; there the scaled values keep fewer bits than the fp64
// reference's, a case no bf16 activation or weight of normal magnitude meets.
__device__ __forceinline__ uint32_t ue8m0_code(float amax) {
  if (!(amax > 0.f)) return 127u;
  const uint32_t b = __float_as_uint(amax);
  const int code = (int)(b >> 23) - 8 + ((b & 0x7FFFFFu) > 0x600000u ? 1 : 0);
  return code < 0 ? 0u : (uint32_t)code;
}
// 1 / scale = 2^(127 - code), exact (a normal fp32 for every code 0..253).
__device__ __forceinline__ float ue8m0_inv(uint32_t code) {
  return __uint_as_float((254u - code) << 23);
}

// E4M3 codes of eight values divided by a power-of-two scale (exact): bytes in
// element order.
__device__ __forceinline__ uint2 e4m3x8(const float (&f)[8], float inv_s) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint16_t h;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;"
        : "=h"(h) : "f"(f[2 * i + 1] * inv_s), "f"(f[2 * i] * inv_s));
    w[i] = h;
  }
  return make_uint2(w[0] | (w[1] << 16), w[2] | (w[3] << 16));
}

// The same with a scale per value (eight columns, each its own 128 x 1 block).
__device__ __forceinline__ uint2 e4m3x8_each(const float (&f)[8], const float* inv_s) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint16_t h;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;"
        : "=h"(h) : "f"(f[2 * i + 1] * inv_s[2 * i + 1]), "f"(f[2 * i] * inv_s[2 * i]));
    w[i] = h;
  }
  return make_uint2(w[0] | (w[1] << 16), w[2] | (w[3] << 16));
}

__device__ __forceinline__ float amax8(const float (&f)[8]) {
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(f[i]));
  return m;
}

}  // namespace moe
