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
#pragma once

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

}  // namespace f8
}  // namespace moe
