// FP8 E4M3 block quantisation for the FP8 layer configuration.
//
// "Scalable Training of Mixture-of-Experts Models with Megatron Core" (es
// summary, Resumen técnico §2.4) quantises the expert GEMMs and their
// activations to FP8 (MXFP8 on Blackwell) while the router stays in high
// precision. Here every GEMM operand is replaced by its E4M3 value times a
// power-of-two block scale, scale = 2^ceil(log2(amax/448)) (1 for an all-zero
// block):
//   tiles  128 x 128 blocks of the expert weights,
//   rows   1 x 128 slices along a row (activations entering a GEMM that
//          reduces along that row),
//   cols   128 x 1 slices along the tokens of each 128-row block of the
//          permuted buffer (weight-gradient operands).
// The MXFP8 configuration uses 32-element blocks instead (1 x 32 rows, 32 x 1
// columns) and quantises each expert weight twice: 1 x 32 along its input
// dimension (forward GEMMs) and 32 x 1 along its output dimension (data
// gradients).
// Output: 1-byte E4M3 codes with UE8M0 scale atoms (fp8_layout.cuh), the
// operands of the block-scaled FP8 tensor-core GEMMs. For the column slices
// the atom's rows are the buffer's columns and its K blocks the 128-row
// blocks of the permuted buffer (the weight gradients reduce over tokens).
// E4M3 rounding (to nearest even, saturating) uses the hardware conversion.
#include "common.cuh"
#include "fp8_layout.cuh"
#include "internal.h"

namespace moe {

// Whether 128-row block rb of the permuted buffer holds any row a GEMM reads:
// group g's segment starts at offsets[g], and the GEMMs read its first
// ceil(counts[g] / 128) blocks (capacity segments and dropless padding past
// them are never read, so they are not quantised).
__device__ __forceinline__ bool live_block(const int32_t* __restrict__ offsets,
                                           const int32_t* __restrict__ counts, int G, long long rb) {
  const long long r0 = rb * 128;
  int lo = 0, hi = G - 1;                                 // last g with offsets[g] <= r0
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (offsets[mid] <= r0) lo = mid;
    else hi = mid - 1;
  }
  return r0 - offsets[lo] < (long long)((counts[lo] + 127) / 128) * 128;
}

// BLK x 1 slices (BLK = 128, or 32 for MX): every live 128-row block of
// [0, offsets[G]) (group segments are multiples of 128 rows, so blocks never
// straddle two experts) -> E4M3 bytes plus the UE8M0 scale atoms [cols / 128]
// [along the rows]. One block of 256 threads per (128-row block, 128-column
// slab): the 128 x 128 tile is read once into shared memory with 16-byte
// loads (eight per thread in flight), the maxima of each column's four
// 32-row pieces are taken there (a bf16 pair of columns per read; combined into
// one for BLK = 128), and every
// thread quantises eight 8-column vectors read back from the tile and stores
// their codes (8 bytes each). With ROWS, the same pass also writes the tile's
// 1 x BLK row form (Xr, sfr; a row's 16 vectors sit in 16 consecutive lanes,
// whose maxima meet by shuffles), so a tensor both GEMM directions need is read
// once.
template <int BLK, bool ROWS>
__global__ void __launch_bounds__(256)
quant_cols8_kernel(const __nv_bfloat16* __restrict__ X, uint8_t* __restrict__ Xq,
                   uint8_t* __restrict__ sf, const int32_t* __restrict__ offsets,
                   const int32_t* __restrict__ counts, int G, int cols, long long kg,
                   uint8_t* __restrict__ Xr, uint8_t* __restrict__ sfr, long long kgr,
                   const int32_t* __restrict__ pages) {
  static_assert(BLK == 128 || BLK == 32, "block length");
  extern __shared__ uint4 qc_smem[];
  uint4 (*tile)[16] = reinterpret_cast<uint4 (*)[16]>(qc_smem);   // 128 rows x 128 bf16
  float* part = reinterpret_cast<float*>(qc_smem + 128 * 16);      // [4 pieces][128]
  float* inv = part + 512;                                         // [4 pieces][128]
  const long long rblocks = offsets[G] / 128;
  const int slabs = cols >> 7;
  const int tid = threadIdx.x;
  for (long long w = blockIdx.x; w < rblocks * slabs; w += gridDim.x) {
    const long long rb = w / slabs;
    const int cs = (int)(w - rb * slabs);
    const int c0 = cs * 128;
    if (!live_block(offsets, counts, G, rb)) continue;
    // (a paged stash tensor keeps the block in one page)
    const __nv_bfloat16* src = X + (size_t)stash_row(pages, (int)rb * 128) * cols + c0;
    {
      uint4 in[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int v = tid + 256 * i, r = v >> 4, q = v & 15;
        in[i] = ldg_nc_v4(src + (size_t)r * cols + q * 8);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int v = tid + 256 * i;
        tile[v >> 4][v & 15] = in[i];
      }
    }
    __syncthreads();
    {
      // columns c and c + 1 (one bf16 pair per 4-byte read, consecutive lanes on
      // consecutive words), 32-row piece j
      const int c = 2 * (tid & 63), j = tid >> 6;
      const uint32_t* pair = reinterpret_cast<const uint32_t*>(&tile[0][0]) + (c >> 1);
      float m0 = 0.f, m1 = 0.f;
#pragma unroll 8
      for (int r = 32 * j; r < 32 * j + 32; ++r) {
        const uint32_t w2 = pair[r * 64];
        m0 = fmaxf(m0, fabsf(bf16_lo(w2)));
        m1 = fmaxf(m1, fabsf(bf16_hi(w2)));
      }
      part[j * 128 + c] = m0;
      part[j * 128 + c + 1] = m1;
    }
    __syncthreads();
    if (BLK == 128) {
      if (tid < 128) {
        const float m = fmaxf(fmaxf(part[tid], part[128 + tid]), fmaxf(part[256 + tid], part[384 + tid]));
        const uint32_t code = ue8m0_code(m);
        const float iv = ue8m0_inv(code);
#pragma unroll
        for (int j = 0; j < 4; ++j) inv[j * 128 + tid] = iv;
        sf[f8::atom_offset(cs, rb, kg) + f8::atom_byte(tid, (int)rb)] = (uint8_t)code;
      }
    } else {
      // column c = tid & 127, pieces 2h, 2h + 1 (one scale byte each)
      const int c = tid & 127, h = tid >> 7;
#pragma unroll
      for (int j = 2 * h; j < 2 * h + 2; ++j) {
        const uint32_t code = ue8m0_code(part[j * 128 + c]);
        inv[j * 128 + c] = ue8m0_inv(code);
        sf[f8::mx_atom_offset(cs, rb, kg) + f8::atom_byte(c, j)] = (uint8_t)code;
      }
    }
    __syncthreads();
    uint8_t* dst = Xq + (size_t)rb * 128 * cols + c0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int v = tid + 256 * i, r = v >> 4, q = v & 15;
      float f[8];
      unpack8(tile[r][q], f);
      *reinterpret_cast<uint2*>(dst + (size_t)r * cols + q * 8) =
          e4m3x8_each(f, inv + (r >> 5) * 128 + q * 8);
      if (ROWS) {
        // row r's 1 x BLK pieces of this 128-column K block
        constexpr int LANES = BLK / 8;
        float m = amax8(f);
#pragma unroll
        for (int o = LANES / 2; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        const uint32_t code = ue8m0_code(m);
        *reinterpret_cast<uint2*>(Xr + ((size_t)rb * 128 + r) * cols + c0 + q * 8) =
            e4m3x8(f, ue8m0_inv(code));
        if ((q & (LANES - 1)) == 0) {
          if (BLK == 128)
            sfr[f8::atom_offset(rb, cs, kgr) + f8::atom_byte(r, cs)] = (uint8_t)code;
          else
            sfr[f8::mx_atom_offset(rb, cs, kgr) + f8::atom_byte(r, q / LANES)] = (uint8_t)code;
        }
      }
    }
    __syncthreads();
  }
}

// 128 x 128 weight tiles -> E4M3 bytes plus the tile's UE8M0 scale, written
// into two atom arrays: sf_f with the weight's rows as the GEMM's N index and
// its columns as K (the forward GEMMs), sf_d with the roles swapped (the data
// gradients, which read the weight transposed). One block per tile.
__global__ void __launch_bounds__(256, 3)
quant_tiles8_kernel(const __nv_bfloat16* __restrict__ W, uint8_t* __restrict__ Wq,
                    uint8_t* __restrict__ sf_f, uint8_t* __restrict__ sf_d, long long n_tiles,
                    int rows, int cols) {
  // the tile is staged in shared memory between its maximum and its
  // conversion (few registers: three blocks share an SM)
  __shared__ uint4 tile[2048];                            // 128 rows x 128 bf16
  __shared__ float red[8];
  const int tc = cols / 128, tr = rows / 128;
  const int64_t kg_f = f8::atoms_k(cols), kg_d = f8::atoms_k(rows);
  for (long long t = blockIdx.x; t < n_tiles; t += gridDim.x) {
    const long long g = t / ((long long)tr * tc);
    const int rem = (int)(t % ((long long)tr * tc));
    const int rt = rem / tc, ct = rem % tc;
    const int r0 = rt * 128, c0 = ct * 128;
    const size_t base = (size_t)g * rows * cols;
    float m = 0.f;
    {
      uint4 in[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int v = threadIdx.x + 256 * i;              // 2048 vectors per tile
        const int r = v >> 4, c = (v & 15) * 8;
        in[i] = ldg_nc_v4(W + base + (size_t)(r0 + r) * cols + c0 + c);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        float f[8];
        unpack8(in[i], f);
        m = fmaxf(m, amax8(f));
        tile[threadIdx.x + 256 * i] = in[i];
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    float amax = red[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
    const uint32_t code = ue8m0_code(amax);
    const float inv = ue8m0_inv(code);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int v = threadIdx.x + 256 * i;                // each thread reads back its own
      const int r = v >> 4, c = (v & 15) * 8;
      float f[8];
      unpack8(tile[v], f);
      *reinterpret_cast<uint2*>(Wq + base + (size_t)(r0 + r) * cols + c0 + c) = e4m3x8(f, inv);
    }
    const int n = threadIdx.x & 127;
    if (threadIdx.x < 128)
      sf_f[f8::atom_offset(g * tr + rt, ct, kg_f) + f8::atom_byte(n, ct)] = (uint8_t)code;
    else
      sf_d[f8::atom_offset(g * tc + ct, rt, kg_d) + f8::atom_byte(n, rt)] = (uint8_t)code;
    __syncthreads();
  }
}

// MX weights: every 128 x 128 tile of W [G, rows, cols] (bf16) -> two E4M3
// forms. Forward (Wf, sf_f): 1 x 32 pieces along the columns (the forward
// GEMM's K), atoms with the weight's rows as N. Data gradient (Wd, sf_d):
// 32 x 1 pieces along the rows (the data gradient's K), atoms with the
// columns as N. One block of 256 threads per tile: the tile is staged in
// shared memory once and both forms are written from there (few registers, so
// six blocks share an SM and keep their loads in flight together).
__global__ void __launch_bounds__(256, 3)
quant_wmx_kernel(const __nv_bfloat16* __restrict__ W, uint8_t* __restrict__ Wf,
                 uint8_t* __restrict__ Wd, uint8_t* __restrict__ sf_f, uint8_t* __restrict__ sf_d,
                 long long n_tiles, int rows, int cols) {
  __shared__ uint4 tile[128][16];                         // 128 rows x 128 bf16
  __shared__ float inv_d[4][128];                         // [row piece][column]
  const int tc = cols / 128, tr = rows / 128;
  const int tid = threadIdx.x;
  for (long long t = blockIdx.x; t < n_tiles; t += gridDim.x) {
    const long long g = t / ((long long)tr * tc);
    const int rem = (int)(t % ((long long)tr * tc));
    const int rt = rem / tc, ct = rem % tc;
    const size_t base = (size_t)g * rows * cols + (size_t)rt * 128 * cols + (size_t)ct * 128;
    uint4 in[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int v = tid + 256 * i, r = v >> 4, q = v & 15;
      in[i] = ldg_nc_v4(W + base + (size_t)r * cols + q * 8);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int v = tid + 256 * i;
      tile[v >> 4][v & 15] = in[i];
    }
    // forward form: a 1 x 32 piece is four consecutive lanes' vectors (from the
    // registers the tile was loaded into)
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int v = tid + 256 * i, r = v >> 4, q = v & 15;
      float f[8];
      unpack8(in[i], f);
      float m = amax8(f);
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
      const uint32_t code = ue8m0_code(m);
      *reinterpret_cast<uint2*>(Wf + base + (size_t)r * cols + q * 8) = e4m3x8(f, ue8m0_inv(code));
      if ((q & 3) == 0)
        sf_f[f8::mx_atom_offset(g * tr + rt, ct, tc) + f8::atom_byte(r, q >> 2)] = (uint8_t)code;
    }
    __syncthreads();
    {
      // data-gradient form: columns c and c + 1 (one bf16 pair per 4-byte read,
      // consecutive lanes on consecutive words), 32-row piece j
      const int c = 2 * (tid & 63), j = tid >> 6;
      const uint32_t* pair = reinterpret_cast<const uint32_t*>(&tile[0][0]) + (c >> 1);
      float m0 = 0.f, m1 = 0.f;
#pragma unroll 8
      for (int r = 32 * j; r < 32 * j + 32; ++r) {
        const uint32_t w2 = pair[r * 64];
        m0 = fmaxf(m0, fabsf(bf16_lo(w2)));
        m1 = fmaxf(m1, fabsf(bf16_hi(w2)));
      }
      const uint32_t code0 = ue8m0_code(m0), code1 = ue8m0_code(m1);
      inv_d[j][c] = ue8m0_inv(code0);
      inv_d[j][c + 1] = ue8m0_inv(code1);
      const int64_t at = f8::mx_atom_offset(g * tc + ct, rt, tr);
      sf_d[at + f8::atom_byte(c, j)] = (uint8_t)code0;
      sf_d[at + f8::atom_byte(c + 1, j)] = (uint8_t)code1;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int v = tid + 256 * i, r = v >> 4, q = v & 15;
      float f[8];
      unpack8(tile[r][q], f);
      *reinterpret_cast<uint2*>(Wd + base + (size_t)r * cols + q * 8) =
          e4m3x8_each(f, &inv_d[r >> 5][q * 8]);
    }
    __syncthreads();
  }
}

// Scale atoms of E4M3 weights quantised by the caller: one UE8M0 code per
// 128 x 128 tile (scale [G][rows / 128][cols / 128]) into the same two atom
// arrays quant_tiles8_kernel writes (the tile's code for each of its 128 rows
// in sf_f, for each of its 128 columns in sf_d). One thread per (tile, row).
__global__ void __launch_bounds__(256)
load_fp8_scales_kernel(const uint8_t* __restrict__ scale, uint8_t* __restrict__ sf_f,
                       uint8_t* __restrict__ sf_d, long long n_tiles, int rows, int cols) {
  const int tc = cols / 128, tr = rows / 128;
  const int64_t kg_f = f8::atoms_k(cols), kg_d = f8::atoms_k(rows);
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n_tiles * 128;
       i += (long long)gridDim.x * blockDim.x) {
    const long long t = i >> 7;
    const int n = (int)(i & 127);
    const long long g = t / ((long long)tr * tc);
    const int rem = (int)(t % ((long long)tr * tc));
    const int rt = rem / tc, ct = rem % tc;
    const uint8_t code = scale[t];
    sf_f[f8::atom_offset(g * tr + rt, ct, kg_f) + f8::atom_byte(n, ct)] = code;
    sf_d[f8::atom_offset(g * tc + ct, rt, kg_d) + f8::atom_byte(n, rt)] = code;
  }
}

static int grid_cap(long long work_items, int per_block) {
  long long b = (work_items + per_block - 1) / per_block;
  const long long cap = (long long)num_sms() * 16;
  if (b > cap) b = cap;
  return b > 0 ? (int)b : 1;
}

cudaError_t launch_quant_tiles8(const void* W, uint8_t* Wq, uint8_t* sf_f, uint8_t* sf_d, int G,
                                int rows, int cols, cudaStream_t s) {
  const long long n = (long long)G * (rows / 128) * (cols / 128);
  quant_tiles8_kernel<<<grid_cap(n, 1), 256, 0, s>>>(static_cast<const __nv_bfloat16*>(W), Wq,
                                                     sf_f, sf_d, n, rows, cols);
  return cudaGetLastError();
}

cudaError_t launch_load_fp8_scales(const uint8_t* scale, uint8_t* sf_f, uint8_t* sf_d, int G,
                                   int rows, int cols, cudaStream_t s) {
  const long long n = (long long)G * (rows / 128) * (cols / 128);
  load_fp8_scales_kernel<<<grid_cap(n * 128, 256), 256, 0, s>>>(scale, sf_f, sf_d, n, rows, cols);
  return cudaGetLastError();
}

cudaError_t launch_quant_wmx(const void* W, uint8_t* Wf, uint8_t* Wd, uint8_t* sf_f, uint8_t* sf_d,
                             int G, int rows, int cols, cudaStream_t s) {
  const long long n = (long long)G * (rows / 128) * (cols / 128);
  quant_wmx_kernel<<<grid_cap(n, 1), 256, 0, s>>>(static_cast<const __nv_bfloat16*>(W), Wf, Wd,
                                                  sf_f, sf_d, n, rows, cols);
  return cudaGetLastError();
}

cudaError_t launch_quant_cols8(const void* X, uint8_t* Xq, uint8_t* sf, const int32_t* offsets,
                               const int32_t* counts, int G, int64_t rows_max, int cols,
                               cudaStream_t s, bool mx, const int32_t* pages) {
  constexpr int smem = 128 * 16 * 16 + 8 * 128 * 4;     // tile + piece maxima + 1/scales
  const int grid = grid_cap(rows_max / 128 * (cols / 128), 1);
  const long long kg = f8::sf_stride(rows_max, mx);
  const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(X);
  if (mx)
    quant_cols8_kernel<32, false><<<grid, 256, smem, s>>>(x, Xq, sf, offsets, counts, G, cols, kg,
                                                           nullptr, nullptr, 0, pages);
  else
    quant_cols8_kernel<128, false><<<grid, 256, smem, s>>>(x, Xq, sf, offsets, counts, G, cols,
                                                            kg, nullptr, nullptr, 0, pages);
  return cudaGetLastError();
}

cudaError_t launch_quant_rows_cols8(const void* X, uint8_t* Xr, uint8_t* sfr, uint8_t* Xc,
                                    uint8_t* sfc, const int32_t* offsets, const int32_t* counts,
                                    int G, int64_t rows_max, int cols, cudaStream_t s, bool mx) {
  constexpr int smem = 128 * 16 * 16 + 8 * 128 * 4;
  const int grid = grid_cap(rows_max / 128 * (cols / 128), 1);
  const long long kgc = f8::sf_stride(rows_max, mx), kgr = f8::sf_stride(cols, mx);
  const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(X);
  if (mx)
    quant_cols8_kernel<32, true><<<grid, 256, smem, s>>>(x, Xc, sfc, offsets, counts, G, cols,
                                                          kgc, Xr, sfr, kgr, nullptr);
  else
    quant_cols8_kernel<128, true><<<grid, 256, smem, s>>>(x, Xc, sfc, offsets, counts, G, cols,
                                                           kgc, Xr, sfr, kgr, nullptr);
  return cudaGetLastError();
}

}  // namespace moe
