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
#include <algorithm>

#include "common.cuh"
#include "fp8_layout.cuh"
#include "internal.h"

namespace moe {

// The live 128-row blocks of the permuted buffer: group g's segment starts at
// offsets[g] (a multiple of 128 rows), and the GEMMs read its first
// ceil(counts[g] / 128) blocks (capacity segments and dropless padding past
// them are never read, so they are not quantised). Every block of 256 threads
// writes pre[g] = the live blocks of the groups before g, for g = 0 .. G
// (pre[G] = all of them), into its shared memory; G <= 511.
__device__ __forceinline__ int live_block_prefix(const int32_t* __restrict__ counts, int G,
                                                 int* pre, int* wsum) {
  const int t = threadIdx.x, lane = t & 31, wid = t >> 5;
  const int g0 = 2 * t, g1 = 2 * t + 1;
  const int n0 = g0 < G ? (counts[g0] + 127) / 128 : 0;
  const int n1 = g1 < G ? (counts[g1] + 127) / 128 : 0;
  int v = n0 + n1;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
  if (lane == 31) wsum[wid] = v;
  __syncthreads();
  int excl = v - n0 - n1;
  for (int w = 0; w < wid; ++w) excl += wsum[w];
  if (g0 <= G) pre[g0] = excl;
  if (g1 <= G) pre[g1] = excl + n0;
  __syncthreads();
  return pre[G];
}

// Row block of live block lb: the last group g with pre[g] <= lb holds it.
__device__ __forceinline__ long long live_row_block(const int* pre, const int32_t* offsets, int G,
                                                    int lb) {
  int lo = 0, hi = G - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pre[mid] <= lb) lo = mid;
    else hi = mid - 1;
  }
  return offsets[lo] / 128 + (lb - pre[lo]);
}

// BLK x 1 slices (BLK = 128, or 32 for MX): every live 128-row block (group
// segments are multiples of 128 rows, so blocks never straddle two experts)
// -> E4M3 bytes plus the UE8M0 scale atoms [cols / 128][along the rows]. One
// block of 256 threads per (128-row block, 128-column slab), looping over the
// live tiles: thread (m, q) = (tid / 16, tid % 16) holds rows m + 16 i (i < 8)
// of the slab's columns 8q .. 8q + 7 in registers (16-byte loads, two 256-byte
// rows per warp instruction), takes its maxima of each column's 32-row pieces
// there, meets lane q + 16 (rows m ^ 1) by one shuffle and the other seven
// warps in shared memory, and quantises its own vectors; the next tile's eight
// loads are issued before this tile is processed, so they are in flight during
// it. With ROWS, the same pass also writes the tile's 1 x BLK row form (Xr,
// sfr; a row's 16 vectors sit in 16 consecutive lanes, whose maxima meet by
// shuffles), so a tensor both GEMM directions need is read once.
template <int BLK, bool ROWS>
__global__ void __launch_bounds__(256, 2)
quant_cols8_kernel(const __nv_bfloat16* __restrict__ X, uint8_t* __restrict__ Xq,
                   uint8_t* __restrict__ sf, const int32_t* __restrict__ offsets,
                   const int32_t* __restrict__ counts, int G, int cols, long long kg,
                   uint8_t* __restrict__ Xr, uint8_t* __restrict__ sfr, long long kgr,
                   const int32_t* __restrict__ pages) {
  static_assert(BLK == 128 || BLK == 32, "block length");
  constexpr int NP = 128 / BLK;                  // pieces of a 128-row block
  constexpr int IP = 8 / NP;                     // a thread's rows per piece
  __shared__ int pre[kMaxGroups + 1];
  __shared__ int wsum[8];
  __shared__ uint32_t part[8][NP][64];          // [warp][piece][column pair] bf16 maxima
  __shared__ __align__(16) float inv[NP][128];   // [piece][column] 1 / scale
  const int slabs = cols >> 7;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int q = tid & 15, m = tid >> 4;
  // (live tiles only, dealt round-robin: every block of the resident grid
  // gets the same number of tiles, to within one)
  const long long work = (long long)live_block_prefix(counts, G, pre, wsum) * slabs;
  auto tile_of = [&](long long w, int& cs) -> long long {
    const int lb = (int)(w / slabs);
    cs = (int)(w - (long long)lb * slabs);
    return live_row_block(pre, offsets, G, lb);
  };
  // (a paged stash tensor keeps the block in one page)
  auto load = [&](long long w, uint4 (&v)[8]) {
    int cs;
    const long long rb = tile_of(w, cs);
    const __nv_bfloat16* src = X + (size_t)stash_row(pages, (int)rb * 128) * cols + cs * 128;
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = ldg_nc_v4(src + (size_t)(m + 16 * i) * cols + q * 8);
  };
  uint4 cur[8], nxt[8];
  long long w = blockIdx.x;
  if (w < work) load(w, cur);
  for (; w < work; w += gridDim.x) {
    if (w + gridDim.x < work) load(w + gridDim.x, nxt);
    int cs;
    const long long rb = tile_of(w, cs);
    const int c0 = cs * 128;
    // |x| maxima on packed bf16 pairs (exact: the maximum of bf16 values is one of them)
#pragma unroll
    for (int p = 0; p < NP; ++p) {
      __nv_bfloat162 mx[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) mx[j] = __float2bfloat162_rn(0.f);
#pragma unroll
      for (int i = p * IP; i < (p + 1) * IP; ++i) {
        const __nv_bfloat162* v = reinterpret_cast<const __nv_bfloat162*>(&cur[i]);
#pragma unroll
        for (int j = 0; j < 4; ++j) mx[j] = __hmax2(mx[j], __habs2(v[j]));
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t u = *reinterpret_cast<const uint32_t*>(&mx[j]);
        u = __shfl_xor_sync(0xffffffffu, u, 16);
        mx[j] = __hmax2(mx[j], *reinterpret_cast<const __nv_bfloat162*>(&u));
      }
      if (lane < 16) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          part[wid][p][q * 4 + j] = *reinterpret_cast<const uint32_t*>(&mx[j]);
      }
    }
    __syncthreads();
    for (int x = tid; x < NP * 128; x += 256) {
      const int p = x >> 7, c = x & 127;
      float a = 0.f;
#pragma unroll
      for (int w2 = 0; w2 < 8; ++w2) {
        const uint32_t u = part[w2][p][c >> 1];
        a = fmaxf(a, (c & 1) ? bf16_hi(u) : bf16_lo(u));
      }
      const uint32_t code = ue8m0_code(a);
      inv[p][c] = ue8m0_inv(code);
      if (BLK == 128)
        sf[f8::atom_offset(cs, rb, kg) + f8::atom_byte(c, (int)rb)] = (uint8_t)code;
      else
        sf[f8::mx_atom_offset(cs, rb, kg) + f8::atom_byte(c, p)] = (uint8_t)code;
    }
    __syncthreads();
    uint8_t* dst = Xq + (size_t)rb * 128 * cols + c0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = m + 16 * i;
      float f[8];
      unpack8(cur[i], f);
      *reinterpret_cast<uint2*>(dst + (size_t)r * cols + q * 8) =
          e4m3x8_each(f, &inv[i / IP][q * 8]);
      if (ROWS) {
        // row r's 1 x BLK pieces of this 128-column K block
        constexpr int LANES = BLK / 8;
        float a = amax8(f);
#pragma unroll
        for (int o = LANES / 2; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
        const uint32_t code = ue8m0_code(a);
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
#pragma unroll
    for (int i = 0; i < 8; ++i) cur[i] = nxt[i];
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

// Grid of a kernel whose blocks loop over equal work items: the blocks that
// fit on the GPU at once, or fewer when there is less work. A larger grid runs
// in rounds, and its last partial round of long-lived blocks leaves most SMs
// idle for the length of a whole block's loop.
template <typename Kern>
static int resident_grid(Kern kern, size_t smem, long long work_items) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 256, smem) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  long long b = (long long)num_sms() * per_sm;
  if (b > work_items) b = work_items;
  return b > 0 ? (int)b : 1;
}

cudaError_t launch_quant_tiles8(const void* W, uint8_t* Wq, uint8_t* sf_f, uint8_t* sf_d, int G,
                                int rows, int cols, cudaStream_t s) {
  const long long n = (long long)G * (rows / 128) * (cols / 128);
  static const int resident = resident_grid(quant_tiles8_kernel, 0, 1LL << 40);
  quant_tiles8_kernel<<<(int)(n < resident ? (n > 0 ? n : 1) : resident), 256, 0, s>>>(static_cast<const __nv_bfloat16*>(W), Wq,
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
  static const int resident = resident_grid(quant_wmx_kernel, 0, 1LL << 40);
  quant_wmx_kernel<<<(int)(n < resident ? (n > 0 ? n : 1) : resident), 256, 0, s>>>(static_cast<const __nv_bfloat16*>(W), Wf, Wd,
                                                  sf_f, sf_d, n, rows, cols);
  return cudaGetLastError();
}

cudaError_t launch_quant_cols8(const void* X, uint8_t* Xq, uint8_t* sf, const int32_t* offsets,
                               const int32_t* counts, int G, int64_t rows_max, int cols,
                               cudaStream_t s, bool mx, const int32_t* pages) {
  constexpr int smem = 0;                              // (static shared memory only)
  const long long tiles = rows_max / 128 * (cols / 128);
  static const int res32 = resident_grid(quant_cols8_kernel<32, false>, smem, 1LL << 40);
  static const int res128 = resident_grid(quant_cols8_kernel<128, false>, smem, 1LL << 40);
  const long long kg = f8::sf_stride(rows_max, mx);
  const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(X);
  const int grid = (int)std::max(1LL, std::min(tiles, (long long)(mx ? res32 : res128)));
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
  constexpr int smem = 0;
  const long long tiles = rows_max / 128 * (cols / 128);
  static const int res32 = resident_grid(quant_cols8_kernel<32, true>, smem, 1LL << 40);
  static const int res128 = resident_grid(quant_cols8_kernel<128, true>, smem, 1LL << 40);
  const int grid = (int)std::max(1LL, std::min(tiles, (long long)(mx ? res32 : res128)));
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
