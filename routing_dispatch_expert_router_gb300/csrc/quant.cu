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
// The quantised values are written back as bf16, which holds every E4M3 value
// times a power of two exactly, so the tcgen05 bf16 GEMMs that consume them
// form exactly the products an FP8 block-scaled MMA would (fp32 accumulation).
// E4M3 rounding (to nearest even, saturating) uses the hardware conversion.
#include <cuda_fp16.h>

#include "common.cuh"
#include "internal.h"

namespace moe {

__device__ __forceinline__ float e4m3_scale(float amax) {
  if (!(amax > 0.f)) return 1.f;
  int e;
  const float m = frexpf(__fdiv_rn(amax, 448.f), &e);   // amax/448 = m * 2^e
  return ldexpf(1.f, m == 0.5f ? e - 1 : e);
}

// E4M3(a / s) * s for two values (s a power of two, so a / s and the product
// are exact).
__device__ __forceinline__ void q2(float a, float b, float inv_s, float s, float& qa, float& qb) {
  uint16_t packed;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(packed) : "f"(b * inv_s), "f"(a * inv_s));
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(packed));
  const __half2 hv = *reinterpret_cast<const __half2*>(&h2);
  qa = __low2float(hv) * s;
  qb = __high2float(hv) * s;
}

__device__ __forceinline__ float q1(float a, float inv_s, float s) {
  float qa, unused;
  q2(a, 0.f, inv_s, s, qa, unused);
  return qa;
}

__device__ __forceinline__ uint4 quant8(const float (&f)[8], float s) {
  const float inv = 1.f / s;                              // exact: s is a power of two
  float o[8];
#pragma unroll
  for (int i = 0; i < 8; i += 2) q2(f[i], f[i + 1], inv, s, o[i], o[i + 1]);
  return pack8(o);
}

__device__ __forceinline__ float amax8(const float (&f)[8]) {
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(f[i]));
  return m;
}

// 128 x 128 tiles: one block per tile, thread owns 8 vectors of 8 elements.
__global__ void __launch_bounds__(256)
quant_tiles_kernel(const __nv_bfloat16* __restrict__ W, __nv_bfloat16* __restrict__ Wq,
                   long long n_tiles, int rows, int cols) {
  __shared__ float red[8];
  const int tc = cols / 128, tr = rows / 128;
  for (long long tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
    const long long g = tile / ((long long)tr * tc);
    const int rem = (int)(tile % ((long long)tr * tc));
    const int r0 = (rem / tc) * 128, c0 = (rem % tc) * 128;
    const size_t base = (size_t)g * rows * cols;
    float f[8][8];
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int v = threadIdx.x + 256 * i;                // 2048 vectors per tile
      const int r = v >> 4, c = (v & 15) * 8;
      unpack8(ldg_nc_v4(W + base + (size_t)(r0 + r) * cols + c0 + c), f[i]);
      m = fmaxf(m, amax8(f[i]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    float amax = red[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
    const float s = e4m3_scale(amax);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int v = threadIdx.x + 256 * i;
      const int r = v >> 4, c = (v & 15) * 8;
      stg_v4(Wq + base + (size_t)(r0 + r) * cols + c0 + c, quant8(f[i], s));
    }
    __syncthreads();
  }
}

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

// 1 x 128 slices along the rows of the live 128-row blocks of [0, offsets[G]):
// one block of 256 threads per 128-row block, 16 lanes per slice. (Four
// vectors per thread in flight measured slower than one.)
__global__ void __launch_bounds__(256)
quant_rows_kernel(const __nv_bfloat16* __restrict__ X, __nv_bfloat16* __restrict__ Xq,
                  const int32_t* __restrict__ offsets, const int32_t* __restrict__ counts, int G,
                  int cols) {
  const long long rblocks = offsets[G] / 128;
  const int nvec = cols >> 3;                             // a multiple of 16
  const int per_block = 128 * nvec;
  for (long long rb = blockIdx.x; rb < rblocks; rb += gridDim.x) {
    if (!live_block(offsets, counts, G, rb)) continue;
    const __nv_bfloat16* src = X + (size_t)rb * 128 * cols;
    __nv_bfloat16* dst = Xq + (size_t)rb * 128 * cols;
    for (int v = threadIdx.x; v < per_block; v += 256) {
      float f[8];
      unpack8(ldg_nc_v4(src + (size_t)v * 8), f);
      float m = amax8(f);
      // the 16 lanes of this half-warp hold one 128-element slice (per_block
      // and 256 are multiples of 16: a half-warp is wholly in range or out)
      const unsigned half = (threadIdx.x & 16) ? 0xffff0000u : 0x0000ffffu;
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(half, m, o));
      stg_v4(dst + (size_t)v * 8, quant8(f, e4m3_scale(m)));
    }
  }
}

// 128 x 1 slices: every live 128-row block of [0, offsets[G]) (group segments
// are multiples of 128 rows, so blocks never straddle two experts). One block
// of 256 threads per (128-row block, 128-column slab): the 128 x 128 tile is
// read once into shared memory with 16-byte loads (eight per thread in
// flight), the column maxima are taken there (two partial maxima of 64 rows
// per column), and every thread quantises and stores eight 8-column vectors
// read back from the tile.
__global__ void __launch_bounds__(256)
quant_cols_kernel(const __nv_bfloat16* __restrict__ X, __nv_bfloat16* __restrict__ Xq,
                  const int32_t* __restrict__ offsets, const int32_t* __restrict__ counts, int G,
                  int cols) {
  extern __shared__ uint4 qc_smem[];
  uint4 (*tile)[16] = reinterpret_cast<uint4 (*)[16]>(qc_smem);   // 128 rows x 128 bf16
  float* part = reinterpret_cast<float*>(qc_smem + 128 * 16);      // [2][128]
  float* scale = part + 256;                                       // [128]
  const long long rblocks = offsets[G] / 128;
  const int slabs = cols >> 7;
  const int tid = threadIdx.x;
  for (long long w = blockIdx.x; w < rblocks * slabs; w += gridDim.x) {
    const long long rb = w / slabs;
    const int c0 = (int)(w - rb * slabs) * 128;
    if (!live_block(offsets, counts, G, rb)) continue;
    const __nv_bfloat16* src = X + (size_t)rb * 128 * cols + c0;
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
      const int c = tid & 127, h = tid >> 7;
      const __nv_bfloat16* col = reinterpret_cast<const __nv_bfloat16*>(&tile[0][0]) + c;
      float m = 0.f;
#pragma unroll 8
      for (int r = h * 64; r < h * 64 + 64; ++r) m = fmaxf(m, fabsf(__bfloat162float(col[r * 128])));
      part[h * 128 + c] = m;
    }
    __syncthreads();
    if (tid < 128) scale[tid] = e4m3_scale(fmaxf(part[tid], part[128 + tid]));
    __syncthreads();
    __nv_bfloat16* dst = Xq + (size_t)rb * 128 * cols + c0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int v = tid + 256 * i, r = v >> 4, q = v & 15;
      float f[8], o[8];
      unpack8(tile[r][q], f);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float sc = scale[q * 8 + j];
        o[j] = q1(f[j], 1.f / sc, sc);
      }
      stg_v4(dst + (size_t)r * cols + q * 8, pack8(o));
    }
    __syncthreads();
  }
}

static int grid_cap(long long work_items, int per_block) {
  long long b = (work_items + per_block - 1) / per_block;
  const long long cap = (long long)num_sms() * 16;
  if (b > cap) b = cap;
  return b > 0 ? (int)b : 1;
}

cudaError_t launch_quant_tiles(const void* W, void* Wq, int G, int rows, int cols, cudaStream_t s) {
  const long long n = (long long)G * (rows / 128) * (cols / 128);
  quant_tiles_kernel<<<grid_cap(n, 1), 256, 0, s>>>(static_cast<const __nv_bfloat16*>(W),
                                                    static_cast<__nv_bfloat16*>(Wq), n, rows, cols);
  return cudaGetLastError();
}

cudaError_t launch_quant_rows(const void* X, void* Xq, const int32_t* offsets,
                              const int32_t* counts, int G, int64_t rows_max, int cols,
                              cudaStream_t s) {
  quant_rows_kernel<<<grid_cap(rows_max / 128, 1), 256, 0, s>>>(
      static_cast<const __nv_bfloat16*>(X), static_cast<__nv_bfloat16*>(Xq), offsets, counts, G,
      cols);
  return cudaGetLastError();
}

cudaError_t launch_quant_cols(const void* X, void* Xq, const int32_t* offsets,
                              const int32_t* counts, int G, int64_t rows_max, int cols,
                              cudaStream_t s) {
  constexpr int smem = 128 * 16 * 16 + 3 * 128 * 4;     // tile + two partial maxima + scales
  quant_cols_kernel<<<grid_cap(rows_max / 128 * (cols / 128), 1), 256, smem, s>>>(
      static_cast<const __nv_bfloat16*>(X), static_cast<__nv_bfloat16*>(Xq), offsets, counts, G,
      cols);
  return cudaGetLastError();
}

}  // namespace moe
