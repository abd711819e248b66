// Device helpers shared by the MoE kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe_abi.h"

namespace moe {

constexpr int kMaxExperts = 256;
constexpr int kMaxGroups = kMaxExperts + 4;    // routed + shared
constexpr int kMaxK = 8;
constexpr int kChunkTokens = 256;              // tokens per dispatch-map chunk

// Scratch layout (bytes from the start of the caller's scratch buffer).
constexpr size_t kScratchStatus = 0;           // int32 device status word
constexpr size_t kScratchAuxTicket = 64;       // uint32 arrival counter of the aux-loss blocks
constexpr size_t kScratchPadPrefix = 256;      // int32 [kMaxGroups+1]
constexpr size_t kScratchHist = 4096;          // int32 [n_chunks][E]

// Records the first problem a kernel sees; never traps.
__device__ __forceinline__ void record_status(int32_t* status, int32_t code) {
  if (status) atomicCAS(status, 0, code);
}

// Row of a layer's stash tensors (x_perm, GU, h, y_perm) that holds its row r:
// with a stash page table (paged stashing), row r lives in page pages[r / 128]
// of the pool; without one (pages == nullptr) the layer's own buffers hold it
// at row r.
__device__ __forceinline__ int stash_row(const int32_t* __restrict__ pages, int r) {
  return pages ? (__ldg(pages + (r >> 7)) << 7) | (r & 127) : r;
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// Eight bf16 in one 16-byte vector -> fp32.
__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
  f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
  f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
  f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

// Round-to-nearest-even fp32 pair -> packed bf16x2 (cvt.rn.bf16x2.f32).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two fp32 values -> their three packed bf16 parts (pairs: low half = first):
// hi = bf16(w), mid = bf16(w - hi), lo = w - hi - mid. Each part keeps 8
// significant bits of the 24, so both subtractions are exact, lo is exactly a
// bf16, and hi + mid + lo == w.
__device__ __forceinline__ void split3_pair(float w0, float w1, uint32_t& hi, uint32_t& mid,
                                            uint32_t& lo) {
  hi = pack_bf16x2(w0, w1);
  const float r0 = w0 - bf16_lo(hi), r1 = w1 - bf16_hi(hi);
  mid = pack_bf16x2(r0, r1);
  lo = pack_bf16x2(r0 - bf16_lo(mid), r1 - bf16_hi(mid));
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  uint4 v;
  v.x = pack_bf16x2(f[0], f[1]);
  v.y = pack_bf16x2(f[2], f[3]);
  v.z = pack_bf16x2(f[4], f[5]);
  v.w = pack_bf16x2(f[6], f[7]);
  return v;
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// L2 eviction-priority policies (createpolicy) and loads that carry them: data
// read once is marked evict-first so that it does not push out small tables
// that every token re-reads (marked evict-last).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint4 ldg_nc_v4_pol(const void* p, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p), "l"(pol));
  return v;
}
__device__ __forceinline__ float4 ldg_nc_f4_pol(const void* p, uint64_t pol) {
  float4 v;
  asm volatile("ld.global.nc.L2::cache_hint.v4.f32 {%0,%1,%2,%3}, [%4], %5;"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p), "l"(pol));
  return v;
}

__device__ __forceinline__ void stg_v4(void* p, const uint4& v) {
  *reinterpret_cast<uint4*>(p) = v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Exclusive scan of n <= 4*blockDim int32 values held in shared memory `a`
// (in place); returns the total. All threads of the block must call it.
// `tmp` needs 33 ints of shared memory.
__device__ inline int block_exclusive_scan(int* a, int n, int* tmp) {
  const int tid = threadIdx.x, nt = blockDim.x;
  const int per = (n + nt - 1) / nt;             // <= 4
  int v[4];
  int local = 0;
  for (int i = 0; i < per; ++i) {
    int j = tid * per + i;
    v[i] = (j < n) ? a[j] : 0;
    local += v[i];
  }
  // inclusive warp scan of `local`
  const int lane = tid & 31, wid = tid >> 5;
  int inc = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) tmp[wid] = inc;
  __syncthreads();
  if (wid == 0) {
    const int nw = (nt + 31) >> 5;
    int s = (lane < nw) ? tmp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < nw) tmp[lane] = s;                 // inclusive warp totals
    if (lane == nw - 1) tmp[32] = s;
  }
  __syncthreads();
  int run = inc - local + (wid > 0 ? tmp[wid - 1] : 0);
  for (int i = 0; i < per; ++i) {
    int j = tid * per + i;
    if (j < n) a[j] = run;
    run += v[i];
  }
  const int total = tmp[32];
  __syncthreads();
  return total;
}

}  // namespace moe
