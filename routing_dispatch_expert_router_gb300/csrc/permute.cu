// Stage 2 of the MoE layer, dispatch, done locally: a stable counting sort of
// the (token, slot) assignments by (expert, token), then a copy of every token
// row into its experts' contiguous segments.
//
// Follows the dispatch stage of "Scalable Training of Mixture-of-Experts
// Models with Megatron Core" (es summary, Resumen técnico §2.1 step 2); with
// every expert on one GPU the all-to-all becomes this permutation. The maps
// are computed without atomics whose order matters, so they are
// deterministic and bit-identical from run to run.
//
// Three launches (four with a paged stash):
//   hist    one block per chunk of 256 tokens: per-expert counts of the chunk;
//   rank    one block per chunk: global counts, segment offsets, and the rank
//           of every assignment = (assignments of its expert in earlier
//           chunks) + (earlier tokens of this chunk that chose the same
//           expert, read from a per-expert bitmap of the chunk's tokens);
//   alloc   (paged stash) one block: the layer's stash pages and page table;
//   scatter one warp per token: reads the row once, writes it to each of its
//           rows with 16-byte stores; padding rows are zero-filled.
#include "common.cuh"
#include "fp8_layout.cuh"
#include "internal.h"

namespace moe {

// Whether assignment i = t*k + j names the same expert as an earlier slot of
// token t. Such a repeat (possible only in a caller-given idx, e.g. a replayed
// one) is reported and dropped like an out-of-range id, so that every counted
// row of an expert segment is written exactly once.
__device__ __forceinline__ bool repeats_earlier_slot(const int32_t* __restrict__ idx, int i, int k,
                                                     int e) {
  for (int i0 = i - i % k; i0 < i; ++i0)
    if (idx[i0] == e) return true;
  return false;
}

__global__ void __launch_bounds__(256)
permute_hist_kernel(const int32_t* __restrict__ idx, int32_t* __restrict__ hist, int T, int k,
                    int E, int32_t* status) {
  __shared__ int cnt[kMaxExperts];
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  const int c = blockIdx.x;
  const int t0 = c * kChunkTokens, t1 = min(T, t0 + kChunkTokens);
  for (int i = t0 * k + threadIdx.x; i < t1 * k; i += blockDim.x) {
    const int e = idx[i];
    if ((unsigned)e < (unsigned)E && !repeats_earlier_slot(idx, i, k, e)) atomicAdd(&cnt[e], 1);
    else record_status(status, MOE_ERR_DEVICE_CHECK);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[(size_t)c * E + e] = cnt[e];
}

__global__ void __launch_bounds__(256)
permute_rank_kernel(const int32_t* __restrict__ idx, const int32_t* __restrict__ hist,
                    int n_chunk, int T, int k, int E, int S, int align, int C,
                    int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                    int32_t* __restrict__ row_of, int32_t* __restrict__ token_of,
                    int32_t* __restrict__ sel_offsets, int32_t* __restrict__ sel_tokens,
                    int32_t* __restrict__ pad_prefix) {
  __shared__ int tot[kMaxExperts];
  __shared__ int before[kMaxExperts];
  __shared__ int seg[kMaxGroups + 1];
  __shared__ int kept[kMaxGroups];
  __shared__ int pad[kMaxGroups + 1];
  __shared__ int soff[kMaxExperts + 1];
  __shared__ uint32_t bm[kMaxExperts][kChunkTokens / 32];
  __shared__ int tmp[33];
  const int c = blockIdx.x, G = E + S, tid = threadIdx.x, nt = blockDim.x;

  for (int e = tid; e < E; e += nt) {
    int a = 0, b = 0;
    for (int cc = 0; cc < n_chunk; ++cc) {
      const int h = hist[(size_t)cc * E + e];
      a += h;
      if (cc < c) b += h;
    }
    tot[e] = a;
    before[e] = b;
    soff[e] = a;
  }
  for (int i = tid; i < E * (kChunkTokens / 32); i += nt) (&bm[0][0])[i] = 0u;
  __syncthreads();
  for (int g = tid; g < G; g += nt) {
    int kp, sl;
    if (g < E) {
      kp = C > 0 ? min(tot[g], C) : tot[g];
      sl = C > 0 ? C : (kp + align - 1) / align * align;
    } else {
      kp = T;
      sl = (T + align - 1) / align * align;
    }
    kept[g] = kp;
    seg[g] = sl;
    // padding rows that a GEMM reads: the rest of the segment's last 128-row
    // block (rows past it -- capacity segments, row_align > 128 -- are never read)
    pad[g] = min(sl, (kp + 127) / 128 * 128) - kp;
  }
  __syncthreads();
  const int R = block_exclusive_scan(seg, G, tmp);
  const int P = block_exclusive_scan(pad, G, tmp);
  const int A = block_exclusive_scan(soff, E, tmp);
  if (tid == 0) {
    seg[G] = R;
    pad[G] = P;
    soff[E] = A;
  }
  __syncthreads();
  if (c == 0) {
    for (int g = tid; g < G; g += nt) counts[g] = kept[g];
    for (int g = tid; g <= G; g += nt) {
      offsets[g] = seg[g];
      pad_prefix[g] = pad[g];
    }
    for (int e = tid; e <= E; e += nt) sel_offsets[e] = soff[e];
  }
  const int t0 = c * kChunkTokens, t1 = min(T, t0 + kChunkTokens);
  for (int i = t0 * k + tid; i < t1 * k; i += nt) {
    const int e = idx[i];
    if ((unsigned)e >= (unsigned)E || repeats_earlier_slot(idx, i, k, e)) continue;
    const int tl = i / k - t0;
    atomicOr(&bm[e][tl >> 5], 1u << (tl & 31));
  }
  __syncthreads();
  for (int i = t0 * k + tid; i < t1 * k; i += nt) {
    const int e = idx[i];
    if ((unsigned)e >= (unsigned)E || repeats_earlier_slot(idx, i, k, e)) {
      row_of[i] = -1;
      continue;
    }
    const int t = i / k, tl = t - t0, wd = tl >> 5;
    int local = __popc(bm[e][wd] & ((1u << (tl & 31)) - 1u));
    for (int q = 0; q < wd; ++q) local += __popc(bm[e][q]);
    const int rank = before[e] + local;
    sel_tokens[soff[e] + rank] = t;
    int row = -1;
    if (C == 0 || rank < C) {
      row = seg[e] + rank;
      token_of[row] = t;
    }
    row_of[i] = row;
  }
  for (int s = 0; s < S; ++s)
    for (int t = t0 + tid; t < t1; t += nt) token_of[seg[E + s] + t] = t;
  // padding rows of groups g = c, c + gridDim.x, ... (gridDim.x >= 1 even when T == 0)
  for (int g = c; g < G; g += gridDim.x)
    for (int r = seg[g] + kept[g] + tid; r < seg[g + 1]; r += nt) token_of[r] = -1;
}

// Paged stashing (es summary §2.3.C: the dynamic buffers are managed inside
// the CUDA graph instead of being reserved for the worst case). The rows a
// layer keeps for its backward live in a pool of 128-row pages shared by the
// layers of a step. Once the segment offsets are on the device, one block
// takes as many pages as the layer has live 128-row blocks -- the
// ceil(counts[g] / 128) blocks of group g from offsets[g] / 128 on, the ones
// the grouped GEMMs' row tiles cover -- from the pool's counter (a
// compare-and-swap, so layers on other streams can allocate too), numbers
// them in block order, and maps every other block, including the one past the
// last row (the odd half of a CTA-pair tile reads there), to the spill page P.
// A layer that does not fit takes no page: all of its blocks map to the spill
// page, MOE_ERR_STASH_FULL is recorded, and every access stays in the pool.
// Entry nblk + 1 keeps the first page taken (the counter's value before),
// which the release writes back.
__global__ void __launch_bounds__(256)
stash_alloc_kernel(const int32_t* __restrict__ counts, const int32_t* __restrict__ offsets,
                   int G, int nblk, int P, int32_t* __restrict__ top,
                   int32_t* __restrict__ table, int32_t* status) {
  __shared__ int pre[kMaxGroups + 1];
  __shared__ int blk0[kMaxGroups + 1];
  __shared__ int tmp[33];
  __shared__ int s_first, s_ok;
  const int tid = threadIdx.x, nt = blockDim.x;
  for (int g = tid; g < G; g += nt) {
    pre[g] = (counts[g] + 127) >> 7;
    blk0[g] = offsets[g] >> 7;
  }
  if (tid == 0) blk0[G] = offsets[G] >> 7;
  __syncthreads();
  const int n = block_exclusive_scan(pre, G, tmp);
  if (tid == 0) {
    pre[G] = n;
    int old = atomicAdd(top, 0);
    int first = -1;
    while (old >= 0 && old <= P - n) {
      const int seen = atomicCAS(top, old, old + n);
      if (seen == old) {
        first = old;
        break;
      }
      old = seen;
    }
    s_ok = first >= 0;
    s_first = first >= 0 ? first : old;
    if (first < 0) record_status(status, MOE_ERR_STASH_FULL);
    table[nblk + 1] = s_first;
  }
  __syncthreads();
  for (int b = tid; b <= nblk; b += nt) {
    int page = P;
    if (s_ok) {
      // the group whose segment holds block b: the last g with blk0[g] <= b
      int lo = 0, hi = G - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (blk0[mid] <= b) lo = mid;
        else hi = mid - 1;
      }
      const int i = b - blk0[lo];
      if (G > 0 && i >= 0 && i < pre[lo + 1] - pre[lo]) page = s_first + pre[lo] + i;
    }
    table[b] = page;
  }
}

__global__ void stash_release_kernel(const int32_t* __restrict__ table, int nblk,
                                     int32_t* __restrict__ top) {
  if (threadIdx.x == 0) *top = table[nblk + 1];
}

// Finds the group whose padding range holds padding row number p.
__device__ __forceinline__ int find_group(const int* prefix, int G, int p) {
  int lo = 0, hi = G - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= p) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Virtual rows v < T copy token v to its rows; v >= T zero one padding row
// (the padding rows inside each segment's last 128-row block, the ones a GEMM
// reads).
// With xq (the FP8 configurations) every row is also written in its 1-byte
// form -- E4M3 codes of its 1 x 128 slices (MXFP8: 1 x 32) and their UE8M0
// scales in the atoms of xsf (fp8_layout.cuh) -- for the FC1 GEMM: each slice
// is quantised once per token and written to each of the token's rows;
// padding rows get zero codes and scale 1.
template <bool MX>
__global__ void __launch_bounds__(256)
permute_scatter_kernel(const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ row_of,
                       const int32_t* __restrict__ counts, const int32_t* __restrict__ offsets,
                       const int32_t* __restrict__ pad_prefix, __nv_bfloat16* __restrict__ x_perm,
                       int T, int H, int k, int E, int S, uint8_t* __restrict__ xq,
                       uint8_t* __restrict__ xsf, const int32_t* __restrict__ pages) {
  __shared__ int s_pp[kMaxGroups + 1];
  __shared__ int s_off[kMaxGroups + 1];
  __shared__ int s_cnt[kMaxGroups];
  const int G = E + S;
  for (int g = threadIdx.x; g <= G; g += blockDim.x) {
    s_pp[g] = pad_prefix[g];
    s_off[g] = offsets[g];
    if (g < G) s_cnt[g] = counts[g];
  }
  __syncthreads();
  const int P = s_pp[G];
  const int lane = threadIdx.x & 31;
  const int nvec = H >> 3;
  const int64_t kg = f8::sf_stride(H, MX);
  const unsigned half = (lane & 16) ? 0xffff0000u : 0x0000ffffu;
  constexpr int piece_lanes = MX ? 4 : 16;         // lanes per scale piece
  const int warps = gridDim.x * (blockDim.x >> 5);
  for (int v = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); v < T + P; v += warps) {
    if (v < T) {
      const int t = v;
      int myrow = (lane < k) ? row_of[(size_t)t * k + lane] : -1;
      if (lane >= k && lane < k + S) myrow = s_off[E + lane - k] + t;
      const int nr = k + S;
      int rows[kMaxK + 4];
#pragma unroll
      for (int j = 0; j < kMaxK + 4; ++j) rows[j] = __shfl_sync(0xffffffffu, myrow, j);
      const __nv_bfloat16* src = x + (size_t)t * H;
      for (int c0 = lane; c0 < nvec; c0 += 32 * 4) {
        uint4 q[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (c0 + 32 * u < nvec) q[u] = ldg_nc_v4(src + (size_t)(c0 + 32 * u) * 8);
        // 1-byte form: a half-warp holds one 128-element slice per u, four
        // lanes one 32-element piece (nvec is a multiple of 16, so a half-warp
        // is wholly in range or out)
        uint2 qb[4];
        uint32_t code[4];
        if (xq) {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            if (c0 + 32 * u >= nvec) continue;
            float f[8];
            unpack8(q[u], f);
            float m = amax8(f);
#pragma unroll
            for (int o = piece_lanes / 2; o > 0; o >>= 1)
              m = fmaxf(m, __shfl_xor_sync(half, m, o));
            code[u] = ue8m0_code(m);
            qb[u] = e4m3x8(f, ue8m0_inv(code[u]));
          }
        }
#pragma unroll
        for (int j = 0; j < kMaxK + 4; ++j) {
          if (j >= nr || rows[j] < 0) continue;
          __nv_bfloat16* dst = x_perm + (size_t)stash_row(pages, rows[j]) * H;
#pragma unroll
          for (int u = 0; u < 4; ++u)
            if (c0 + 32 * u < nvec) stg_v4(dst + (size_t)(c0 + 32 * u) * 8, q[u]);
          if (xq) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int c = c0 + 32 * u;
              if (c >= nvec) continue;
              *reinterpret_cast<uint2*>(xq + (size_t)rows[j] * H + (size_t)c * 8) = qb[u];
              if ((lane & (piece_lanes - 1)) == 0)
                xsf[f8::row_sf_index(rows[j], c, kg, MX)] = (uint8_t)code[u];
            }
          }
        }
      }
    } else {
      const int p = v - T;
      const int g = find_group(s_pp, G, p);
      const int r = s_off[g] + s_cnt[g] + (p - s_pp[g]);
      __nv_bfloat16* dst = x_perm + (size_t)stash_row(pages, r) * H;
      const uint4 z = make_uint4(0u, 0u, 0u, 0u);
      for (int c0 = lane; c0 < nvec; c0 += 32) {
        stg_v4(dst + (size_t)c0 * 8, z);
        if (xq) {
          *reinterpret_cast<uint2*>(xq + (size_t)r * H + (size_t)c0 * 8) = make_uint2(0u, 0u);
          if ((c0 & (piece_lanes - 1)) == 0) xsf[f8::row_sf_index(r, c0, kg, MX)] = 127u;
        }
      }
    }
  }
}

cudaError_t launch_permute(const moe_config& c, const void* x, const int32_t* idx,
                           int32_t* counts, int32_t* offsets, int32_t* row_of, int32_t* token_of,
                           int32_t* sel_offsets, int32_t* sel_tokens, void* x_perm,
                           uint8_t* scratch, cudaStream_t s, const Fp8Scratch* fp8,
                           const StashAlloc* alloc) {
  int32_t* status = reinterpret_cast<int32_t*>(scratch + kScratchStatus);
  int32_t* pad_prefix = reinterpret_cast<int32_t*>(scratch + kScratchPadPrefix);
  int32_t* hist = reinterpret_cast<int32_t*>(scratch + kScratchHist);
  const int nc = n_chunks(c);
  cudaError_t err;
  if (nc > 0) {
    permute_hist_kernel<<<nc, 256, 0, s>>>(idx, hist, c.T, c.k, c.E, status);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }
  permute_rank_kernel<<<nc > 0 ? nc : 1, 256, 0, s>>>(idx, hist, nc, c.T, c.k, c.E, c.n_shared, c.row_align,
                                         (int)capacity_rows(c), counts, offsets, row_of,
                                         token_of, sel_offsets, sel_tokens, pad_prefix);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const int32_t* pages = nullptr;
  if (alloc) {
    stash_alloc_kernel<<<1, 256, 0, s>>>(counts, offsets, c.E + c.n_shared,
                                         (int)(rows_max(c) / 128), alloc->pool_pages, alloc->top,
                                         alloc->table, status);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    pages = alloc->table;
  }
  uint8_t* xq = nullptr;
  uint8_t* xsf = nullptr;
  if (c.dtype != MOE_DTYPE_BF16 && fp8) {
    xq = fp8->xq;
    xsf = fp8->xsf;
  }
  // (the MX pieces of x_perm's 1-byte form are 32 elements, the block recipe's 128)
  auto kern = (c.dtype == MOE_DTYPE_MXFP8 && xq) ? permute_scatter_kernel<true>
                                                 : permute_scatter_kernel<false>;
  kern<<<num_sms() * 8, 256, 0, s>>>(
      static_cast<const __nv_bfloat16*>(x), row_of, counts, offsets, pad_prefix,
      static_cast<__nv_bfloat16*>(x_perm), c.T, c.H, c.k, c.E, c.n_shared, xq, xsf, pages);
  return cudaGetLastError();
}

cudaError_t launch_stash_release(const moe_config& c, const int32_t* table, int32_t* top,
                                 cudaStream_t s) {
  stash_release_kernel<<<1, 32, 0, s>>>(table, (int)(rows_max(c) / 128), top);
  return cudaGetLastError();
}

}  // namespace moe

// ------------------------------------------------------------------------------
// Dispatch without a caller-provided scratch buffer.
//
// Some callers cannot hand this library a scratch allocation: code that runs
// inside a host framework which owns every byte of device memory (a caching
// allocator or plugin host with no way to request an extra workspace), or
// code on a path where calling cudaMalloc is not allowed. For them
// moe_permute_noalloc keeps its scratch -- the per-chunk expert histograms,
// the padding prefix and the status word -- in one file-scope device array of
// fixed size, which every GPU that loads this library holds until the process
// exits. It allocates nothing.
namespace moe {
namespace {

constexpr size_t kNoAllocScratchBytes = 512 * 1024;
static __device__ __align__(256) uint8_t g_permute_scratch[kNoAllocScratchBytes];

// Device address of g_permute_scratch in the current context, looked up on
// every call (cheap): a cached address would go stale after cudaDeviceReset or
// under another context on the same device.
cudaError_t noalloc_scratch(uint8_t** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_permute_scratch);
  if (e != cudaSuccess) return e;
  *out = static_cast<uint8_t*>(p);
  return cudaSuccess;
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_permute_noalloc(const moe_config* cfg, const void* x,
                                          const int32_t* idx, int32_t* counts, int32_t* offsets,
                                          int32_t* row_of, int32_t* token_of,
                                          int32_t* sel_offsets, int32_t* sel_tokens,
                                          void* x_perm, void* stream) {
  using namespace moe;
  const moe_status st = check_config(cfg);
  if (st != MOE_OK) return st;
  // an FP8 dispatch also writes x_perm's E4M3 form into the caller's scratch,
  // which this entry point does not take
  if (cfg->dtype != MOE_DTYPE_BF16) return MOE_ERR_UNSUPPORTED;
  auto a16 = [](const void* p) { return p && ((uintptr_t)p & 15u) == 0; };
  auto a4 = [](const void* p) { return p && ((uintptr_t)p & 3u) == 0; };
  const bool empty = cfg->T == 0;
  if (!((empty && !x) || a16(x)) || !((empty && !idx) || a4(idx)) || !a4(counts) ||
      !a4(offsets) || !((empty && !row_of) || a4(row_of)) || !a4(token_of) ||
      !a4(sel_offsets) || !((empty && !sel_tokens) || a4(sel_tokens)) || !a16(x_perm))
    return MOE_ERR_INVALID_ARG;
  if ((size_t)permute_scratch_bytes(*cfg) > kNoAllocScratchBytes) return MOE_ERR_WORKSPACE;
  uint8_t* sc = nullptr;
  if (noalloc_scratch(&sc) != cudaSuccess) return MOE_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
  // the status word is the only part that must start at zero; the histograms
  // and the padding prefix are fully rewritten by every call
  if (cudaMemsetAsync(sc + kScratchStatus, 0, sizeof(int32_t), s) != cudaSuccess)
    return MOE_ERR_CUDA;
  const cudaError_t e = launch_permute(*cfg, x, idx, counts, offsets, row_of, token_of,
                                       sel_offsets, sel_tokens, x_perm, sc, s, nullptr);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// Reads back what the last moe_permute_noalloc call recorded in its status
// word (an index out of range or repeated): synchronises `stream`, then copies
// the word from the library's array on the current device.
extern "C" moe_status moe_permute_noalloc_status(int32_t* code, void* stream) {
  using namespace moe;
  if (!code) return MOE_ERR_INVALID_ARG;
  uint8_t* sc = nullptr;
  if (noalloc_scratch(&sc) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemcpy(code, sc + kScratchStatus, sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
