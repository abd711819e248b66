// Stage 4 of the MoE layer (combine, done locally), its backward, the backward
// of stage 2 (dispatch) and of the router.
//
// Follows the combine stage of "Scalable Training of Mixture-of-Experts Models
// with Megatron Core" (es summary, Resumen técnico §2.1 step 4: results return
// to their tokens and are weighted by the router). Every kernel here is
// bandwidth-bound: one warp per token, 16-byte vector accesses, fp32
// accumulation in a fixed order.
#include "common.cuh"
#include "fp8_layout.cuh"
#include "internal.h"

namespace moe {

// Loads the k rows/weights of token t into lane-indexed registers and appends
// the shared experts' rows (weight 1).
__device__ __forceinline__ void token_rows(const int32_t* row_of, const float* w,
                                           const int32_t* offsets, int t, int k, int E, int S,
                                           int lane, int& row, float& wt) {
  row = -1;
  wt = 0.f;
  if (lane < k) {
    row = row_of[(size_t)t * k + lane];
    wt = w ? w[(size_t)t * k + lane] : 1.f;
  } else if (lane < k + S) {
    row = offsets[E + lane - k] + t;
    wt = 1.f;
  }
}

// Row indices and weights of token t, slot j (j >= k: shared experts, weight 1).
__device__ __forceinline__ void slot_row(const int32_t* row_of, const float* w,
                                         const int32_t* offsets, int t, int j, int k, int E,
                                         int& r, float& wt) {
  if (j < k) {
    r = row_of[(size_t)t * k + j];
    wt = w ? w[(size_t)t * k + j] : 1.f;
  } else {
    r = offsets[E + j - k] + t;
    wt = 1.f;
  }
}

// Gather-reduce, one warp per token (grid-stride):
//   unpermute     out[t] = bf16( sum_j w_tj y[row_tj] + sum_s y[shared row s] )
//   permute bwd   dx[t]  = bf16( sum_j dX[row_tj] + sum_s dX[shared row s]
//                                + sum_{j dropped} dl_tj W_r[e_tj] )          (ROUTER)
// (the FC1 data-gradient GEMM has already added dl_tj W_r[e_tj] to the row of
// every kept assignment; only capacity-dropped assignments have no row, and
// without a capacity limit the permute backward is a plain gather with unit
// weights)
// Lanes j < k+S fetch the token's rows (and weights, experts and dlogits) once;
// then each lane walks its 16-byte slices U at a time with the U * (k+S) row
// loads of a step in flight together, summing in slot order (fp32, fixed
// order). The permuted rows are read once (L2 evict-first); the W_r rows are
// read by every token (L2 evict-last).
template <int MAXR, int U, bool ROUTER>
__global__ void __launch_bounds__(256, (MAXR > 4) ? 2 : 3)
gather_reduce_kernel(const __nv_bfloat16* __restrict__ src, const int32_t* __restrict__ row_of,
                     const float* __restrict__ w, const int32_t* __restrict__ offsets,
                     const int32_t* __restrict__ idx, const float* __restrict__ dlogits,
                     const float* __restrict__ W_r, __nv_bfloat16* __restrict__ out, int T,
                     int H, int k, int E, int S, const int32_t* __restrict__ pages) {
  const int lane = threadIdx.x & 31;
  const int nvec = H >> 3, nr = k + S;
  const int warps = gridDim.x * (blockDim.x >> 5);
  const uint64_t stream_pol = l2_evict_first_policy();
  const uint64_t keep_pol = ROUTER ? l2_evict_last_policy() : 0ull;
  for (int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < T; t += warps) {
    int myrow = -1, mye = -1;
    float mywt = 0.f, mydl = 0.f;
    if (lane < nr) {
      slot_row(row_of, w, offsets, t, lane, k, E, myrow, mywt);
      if (myrow >= 0) myrow = stash_row(pages, myrow);
    }
    if (ROUTER && lane < k) {
      mye = idx[(size_t)t * k + lane];
      if ((unsigned)mye < (unsigned)E) mydl = dlogits[(size_t)t * E + mye];
      else mye = -1;
    }
    // (router terms exist for the k routed slots only, k <= kMaxK)
    constexpr int RK = MAXR < kMaxK ? MAXR : kMaxK;
    int rows[MAXR], es[RK];
    float wts[MAXR], dls[RK];
#pragma unroll
    for (int j = 0; j < MAXR; ++j) {
      rows[j] = __shfl_sync(0xffffffffu, myrow, j);
      wts[j] = __shfl_sync(0xffffffffu, mywt, j);
      if (ROUTER && j < RK) {
        es[j] = __shfl_sync(0xffffffffu, mye, j);
        dls[j] = __shfl_sync(0xffffffffu, mydl, j);
      }
    }
    for (int c0 = lane; c0 < nvec; c0 += 32 * U) {
      uint4 q[U][MAXR];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = c0 + 32 * u;
#pragma unroll
        for (int j = 0; j < MAXR; ++j)
          if (j < nr && rows[j] >= 0 && c < nvec)
            q[u][j] = ldg_nc_v4_pol(src + (size_t)rows[j] * H + (size_t)c * 8, stream_pol);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = c0 + 32 * u;
        if (c >= nvec) continue;
        float acc[8];
#pragma unroll
        for (int m = 0; m < 8; ++m) acc[m] = 0.f;
#pragma unroll
        for (int j = 0; j < MAXR; ++j) {
          if (j >= nr || rows[j] < 0) continue;
          float f[8];
          unpack8(q[u][j], f);
          if (ROUTER) {
#pragma unroll
            for (int m = 0; m < 8; ++m) acc[m] += f[m];
          } else {
#pragma unroll
            for (int m = 0; m < 8; ++m) acc[m] = fmaf(wts[j], f[m], acc[m]);
          }
        }
        if (ROUTER) {
#pragma unroll
          for (int j = 0; j < RK; ++j) {
            if (j >= k || es[j] < 0 || rows[j] >= 0) continue;
            const float d = dls[j];
            const float* wr = W_r + (size_t)es[j] * H + (size_t)c * 8;
            const float4 a = ldg_nc_f4_pol(wr, keep_pol), b = ldg_nc_f4_pol(wr + 4, keep_pol);
            acc[0] = fmaf(d, a.x, acc[0]);
            acc[1] = fmaf(d, a.y, acc[1]);
            acc[2] = fmaf(d, a.z, acc[2]);
            acc[3] = fmaf(d, a.w, acc[3]);
            acc[4] = fmaf(d, b.x, acc[4]);
            acc[5] = fmaf(d, b.y, acc[5]);
            acc[6] = fmaf(d, b.z, acc[6]);
            acc[7] = fmaf(d, b.w, acc[7]);
          }
        }
        stg_v4(out + (size_t)t * H + (size_t)c * 8, pack8(acc));
      }
    }
  }
}

__device__ __forceinline__ int find_pad_group(const int* prefix, int G, int p) {
  int lo = 0, hi = G - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= p) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// dO[row_tj] = bf16(w_tj dY[t]); dw_tj = <dY[t], y[row_tj]>; shared rows get dY.
// One warp per token (grid-stride over tokens, then over the zero padding rows
// of dO). Lanes j < k+S fetch the token's rows and weights once; then each
// lane walks its 16-byte slices U at a time, keeping the U dY slices and the
// U*k y slices of one step in flight together. Every lane sums its slices in
// order and the warp combines lanes by a fixed butterfly, so dw is
// deterministic. No block-wide synchronisation on the token path.
// COPY (the layer with the routing weight inside the expert): dO[row_tj] =
// dY[t] unweighted, y is not read and dw is not written (it comes from the FC2
// data gradient there). With dOq (the FP8 configurations) every row written is
// also written in its 1-byte form -- E4M3 codes of the bf16 values' 1 x 128
// slices (MXFP8: 1 x 32) with their UE8M0 scales in dOsf's atoms -- for the
// FC2 data gradient.
template <int MAXR, int U, bool COPY = false, bool MX = false>
__global__ void __launch_bounds__(256, (MAXR <= 2) ? 3 : 2)
unpermute_bwd_kernel(const __nv_bfloat16* __restrict__ dY, const __nv_bfloat16* __restrict__ y,
                     const int32_t* __restrict__ row_of, const float* __restrict__ w,
                     const int32_t* __restrict__ counts, const int32_t* __restrict__ offsets,
                     __nv_bfloat16* __restrict__ dO, float* __restrict__ dw, int T, int H, int k,
                     int E, int S, uint8_t* __restrict__ dOq, uint8_t* __restrict__ dOsf,
                     const int32_t* __restrict__ pages) {
  __shared__ int s_pp[kMaxGroups + 1];
  __shared__ int s_off[kMaxGroups + 1];
  __shared__ int s_cnt[kMaxGroups];
  __shared__ int s_tmp[33];
  const int G = E + S;
  for (int g = threadIdx.x; g <= G; g += blockDim.x) s_off[g] = offsets[g];
  for (int g = threadIdx.x; g < G; g += blockDim.x) s_cnt[g] = counts[g];
  __syncthreads();
  // padding rows to zero: the rest of each segment's last 128-row block (the
  // rows a GEMM reads; rows past it are never read)
  for (int g = threadIdx.x; g < G; g += blockDim.x)
    s_pp[g] = min(s_off[g + 1] - s_off[g], (s_cnt[g] + 127) / 128 * 128) - s_cnt[g];
  __syncthreads();
  const int P = block_exclusive_scan(s_pp, G, s_tmp);
  if (threadIdx.x == 0) s_pp[G] = P;
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int nvec = H >> 3, nr = k + S;
  const int warps = gridDim.x * (blockDim.x >> 5);
  const int64_t kg = f8::sf_stride(H, MX);
  const unsigned half = (lane & 16) ? 0xffff0000u : 0x0000ffffu;
  constexpr int piece_lanes = MX ? 4 : 16;         // lanes per scale piece
  for (int v = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); v < T + P; v += warps) {
    if (v >= T) {
      const int p = v - T;
      const int g = find_pad_group(s_pp, G, p);
      const int r = s_off[g] + s_cnt[g] + (p - s_pp[g]);
      const uint4 z = make_uint4(0u, 0u, 0u, 0u);
      for (int c = lane; c < nvec; c += 32) {
        stg_v4(dO + (size_t)r * H + (size_t)c * 8, z);
        if (dOq) {
          *reinterpret_cast<uint2*>(dOq + (size_t)r * H + (size_t)c * 8) = make_uint2(0u, 0u);
          if ((c & (piece_lanes - 1)) == 0) dOsf[f8::row_sf_index(r, c, kg, MX)] = 127u;
        }
      }
      continue;
    }
    const int t = v;
    int myrow = -1;
    float mywt = 0.f;
    if (lane < k) {
      myrow = row_of[(size_t)t * k + lane];
      mywt = COPY ? 1.f : w[(size_t)t * k + lane];    // the copy has no weights (w NULL)
    } else if (lane < nr) {
      myrow = s_off[E + lane - k] + t;
    }
    int rows[MAXR];
    float wts[MAXR], dot[MAXR];
#pragma unroll
    for (int j = 0; j < MAXR; ++j) {
      rows[j] = __shfl_sync(0xffffffffu, myrow, j);
      wts[j] = __shfl_sync(0xffffffffu, mywt, j);
      dot[j] = 0.f;
    }
    const __nv_bfloat16* gsrc = dY + (size_t)t * H;
    for (int c0 = lane; c0 < nvec; c0 += 32 * U) {
      uint4 gq[U], yq[U][MAXR];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = c0 + 32 * u;
        if (c >= nvec) continue;
        gq[u] = ldg_nc_v4(gsrc + (size_t)c * 8);
#pragma unroll
        for (int j = 0; j < MAXR; ++j)
          if (!COPY && j < k && rows[j] >= 0)     // y_perm may live in stash pages, dO_perm not
            yq[u][j] = ldg_nc_v4(y + (size_t)stash_row(pages, rows[j]) * H + (size_t)c * 8);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = c0 + 32 * u;
        if (c >= nvec) continue;
        float g[8];
        unpack8(gq[u], g);
#pragma unroll
        for (int j = 0; j < MAXR; ++j) {
          if (j >= nr || rows[j] < 0) continue;
          __nv_bfloat16* dst = dO + (size_t)rows[j] * H + (size_t)c * 8;
          uint4 ov;
          if (COPY || j >= k) {
            ov = gq[u];
          } else {
            float f[8], o[8];
            unpack8(yq[u][j], f);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              dot[j] = fmaf(g[i], f[i], dot[j]);
              o[i] = wts[j] * g[i];
            }
            ov = pack8(o);
          }
          stg_v4(dst, ov);
          if (dOq) {
            // a half-warp holds one 128-element slice, four lanes a 32-element
            // piece (nvec % 32 == 0 in this mode)
            float fq[8];
            unpack8(ov, fq);
            float m = amax8(fq);
#pragma unroll
            for (int o = piece_lanes / 2; o > 0; o >>= 1)
              m = fmaxf(m, __shfl_xor_sync(half, m, o));
            const uint32_t code = ue8m0_code(m);
            *reinterpret_cast<uint2*>(dOq + (size_t)rows[j] * H + (size_t)c * 8) =
                e4m3x8(fq, ue8m0_inv(code));
            if ((lane & (piece_lanes - 1)) == 0)
              dOsf[f8::row_sf_index(rows[j], c, kg, MX)] = (uint8_t)code;
          }
        }
      }
    }
    if (COPY) continue;
    float mine = 0.f;
#pragma unroll
    for (int j = 0; j < MAXR; ++j) {
      if (j >= k) break;
      const float sj = warp_sum(dot[j]);
      if (lane == j) mine = (rows[j] >= 0) ? sj : 0.f;
    }
    if (lane < k) dw[(size_t)t * k + lane] = mine;
  }
}

// Routing weight of every used row of the permuted buffer, for the layer with
// the weight inside the expert: w[t, j] for the row of assignment (t, j), 1 for
// a shared expert's row, 0 for padding. One thread per row.
__global__ void __launch_bounds__(256)
row_weights_kernel(const int32_t* __restrict__ token_of, const int32_t* __restrict__ row_of,
                   const float* __restrict__ w, const int32_t* __restrict__ offsets,
                   float* __restrict__ row_w, int k, int E, int S) {
  const int used = offsets[E + S];
  const int routed_end = offsets[E];
  for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < used; r += gridDim.x * blockDim.x) {
    const int t = token_of[r];
    float v = 0.f;
    if (t >= 0) {
      if (r >= routed_end) {
        v = 1.f;
      } else {
        for (int j = 0; j < k; ++j)
          if (row_of[(size_t)t * k + j] == r) {
            v = w[(size_t)t * k + j];
            break;
          }
      }
    }
    row_w[r] = v;
  }
}

// dw[t, j] = sum over the FC2 data gradient's n-tiles (in order) of the partial
// <dh_s, h> of the row of assignment (t, j); 0 for a dropped assignment.
__global__ void __launch_bounds__(256)
dw_reduce_kernel(const float* __restrict__ part, int nt, const int32_t* __restrict__ row_of,
                 float* __restrict__ dw, int n) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    const int r = row_of[i];
    float acc = 0.f;
    if (r >= 0)
      for (int q = 0; q < nt; ++q) acc += part[(size_t)r * nt + q];
    dw[i] = acc;
  }
}

// dlogits[t,:] = 0 except the selected experts:
//   softmax: dl_j = w_j (dw_j - sum_i w_i dw_i)
//   sigmoid: ds_j = (r/S)(dw_j - sum_i (s_i/S) dw_i), dl_j = ds_j s_j (1 - s_j)
__global__ void __launch_bounds__(256)
route_bwd_kernel(const float* __restrict__ logits, const int32_t* __restrict__ idx,
                 const float* __restrict__ w, const float* __restrict__ dw,
                 float* __restrict__ dlogits, int T, int E, int k, int score_fn,
                 float route_scale) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  float* row = dlogits + (size_t)t * E;
  for (int e = lane; e < E; e += 32) row[e] = 0.f;
  __syncwarp();
  int e = 0;
  float wj = 0.f, dwj = 0.f, sj = 0.f;
  if (lane < k) {
    e = idx[(size_t)t * k + lane];
    wj = w[(size_t)t * k + lane];
    dwj = dw[(size_t)t * k + lane];
    if ((unsigned)e < (unsigned)E) sj = __fdiv_rn(1.f, 1.f + expf(-logits[(size_t)t * E + e]));
  }
  // fp32 throughout (at most 8 terms, relative error ~1e-6); fp64 arithmetic
  // is slow on this GPU
  float v;
  if (score_fn == MOE_SCORE_SOFTMAX) {
    const float inner = warp_sum(wj * dwj);
    v = wj * (dwj - inner);
  } else {
    const float ssum = warp_sum(sj);
    const float sdw = warp_sum(sj * dwj);
    const float ds = (route_scale / ssum) * (dwj - sdw / ssum);
    v = ds * sj * (1.f - sj);
  }
  if (lane < k && (unsigned)e < (unsigned)E) row[e] = v;
}

// dW_r[e, cols] = sum over the tokens that selected e of dlogits[t,e] x[t, cols]
// (sel_offsets == NULL: over all T tokens; accumulate: added to dW_r).
// Block (e, slab of 32*CPL columns); lane owns CPL columns. The expert's
// selecting tokens are taken in chunks of 8 (chunk i by warp i mod 16): lanes
// 0..7 load the chunk's token ids and dlogits, then the warp walks the chunk in
// token order with 4 x rows in flight. Warp partial sums are combined in warp
// order, so the summation order is fixed (deterministic).
template <int CPL>
__global__ void __launch_bounds__(512, 2)
router_wgrad_kernel(const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ sel_offsets,
                    const int32_t* __restrict__ sel_tokens, const float* __restrict__ dlogits,
                    float* __restrict__ dW_r, int H, int E, int T, int accumulate) {
  constexpr int NW = 16, CH = 8, U = 4, SLAB = 32 * CPL;
  __shared__ float part[NW][SLAB];
  const int e = blockIdx.x;
  const int col0 = blockIdx.y * SLAB;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int c = col0 + lane * CPL;
  const bool on = c < H;
  const int beg = sel_offsets ? sel_offsets[e] : 0, end = sel_offsets ? sel_offsets[e + 1] : T;
  float acc[CPL];
#pragma unroll
  for (int i = 0; i < CPL; ++i) acc[i] = 0.f;
  for (int base = beg + CH * wid; base < end; base += CH * NW) {
    const int n = min(CH, end - base);
    int my_t = 0;
    float my_d = 0.f;
    if (lane < n) {
      my_t = sel_tokens ? sel_tokens[base + lane] : base + lane;
      my_d = dlogits[(size_t)my_t * E + e];
    }
#pragma unroll
    for (int u0 = 0; u0 < CH; u0 += U) {
      uint4 q[U];
      float d[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int t = __shfl_sync(0xffffffffu, my_t, u0 + u);
        d[u] = __shfl_sync(0xffffffffu, my_d, u0 + u);
        if (on && u0 + u < n) {
          if (CPL == 8) {
            q[u] = ldg_nc_v4(x + (size_t)t * H + c);
          } else {
            const uint2 h2 = __ldg(reinterpret_cast<const uint2*>(x + (size_t)t * H + c));
            q[u] = make_uint4(h2.x, h2.y, 0u, 0u);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (!on || u0 + u >= n) continue;
        float f[8];
        unpack8(q[u], f);
#pragma unroll
        for (int m = 0; m < CPL; ++m) acc[m] = fmaf(d[u], f[m], acc[m]);
      }
    }
  }
#pragma unroll
  for (int m = 0; m < CPL; ++m) part[wid][lane * CPL + m] = acc[m];
  __syncthreads();
  for (int i = threadIdx.x; i < SLAB; i += blockDim.x) {
    const int col = col0 + i;
    if (col < H) {
      float s = 0.f;
#pragma unroll
      for (int q2 = 0; q2 < NW; ++q2) s += part[q2][i];
      dW_r[(size_t)e * H + col] = accumulate ? dW_r[(size_t)e * H + col] + s : s;
    }
  }
}

static int grid_for_warps(int n_items) {
  const int blocks = (n_items + 7) / 8;
  const int cap = num_sms() * 16;
  return blocks < cap ? (blocks > 0 ? blocks : 1) : cap;
}

template <bool ROUTER>
static cudaError_t launch_gather_reduce(const moe_config& c, const void* src,
                                        const int32_t* row_of, const float* w,
                                        const int32_t* offsets, const int32_t* idx,
                                        const float* dlogits, const float* W_r, void* out,
                                        cudaStream_t s, const int32_t* pages = nullptr) {
  auto sp = static_cast<const __nv_bfloat16*>(src);
  auto o = static_cast<__nv_bfloat16*>(out);
  const int nr = c.k + c.n_shared;
  const int grid = grid_for_warps(c.T);
  if (nr <= 2)
    gather_reduce_kernel<2, 4, ROUTER><<<grid, 256, 0, s>>>(sp, row_of, w, offsets, idx, dlogits,
                                                           W_r, o, c.T, c.H, c.k, c.E,
                                                           c.n_shared, pages);
  else if (nr <= 4)
    gather_reduce_kernel<4, 2, ROUTER><<<grid, 256, 0, s>>>(sp, row_of, w, offsets, idx, dlogits,
                                                           W_r, o, c.T, c.H, c.k, c.E,
                                                           c.n_shared, pages);
  else if (nr <= 8)    // top-8 without shared experts: a third fewer registers than 12
    gather_reduce_kernel<8, 1, ROUTER><<<grid, 256, 0, s>>>(sp, row_of, w, offsets, idx, dlogits,
                                                           W_r, o, c.T, c.H, c.k, c.E,
                                                           c.n_shared, pages);
  else
    gather_reduce_kernel<kMaxK + 4, 1, ROUTER><<<grid, 256, 0, s>>>(
        sp, row_of, w, offsets, idx, dlogits, W_r, o, c.T, c.H, c.k, c.E, c.n_shared, pages);
  return cudaGetLastError();
}

cudaError_t launch_unpermute(const moe_config& c, const void* y_perm, const int32_t* row_of,
                             const float* w, const int32_t* offsets, void* out, cudaStream_t s,
                             const int32_t* pages) {
  return launch_gather_reduce<false>(c, y_perm, row_of, w, offsets, nullptr, nullptr, nullptr, out,
                                     s, pages);
}

template <bool MX>
static void unpermute_bwd_launch(const moe_config& c, const __nv_bfloat16* dYp,
                                 const __nv_bfloat16* yp, const int32_t* row_of, const float* w,
                                 const int32_t* counts, const int32_t* offsets,
                                 __nv_bfloat16* dOp, float* dw, cudaStream_t s, uint8_t* dOq,
                                 uint8_t* dOsf, const int32_t* pages) {
  // one warp per token (8 per block), capped at 16 blocks per SM
  const int grid = grid_for_warps(c.T);
  const int nr = c.k + c.n_shared;
  if (nr <= 2)
    unpermute_bwd_kernel<2, 4, false, MX><<<grid, 256, 0, s>>>(
        dYp, yp, row_of, w, counts, offsets, dOp, dw, c.T, c.H, c.k, c.E, c.n_shared, dOq, dOsf,
        pages);
  else if (nr <= 4)
    unpermute_bwd_kernel<4, 4, false, MX><<<grid, 256, 0, s>>>(
        dYp, yp, row_of, w, counts, offsets, dOp, dw, c.T, c.H, c.k, c.E, c.n_shared, dOq, dOsf,
        pages);
  else if (nr <= 8)
    unpermute_bwd_kernel<8, 1, false, MX><<<grid, 256, 0, s>>>(
        dYp, yp, row_of, w, counts, offsets, dOp, dw, c.T, c.H, c.k, c.E, c.n_shared, dOq, dOsf,
        pages);
  else
    unpermute_bwd_kernel<kMaxK + 4, 1, false, MX><<<grid, 256, 0, s>>>(
        dYp, yp, row_of, w, counts, offsets, dOp, dw, c.T, c.H, c.k, c.E, c.n_shared, dOq, dOsf,
        pages);
}

cudaError_t launch_unpermute_bwd(const moe_config& c, const void* dY, const void* y_perm,
                                 const int32_t* row_of, const float* w, const int32_t* counts,
                                 const int32_t* offsets, void* dO_perm, float* dw,
                                 cudaStream_t s, uint8_t* dOq, uint8_t* dOsf,
                                 const int32_t* pages) {
  auto dYp = static_cast<const __nv_bfloat16*>(dY);
  auto yp = static_cast<const __nv_bfloat16*>(y_perm);
  auto dOp = static_cast<__nv_bfloat16*>(dO_perm);
  // (the MX pieces of dO's 1-byte form are 32 elements, the block recipe's 128)
  if (c.dtype == MOE_DTYPE_MXFP8 && dOq)
    unpermute_bwd_launch<true>(c, dYp, yp, row_of, w, counts, offsets, dOp, dw, s, dOq, dOsf,
                               pages);
  else
    unpermute_bwd_launch<false>(c, dYp, yp, row_of, w, counts, offsets, dOp, dw, s, dOq, dOsf,
                                pages);
  return cudaGetLastError();
}

cudaError_t launch_unpermute_bwd_copy(const moe_config& c, const void* dY, const int32_t* row_of,
                                      const int32_t* counts, const int32_t* offsets,
                                      void* dO_perm, cudaStream_t s) {
  auto dYp = static_cast<const __nv_bfloat16*>(dY);
  auto dOp = static_cast<__nv_bfloat16*>(dO_perm);
  const int grid = grid_for_warps(c.T);
  if (c.k + c.n_shared <= 2)
    unpermute_bwd_kernel<2, 4, true><<<grid, 256, 0, s>>>(dYp, nullptr, row_of, nullptr, counts,
                                                          offsets, dOp, nullptr, c.T, c.H, c.k,
                                                          c.E, c.n_shared, nullptr, nullptr,
                                                          nullptr);
  else if (c.k + c.n_shared <= 4)
    unpermute_bwd_kernel<4, 4, true><<<grid, 256, 0, s>>>(dYp, nullptr, row_of, nullptr, counts,
                                                          offsets, dOp, nullptr, c.T, c.H, c.k,
                                                          c.E, c.n_shared, nullptr, nullptr,
                                                          nullptr);
  else
    unpermute_bwd_kernel<kMaxK + 4, 1, true><<<grid, 256, 0, s>>>(
        dYp, nullptr, row_of, nullptr, counts, offsets, dOp, nullptr, c.T, c.H, c.k, c.E,
        c.n_shared, nullptr, nullptr, nullptr);
  return cudaGetLastError();
}

cudaError_t launch_row_weights(const moe_config& c, const int32_t* token_of,
                               const int32_t* row_of, const float* w, const int32_t* offsets,
                               float* row_w, cudaStream_t s) {
  const int64_t R = rows_max(c);
  long long blocks = (R + 255) / 256;
  if (blocks > (long long)num_sms() * 8) blocks = (long long)num_sms() * 8;
  row_weights_kernel<<<blocks > 0 ? (int)blocks : 1, 256, 0, s>>>(token_of, row_of, w, offsets,
                                                                  row_w, c.k, c.E, c.n_shared);
  return cudaGetLastError();
}

cudaError_t launch_dw_reduce(const moe_config& c, const float* dw_part, const int32_t* row_of,
                             float* dw, cudaStream_t s) {
  const int n = c.T * c.k;
  long long blocks = (n + 255) / 256;
  if (blocks > (long long)num_sms() * 8) blocks = (long long)num_sms() * 8;
  dw_reduce_kernel<<<blocks > 0 ? (int)blocks : 1, 256, 0, s>>>(dw_part, dw_tiles(c), row_of, dw,
                                                                 n);
  return cudaGetLastError();
}

cudaError_t launch_route_bwd(const moe_config& c, const float* logits, const int32_t* idx,
                             const float* w, const float* dw, float* dlogits, cudaStream_t s) {
  route_bwd_kernel<<<(c.T + 7) / 8, 256, 0, s>>>(logits, idx, w, dw, dlogits, c.T, c.E, c.k,
                                                 c.score_fn, c.route_scale);
  return cudaGetLastError();
}

cudaError_t launch_permute_bwd(const moe_config& c, const void* dX_perm, const int32_t* row_of,
                               const int32_t* offsets, const int32_t* idx, const float* dlogits,
                               const float* W_r, void* dx, cudaStream_t s) {
  if (!(c.capacity_factor > 0.f))   // no assignment is dropped
    return launch_gather_reduce<false>(c, dX_perm, row_of, nullptr, offsets, nullptr, nullptr,
                                       nullptr, dx, s);
  return launch_gather_reduce<true>(c, dX_perm, row_of, nullptr, offsets, idx, dlogits, W_r, dx,
                                    s);
}

// dlogits [T, E] -> its three bf16 parts stacked along rows, D3 [3 * Tp, E]
// (part q at rows q * Tp; rows T..Tp-1 of every part zero). 8 columns per
// thread (E % 128 == 0).
__global__ void __launch_bounds__(256)
split_dlogits_kernel(const float* __restrict__ dl, __nv_bfloat16* __restrict__ D3, int T,
                     long long Tp, int E) {
  const int per_row = E >> 3;
  const long long n = Tp * per_row;
  for (long long v = (long long)blockIdx.x * blockDim.x + threadIdx.x; v < n;
       v += (long long)gridDim.x * blockDim.x) {
    const long long t = v / per_row;
    const int e = (int)(v - t * per_row) << 3;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
    if (t < T) {
      const float4* src = reinterpret_cast<const float4*>(dl + t * E + e);
      a = __ldg(src);
      b = __ldg(src + 1);
    }
    uint4 hi, mid, lo;
    split3_pair(a.x, a.y, hi.x, mid.x, lo.x);
    split3_pair(a.z, a.w, hi.y, mid.y, lo.y);
    split3_pair(b.x, b.y, hi.z, mid.z, lo.z);
    split3_pair(b.z, b.w, hi.w, mid.w, lo.w);
    __nv_bfloat16* dst = D3 + t * E + e;
    *reinterpret_cast<uint4*>(dst) = hi;
    *reinterpret_cast<uint4*>(dst + Tp * E) = mid;
    *reinterpret_cast<uint4*>(dst + 2 * Tp * E) = lo;
  }
}

// dW_r[e, h] = sum over chunks g in order of P[g * H + h, e] (fp32), through a
// 32 x 32 shared-memory transpose: both the reads (16 bytes along e) and the
// writes (along h) are coalesced. Thread (row r, quad j) sums P[g][h0 + r][e0 +
// 4j .. 4j+3] over g with four chunks' loads in flight.
__global__ void __launch_bounds__(256)
sum_chunks_transpose_kernel(const float* __restrict__ P, float* __restrict__ dW_r, int NG, int H,
                            int E, int accumulate) {
  __shared__ float tile[32][33];
  const int j = threadIdx.x & 7, r = threadIdx.x >> 3;
  const int h0 = blockIdx.x * 32, e0 = blockIdx.y * 32;
  const float* src = P + (size_t)(h0 + r) * E + e0 + 4 * j;
  const size_t gstride = (size_t)H * E;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  int g = 0;
  for (; g + 4 <= NG; g += 4) {
    float4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = __ldg(reinterpret_cast<const float4*>(src + (g + u) * gstride));
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      acc.x += v[u].x;
      acc.y += v[u].y;
      acc.z += v[u].z;
      acc.w += v[u].w;
    }
  }
  for (; g < NG; ++g) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(src + g * gstride));
    acc.x += v.x;
    acc.y += v.y;
    acc.z += v.z;
    acc.w += v.w;
  }
  tile[r][4 * j] = acc.x;
  tile[r][4 * j + 1] = acc.y;
  tile[r][4 * j + 2] = acc.z;
  tile[r][4 * j + 3] = acc.w;
  __syncthreads();
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float* o = dW_r + (size_t)(e0 + ty + 8 * i) * H + h0 + tx;
    *o = accumulate ? *o + tile[tx][ty + 8 * i] : tile[tx][ty + 8 * i];
  }
}

cudaError_t launch_router_wgrad(const moe_config& c, const void* x, const int32_t* sel_offsets,
                                const int32_t* sel_tokens, const float* dlogits, float* dW_r,
                                uint8_t* scratch, cudaStream_t s, bool accumulate) {
  if (router_on_tensor_cores(c)) {
    // tensor cores: dW_r^T chunk sums x^T . dlogits over chunks of tokens, then
    // the chunks added in order (every x row read once)
    if (c.T == 0)
      return accumulate ? cudaSuccess : cudaMemsetAsync(dW_r, 0, (size_t)c.E * c.H * 4, s);
    uint8_t* base = scratch + router_split_offset(c);
    const long long Tp = ((long long)c.T + 63) / 64 * 64;
    auto D3 = reinterpret_cast<__nv_bfloat16*>(base);
    auto P = reinterpret_cast<float*>(base + router_wgrad_split_bytes(c));
    const int chunk = router_wgrad_chunk(c);
    const int NG = (c.T + chunk - 1) / chunk;
    long long blocks = (Tp * (c.E / 8) + 255) / 256;
    if (blocks > (long long)num_sms() * 16) blocks = (long long)num_sms() * 16;
    split_dlogits_kernel<<<(int)blocks, 256, 0, s>>>(dlogits, D3, c.T, Tp, c.E);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    err = launch_router_wgrad_tc(c, x, D3, Tp, P, chunk,
                                 reinterpret_cast<int32_t*>(scratch + kScratchStatus), s);
    if (err != cudaSuccess) return err;
    sum_chunks_transpose_kernel<<<dim3(c.H / 32, c.E / 32), 256, 0, s>>>(P, dW_r, NG, c.H, c.E,
                                                                         accumulate ? 1 : 0);
    return cudaGetLastError();
  }
  auto xb = static_cast<const __nv_bfloat16*>(x);
  // few experts: 128-column slabs so that every SM gets blocks
  if ((long long)c.E * ((c.H + 255) / 256) < 2LL * num_sms()) {
    dim3 grid(c.E, (c.H + 127) / 128);
    router_wgrad_kernel<4><<<grid, 512, 0, s>>>(xb, sel_offsets, sel_tokens, dlogits, dW_r, c.H,
                                                c.E, c.T, accumulate ? 1 : 0);
  } else {
    dim3 grid(c.E, (c.H + 255) / 256);
    router_wgrad_kernel<8><<<grid, 512, 0, s>>>(xb, sel_offsets, sel_tokens, dlogits, dW_r, c.H,
                                                c.E, c.T, accumulate ? 1 : 0);
  }
  return cudaGetLastError();
}

}  // namespace moe
