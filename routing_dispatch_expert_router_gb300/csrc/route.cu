// Stage 1 of the MoE layer, route: fp32 router logits and top-k selection.
//
// Follows the route stage of "Scalable Training of Mixture-of-Experts Models
// with Megatron Core" (es summary, Resumen técnico §2.1 step 1: a router sends
// every token to its k best experts), with the router kept in fp32 (§2.4).
#include "common.cuh"
#include "internal.h"

namespace moe {

// logits[t,e] = sum_h x[t,h] W_r[e,h] in fp32, one thread owning a 4x4 block of
// (token, expert) outputs; x and W_r staged through shared memory in 32-wide
// slices of H. The summation order over h is fixed (sequential FMA).
template <int BT, int BE>
__global__ void __launch_bounds__(256)
route_logits_kernel(const __nv_bfloat16* __restrict__ x, const float* __restrict__ W,
                    float* __restrict__ logits, int T, int H, int E) {
  constexpr int HC = 32;
  constexpr int TX = BE / 4;
  constexpr int TY = BT / 4;
  static_assert(TX * TY == 256, "256 threads");
  __shared__ __align__(16) float xs[HC][BT + 4];
  __shared__ __align__(16) float ws[HC][BE + 4];
  const int t0 = blockIdx.x * BT, e0 = blockIdx.y * BE;
  const int tx = threadIdx.x % TX, ty = threadIdx.x / TX;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

  for (int h0 = 0; h0 < H; h0 += HC) {
    for (int v = threadIdx.x; v < BT * 4; v += 256) {
      const int tt = v >> 2, hq = (v & 3) * 8, t = t0 + tt;
      float f[8];
      if (t < T) {
        unpack8(ldg_nc_v4(x + (size_t)t * H + h0 + hq), f);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) f[i] = 0.f;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) xs[hq + i][tt] = f[i];
    }
    for (int v = threadIdx.x; v < BE * 8; v += 256) {
      const int ee = v >> 3, hq = (v & 7) * 4, e = e0 + ee;
      float4 q = make_float4(0.f, 0.f, 0.f, 0.f);
      if (e < E) q = *reinterpret_cast<const float4*>(W + (size_t)e * H + h0 + hq);
      ws[hq][ee] = q.x;
      ws[hq + 1][ee] = q.y;
      ws[hq + 2][ee] = q.z;
      ws[hq + 3][ee] = q.w;
    }
    __syncthreads();
#pragma unroll 8
    for (int h = 0; h < HC; ++h) {
      const float4 a = *reinterpret_cast<const float4*>(&xs[h][ty * 4]);
      const float4 b = *reinterpret_cast<const float4*>(&ws[h][tx * 4]);
      const float av[4] = {a.x, a.y, a.z, a.w};
      const float bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + ty * 4 + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + tx * 4 + j;
      if (e < E) logits[(size_t)t * E + e] = acc[i][j];
    }
  }
}

// Few experts (E <= 16): logits on the warp-level tensor-core MMA (mma.sync
// m16n8k16, bf16 operands, fp32 accumulation): with 8 or 16 output columns a
// tile needs no tensor memory or TMA pipeline, and the kernel is a stream over
// x. W_r is split in registers into three bf16 parts, hi = bf16(w),
// mid = bf16(w - hi), lo = w - hi - mid (exact: hi + mid + lo == w), so the
// products are those of the fp32 weights. A block of 8 warps owns 16 tokens;
// warp w takes the 32-column chunks w, w + 8, ... of H, D chunks in flight.
// Inside a chunk the reduction index is permuted the same way in A and B so
// that every lane's fragments are 16-byte loads: lane (g = lane / 4,
// q = lane % 4) loads columns 8q..8q+7 of token rows g and g + 8 and of weight
// row g (+ 8 per n-tile); the chunk's first MMA covers columns 8q..8q+3 of
// every lane, the second 8q+4..8q+7. The warps' partial sums are added in warp
// order through shared memory, so the summation order is fixed.
__device__ __forceinline__ void mma_m16n8k16_bf16(float (&d)[4], uint32_t a0, uint32_t a1,
                                                  uint32_t a2, uint32_t a3, uint32_t b0,
                                                  uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <int NT>
__global__ void __launch_bounds__(256)
route_logits_mma_kernel(const __nv_bfloat16* __restrict__ x, const float* __restrict__ W,
                        float* __restrict__ logits, int T, int H, int E) {
  constexpr int D = NT == 1 ? 4 : 2;               // chunks in flight per warp
  __shared__ float part[8][16][8 * NT];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int g = lane >> 2, q = lane & 3;
  const int t0 = blockIdx.x * 16;
  const bool ok0 = t0 + g < T, ok1 = t0 + g + 8 < T;
  const __nv_bfloat16* x0 = x + (size_t)(t0 + g) * H + 8 * q;
  const __nv_bfloat16* x1 = x0 + (size_t)8 * H;
  bool wok[NT];
  const float* wrow[NT];
#pragma unroll
  for (int n = 0; n < NT; ++n) {
    wok[n] = 8 * n + g < E;
    wrow[n] = W + (size_t)(8 * n + g) * H + 8 * q;
  }
  const int nchunks = H >> 5;
  const int mine = nchunks > wid ? (nchunks - wid + 7) >> 3 : 0;
  uint4 xa[D], xb[D];
  float4 wa[D][NT], wb[D][NT];
  auto load = [&](int d, int i) {
    const int col = (wid + 8 * i) * 32;
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    xa[d] = ok0 ? ldg_nc_v4(x0 + col) : z;
    xb[d] = ok1 ? ldg_nc_v4(x1 + col) : z;
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      const float4 zf = make_float4(0.f, 0.f, 0.f, 0.f);
      wa[d][n] = wok[n] ? __ldg(reinterpret_cast<const float4*>(wrow[n] + col)) : zf;
      wb[d][n] = wok[n] ? __ldg(reinterpret_cast<const float4*>(wrow[n] + col) + 1) : zf;
    }
  };
  float acc[NT][4];
#pragma unroll
  for (int n = 0; n < NT; ++n)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[n][j] = 0.f;
#pragma unroll
  for (int d = 0; d < D; ++d)
    if (d < mine) load(d, d);
  for (int i = 0; i < mine; i += D) {
#pragma unroll
    for (int d = 0; d < D; ++d) {
      if (i + d >= mine) break;
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        uint32_t h[4], m[4], l[4];
        split3_pair(wa[d][n].x, wa[d][n].y, h[0], m[0], l[0]);
        split3_pair(wa[d][n].z, wa[d][n].w, h[1], m[1], l[1]);
        split3_pair(wb[d][n].x, wb[d][n].y, h[2], m[2], l[2]);
        split3_pair(wb[d][n].z, wb[d][n].w, h[3], m[3], l[3]);
        mma_m16n8k16_bf16(acc[n], xa[d].x, xb[d].x, xa[d].y, xb[d].y, h[0], h[1]);
        mma_m16n8k16_bf16(acc[n], xa[d].z, xb[d].z, xa[d].w, xb[d].w, h[2], h[3]);
        mma_m16n8k16_bf16(acc[n], xa[d].x, xb[d].x, xa[d].y, xb[d].y, m[0], m[1]);
        mma_m16n8k16_bf16(acc[n], xa[d].z, xb[d].z, xa[d].w, xb[d].w, m[2], m[3]);
        mma_m16n8k16_bf16(acc[n], xa[d].x, xb[d].x, xa[d].y, xb[d].y, l[0], l[1]);
        mma_m16n8k16_bf16(acc[n], xa[d].z, xb[d].z, xa[d].w, xb[d].w, l[2], l[3]);
      }
      if (i + d + D < mine) load(d, i + d + D);
    }
  }
  // accumulator fragment: (row g, columns 2q, 2q+1) and (row g + 8, same)
#pragma unroll
  for (int n = 0; n < NT; ++n) {
    part[wid][g][8 * n + 2 * q] = acc[n][0];
    part[wid][g][8 * n + 2 * q + 1] = acc[n][1];
    part[wid][g + 8][8 * n + 2 * q] = acc[n][2];
    part[wid][g + 8][8 * n + 2 * q + 1] = acc[n][3];
  }
  __syncthreads();
  for (int v = threadIdx.x; v < 16 * 8 * NT; v += 256) {
    const int r = v / (8 * NT), e = v % (8 * NT);
    if (t0 + r < T && e < E) {
      float sum = part[0][r][e];
#pragma unroll
      for (int w = 1; w < 8; ++w) sum += part[w][r][e];
      logits[(size_t)(t0 + r) * E + e] = sum;
    }
  }
}

// ---------------------------------------------------------------- selection
// Selection compares keys as unsigned integers whose order is the numeric
// order of the (non-NaN) floating-point keys: one integer compare instead of
// a floating-point one (fp64 compares are slow on this part), and a 32-bit key
// packed with the expert index makes "larger key, then lower index" a single
// 64-bit max.
__device__ __forceinline__ uint32_t ord32(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float unord32(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}
__device__ __forceinline__ uint64_t ord64(double d) {
  const uint64_t u = (uint64_t)__double_as_longlong(d);
  return (u >> 63) ? ~u : (u | (1ull << 63));
}
__device__ __forceinline__ double unord64(uint64_t k) {
  return __longlong_as_double((long long)((k >> 63) ? (k & ~(1ull << 63)) : ~k));
}
// (key, expert) packed so that the maximum is the largest key, ties to the
// lower expert; 0 = no candidate (every real key packs above it).
__device__ __forceinline__ uint64_t pack_key(float key, int e) {
  return ((uint64_t)ord32(key) << 32) | (uint64_t)(0xffffffffu - (uint32_t)e);
}
__device__ __forceinline__ int packed_expert(uint64_t p) {
  return (int)(0xffffffffu - (uint32_t)(p & 0xffffffffu));
}

__device__ __forceinline__ uint64_t warp_max_u64(uint64_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint64_t w = __shfl_xor_sync(0xffffffffu, v, o);
    v = w > v ? w : v;
  }
  return v;
}

// Largest (key, lowest expert) over the warp for 64-bit keys; key 0 = none.
__device__ __forceinline__ void warp_best_pair(uint64_t& key, int& e) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint64_t k2 = __shfl_xor_sync(0xffffffffu, key, o);
    const int e2 = __shfl_xor_sync(0xffffffffu, e, o);
    if (k2 > key || (k2 == key && e2 < e)) {
      key = k2;
      e = e2;
    }
  }
}

// The two largest values held by the warp (duplicates count twice).
__device__ __forceinline__ void warp_top2_u64(uint64_t& a1, uint64_t& a2) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint64_t b1 = __shfl_xor_sync(0xffffffffu, a1, o);
    const uint64_t b2 = __shfl_xor_sync(0xffffffffu, a2, o);
    const uint64_t hi = a1 > b1 ? a1 : b1;
    const uint64_t lo1 = a1 > b1 ? b1 : a1;
    const uint64_t lo2 = a2 > b2 ? a2 : b2;
    a1 = hi;
    a2 = lo1 > lo2 ? lo1 : lo2;
  }
}
__device__ __forceinline__ void warp_top2_f(float& a1, float& a2) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float b1 = __shfl_xor_sync(0xffffffffu, a1, o);
    const float b2 = __shfl_xor_sync(0xffffffffu, a2, o);
    const float hi = fmaxf(a1, b1);
    a2 = fmaxf(fminf(a1, b1), fmaxf(a2, b2));
    a1 = hi;
  }
}

__device__ __forceinline__ void top2_insert(uint64_t v, uint64_t& a1, uint64_t& a2) {
  if (v > a1) {
    a2 = a1;
    a1 = v;
  } else if (v > a2) {
    a2 = v;
  }
}
__device__ __forceinline__ void top2_insert_f(float v, float& a1, float& a2) {
  if (v > a1) {
    a2 = a1;
    a1 = v;
  } else if (v > a2) {
    a2 = v;
  }
}

// Keeps the topk_groups best groups given the group scores (lane g holds group
// g's ordered fp64 score; ties to the lower group) and clears the availability
// of every expert outside them.
template <int NPL>
__device__ __forceinline__ void keep_best_groups(uint64_t gs_mine, int lane, int n_groups,
                                                 int topk_groups, const int (&gid)[NPL],
                                                 bool (&avail)[NPL]) {
  uint32_t kept = 0;
  for (int r = 0; r < topk_groups; ++r) {
    uint64_t key = (lane < n_groups && !((kept >> lane) & 1u)) ? gs_mine : 0ull;
    int g = lane;
    warp_best_pair(key, g);
    kept |= 1u << g;
  }
#pragma unroll
  for (int i = 0; i < NPL; ++i)
    if (gid[i] >= 0 && !((kept >> gid[i]) & 1u)) avail[i] = false;
}

// Group of each owned expert (-1 past E), computed once: the group loops
// below would otherwise divide in their inner loops.
template <int NPL>
__device__ __forceinline__ void group_ids(int lane, int E, int per, int (&gid)[NPL]) {
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = lane + 32 * i;
    gid[i] = e < E ? e / per : -1;
  }
}

// One warp per token, softmax router: selection key = fp32 (logit + bias)
// (NaN ranks last), optional group limit (group score = top-1 or top-2 sum of
// the group's keys in fp64), top-k with ties to the lower expert, weights =
// softmax over the selected (logit + bias). Lane l owns experts l, l+32, ...
template <int NPL>
__global__ void __launch_bounds__(256)
route_select_softmax_kernel(const float* __restrict__ logits, const float* __restrict__ bias,
                            int32_t* __restrict__ idx, float* __restrict__ wout, int T, int E,
                            int k, int n_groups, int topk_groups, int group_score) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  const float* lrow = logits + (size_t)t * E;
  float key[NPL];
  bool avail[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = lane + 32 * i;
    avail[i] = e < E;
    key[i] = -INFINITY;
    if (e < E) {
      // (+ 0 turns a -0 sum into +0, which compares equal to it)
      const float v = __fadd_rn(__fadd_rn(lrow[e], bias ? bias[e] : 0.f), 0.f);
      key[i] = isnan(v) ? -INFINITY : v;
    }
  }
  if (n_groups > 1) {
    const int per = E / n_groups;
    const bool two = group_score == MOE_GROUP_TOP2_SUM && per >= 2;
    int gid[NPL];
    group_ids<NPL>(lane, E, per, gid);
    uint64_t gs_mine = 0;
    for (int g = 0; g < n_groups; ++g) {
      float a1 = -INFINITY, a2 = -INFINITY;
#pragma unroll
      for (int i = 0; i < NPL; ++i)
        if (gid[i] == g) top2_insert_f(key[i], a1, a2);
      warp_top2_f(a1, a2);
      const double gsc = two ? (double)a1 + (double)a2 : (double)a1;
      if (lane == g) gs_mine = ord64(gsc);
    }
    keep_best_groups<NPL>(gs_mine, lane, n_groups, topk_groups, gid, avail);
  }
  // packed keys of the available experts (0 = not available), then k rounds
  // of a warp maximum; the winner's slot is cleared
  uint64_t pk[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) pk[i] = avail[i] ? pack_key(key[i], lane + 32 * i) : 0ull;
  int my_e = 0;
  for (int j = 0; j < k; ++j) {
    uint64_t best = pk[0];
#pragma unroll
    for (int i = 1; i < NPL; ++i) best = pk[i] > best ? pk[i] : best;
    best = warp_max_u64(best);
#pragma unroll
    for (int i = 0; i < NPL; ++i)
      if (pk[i] == best) pk[i] = 0ull;
    if (lane == j) my_e = packed_expert(best);
  }
  // weights: softmax over the selected (logit + bias), relative to the first
  float z = 0.f, z0 = 0.f;
  {
    const int e0 = __shfl_sync(0xffffffffu, my_e, 0);
    z0 = __fadd_rn(lrow[e0], bias ? bias[e0] : 0.f);
    if (lane < k) z = expf(__fadd_rn(lrow[my_e], bias ? bias[my_e] : 0.f) - z0);
  }
  float zs = 0.f;
  for (int j = 0; j < k; ++j) zs += __shfl_sync(0xffffffffu, z, j);
  if (lane < k) {
    idx[(size_t)t * k + lane] = my_e;
    wout[(size_t)t * k + lane] = z / zs;
  }
}

// fp64 sigmoid of every owned expert whose bit is set in `need` (bit i =
// expert lane + 32 i), spread over the warp: the candidates of all lanes are
// numbered (by i, then lane) and lane n evaluates candidate n (32 per round),
// then every owner picks its values up by shuffle. A warp instruction on the
// fp64 pipe costs the same with one lane active as with 32, so this is up to
// 32 times cheaper than every lane evaluating its own candidates.
template <int NPL>
__device__ __forceinline__ void exact_sigmoids(const float* __restrict__ lrow, uint32_t need,
                                               int lane, double (&s64)[NPL]) {
  uint32_t b[NPL];
  int base[NPL + 1];
  base[0] = 0;
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    b[i] = __ballot_sync(0xffffffffu, (need >> i) & 1u);
    base[i + 1] = base[i] + __popc(b[i]);
  }
  const int total = base[NPL];
  for (int r0 = 0; r0 < total; r0 += 32) {
    const int n = r0 + lane;
    double sv = 0.0;
    if (n < total) {
      int e = 0;
#pragma unroll
      for (int i = 0; i < NPL; ++i)
        if (n >= base[i] && n < base[i + 1]) e = (int)__fns(b[i], 0u, n - base[i] + 1) + 32 * i;
      sv = 1.0 / (1.0 + exp(-(double)lrow[e]));
    }
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      const int slot = base[i] + __popc(b[i] & ((1u << lane) - 1u));
      const double got = __shfl_sync(0xffffffffu, sv, (slot - r0) & 31);
      if (((b[i] >> lane) & 1u) && slot >= r0 && slot < r0 + 32) s64[i] = got;
    }
  }
}

// One warp per token, sigmoid router: s = sigmoid(logit) and selection key
// s + bias, both in fp64 (NaN ranks last); optional group limit; top-k with
// ties to the lower expert; weights route_scale * s / sum(s) over the
// selected.
//
// fp64 is slow on this part, so the fp64 keys are computed only where they can
// decide anything. Every key is first formed in fp32 (A, off the fp64 key by
// at most 3.6e-7 + 6e-8 |A|; margin(x) = 1e-5 (1 + |x|) is well above twice
// that).
//   Fast path: the group scores and the top-k are taken on the fp32 keys, and
//   the result stands when every decision is clear by the margins: every kept
//   group's score minus its margin (the sum of its top-m keys' margins) above
//   every dropped group's score plus its margin, and each of the k selected
//   keys above the next one in the order (the (k+1)-th included) by more than
//   margin(larger |key|). The fp64 keys then select and order exactly the same
//   way. The weights come from the fp32 sigmoids (a few ulp).
//   Exact path (a decision within a margin): a group's top-m (m = 2 for the
//   top-2 sum, else 1) can only contain experts with A >= (the group's m-th
//   best A) - margin, and the final top-k only experts with A >= (the k-th best
//   A among the kept groups) - margin: any other expert has m (or k) experts
//   whose fp64 key is strictly larger. Those candidates get their fp64 keys,
//   and the group scores and the selection are taken on fp64 keys alone, so the
//   result is the one the fp64 keys of all experts give.
template <int NPL>
__global__ void __launch_bounds__(128, 6)
route_select_sigmoid_kernel(const float* __restrict__ logits, const float* __restrict__ bias,
                            int32_t* __restrict__ idx, float* __restrict__ wout, int T, int E,
                            int k, int n_groups, int topk_groups, int group_score,
                            float route_scale) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  const float* lrow = logits + (size_t)t * E;
  float A[NPL];
  bool avail[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = lane + 32 * i;
    avail[i] = e < E;
    A[i] = -INFINITY;
    if (e < E) {
      const float s32 = __fdiv_rn(1.f, 1.f + expf(-lrow[e]));
      const float v = __fadd_rn(s32, bias ? bias[e] : 0.f);
      A[i] = isnan(v) ? -INFINITY : v;
    }
  }
  auto margin = [](float thr) { return 1e-5f * (1.f + fabsf(thr)); };
  // ------------------------------------------------ fast path (fp32 decisions)
  {
    bool clear = true;
    uint32_t kept = 0xffffffffu;
    int gid[NPL];
    if (n_groups > 1) {
      const int per = E / n_groups;
      const bool two = group_score == MOE_GROUP_TOP2_SUM && per >= 2;
      group_ids<NPL>(lane, E, per, gid);
      // fp32 group scores (no fp64 instruction on this path: the fp64 pipe is
      // narrow on this part)
      float gs_mine = -INFINITY, gm_mine = 0.f;
      if (per == 32) {
        // lane l's expert of group g is l + 32 g: the groups' reductions are
        // independent and unrolled
#pragma unroll
        for (int g = 0; g < NPL; ++g) {
          if (g >= n_groups) break;
          float a1 = A[g], a2 = -INFINITY;
          warp_top2_f(a1, a2);
          if (lane == g) {
            gs_mine = two ? a1 + a2 : a1;
            gm_mine = two ? margin(a1) + margin(a2) : margin(a1);
          }
        }
      } else {
        for (int g = 0; g < n_groups; ++g) {
          float a1 = -INFINITY, a2 = -INFINITY;
#pragma unroll
          for (int i = 0; i < NPL; ++i)
            if (gid[i] == g) top2_insert_f(A[i], a1, a2);
          warp_top2_f(a1, a2);
          if (lane == g) {
            gs_mine = two ? a1 + a2 : a1;
            gm_mine = two ? margin(a1) + margin(a2) : margin(a1);
          }
        }
      }
      kept = 0;
      for (int r = 0; r < topk_groups; ++r) {
        uint64_t key = (lane < n_groups && !((kept >> lane) & 1u)) ? pack_key(gs_mine, lane) : 0ull;
        key = warp_max_u64(key);
        kept |= 1u << packed_expert(key);
      }
      // clear when every kept group's lowest possible score is above every
      // dropped group's highest possible one
      float lo = INFINITY, hi = -INFINITY;
      if (lane < n_groups) {
        if ((kept >> lane) & 1u) lo = gs_mine - gm_mine;
        else hi = gs_mine + gm_mine;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
        hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
      }
      clear = lo > hi;
    }
    // packed keys of the available experts (0 = not available), then k + 1
    // rounds of a warp maximum; the winner's slot is cleared
    uint64_t pk[NPL];
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      const bool in = avail[i] && (n_groups <= 1 || ((kept >> gid[i]) & 1u));
      pk[i] = in ? pack_key(A[i], lane + 32 * i) : 0ull;
    }
    int my_e = 0;
    float prev = 0.f;
    for (int j = 0; j <= k && clear; ++j) {
      uint64_t best = pk[0];
#pragma unroll
      for (int i = 1; i < NPL; ++i) best = pk[i] > best ? pk[i] : best;
      best = warp_max_u64(best);
      if (best == 0) break;                        // fewer than k + 1 experts available
      const float a = unord32((uint32_t)(best >> 32));
      if (j > 0) clear = (prev - a) > margin(fmaxf(fabsf(prev), fabsf(a)));
      prev = a;
      if (j == k) break;
#pragma unroll
      for (int i = 0; i < NPL; ++i)
        if (pk[i] == best) pk[i] = 0ull;
      if (lane == j) my_e = packed_expert(best);
    }
    if (clear) {
      // the selected experts' fp32 sigmoids, recomputed as above
      const float my_s = lane < k ? __fdiv_rn(1.f, 1.f + expf(-lrow[my_e])) : 0.f;
      float ss = 0.f;
      for (int j = 0; j < k; ++j) ss += __shfl_sync(0xffffffffu, my_s, j);
      if (lane < k) {
        idx[(size_t)t * k + lane] = my_e;
        wout[(size_t)t * k + lane] = route_scale * my_s / ss;
      }
      return;
    }
  }
  double s64[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) s64[i] = 0.0;
  // ------------------------------------------------ exact path (fp64 decisions)
  // ordered fp64 key of owned expert i (its s64 must have been evaluated)
  auto key64 = [&](int i) -> uint64_t {
    const double v = s64[i] + (double)(bias ? bias[lane + 32 * i] : 0.f);
    return isnan(v) ? ord64(-INFINITY) : ord64(v);
  };
  uint32_t have = 0;                               // bit i: s64[i] evaluated
  if (n_groups > 1) {
    const int per = E / n_groups;
    const bool two = group_score == MOE_GROUP_TOP2_SUM && per >= 2;
    int gid[NPL];
    group_ids<NPL>(lane, E, per, gid);
    // candidates for every group's top-m, from the fp32 keys
    uint32_t gc = 0;
    uint64_t gs_mine = 0;
    if (per == 32) {
      // groups of 32 experts: lane l's expert of group g is l + 32 g (i = g), so
      // the per-lane scans over i disappear (fully unrolled, n_groups <= NPL)
#pragma unroll
      for (int g = 0; g < NPL; ++g) {
        if (g >= n_groups) break;
        float a1 = A[g], a2 = -INFINITY;
        warp_top2_f(a1, a2);
        const float am = two ? a2 : a1;
        if (A[g] >= am - margin(am)) gc |= 1u << g;
      }
      exact_sigmoids<NPL>(lrow, gc, lane, s64);
#pragma unroll
      for (int g = 0; g < NPL; ++g) {
        if (g >= n_groups) break;
        uint64_t k1 = ((gc >> g) & 1u) ? key64(g) : 0ull, k2 = 0;
        warp_top2_u64(k1, k2);
        const double gsc = two ? unord64(k1) + unord64(k2) : unord64(k1);
        if (lane == g) gs_mine = ord64(gsc);
      }
    } else {
      for (int g = 0; g < n_groups; ++g) {
        float a1 = -INFINITY, a2 = -INFINITY;
#pragma unroll
        for (int i = 0; i < NPL; ++i)
          if (gid[i] == g) top2_insert_f(A[i], a1, a2);
        warp_top2_f(a1, a2);
        const float am = two ? a2 : a1;
        const float thr = am - margin(am);
#pragma unroll
        for (int i = 0; i < NPL; ++i)
          if (gid[i] == g && A[i] >= thr) gc |= 1u << i;
      }
      exact_sigmoids<NPL>(lrow, gc, lane, s64);
      // group scores on the fp64 keys of the candidates
      for (int g = 0; g < n_groups; ++g) {
        uint64_t k1 = 0, k2 = 0;
#pragma unroll
        for (int i = 0; i < NPL; ++i)
          if (((gc >> i) & 1u) && gid[i] == g) top2_insert(key64(i), k1, k2);
        warp_top2_u64(k1, k2);
        const double gsc = two ? unord64(k1) + unord64(k2) : unord64(k1);
        if (lane == g) gs_mine = ord64(gsc);
      }
    }
    have = gc;
    keep_best_groups<NPL>(gs_mine, lane, n_groups, topk_groups, gid, avail);
  }
  // the k-th best fp32 key among the available experts
  uint64_t kth = 0;
  {
    bool taken[NPL];
#pragma unroll
    for (int i = 0; i < NPL; ++i) taken[i] = false;
    for (int j = 0; j < k; ++j) {
      uint64_t best = 0;
#pragma unroll
      for (int i = 0; i < NPL; ++i) {
        if (!avail[i] || taken[i]) continue;
        const uint64_t p = pack_key(A[i], lane + 32 * i);
        best = p > best ? p : best;
      }
      best = warp_max_u64(best);
      const int e = packed_expert(best);
#pragma unroll
      for (int i = 0; i < NPL; ++i)
        if (lane + 32 * i == e) taken[i] = true;
      kth = best;
    }
  }
  const float ak = unord32((uint32_t)(kth >> 32));
  const float thr = ak - margin(ak);
  uint32_t fc = 0;                                 // candidates for the final top-k
#pragma unroll
  for (int i = 0; i < NPL; ++i)
    if (avail[i] && A[i] >= thr) fc |= 1u << i;
  if (__any_sync(0xffffffffu, (fc & ~have) != 0u)) exact_sigmoids<NPL>(lrow, fc & ~have, lane, s64);
  uint64_t ck[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) ck[i] = ((fc >> i) & 1u) ? key64(i) : 0ull;
  int my_e = 0;
  double my_s = 0.0;
  for (int j = 0; j < k; ++j) {
    uint64_t best = 0;
    int be = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      const int e = lane + 32 * i;
      if (ck[i] > best || (ck[i] == best && ck[i] != 0ull && e < be)) {
        best = ck[i];
        be = e;
      }
    }
    warp_best_pair(best, be);
    double sv = 0.0;
#pragma unroll
    for (int i = 0; i < NPL; ++i)
      if (lane + 32 * i == be) {
        ck[i] = 0ull;
        sv = s64[i];
      }
    sv = __shfl_sync(0xffffffffu, sv, be & 31);
    if (lane == j) {
      my_e = be;
      my_s = sv;
    }
  }
  double ss = 0.0;
  for (int j = 0; j < k; ++j) ss += __shfl_sync(0xffffffffu, my_s, j);
  if (lane < k) {
    idx[(size_t)t * k + lane] = my_e;
    wout[(size_t)t * k + lane] = (float)((double)route_scale * my_s / ss);
  }
}

// W3[e] = the three bf16 parts of row e of W_r, hi = bf16(w), mid = bf16(w - hi),
// lo = bf16(w - hi - mid) (each keeps 8 significant bits, so hi + mid + lo == w
// exactly for every fp32 w: the two subtractions are exact), interleaved per
// 64 columns: columns 64j..64j+63 of hi, of mid, of lo, then the next 64.
// One thread per 8 consecutive columns (H % 64 == 0): two 16-byte loads, three
// 16-byte stores.
__global__ void __launch_bounds__(256)
split3_kernel(const float* __restrict__ W, __nv_bfloat16* __restrict__ W3, int E, int H) {
  const int per_row = H >> 3;
  const long long n = (long long)E * per_row;
  for (long long v = (long long)blockIdx.x * blockDim.x + threadIdx.x; v < n;
       v += (long long)gridDim.x * blockDim.x) {
    const int e = (int)(v / per_row), h = (int)(v - (long long)e * per_row) << 3;
    const float4* src = reinterpret_cast<const float4*>(W + (size_t)e * H + h);
    const float4 a = __ldg(src), b = __ldg(src + 1);
    const float f[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    float hi[8], mid[8], lo[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      hi[q] = __bfloat162float(__float2bfloat16_rn(f[q]));
      const float r1 = f[q] - hi[q];
      mid[q] = __bfloat162float(__float2bfloat16_rn(r1));
      lo[q] = r1 - mid[q];
    }
    uint4* blk = reinterpret_cast<uint4*>(W3 + (size_t)e * 3 * H + (size_t)(h >> 6) * 192 + (h & 63));
    blk[0] = pack8(hi);
    blk[8] = pack8(mid);                          // + 64 columns
    blk[16] = pack8(lo);                          // + 128 columns
  }
}

bool router_on_tensor_cores(const moe_config& c) { return c.E >= 128 && c.E % 128 == 0; }

int router_wgrad_chunk(const moe_config& c) {
  const int by_count = ((c.T + 255) / 256 + 63) / 64 * 64;   // at most 256 chunks
  return by_count > 1024 ? by_count : 1024;
}

int64_t router_wgrad_split_bytes(const moe_config& c) {
  const int64_t Tp = ((int64_t)c.T + 63) / 64 * 64;
  return (3 * Tp * c.E * 2 + 255) / 256 * 256;
}

// The router region of scratch: the forward's split W_r, the backward's split
// dlogits and the chunk partial sums of dW_r^T, or the load-balancing loss's
// split dx operands ([T, 3E] and [H, 3E] bf16), whichever is largest.
int64_t router_split_bytes(const moe_config& c) {
  if (!router_on_tensor_cores(c)) return 0;
  const int64_t fwd = ((int64_t)c.E * 3 * c.H * 2 + 255) / 256 * 256;
  const int64_t chunks = (c.T + router_wgrad_chunk(c) - 1) / router_wgrad_chunk(c);
  const int64_t bwd = router_wgrad_split_bytes(c) + (chunks * c.H * c.E * 4 + 255) / 256 * 256;
  const int64_t aux = aux_dx_split_bytes(c);
  const int64_t m = fwd > bwd ? fwd : bwd;
  return m > aux ? m : aux;
}

int64_t aux_dx_split_bytes(const moe_config& c) {
  return ((int64_t)c.T * 3 * c.E * 2 + 255) / 256 * 256 +
         ((int64_t)c.H * 3 * c.E * 2 + 255) / 256 * 256;
}

// Router Replay: the weights of recorded experts idx [T,k] (in that order)
// from the logits, with the selection kernels' own arithmetic (softmax router:
// exp of the chosen logit + bias relative to slot 0's, over their sum in slot
// order; sigmoid router: route_scale times the fp32 sigmoid over the sum of the
// chosen ones), so replaying the router's own choice reproduces its weights.
// One warp per token, lane j < k takes slot j. An expert index outside [0, E)
// records MOE_ERR_DEVICE_CHECK and counts as weight 0.
__global__ void __launch_bounds__(256)
route_replay_weights_kernel(const float* __restrict__ logits, const float* __restrict__ bias,
                            const int32_t* __restrict__ idx, float* __restrict__ wout, int T,
                            int E, int k, int score_fn, float route_scale, int32_t* status) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  const float* lrow = logits + (size_t)t * E;
  int e = lane < k ? idx[(size_t)t * k + lane] : -1;
  // an id out of range, or one that repeats an earlier slot of the token, is
  // reported and gets weight 0 (the dispatch drops it the same way)
  bool rep = false;
  for (int j = 0; j < k; ++j) {
    const int ej = __shfl_sync(0xffffffffu, e, j);
    if (j < lane && ej == e) rep = true;
  }
  const bool bad = lane < k && ((unsigned)e >= (unsigned)E || rep);
  if (bad) record_status(status, MOE_ERR_DEVICE_CHECK);
  if (bad || lane >= k) e = 0;
  float v = 0.f;
  if (score_fn == MOE_SCORE_SOFTMAX) {
    const int e0 = __shfl_sync(0xffffffffu, e, 0);
    const float z0 = __fadd_rn(lrow[e0], bias ? bias[e0] : 0.f);
    if (lane < k && !bad) v = expf(__fadd_rn(lrow[e], bias ? bias[e] : 0.f) - z0);
  } else if (lane < k && !bad) {
    v = __fdiv_rn(1.f, 1.f + expf(-lrow[e]));
  }
  float sum = 0.f;
  for (int j = 0; j < k; ++j) sum += __shfl_sync(0xffffffffu, v, j);
  if (lane < k)
    wout[(size_t)t * k + lane] = score_fn == MOE_SCORE_SOFTMAX ? v / sum : route_scale * v / sum;
}

// logits[T,E] = x . W_r^T in fp32, by the path the expert count selects.
static cudaError_t launch_router_logits(const moe_config& c, const void* x, const float* W_r,
                                        float* logits, uint8_t* scratch, cudaStream_t s) {
  const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
  if (router_on_tensor_cores(c)) {
    // logits on the tensor cores from the exact three-way bf16 split of W_r
    __nv_bfloat16* W3 = reinterpret_cast<__nv_bfloat16*>(scratch + router_split_offset(c));
    const long long n = (long long)c.E * (c.H / 8);
    long long blocks = (n + 255) / 256;
    if (blocks > (long long)num_sms() * 16) blocks = (long long)num_sms() * 16;
    split3_kernel<<<(int)blocks, 256, 0, s>>>(W_r, W3, c.E, c.H);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    err = launch_router_logits_tc(c, x, W3, logits,
                                  reinterpret_cast<int32_t*>(scratch + kScratchStatus), s);
    if (err != cudaSuccess) return err;
  } else if (c.E <= 16) {
    const int blocks = (c.T + 15) / 16;      // 16 tokens per block of 8 warps
    if (c.E <= 8)
      route_logits_mma_kernel<1><<<blocks, 256, 0, s>>>(xb, W_r, logits, c.T, c.H, c.E);
    else
      route_logits_mma_kernel<2><<<blocks, 256, 0, s>>>(xb, W_r, logits, c.T, c.H, c.E);
  } else {
    dim3 grid((c.T + 63) / 64, (c.E + 63) / 64);
    route_logits_kernel<64, 64><<<grid, 256, 0, s>>>(xb, W_r, logits, c.T, c.H, c.E);
  }
  return cudaGetLastError();
}

cudaError_t launch_route(const moe_config& c, const void* x, const float* W_r, const float* bias,
                         float* logits, int32_t* idx, float* w, uint8_t* scratch, cudaStream_t s) {
  if (cudaError_t err = launch_router_logits(c, x, W_r, logits, scratch, s); err != cudaSuccess)
    return err;
  // experts per lane: the smallest of 1, 2, 4, 8 that covers E
  const int npl = c.E <= 32 ? 1 : c.E <= 64 ? 2 : c.E <= 128 ? 4 : 8;
  if (c.score_fn == MOE_SCORE_SOFTMAX) {
    auto kern = npl == 1 ? route_select_softmax_kernel<1>
              : npl == 2 ? route_select_softmax_kernel<2>
              : npl == 4 ? route_select_softmax_kernel<4> : route_select_softmax_kernel<8>;
    kern<<<(c.T + 7) / 8, 256, 0, s>>>(logits, bias, idx, w, c.T, c.E, c.k, c.n_groups,
                                       c.topk_groups, c.group_score);
  } else {
    auto kern = npl == 1 ? route_select_sigmoid_kernel<1>
              : npl == 2 ? route_select_sigmoid_kernel<2>
              : npl == 4 ? route_select_sigmoid_kernel<4> : route_select_sigmoid_kernel<8>;
    kern<<<(c.T + 3) / 4, 128, 0, s>>>(logits, bias, idx, w, c.T, c.E, c.k, c.n_groups,
                                       c.topk_groups, c.group_score, c.route_scale);
  }
  return cudaGetLastError();
}

cudaError_t launch_route_replay(const moe_config& c, const void* x, const float* W_r,
                                const float* bias, const int32_t* idx, float* logits, float* w,
                                uint8_t* scratch, cudaStream_t s) {
  if (cudaError_t err = launch_router_logits(c, x, W_r, logits, scratch, s); err != cudaSuccess)
    return err;
  route_replay_weights_kernel<<<(c.T + 7) / 8, 256, 0, s>>>(
      logits, bias, idx, w, c.T, c.E, c.k, c.score_fn, c.route_scale,
      reinterpret_cast<int32_t*>(scratch + kScratchStatus));
  return cudaGetLastError();
}

}  // namespace moe
