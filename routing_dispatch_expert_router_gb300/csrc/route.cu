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

// Few experts (E <= 16): the logits are a pure stream over x. A block of 4
// warps owns 4 consecutive tokens; warp w walks the w-th quarter of H, each
// lane loading 16-byte slices of the 4 rows (two slices in flight per row)
// and the matching W_r slices, which the 4 tokens share. Lane partial sums are
// combined by a fixed butterfly, then the 4 warps' sums in warp order, so the
// summation order is deterministic.
template <int EP>
__global__ void __launch_bounds__(128)
route_logits_few_kernel(const __nv_bfloat16* __restrict__ x, const float* __restrict__ W,
                        float* __restrict__ logits, int T, int H, int E) {
  constexpr int TPB = 4;
  __shared__ float part[4][TPB][EP];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int t0 = blockIdx.x * TPB;
  float acc[TPB][EP];
#pragma unroll
  for (int i = 0; i < TPB; ++i)
#pragma unroll
    for (int e = 0; e < EP; ++e) acc[i][e] = 0.f;
  const int nvec = H >> 3, per = nvec >> 2;
  const int cbeg = wid * per, cend = cbeg + per;
  for (int c0 = cbeg + lane; c0 < cend; c0 += 64) {
    float xf[2][TPB][8];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int c = c0 + 32 * u;
#pragma unroll
      for (int i = 0; i < TPB; ++i) {
        if (c < cend && t0 + i < T) {
          unpack8(ldg_nc_v4(x + (size_t)(t0 + i) * H + (size_t)c * 8), xf[u][i]);
        } else {
#pragma unroll
          for (int q = 0; q < 8; ++q) xf[u][i][q] = 0.f;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int c = c0 + 32 * u;
      if (c >= cend) break;
#pragma unroll
      for (int e = 0; e < EP; ++e) {
        if (e >= E) break;
        const float4* wp = reinterpret_cast<const float4*>(W + (size_t)e * H + (size_t)c * 8);
        const float4 a = __ldg(wp), b = __ldg(wp + 1);
        const float wv[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int i = 0; i < TPB; ++i)
#pragma unroll
          for (int q = 0; q < 8; ++q) acc[i][e] = fmaf(xf[u][i][q], wv[q], acc[i][e]);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < TPB; ++i)
#pragma unroll
    for (int e = 0; e < EP; ++e) {
      const float v = warp_sum(acc[i][e]);
      if (lane == 0) part[wid][i][e] = v;
    }
  __syncthreads();
  if (threadIdx.x < TPB * EP) {
    const int i = threadIdx.x / EP, e = threadIdx.x % EP;
    if (e < E && t0 + i < T) {
      const float v = ((part[0][i][e] + part[1][i][e]) + part[2][i][e]) + part[3][i][e];
      logits[(size_t)(t0 + i) * E + e] = v;
    }
  }
}

struct Cand {
  double key;
  int e;  // -1 = no candidate
};

__device__ __forceinline__ bool better(const Cand& a, const Cand& b) {
  if (a.e < 0) return false;
  if (b.e < 0) return true;
  if (a.key > b.key) return true;
  if (a.key < b.key) return false;
  return a.e < b.e;
}

__device__ __forceinline__ Cand warp_best(Cand c) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    Cand d;
    d.key = __shfl_xor_sync(0xffffffffu, c.key, o);
    d.e = __shfl_xor_sync(0xffffffffu, c.e, o);
    if (better(d, c)) c = d;
  }
  return c;
}

// The two largest values held by the warp (duplicates count twice).
__device__ __forceinline__ void warp_top2(double& a1, double& a2) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const double b1 = __shfl_xor_sync(0xffffffffu, a1, o);
    const double b2 = __shfl_xor_sync(0xffffffffu, a2, o);
    const double hi = fmax(a1, b1);
    const double lo = fmax(fmin(a1, b1), fmax(a2, b2));
    a1 = hi;
    a2 = lo;
  }
}

// One warp per token: selection keys, optional group limit, top-k, weights.
// Lane l owns experts l, l+32, l+64, ... (at most 8).
__global__ void __launch_bounds__(256)
route_select_kernel(const float* __restrict__ logits, const float* __restrict__ bias,
                    int32_t* __restrict__ idx, float* __restrict__ wout, int T, int E, int k,
                    int score_fn, int n_groups, int topk_groups, int group_score,
                    float route_scale) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  const float* lrow = logits + (size_t)t * E;
  constexpr int NPL = kMaxExperts / 32;
  double key[NPL];
  bool avail[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = lane + 32 * i;
    avail[i] = e < E;
    key[i] = -INFINITY;
    if (e < E) {
      const float l = lrow[e];
      const float b = bias ? bias[e] : 0.f;
      double v;
      if (score_fn == MOE_SCORE_SOFTMAX) {
        v = (double)__fadd_rn(l, b);
      } else {
        const double s = 1.0 / (1.0 + exp(-(double)l));
        v = s + (double)b;
      }
      key[i] = isnan(v) ? -INFINITY : v;
    }
  }
  if (n_groups > 1) {
    const int per = E / n_groups;
    double gs_mine = -INFINITY;   // lane g keeps group g's score
    for (int g = 0; g < n_groups; ++g) {
      double a1 = -INFINITY, a2 = -INFINITY;
#pragma unroll
      for (int i = 0; i < NPL; ++i) {
        const int e = lane + 32 * i;
        if (e < E && e / per == g) {
          const double v = key[i];
          if (v > a1) { a2 = a1; a1 = v; }
          else if (v > a2) { a2 = v; }
        }
      }
      warp_top2(a1, a2);
      const double gsc = (group_score == MOE_GROUP_TOP2_SUM && per >= 2) ? a1 + a2 : a1;
      if (lane == g) gs_mine = gsc;
    }
    // keep the topk_groups best groups (ties -> lower group)
    uint32_t kept = 0;
    for (int r = 0; r < topk_groups; ++r) {
      Cand c;
      c.key = gs_mine;
      c.e = (lane < n_groups && !((kept >> lane) & 1u)) ? lane : -1;
      c = warp_best(c);
      if (c.e >= 0) kept |= 1u << c.e;
    }
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !((kept >> (e / per)) & 1u)) avail[i] = false;
    }
  }
  int sel_e[kMaxK];
  for (int j = 0; j < k; ++j) {
    Cand c;
    c.key = -INFINITY;
    c.e = -1;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      Cand d;
      d.key = key[i];
      d.e = avail[i] ? lane + 32 * i : -1;
      if (better(d, c)) c = d;
    }
    c = warp_best(c);
    sel_e[j] = c.e;
#pragma unroll
    for (int i = 0; i < NPL; ++i)
      if (lane + 32 * i == c.e) avail[i] = false;
  }
  // weights: every lane computes them; lane j writes slot j
  if (score_fn == MOE_SCORE_SOFTMAX) {
    float z[kMaxK];
    float zs = 0.f;
    for (int j = 0; j < k; ++j) {
      const int e = sel_e[j];
      z[j] = __fadd_rn(lrow[e], bias ? bias[e] : 0.f);
    }
    const float z0 = z[0];
    for (int j = 0; j < k; ++j) {
      z[j] = expf(z[j] - z0);
      zs += z[j];
    }
    if (lane < k) {
      float v = 0.f;
      int ee = 0;
      for (int j = 0; j < k; ++j)
        if (j == lane) { v = z[j]; ee = sel_e[j]; }
      idx[(size_t)t * k + lane] = ee;
      wout[(size_t)t * k + lane] = v / zs;
    }
  } else {
    double s[kMaxK];
    double ss = 0.0;
    for (int j = 0; j < k; ++j) {
      s[j] = 1.0 / (1.0 + exp(-(double)lrow[sel_e[j]]));
      ss += s[j];
    }
    if (lane < k) {
      double v = 0.0;
      int ee = 0;
      for (int j = 0; j < k; ++j)
        if (j == lane) { v = s[j]; ee = sel_e[j]; }
      idx[(size_t)t * k + lane] = ee;
      wout[(size_t)t * k + lane] = (float)((double)route_scale * v / ss);
    }
  }
}

// W3[e] = [hi | mid | lo] with hi = bf16(w), mid = bf16(w - hi), lo = bf16(w - hi - mid):
// each part keeps 8 significant bits, so hi + mid + lo == w exactly for every
// fp32 w (the two subtractions are exact).
__global__ void __launch_bounds__(256)
split3_kernel(const float* __restrict__ W, __nv_bfloat16* __restrict__ W3, int E, int H) {
  const long long n = (long long)E * H;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const int e = (int)(i / H), h = (int)(i % H);
    const float v = W[i];
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    const float r1 = v - __bfloat162float(hi);
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(mid);
    __nv_bfloat16* row = W3 + (size_t)e * 3 * H;
    row[h] = hi;
    row[H + h] = mid;
    row[2 * H + h] = __float2bfloat16_rn(r2);
  }
}

bool router_on_tensor_cores(const moe_config& c) { return c.E >= 128 && c.E % 128 == 0; }

int64_t router_split_bytes(const moe_config& c) {
  return router_on_tensor_cores(c) ? ((int64_t)c.E * 3 * c.H * 2 + 255) / 256 * 256 : 0;
}

cudaError_t launch_route(const moe_config& c, const void* x, const float* W_r, const float* bias,
                         float* logits, int32_t* idx, float* w, uint8_t* scratch, cudaStream_t s) {
  const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
  if (router_on_tensor_cores(c)) {
    // logits on the tensor cores from the exact three-way bf16 split of W_r
    __nv_bfloat16* W3 = reinterpret_cast<__nv_bfloat16*>(scratch + router_split_offset(c));
    const long long n = (long long)c.E * c.H;
    long long blocks = (n + 255) / 256;
    if (blocks > (long long)num_sms() * 16) blocks = (long long)num_sms() * 16;
    split3_kernel<<<(int)blocks, 256, 0, s>>>(W_r, W3, c.E, c.H);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    err = launch_router_logits_tc(c, x, W3, logits,
                                  reinterpret_cast<int32_t*>(scratch + kScratchStatus), s);
    if (err != cudaSuccess) return err;
  } else if (c.E <= 16) {
    const int blocks = (c.T + 3) / 4;        // 4 tokens per block of 4 warps
    if (c.E <= 8)
      route_logits_few_kernel<8><<<blocks, 128, 0, s>>>(xb, W_r, logits, c.T, c.H, c.E);
    else
      route_logits_few_kernel<16><<<blocks, 128, 0, s>>>(xb, W_r, logits, c.T, c.H, c.E);
  } else {
    dim3 grid((c.T + 63) / 64, (c.E + 63) / 64);
    route_logits_kernel<64, 64><<<grid, 256, 0, s>>>(xb, W_r, logits, c.T, c.H, c.E);
  }
  if (cudaError_t err = cudaGetLastError(); err != cudaSuccess) return err;
  route_select_kernel<<<(c.T + 7) / 8, 256, 0, s>>>(logits, bias, idx, w, c.T, c.E, c.k,
                                                    c.score_fn, c.n_groups, c.topk_groups,
                                                    c.group_score, c.route_scale);
  return cudaGetLastError();
}

}  // namespace moe
