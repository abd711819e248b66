// Load-balancing auxiliary loss of the router, its gradient, and the
// auxiliary-loss-free update of the selection bias.
//
// "Scalable Training of Mixture-of-Experts Models with Megatron Core"
// (gist.science summaries; es: "Resumen técnico" §2.3.C, "Fusión de Kernels")
// fuses routing, permutation and the auxiliary-loss computation to save
// kernel launches; it gives no formula. The loss here is the switch-style
// balance loss
//   loss = coeff * E * sum_e f_e P_e,
//   f_e = (tokens that selected e) / (T k),  P_e = mean over tokens of p[t,e],
// p[t,:] the router's probability of every expert (softmax of l + b over all
// E; sigmoid router: s / sum_e s, s = sigmoid(l)).
//
// Forward: one launch. Every block takes 64 tokens (8 per warp, one token at a
// time, lane l owns experts l, l + 32, ...), sums p per expert in registers
// and the selections in shared memory, and writes its partial sums; the last
// block to finish adds the partials in a fixed order (deterministic), writes
// counts, P and the loss, and applies the bias update.
// Backward: dlogits of the loss (dense [T,E]), then dx += dl W_r (tensor
// cores from the hi + mid bf16 parts of both operands when E % 128 == 0, else
// the CUDA cores in fp32; one bf16 rounding) and dW_r += dl^T x through the
// router weight-gradient path.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace moe {

constexpr int kAuxTokens = 64;    // tokens per block of the statistics kernel
constexpr int kAuxWarps = 8;      // (8 per warp)

int64_t aux_partial_bytes(const moe_config& c) {
  const int64_t nb = c.T > 0 ? ((int64_t)c.T + kAuxTokens - 1) / kAuxTokens : 1;
  return (2 * nb * c.E * 4 + 255) / 256 * 256;
}

// One token's logits for the lane's experts lane + 32 i (0 beyond E).
template <int NPL>
__device__ __forceinline__ void aux_load(const float* __restrict__ lrow, int E, int lane,
                                         float (&v)[NPL]) {
#pragma unroll
  for (int i = 0; i < NPL; ++i) v[i] = lane + 32 * i < E ? lrow[lane + 32 * i] : 0.f;
}

// p[i] = the router probability of expert lane + 32 i (0 beyond E) from the
// token's logits v and the lane's biases bb; s[i] = its sigmoid and S their
// sum (sigmoid router only).
template <int NPL>
__device__ __forceinline__ void aux_probs(const float (&v)[NPL], const float (&bb)[NPL], int E,
                                          int score_fn, int lane, float (&p)[NPL],
                                          float (&s)[NPL], float& S) {
  if (score_fn == MOE_SCORE_SOFTMAX) {
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      p[i] = lane + 32 * i < E ? __fadd_rn(v[i], bb[i]) : -INFINITY;
      m = fmaxf(m, p[i]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float z = 0.f;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      p[i] = lane + 32 * i < E ? expf(p[i] - m) : 0.f;
      z += p[i];
    }
    z = warp_sum(z);
#pragma unroll
    for (int i = 0; i < NPL; ++i) p[i] = __fdiv_rn(p[i], z);
    S = 0.f;
  } else {
    float z = 0.f;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      s[i] = lane + 32 * i < E ? __fdiv_rn(1.f, 1.f + expf(-v[i])) : 0.f;
      z += s[i];
    }
    S = warp_sum(z);
#pragma unroll
    for (int i = 0; i < NPL; ++i) p[i] = __fdiv_rn(s[i], S);
  }
}

template <int NPL>
__device__ __forceinline__ void aux_lane_bias(const float* bias, int E, int lane,
                                              float (&bb)[NPL]) {
#pragma unroll
  for (int i = 0; i < NPL; ++i) bb[i] = (bias && lane + 32 * i < E) ? bias[lane + 32 * i] : 0.f;
}

template <int NPL>
__global__ void __launch_bounds__(256)
route_aux_stats_kernel(const float* __restrict__ logits, const float* bias,
                       const int32_t* __restrict__ idx, int T, int E, int k, int score_fn,
                       float coeff, float rate, float* __restrict__ Pp, int32_t* __restrict__ Cp,
                       unsigned* ticket, int32_t* __restrict__ counts_out,
                       float* __restrict__ p_mean, float* __restrict__ loss,
                       float* bias_out, int32_t* status) {
  constexpr int TPW = kAuxTokens / kAuxWarps;
  __shared__ float part[kAuxWarps * kMaxExperts];
  __shared__ int cnt[kMaxExperts];
  __shared__ float red[kAuxWarps];
  __shared__ bool last;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  float acc[NPL], bb[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) acc[i] = 0.f;
  aux_lane_bias<NPL>(bias, E, lane, bb);
  // the warp's tokens in order, the next token's logits and selections loaded
  // while the current one is reduced
  const int t0 = blockIdx.x * kAuxTokens + wid * TPW;
  const int n = min(TPW, T - t0);                 // the same for the whole warp
  float v[NPL];
  int ie = 0;
  if (n > 0) {
    aux_load<NPL>(logits + (size_t)t0 * E, E, lane, v);
    if (lane < k) ie = idx[(size_t)t0 * k + lane];
  }
  for (int u = 0; u < n; ++u) {
    float cur[NPL];
#pragma unroll
    for (int i = 0; i < NPL; ++i) cur[i] = v[i];
    const int ce = ie;
    if (u + 1 < n) {
      aux_load<NPL>(logits + (size_t)(t0 + u + 1) * E, E, lane, v);
      if (lane < k) ie = idx[(size_t)(t0 + u + 1) * k + lane];
    }
    float p[NPL], s[NPL], S;
    aux_probs<NPL>(cur, bb, E, score_fn, lane, p, s, S);
#pragma unroll
    for (int i = 0; i < NPL; ++i) acc[i] += p[i];
    if (lane < k) {
      if ((unsigned)ce < (unsigned)E) atomicAdd(&cnt[ce], 1);
      else record_status(status, MOE_ERR_DEVICE_CHECK);
    }
  }
#pragma unroll
  for (int i = 0; i < NPL; ++i)
    if (lane + 32 * i < E) part[wid * kMaxExperts + lane + 32 * i] = acc[i];
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < kAuxWarps; ++w) sum += part[w * kMaxExperts + e];
    Pp[(size_t)blockIdx.x * E + e] = sum;
    Cp[(size_t)blockIdx.x * E + e] = cnt[e];
  }
  // the last block to arrive adds every block's partials
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(ticket, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  // R = blockDim / E threads per expert: thread (r, e) adds blocks r, r + R,
  // ... (eight loads in flight), then expert e adds its R sums in r order
  const int nb = gridDim.x, R = blockDim.x / E;
  if (threadIdx.x < R * E) {
    const int e = threadIdx.x % E, r = threadIdx.x / E;
    constexpr int U = 8;
    float ps = 0.f;
    int c = 0;
    for (int b0 = r; b0 < nb; b0 += U * R) {
      float pv[U];
      int cv[U];
#pragma unroll
      for (int q = 0; q < U; ++q) {
        const int b = b0 + q * R;
        pv[q] = b < nb ? __ldcg(Pp + (size_t)b * E + e) : 0.f;
        cv[q] = b < nb ? __ldcg(Cp + (size_t)b * E + e) : 0;
      }
#pragma unroll
      for (int q = 0; q < U; ++q) {
        ps += pv[q];
        c += cv[q];
      }
    }
    part[threadIdx.x] = ps;
    cnt[threadIdx.x] = c;                          // (E <= blockDim: cnt has room for R E)
  }
  __syncthreads();
  float term = 0.f, ps = 0.f;
  int c = 0;
  const int e = threadIdx.x;
  if (e < E) {
    for (int r = 0; r < R; ++r) {
      ps += part[r * E + e];
      c += cnt[r * E + e];
    }
  }
  __syncthreads();
  if (e < E) {
    const float P = T > 0 ? __fdiv_rn(ps, (float)T) : 0.f;
    const float f = T > 0 ? __fdiv_rn((float)c, (float)((int64_t)T * k)) : 0.f;
    counts_out[e] = c;
    p_mean[e] = P;
    term = f * P;
    if (bias_out) {
      // b + rate * sign(mean load - load), mean load = T k / E (in integers)
      const int64_t d = (int64_t)T * k - (int64_t)E * c;
      const float sgn = d > 0 ? 1.f : d < 0 ? -1.f : 0.f;
      bias_out[e] = __fadd_rn(bias ? bias[e] : 0.f, __fmul_rn(rate, sgn));
    }
  }
  term = warp_sum(term);
  if (lane == 0) red[wid] = term;
  __syncthreads();
  if (threadIdx.x == 0) {
    float tot = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += red[w];
    *loss = coeff * (float)E * tot;
    *ticket = 0u;                                  // ready for the next call
  }
}

// dl[t,:] = dloss * d loss / d l[t,:] with g_e = gscale * counts[e]
// (gscale = dloss coeff E / (T^2 k)): softmax p (g - p.g); sigmoid
// s (1 - s) / S (g - p.g). One warp per token.
template <int NPL>
__global__ void __launch_bounds__(256)
route_aux_dlogits_kernel(const float* __restrict__ logits, const float* __restrict__ bias,
                         const int32_t* __restrict__ counts, int T, int E, int score_fn,
                         float gscale, float* __restrict__ dl) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  float v[NPL], bb[NPL], p[NPL], s[NPL], S;
  aux_load<NPL>(logits + (size_t)t * E, E, lane, v);
  aux_lane_bias<NPL>(bias, E, lane, bb);
  aux_probs<NPL>(v, bb, E, score_fn, lane, p, s, S);
  float g[NPL], pg = 0.f;
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = lane + 32 * i;
    g[i] = e < E ? gscale * (float)counts[e] : 0.f;
    pg += p[i] * g[i];
  }
  pg = warp_sum(pg);
  float* row = dl + (size_t)t * E;
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = lane + 32 * i;
    if (e >= E) continue;
    const float c = g[i] - pg;
    row[e] = score_fn == MOE_SCORE_SOFTMAX ? p[i] * c
                                           : __fdiv_rn(s[i] * (1.f - s[i]), S) * c;
  }
}

// dx[t, h] = bf16(dx[t, h] + sum_e dl[t, e] W_r[e, h]), e in increasing order.
// Block: 64 tokens x 128 columns; warp w takes tokens 8w..8w+7, lane l columns
// 4l..4l+3. Experts in chunks of kDxChunk (8 when E <= 8, else 32): dl^T and
// W_r chunks staged in shared memory, every thread 8 x 4 fp32 accumulators.
constexpr int kDxTokens = 64, kDxCols = 128;

template <int kDxChunk>
__global__ void __launch_bounds__(256)
router_dx_dense_kernel(const float* __restrict__ dl, const float* __restrict__ W_r,
                       __nv_bfloat16* __restrict__ dx, int T, int H, int E) {
  __shared__ __align__(16) float sd[kDxChunk][kDxTokens + 4];
  __shared__ __align__(16) float sw[kDxChunk][kDxCols];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int t0 = blockIdx.x * kDxTokens, h0 = blockIdx.y * kDxCols;
  float acc[8][4];
#pragma unroll
  for (int r = 0; r < 8; ++r)
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[r][q] = 0.f;
  for (int e0 = 0; e0 < E; e0 += kDxChunk) {
    for (int i = threadIdx.x; i < kDxTokens * kDxChunk; i += blockDim.x) {
      const int tt = i / kDxChunk, ee = i % kDxChunk;
      const int t = t0 + tt, e = e0 + ee;
      sd[ee][tt] = (t < T && e < E) ? dl[(size_t)t * E + e] : 0.f;
    }
    for (int i = threadIdx.x; i < kDxChunk * (kDxCols / 4); i += blockDim.x) {
      const int ee = i / (kDxCols / 4), c4 = (i % (kDxCols / 4)) * 4;
      const int e = e0 + ee;
      const float4 v = e < E ? __ldg(reinterpret_cast<const float4*>(W_r + (size_t)e * H + h0 + c4))
                             : make_float4(0.f, 0.f, 0.f, 0.f);
      *reinterpret_cast<float4*>(&sw[ee][c4]) = v;
    }
    __syncthreads();
#pragma unroll 4
    for (int ee = 0; ee < kDxChunk; ++ee) {
      const float4 w = *reinterpret_cast<const float4*>(&sw[ee][lane * 4]);
      const float4 d0 = *reinterpret_cast<const float4*>(&sd[ee][wid * 8]);
      const float4 d1 = *reinterpret_cast<const float4*>(&sd[ee][wid * 8 + 4]);
      const float d[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        acc[r][0] = fmaf(d[r], w.x, acc[r][0]);
        acc[r][1] = fmaf(d[r], w.y, acc[r][1]);
        acc[r][2] = fmaf(d[r], w.z, acc[r][2]);
        acc[r][3] = fmaf(d[r], w.w, acc[r][3]);
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const int t = t0 + wid * 8 + r;
    if (t >= T) break;
    uint2* p = reinterpret_cast<uint2*>(dx + (size_t)t * H + h0 + lane * 4);
    const uint2 v = *p;
    uint2 o;
    o.x = pack_bf16x2(bf16_lo(v.x) + acc[r][0], bf16_hi(v.x) + acc[r][1]);
    o.y = pack_bf16x2(bf16_lo(v.y) + acc[r][2], bf16_hi(v.y) + acc[r][3]);
    *p = o;
  }
}

// A3[t, :] = [hi(dl[t,:]) | hi(dl[t,:]) | mid(dl[t,:])], 3E bf16 columns, with
// hi = bf16(v) and mid = bf16(v - hi); one thread per 8 consecutive experts.
__global__ void __launch_bounds__(256)
aux_split_dl_kernel(const float* __restrict__ dl, __nv_bfloat16* __restrict__ A3, int T, int E) {
  const int per_row = E >> 3;
  const long long n = (long long)T * per_row;
  for (long long v = (long long)blockIdx.x * blockDim.x + threadIdx.x; v < n;
       v += (long long)gridDim.x * blockDim.x) {
    const int t = (int)(v / per_row), e = (int)(v - (long long)t * per_row) << 3;
    const float4* src = reinterpret_cast<const float4*>(dl + (size_t)t * E + e);
    const float4 a = __ldg(src), b = __ldg(src + 1);
    const float f[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    float hi[8], mid[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      hi[q] = __bfloat162float(__float2bfloat16_rn(f[q]));
      mid[q] = f[q] - hi[q];
    }
    const uint4 h = pack8(hi);
    uint4* row = reinterpret_cast<uint4*>(A3 + (size_t)t * 3 * E + e);
    row[0] = h;
    row[E / 8] = h;                                // + E columns
    row[E / 4] = pack8(mid);                       // + 2E columns
  }
}

// B3[h, :] = [hi(W_r[:,h]) | mid(W_r[:,h]) | hi(W_r[:,h])], 3E bf16 columns
// (W_r transposed through a 32 x 32 shared tile).
__global__ void __launch_bounds__(256)
aux_split_wr_kernel(const float* __restrict__ W_r, __nv_bfloat16* __restrict__ B3, int E, int H) {
  __shared__ float tile[32][33];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int h0 = blockIdx.x * 32, e0 = blockIdx.y * 32;
#pragma unroll
  for (int i = 0; i < 4; ++i) tile[ty + 8 * i][tx] = W_r[(size_t)(e0 + ty + 8 * i) * H + h0 + tx];
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int h = h0 + ty + 8 * i;
    const float w = tile[tx][ty + 8 * i];
    const __nv_bfloat16 hi = __float2bfloat16_rn(w);
    const __nv_bfloat16 mid = __float2bfloat16_rn(w - __bfloat162float(hi));
    __nv_bfloat16* row = B3 + (size_t)h * 3 * E + e0 + tx;
    row[0] = hi;
    row[E] = mid;
    row[2 * E] = hi;
  }
}

static int experts_per_lane(int E) { return E <= 32 ? 1 : E <= 64 ? 2 : E <= 128 ? 4 : 8; }

cudaError_t launch_route_aux(const moe_config& c, const float* logits, const float* bias,
                             const int32_t* idx, float coeff, float rate, int32_t* counts,
                             float* p_mean, float* loss, float* bias_out, uint8_t* scratch,
                             cudaStream_t s) {
  const int nb = c.T > 0 ? (c.T + kAuxTokens - 1) / kAuxTokens : 1;
  uint8_t* base = scratch + aux_partial_offset(c);
  float* Pp = reinterpret_cast<float*>(base);
  int32_t* Cp = reinterpret_cast<int32_t*>(base + (size_t)nb * c.E * 4);
  unsigned* ticket = reinterpret_cast<unsigned*>(scratch + kScratchAuxTicket);
  int32_t* status = reinterpret_cast<int32_t*>(scratch + kScratchStatus);
  const int npl = experts_per_lane(c.E);
  auto kern = npl == 1 ? route_aux_stats_kernel<1>
            : npl == 2 ? route_aux_stats_kernel<2>
            : npl == 4 ? route_aux_stats_kernel<4> : route_aux_stats_kernel<8>;
  kern<<<nb, 32 * kAuxWarps, 0, s>>>(logits, bias, idx, c.T, c.E, c.k, c.score_fn, coeff, rate,
                                      Pp, Cp, ticket, counts, p_mean, loss, bias_out, status);
  return cudaGetLastError();
}

cudaError_t launch_route_aux_bwd(const moe_config& c, const void* x, const float* logits,
                                 const float* bias, const float* W_r, const int32_t* counts,
                                 float coeff, float dloss, float* dl, void* dx, float* dW_r,
                                 uint8_t* scratch, cudaStream_t s) {
  if (c.T == 0) return cudaSuccess;                 // nothing to add
  const double gscale = (double)dloss * coeff * c.E / ((double)c.T * c.T * c.k);
  const int npl = experts_per_lane(c.E);
  auto kern = npl == 1 ? route_aux_dlogits_kernel<1>
            : npl == 2 ? route_aux_dlogits_kernel<2>
            : npl == 4 ? route_aux_dlogits_kernel<4> : route_aux_dlogits_kernel<8>;
  kern<<<(c.T + 7) / 8, 256, 0, s>>>(logits, bias, counts, c.T, c.E, c.score_fn, (float)gscale,
                                     dl);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  if (router_on_tensor_cores(c)) {
    // dx on the tensor cores: dl and W_r each as hi + mid bf16 parts; the three
    // products hi.hi + hi.mid + mid.hi (what they leave out is ~2^-16 of
    // |dl| |W_r|, far below the bf16 rounding of dx) as one K = 3E GEMM
    uint8_t* base = scratch + router_split_offset(c);
    auto A3 = reinterpret_cast<__nv_bfloat16*>(base);
    auto B3 = reinterpret_cast<__nv_bfloat16*>(base + ((int64_t)c.T * 3 * c.E * 2 + 255) / 256 * 256);
    long long blocks = ((long long)c.T * (c.E / 8) + 255) / 256;
    if (blocks > (long long)num_sms() * 16) blocks = (long long)num_sms() * 16;
    aux_split_dl_kernel<<<(int)blocks, 256, 0, s>>>(dl, A3, c.T, c.E);
    aux_split_wr_kernel<<<dim3(c.H / 32, c.E / 32), 256, 0, s>>>(W_r, B3, c.E, c.H);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    err = launch_router_dx_tc(c, A3, B3, 3 * c.E, dx,
                              reinterpret_cast<int32_t*>(scratch + kScratchStatus), s);
  } else {
    const dim3 grid((c.T + kDxTokens - 1) / kDxTokens, c.H / kDxCols);
    auto dxp = static_cast<__nv_bfloat16*>(dx);
    if (c.E <= 8)
      router_dx_dense_kernel<8><<<grid, 256, 0, s>>>(dl, W_r, dxp, c.T, c.H, c.E);
    else
      router_dx_dense_kernel<32><<<grid, 256, 0, s>>>(dl, W_r, dxp, c.T, c.H, c.E);
    err = cudaGetLastError();
  }
  if (err != cudaSuccess) return err;
  // every token contributes to every expert's row of dW_r
  return launch_router_wgrad(c, x, nullptr, nullptr, dl, dW_r, scratch, s, true);
}

}  // namespace moe
