// Pieces shared by the grouped-GEMM kernel families (bf16 in grouped_gemm.cu,
// FP8 block-scaled in grouped_gemm_fp8.cu): launch constants, the parameter
// block, the persistent tile scheduler's decode, the SwiGLU arithmetic of the
// epilogues, the output staging layout, and the host-side TMA tensor maps.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace gg {

constexpr int BM = 128;
constexpr int BK = 64;                       // 64 bf16 = one 128-byte swizzle row
constexpr int kThreads = 192;
constexpr int kCtrlBytes = 5120;
constexpr int kBoxBytes = 32 * 32 * 2;           // one 32 x 32 bf16 output box
constexpr int kStageBytes = 3 * kBoxBytes;       // output staging per epilogue warp
constexpr long long kWaitBudget = 4000000000LL;   // clock64 cycles (~2 s)

enum Epi : int { kEpiSwigluFwd = 0, kEpiStore = 1, kEpiSwigluBwd = 2, kEpiWgrad = 3,
                 kEpiStoreF32 = 4, kEpiDgradRouter = 5, kEpiAddBf16 = 6,
                 // the layer with the routing weight inside the expert: FC1 writes
                 // h_s = w_row silu(G) U; the FC2 data gradient scales dh_s by w_row
                 // and writes each row's partial <dh_s, h> for the weight's gradient
                 kEpiSwigluFwdW = 7, kEpiSwigluBwdW = 8 };
constexpr bool swiglu_fwd(int epi) { return epi == kEpiSwigluFwd || epi == kEpiSwigluFwdW; }
constexpr bool swiglu_bwd(int epi) { return epi == kEpiSwigluBwd || epi == kEpiSwigluBwdW; }

struct Params {
  int kgrouped;               // 0: row-grouped, 1: K-grouped
  int G;
  int N;                      // output columns per group (unused by SwiGLU-fwd)
  int K;                      // reduction length (row-grouped)
  int Mw;                     // output rows per group (K-grouped)
  int F;                      // SwiGLU width
  int b_rows;                 // rows of one group in B's 2D view (row-grouped)
  const int32_t* counts;
  const int32_t* offsets;
  __nv_bfloat16* out;
  long long ldo;
  long long out_gstride;      // K-grouped: elements between groups' outputs
  __nv_bfloat16* out2;        // SwiGLU-fwd: h
  long long ldo2;
  const __nv_bfloat16* aux;   // SwiGLU-bwd: GU; add-to-output (kEpiAddBf16): the output
  long long ldaux;            // itself, read before it is overwritten
  int32_t* status;
  int dense_rows;             // > 0: one group of this many rows at row 0 (no counts/offsets),
                              // or, with chunk_rows > 0, that many rows cut into groups of
                              // chunk_rows consecutive rows (the last one shorter)
  int chunk_rows;
  long long part_rows;        // B parts (b_parts > 1) of an MN-major B: part q's rows start
                              // at q * part_rows
  // FC1 data gradient with the router term (kEpiDgradRouter): row r of a
  // routed group g < router_E gains dlogits[token_of[r], g] * W_r[g, :]
  const int32_t* token_of;
  const float* dlogits;
  const float* W_r;
  int router_E;
  int router_T;               // rows of dlogits; a token id outside [0, router_T) adds nothing
  // routing weight inside the expert (kEpiSwigluFwdW / kEpiSwigluBwdW): the
  // weight of every permuted row, and the FC2 data gradient's per-tile partial
  // dot products <dh_s, h> of every row ([R][dw_nt], fp32)
  const float* row_w;
  float* dw_part;
  __nv_bfloat16* h_out;       // SwiGLU-bwd: h rewritten from GU ([rows, F]), or null
  int dw_nt;
  // FP8 block-scaled operands (grouped_gemm_fp8.cu): UE8M0 scale atoms of A
  // ([R/128][sfa_kg]) and of B ([G * sfb_nb][sfb_kg]), fp8_layout.cuh
  const uint8_t* sfa;
  const uint8_t* sfb;
  int sfa_kg;
  int sfb_nb, sfb_kg;
  // and the 1-byte form of the FC1 epilogue's h for FC2 (1 x 128 slices,
  // atoms [R/128][qsf_kg])
  uint8_t* qout;
  uint8_t* qsf;
  int qsf_kg;
  // Tile order: 1 = n-tiles vary fastest, else m-tiles (m-pairs). Weight gradients
  // whose output is taller than wide take n-fastest: the clusters running at
  // once then share the A slice (the group's rows x 256 output rows) and stream
  // B, which is the smaller operand and stays in L2 (Mixtral-sized dW13: the
  // group's dGU is read from DRAM once instead of about four times).
  int n_fast;
  // Paged stash: the row tensors marked in page_ops (kPage*) are pool tensors
  // whose row r is row pages[r / 128] * 128 + r % 128 (every tile and k-block
  // stays inside one 128-row block, so one look-up serves a whole box).
  const int32_t* pages;
  int page_ops;
};

enum PageOps : int {
  kPageA = 1,     // A's rows (row-grouped: the tile's rows; K-grouped: the k-block's)
  kPageB = 2,     // B's k-block rows of a K-grouped launch
  kPageOut = 4,   // the rows the epilogue stores (row-grouped launches)
  kPageAux = 8,   // the SwiGLU backward's GU rows and the rows of h_out
};

__device__ __forceinline__ int page_row(const Params& p, int op, int r) {
  return (p.page_ops & op) ? stash_row(p.pages, r) : r;
}

// Router logits (kEpiStoreF32) multiply each A k-block by the three bf16 parts
// of the fp32 weight, held in B as three consecutive 64-column blocks: one
// stage carries the A block once and the three B blocks.
template <int EPI>
constexpr int b_parts() { return EPI == kEpiStoreF32 ? 3 : 1; }

template <int BN, int STAGES, int BPARTS = 1>
struct Layout {
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE = A_BYTES + BPARTS * B_BYTES;
  static constexpr int TILES = STAGES * STAGE;
  static constexpr int SMEM = TILES + kCtrlBytes + 4 * kStageBytes + 1024;
  static constexpr int TMEM_COLS = 2 * BN;
};

struct Tile {
  int g, mt, nt, nk;
};

__device__ __forceinline__ int find_group(const int* prefix, int G, int tile) {
  int lo = 0, hi = G - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= tile) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ Tile decode(int tile, const int* prefix, const int* mtiles,
                                       const int* cnt, int G, int kgrouped, int K, int NT,
                                       int n_fast) {
  Tile t;
  t.g = find_group(prefix, G, tile);
  const int local = tile - prefix[t.g];
  const int mt = mtiles[t.g];
  if (n_fast) {
    t.nt = local % NT;
    t.mt = local / NT;
  } else {
    t.mt = local % mt;
    t.nt = local / mt;
  }
  t.nk = kgrouped ? (cnt[t.g] + BK - 1) / BK : K / BK;
  return t;
}

// Logistic sigmoid 1 / (1 + e^-z) = 1 / (1 + 2^(-z log2 e)) and SiLU for the
// SwiGLU epilogues, on the special-function unit (a few fp32 ulp; the bf16
// outputs keep 8 significant bits). Large |z| saturate to 0 and 1.
constexpr float kLog2e = 1.4426950408889634f;
__device__ __forceinline__ float sigmoid_f(float z) {
  return ptx::rcp_approx(1.f + ptx::ex2_approx(-kLog2e * z));
}
__device__ __forceinline__ float silu_f(float z) { return z * sigmoid_f(z); }

// SwiGLU backward of 8 consecutive columns. With s = sigmoid(g) and
// silu(g) = g s (h = silu(g) u):
//   dU = dh silu(g),  dG = dh u (s + silu(g) (1 - s))   [= dh u s (1 + g (1 - s))].
// dh: 8 fp32 (tensor-memory bits); g, u: 8 bf16 each. fp32 pairs throughout.
__device__ __forceinline__ void swiglu_bwd8(const uint32_t* dh, const uint4& g, const uint4& u,
                                            uint4& dg, uint4& du) {
  const uint32_t gw[4] = {g.x, g.y, g.z, g.w}, uw[4] = {u.x, u.y, u.z, u.w};
  uint32_t dgw[4], duw[4];
  const uint64_t one = ptx::f2_pack(1.f, 1.f);
  const uint64_t nl2e = ptx::f2_pack(-kLog2e, -kLog2e);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint64_t G = ptx::f2_pack(bf16_lo(gw[j]), bf16_hi(gw[j]));
    const uint64_t U = ptx::f2_pack(bf16_lo(uw[j]), bf16_hi(uw[j]));
    const uint64_t D = ptx::f2_pack(__uint_as_float(dh[2 * j]), __uint_as_float(dh[2 * j + 1]));
    float e0, e1;
    ptx::f2_unpack(ptx::f2_mul(G, nl2e), e0, e1);
    float d0, d1;
    ptx::f2_unpack(ptx::f2_add(ptx::f2_pack(ptx::ex2_approx(e0), ptx::ex2_approx(e1)), one), d0, d1);
    const uint64_t S = ptx::f2_pack(ptx::rcp_approx(d0), ptx::rcp_approx(d1));
    const uint64_t SILU = ptx::f2_mul(G, S);
    const uint64_t DU = ptx::f2_mul(D, SILU);
    const uint64_t T = ptx::f2_fma(SILU, ptx::f2_sub(one, S), S);
    const uint64_t DG = ptx::f2_mul(ptx::f2_mul(D, U), T);
    float a0, a1, b0, b1;
    ptx::f2_unpack(DG, a0, a1);
    ptx::f2_unpack(DU, b0, b1);
    dgw[j] = pack_bf16x2(a0, a1);
    duw[j] = pack_bf16x2(b0, b1);
  }
  dg = make_uint4(dgw[0], dgw[1], dgw[2], dgw[3]);
  du = make_uint4(duw[0], duw[1], duw[2], duw[3]);
}

// h = bf16(silu(g) u), times the row's routing weight when it sits inside the
// expert, of 8 columns from the stored bf16 G and U: the forward epilogue's
// arithmetic exactly, so the h recomputed in the backward (fine-grained
// recompute of the activation function) equals the forward's bit for bit.
template <bool WGT>
__device__ __forceinline__ uint4 swiglu_h8(const uint4& g, const uint4& u, float rwt) {
  float gr[8], ur[8], hf[8];
  unpack8(g, gr);
  unpack8(u, ur);
#pragma unroll
  for (int i = 0; i < 8; ++i) hf[i] = WGT ? silu_f(gr[i]) * ur[i] * rwt : silu_f(gr[i]) * ur[i];
  return pack8(hf);
}

// The same with the routing weight inside the expert: dh_s (the accumulator)
// is the gradient of h_s = w h, so dh = w dh_s, and the weight's gradient gains
// <dh_s, h> with h = silu(g) u recomputed here (added to `dot` in column order).
__device__ __forceinline__ void swiglu_bwd8_w(const uint32_t* dhs, const uint4& g, const uint4& u,
                                              float w, uint4& dg, uint4& du, float& dot) {
  const uint32_t gw[4] = {g.x, g.y, g.z, g.w}, uw[4] = {u.x, u.y, u.z, u.w};
  uint32_t dgw[4], duw[4];
  const uint64_t one = ptx::f2_pack(1.f, 1.f);
  const uint64_t nl2e = ptx::f2_pack(-kLog2e, -kLog2e);
  const uint64_t W2v = ptx::f2_pack(w, w);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint64_t G = ptx::f2_pack(bf16_lo(gw[j]), bf16_hi(gw[j]));
    const uint64_t U = ptx::f2_pack(bf16_lo(uw[j]), bf16_hi(uw[j]));
    const uint64_t Ds = ptx::f2_pack(__uint_as_float(dhs[2 * j]), __uint_as_float(dhs[2 * j + 1]));
    float e0, e1;
    ptx::f2_unpack(ptx::f2_mul(G, nl2e), e0, e1);
    float d0, d1;
    ptx::f2_unpack(ptx::f2_add(ptx::f2_pack(ptx::ex2_approx(e0), ptx::ex2_approx(e1)), one), d0, d1);
    const uint64_t S = ptx::f2_pack(ptx::rcp_approx(d0), ptx::rcp_approx(d1));
    const uint64_t SILU = ptx::f2_mul(G, S);
    float p0, p1;
    ptx::f2_unpack(ptx::f2_mul(Ds, ptx::f2_mul(SILU, U)), p0, p1);
    dot += p0;
    dot += p1;
    const uint64_t D = ptx::f2_mul(Ds, W2v);
    const uint64_t DU = ptx::f2_mul(D, SILU);
    const uint64_t T = ptx::f2_fma(SILU, ptx::f2_sub(one, S), S);
    const uint64_t DG = ptx::f2_mul(ptx::f2_mul(D, U), T);
    float a0, a1, b0, b1;
    ptx::f2_unpack(DG, a0, a1);
    ptx::f2_unpack(DU, b0, b1);
    dgw[j] = pack_bf16x2(a0, a1);
    duw[j] = pack_bf16x2(b0, b1);
  }
  dg = make_uint4(dgw[0], dgw[1], dgw[2], dgw[3]);
  du = make_uint4(duw[0], duw[1], duw[2], duw[3]);
}

// Output staging: every epilogue warp owns kStageBytes of shared memory (1024-
// byte aligned), stored to global memory by TMA (coalesced, asynchronous). The
// SwiGLU epilogues stage up to three 32 x 32 bf16 boxes with the 64-byte
// swizzle of their output maps (16-byte chunk j of row r at slot j ^ ((r>>1)&3));
// the plain-store epilogues one 32 x 64 box with the 128-byte swizzle (chunk j
// of row r at slot j ^ (r & 7)). Either way the 32 lanes' row writes hit
// distinct banks.

__device__ __forceinline__ void stage_row(uint8_t* stage, int box, int lane, const uint4 (&v)[4]) {
  uint8_t* row = stage + box * kBoxBytes + lane * 64;
  const int sw = (lane >> 1) & 3;
#pragma unroll
  for (int j = 0; j < 4; ++j) *reinterpret_cast<uint4*>(row + ((j ^ sw) << 4)) = v[j];
}

__device__ __forceinline__ void pack_slice(const uint32_t (&r)[32], uint4 (&o)[4]) {
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    float f[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) f[i] = __uint_as_float(r[v * 8 + i]);
    o[v] = pack8(f);
  }
}


// ----------------------------------------------------------------- host side
static inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// 2D bf16 view [outer rows, inner columns] with a {64, box_outer} box and
// 128-byte swizzle; elements outside the view read as zero.
static inline bool make_map(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer,
                     uint32_t box_outer) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {64, box_outer};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Output view [outer rows, inner columns] for TMA stores of 32 x 32 boxes with
// the 64-byte swizzle of the epilogue's staging layout.
static inline bool make_out_map(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 output view for TMA stores of 32-row x 64-column boxes (128-byte rows,
// 128-byte swizzle): the plain-store epilogues.
static inline bool make_out_map_w64(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {64, 32};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2D view of 1-byte (E4M3) elements [outer rows, inner columns] with a 128 x
// box_outer box (128 or 256 rows) and the 128-byte swizzle (one box row = one
// 128-byte swizzle row).
static inline bool make_map_u8(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer,
                               uint32_t box_outer = 128) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner};
  cuuint32_t box[2] = {128, box_outer};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// An MN-major operand of 1-byte elements [outer rows, inner columns] seen as
// 128-column chunks: dims {128 columns of a chunk, rows, chunk index} with
// strides {inner bytes per row, 128 bytes per chunk}, a {128, 128, chunks} box
// and the 128-byte swizzle. One load brings `chunks` consecutive 128-column
// slices of 128 rows, each slice 16 KB after the previous in shared memory --
// the layout of `chunks` separate 2D boxes, in one request.
static inline bool make_map_u8_chunks(CUtensorMap* m, const void* ptr, uint64_t inner,
                                      uint64_t outer, uint32_t chunks) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn || inner % 128) return false;
  cuuint64_t dims[3] = {128, outer, inner / 128};
  cuuint64_t strides[2] = {inner, 128};
  cuuint32_t box[3] = {128, 128, chunks};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The bf16 form of the chunked view: dims {64 columns of a chunk, rows, chunk
// index}, strides {inner * 2 bytes per row, 128 bytes per chunk}, a {64, 64,
// chunks} box (64 rows = one bf16 k-block): `chunks` 64-column slices of 64 rows,
// 8 KB apart in shared memory, in one request.
static inline bool make_map_chunks(CUtensorMap* m, const void* ptr, uint64_t inner,
                                   uint64_t outer, uint32_t chunks) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn || inner % 64) return false;
  cuuint64_t dims[3] = {64, outer, inner / 64};
  cuuint64_t strides[2] = {inner * 2, 128};
  cuuint32_t box[3] = {64, 64, chunks};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 output view for TMA stores of 32 x 32 boxes (128-byte rows, 128-byte swizzle).
static inline bool make_out_map_f32(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 4};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(ptr), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}


static inline Params base_params(const moe_config& c, const int32_t* counts, const int32_t* offsets,
                          int32_t* status) {
  Params p{};
  p.G = c.E + c.n_shared;
  p.F = c.F;
  p.counts = counts;
  p.offsets = offsets;
  p.status = status;
  return p;
}


}  // namespace gg
}  // namespace moe
