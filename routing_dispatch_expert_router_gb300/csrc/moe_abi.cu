// The library's C entry points: argument checks, buffer sizes, and the layer
// composition. Every compute step runs in this library's own kernels; nothing
// here falls back to another implementation.
#include <math.h>
#include <stdio.h>

#include "common.cuh"
#include "fp8_layout.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace moe {

int64_t capacity_rows(const moe_config& c) {
  if (!(c.capacity_factor > 0.f)) return 0;
  const double cf = (double)c.capacity_factor;
  const int64_t cap = (int64_t)ceil(cf * (double)c.T * (double)c.k / (double)c.E);
  return (cap + c.row_align - 1) / c.row_align * c.row_align;
}

int64_t rows_max(const moe_config& c) {
  const int64_t a = c.row_align;
  const int64_t shared = (int64_t)c.n_shared * (((int64_t)c.T + a - 1) / a * a);
  const int64_t C = capacity_rows(c);
  if (C > 0) return (int64_t)c.E * C + shared;
  return (int64_t)c.T * c.k + (int64_t)c.E * (a - 1) + shared;
}

int n_chunks(const moe_config& c) { return (c.T + kChunkTokens - 1) / kChunkTokens; }

int num_sms() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

static int64_t align256(int64_t v) { return (v + 255) / 256 * 256; }

int64_t permute_scratch_bytes(const moe_config& c) {
  return align256((int64_t)kScratchHist + (int64_t)n_chunks(c) * c.E * 4 + 256);
}

int64_t router_split_offset(const moe_config& c) { return permute_scratch_bytes(c); }

int64_t aux_partial_offset(const moe_config& c) {
  return permute_scratch_bytes(c) + router_split_bytes(c);
}

static int64_t base_scratch_bytes(const moe_config& c) {
  return aux_partial_offset(c) + aux_partial_bytes(c);
}

static bool is_fp8(const moe_config& c) {
  return c.dtype == MOE_DTYPE_FP8_E4M3_BLOCK || c.dtype == MOE_DTYPE_MXFP8;
}

// The FP8 modes' region of scratch, in order: the E4M3 weights (the MXFP8
// mode's second, data-gradient form after each) with their scale atoms for
// both orientations, the 1-byte activations (x_perm, h, dO, dGU in slices
// along each row) with their atoms, and the 1-byte weight-gradient operands
// (dO, h, dGU, x_perm in slices along the tokens) with theirs.
static int64_t fp8_region(const moe_config& c, Fp8Scratch* f, uint8_t* p) {
  constexpr int kRegions = 24;
  const int64_t G = c.E + c.n_shared, R = rows_max(c), H = c.H, F = c.F;
  const bool mx = c.dtype == MOE_DTYPE_MXFP8;
  auto sfb = [mx](int64_t rows, int64_t K) { return f8::sf_bytes_of(rows, K, mx); };
  const int64_t sizes[kRegions] = {
      G * 2 * F * H, mx ? G * 2 * F * H : 0, sfb(G * 2 * F, H), sfb(G * H, 2 * F),
      G * H * F,     mx ? G * H * F : 0,     sfb(G * H, F),     sfb(G * F, H),
      R * H, sfb(R, H), R * F, sfb(R, F),
      R * H, sfb(R, H), R * 2 * F, sfb(R, 2 * F),
      R * H, sfb(H, R), R * F, sfb(F, R),
      R * 2 * F, sfb(2 * F, R), R * H, sfb(H, R)};
  uint8_t* ptrs[kRegions];
  int64_t off = 0;
  for (int i = 0; i < kRegions; ++i) {
    ptrs[i] = p ? p + off : nullptr;
    off += align256(sizes[i]);
  }
  if (f) {
    f->mx = mx;
    f->W13q = ptrs[0];
    f->W13qd = mx ? ptrs[1] : ptrs[0];
    f->W13sf = ptrs[2];
    f->W13sft = ptrs[3];
    f->W2q = ptrs[4];
    f->W2qd = mx ? ptrs[5] : ptrs[4];
    f->W2sf = ptrs[6];
    f->W2sft = ptrs[7];
    f->xq = ptrs[8];
    f->xsf = ptrs[9];
    f->hq = ptrs[10];
    f->hsf = ptrs[11];
    f->dOq = ptrs[12];
    f->dOsf = ptrs[13];
    f->dGq = ptrs[14];
    f->dGsf = ptrs[15];
    f->cHq = ptrs[16];
    f->cHsf = ptrs[17];
    f->bFq = ptrs[18];
    f->bFsf = ptrs[19];
    f->d2Fq = ptrs[20];
    f->d2Fsf = ptrs[21];
    f->aHq = ptrs[22];
    f->aHsf = ptrs[23];
  }
  return off;
}

// The region of the layer with the routing weight inside the expert: the
// weight of every permuted row, then the FC2 data gradient's partial dot
// products per row and n-tile.
static int64_t reorder_offset(const moe_config& c) {
  int64_t b = base_scratch_bytes(c);
  if (is_fp8(c)) b += fp8_region(c, nullptr, nullptr);
  return b;
}

static int64_t reorder_bytes(const moe_config& c) {
  if (!c.weights_in_expert) return 0;
  const int64_t R = rows_max(c);
  return align256(R * 4) + align256(R * dw_tiles(c) * 4);
}

ReorderScratch reorder_scratch(const moe_config& c, void* scratch) {
  uint8_t* p = static_cast<uint8_t*>(scratch) + reorder_offset(c);
  ReorderScratch r;
  r.row_w = reinterpret_cast<float*>(p);
  r.dw_part = reinterpret_cast<float*>(p + align256(rows_max(c) * 4));
  return r;
}

int64_t scratch_bytes(const moe_config& c) { return reorder_offset(c) + reorder_bytes(c); }

Fp8Scratch fp8_scratch(const moe_config& c, void* scratch) {
  Fp8Scratch f;
  fp8_region(c, &f, static_cast<uint8_t*>(scratch) + base_scratch_bytes(c));
  return f;
}

moe_status check_config(const moe_config* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (c->T < 0 || c->H < 128 || c->F < 128 || c->E < 1 || c->k < 1) return MOE_ERR_INVALID_ARG;
  if (c->H % 128 || c->F % 128) return MOE_ERR_INVALID_ARG;
  if (c->E > kMaxExperts || c->k > kMaxK || c->k > c->E) return MOE_ERR_INVALID_ARG;
  if (c->n_shared < 0 || c->n_shared > 4) return MOE_ERR_INVALID_ARG;
  if (c->score_fn != MOE_SCORE_SOFTMAX && c->score_fn != MOE_SCORE_SIGMOID)
    return MOE_ERR_INVALID_ARG;
  if (c->n_groups < 1 || c->n_groups > 32 || c->E % c->n_groups) return MOE_ERR_INVALID_ARG;
  if (c->topk_groups < 1 || c->topk_groups > c->n_groups) return MOE_ERR_INVALID_ARG;
  if (c->n_groups > 1 && c->topk_groups * (c->E / c->n_groups) < c->k) return MOE_ERR_INVALID_ARG;
  if (c->group_score != MOE_GROUP_TOP2_SUM && c->group_score != MOE_GROUP_MAX)
    return MOE_ERR_INVALID_ARG;
  if (!(c->capacity_factor >= 0.f) || !isfinite(c->capacity_factor)) return MOE_ERR_INVALID_ARG;
  if (!isfinite(c->route_scale)) return MOE_ERR_INVALID_ARG;
  if (c->row_align < 128 || c->row_align % 128) return MOE_ERR_INVALID_ARG;
  if (c->dtype != MOE_DTYPE_BF16 && !is_fp8(*c)) return MOE_ERR_INVALID_ARG;
  if (is_fp8(*c) && (c->n_shared != 0 || c->H % 256 || c->F % 256))
    return MOE_ERR_UNSUPPORTED;
  if (c->weights_in_expert != 0 && c->weights_in_expert != 1) return MOE_ERR_INVALID_ARG;
  if (c->recompute_h != 0 && c->recompute_h != 1) return MOE_ERR_INVALID_ARG;
  if (c->stash_pool_pages < 0 || ((int64_t)c->stash_pool_pages + 1) * 128 >= (1LL << 31))
    return MOE_ERR_INVALID_ARG;
  if (c->weights_in_expert && c->dtype != MOE_DTYPE_BF16) return MOE_ERR_UNSUPPORTED;
  if ((int64_t)c->T * c->k >= (1LL << 31) || rows_max(*c) >= (1LL << 31))
    return MOE_ERR_INVALID_ARG;
  if ((int64_t)c->E * 2 * c->F >= (1LL << 31) || (int64_t)(c->E + c->n_shared) * c->H >= (1LL << 31))
    return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

int64_t stash_rows(const moe_config& c, const StashMap& sm) {
  return sm.pages ? sm.rows : rows_max(c);
}

static bool al16(const void* p) { return p && ((uintptr_t)p & 15u) == 0; }
static bool al16_or_null(const void* p) { return !p || ((uintptr_t)p & 15u) == 0; }
static bool al4(const void* p) { return p && ((uintptr_t)p & 3u) == 0; }
// Token-indexed buffers may be NULL when the batch is empty (T == 0).
static bool tok16(const moe_config* c, const void* p) { return (c->T == 0 && !p) || al16(p); }
static bool tok4(const moe_config* c, const void* p) { return (c->T == 0 && !p) || al4(p); }

static moe_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return MOE_OK;
  if (e == cudaErrorInvalidValue) return MOE_ERR_INVALID_ARG;
  return MOE_ERR_CUDA;
}

static int32_t* status_word(void* scratch) {
  return reinterpret_cast<int32_t*>(static_cast<uint8_t*>(scratch) + kScratchStatus);
}

// Runs the bounded mbarrier wait that every grouped-GEMM role uses on a barrier
// that nothing ever completes: the wait gives up after `budget` clock64 cycles
// and records MOE_ERR_TIMEOUT in the status word, exactly as a stalled GEMM
// pipeline would.
__global__ void bounded_wait_check_kernel(int32_t* status, long long budget) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  const uint32_t b = ptx::smem_u32(&bar);
  ptx::mbar_init(b, 1);
  ptx::fence_mbar_init();
  if (!ptx::mbar_wait(b, 0, budget, nullptr)) record_status(status, MOE_ERR_TIMEOUT);
}

}  // namespace moe

using namespace moe;

#define MOE_TRY(expr)                    \
  do {                                   \
    moe_status _s = (expr);              \
    if (_s != MOE_OK) return _s;         \
  } while (0)

#define MOE_CUDA(expr)                   \
  do {                                   \
    cudaError_t _e = (expr);             \
    if (_e != cudaSuccess) return cuda_status(_e); \
  } while (0)

#define MOE_REQUIRE(cond)                \
  do {                                   \
    if (!(cond)) return MOE_ERR_INVALID_ARG; \
  } while (0)

// The paged stash of a layer (cfg->stash_pool_pages > 0): its page table and
// the pool's row count; the layer's own buffers otherwise.
static moe_status stash_of(const moe_config* cfg, const moe_fwd_state* st, StashMap* sm) {
  *sm = StashMap();
  if (cfg->stash_pool_pages == 0) return MOE_OK;
  MOE_REQUIRE(al4(st->stash_table) && al4(st->stash_top));
  sm->pages = st->stash_table;
  sm->rows = ((int64_t)cfg->stash_pool_pages + 1) * 128;
  return MOE_OK;
}

// The bf16 expert weights: read by the bf16 GEMMs; in the FP8 modes only by the
// weight quantisation (moe_quantize_weights), so they may be NULL there.
static bool weights_ok(const moe_config* cfg, const void* W13, const void* W2) {
  return is_fp8(*cfg) ? (al16_or_null(W13) && al16_or_null(W2)) : (al16(W13) && al16(W2));
}

// The per-stage entry points take the layer's own rows_max-row buffers; a
// paged stash (whose pool tensors have fewer rows) runs through the layer calls.
static moe_status own_buffers(const moe_config* cfg) {
  if (!cfg) return MOE_ERR_INVALID_ARG;
  return cfg->stash_pool_pages > 0 ? MOE_ERR_UNSUPPORTED : MOE_OK;
}

// The stage bodies, shared by the per-stage entry points (the layer's own
// buffers) and by moe_layer_fwd / moe_layer_bwd (which may keep the stashed
// rows in pool pages).
static moe_status permute_impl(const moe_config* cfg, const void* x, const int32_t* idx, int32_t* counts,
                       int32_t* offsets, int32_t* row_of, int32_t* token_of, int32_t* sel_offsets,
                       int32_t* sel_tokens, void* x_perm, void* scratch, void* stream,
    const StashAlloc* alloc) {
  MOE_TRY(check_config(cfg));
  MOE_REQUIRE(tok16(cfg, x) && tok4(cfg, idx) && al4(counts) && al4(offsets) && tok4(cfg, row_of));
  MOE_REQUIRE(al4(token_of) && al4(sel_offsets) && tok4(cfg, sel_tokens) && al16(x_perm));
  MOE_REQUIRE(al16(scratch));
  Fp8Scratch q;
  const bool fp8 = is_fp8(*cfg);
  if (fp8) q = fp8_scratch(*cfg, scratch);
  cudaStream_t s = (cudaStream_t)stream;
  // x_perm's E4M3 form (1x128, or 1x32 for MXFP8) is written by the scatter itself
  MOE_CUDA(launch_permute(*cfg, x, idx, counts, offsets, row_of, token_of, sel_offsets,
                          sel_tokens, x_perm, static_cast<uint8_t*>(scratch), s,
                          fp8 ? &q : nullptr, alloc));
  return MOE_OK;
}

static moe_status ffn_fwd_impl(const moe_config* cfg, const void* x_perm, const int32_t* counts,
                               const int32_t* offsets, const void* W13, const void* W2, void* GU,
                               void* h, void* y_perm, void* scratch, void* stream,
    const StashMap& sm) {
  MOE_TRY(check_config(cfg));
  MOE_REQUIRE(al16(x_perm) && al4(counts) && al4(offsets) && weights_ok(cfg, W13, W2));
  MOE_REQUIRE(al16(GU) && al16(h) && al16(y_perm) && al16(scratch));
  cudaStream_t s = (cudaStream_t)stream;
  int32_t* st = status_word(scratch);
  if (is_fp8(*cfg)) {
    // the E4M3 weights are the ones moe_quantize_weights left in scratch, the
    // E4M3 x_perm the one moe_permute wrote there with the bf16 rows; h's
    // E4M3 form comes out of the FC1 epilogue
    const Fp8Scratch q = fp8_scratch(*cfg, scratch);
    MOE_CUDA(launch_ffn_fc1_fp8(*cfg, q.xq, q.xsf, counts, offsets, q.W13q, q.W13sf, GU, h, q.hq,
                                q.hsf, st, s, sm));
    MOE_CUDA(launch_ffn_fc2_fp8(*cfg, q.hq, q.hsf, counts, offsets, q.W2q, q.W2sf, y_perm, st, s,
                                sm));
    return MOE_OK;
  }
  MOE_CUDA(launch_ffn_fc1(*cfg, x_perm, counts, offsets, W13, GU, h, st, s, nullptr, sm));
  MOE_CUDA(launch_ffn_fc2(*cfg, h, counts, offsets, W2, y_perm, st, s, sm));
  return MOE_OK;
}

static moe_status unpermute_impl(const moe_config* cfg, const void* y_perm, const int32_t* row_of,
                         const float* w, const int32_t* offsets, void* out, void* stream,
    const int32_t* pages) {
  MOE_TRY(check_config(cfg));
  MOE_REQUIRE(al16(y_perm) && tok4(cfg, row_of) && al4(offsets) && tok16(cfg, out));
  MOE_REQUIRE(w == nullptr || al4(w));
  MOE_CUDA(launch_unpermute(*cfg, y_perm, row_of, w, offsets, out, (cudaStream_t)stream, pages));
  return MOE_OK;
}

static moe_status unpermute_bwd_impl(const moe_config* cfg, const void* dY, const void* y_perm,
                             const int32_t* row_of, const float* w, const int32_t* counts,
                             const int32_t* offsets, void* dO_perm, float* dw, void* scratch,
                             void* stream,
    const int32_t* pages) {
  MOE_TRY(check_config(cfg));
  MOE_REQUIRE(tok16(cfg, dY) && al16(y_perm) && tok4(cfg, row_of) && tok4(cfg, w) && al4(counts));
  MOE_REQUIRE(al4(offsets) && al16(dO_perm) && tok4(cfg, dw) && al16(scratch));
  uint8_t* dOq = nullptr;
  uint8_t* dOsf = nullptr;
  Fp8Scratch q;
  const bool fp8 = is_fp8(*cfg);
  if (fp8) q = fp8_scratch(*cfg, scratch);
  if (fp8) {                          // dO's E4M3 form written by the scatter itself
    dOq = q.dOq;
    dOsf = q.dOsf;
  }
  cudaStream_t s = (cudaStream_t)stream;
  MOE_CUDA(launch_unpermute_bwd(*cfg, dY, y_perm, row_of, w, counts, offsets, dO_perm, dw, s, dOq,
                                dOsf, pages));
  return MOE_OK;
}

static moe_status ffn_dgrad_impl(const moe_config* cfg, const void* dO_perm, const void* GU,
                                 void* h, const int32_t* counts, const int32_t* offsets,
                                 const int32_t* token_of, const float* dlogits, const float* W_r,
                                 const void* W13, const void* W2, void* dGU, void* dX_perm,
                                 void* scratch, void* stream,
    const StashMap& sm) {
  MOE_TRY(check_config(cfg));
  MOE_REQUIRE(al16(dO_perm) && al16(GU) && al4(counts) && al4(offsets) && al4(token_of));
  MOE_REQUIRE(tok4(cfg, dlogits) && al16(W_r) && weights_ok(cfg, W13, W2) && al16(dGU));
  MOE_REQUIRE(al16(dX_perm) && al16(scratch) && (h == nullptr || al16(h)));
  cudaStream_t s = (cudaStream_t)stream;
  int32_t* st = status_word(scratch);
  if (is_fp8(*cfg)) {
    const Fp8Scratch q = fp8_scratch(*cfg, scratch);
    const int G = cfg->E + cfg->n_shared;
    const int64_t R = rows_max(*cfg);
    // dO_perm's E4M3 form is the one moe_unpermute_bwd wrote into scratch;
    // the weights in their data-gradient forms
    MOE_CUDA(launch_ffn_fc2_dgrad_fp8(*cfg, q.dOq, q.dOsf, counts, offsets, q.W2qd, q.W2sft, GU,
                                      dGU, st, s, h, sm));
    // dGU's row form for FC1's data gradient and its column form for the
    // weight gradient, from one read
    MOE_CUDA(launch_quant_rows_cols8(dGU, q.dGq, q.dGsf, q.d2Fq, q.d2Fsf, offsets, counts, G, R,
                                     2 * cfg->F, s, q.mx));
    MOE_CUDA(launch_ffn_fc1_dgrad_fp8(*cfg, q.dGq, q.dGsf, counts, offsets, q.W13qd, q.W13sft,
                                      token_of, dlogits, W_r, dX_perm, st, s));
    return MOE_OK;
  }
  MOE_CUDA(launch_ffn_fc2_dgrad(*cfg, dO_perm, counts, offsets, W2, GU, dGU, st, s, nullptr,
                                nullptr, h, sm));
  MOE_CUDA(launch_ffn_fc1_dgrad(*cfg, dGU, counts, offsets, W13, token_of, dlogits, W_r, dX_perm,
                                st, s));
  return MOE_OK;
}

static moe_status ffn_wgrad_impl(const moe_config* cfg, const void* dO_perm, const void* x_perm,
                                 const void* h, const void* dGU, const int32_t* counts,
                                 const int32_t* offsets, void* dW13, void* dW2, void* scratch,
                                 void* stream,
    const StashMap& sm) {
  MOE_TRY(check_config(cfg));
  MOE_REQUIRE(al16(dO_perm) && al16(x_perm) && al16(h) && al16(dGU) && al4(counts));
  MOE_REQUIRE(al4(offsets) && al16(dW13) && al16(dW2) && al16(scratch));
  cudaStream_t s = (cudaStream_t)stream;
  int32_t* st = status_word(scratch);
  if (is_fp8(*cfg)) {
    // both operands in slices along each expert's tokens (128x1, or 32x1 for
    // MXFP8; E4M3 codes and scale atoms), multiplied on the block-scaled FP8
    // tensor cores
    const Fp8Scratch q = fp8_scratch(*cfg, scratch);
    const int G = cfg->E + cfg->n_shared;
    const int64_t R = rows_max(*cfg);
    const int H = cfg->H, F = cfg->F;
    MOE_CUDA(launch_quant_cols8(dO_perm, q.cHq, q.cHsf, offsets, counts, G, R, H, s, q.mx));
    MOE_CUDA(launch_quant_cols8(h, q.bFq, q.bFsf, offsets, counts, G, R, F, s, q.mx, sm.pages));
    MOE_CUDA(launch_ffn_wgrad_fc2_fp8(*cfg, q.cHq, q.cHsf, q.bFq, q.bFsf, counts, offsets, dW2,
                                      st, s));
    // (dGU's column form is the one moe_grouped_ffn_dgrad left in scratch)
    MOE_CUDA(launch_quant_cols8(x_perm, q.aHq, q.aHsf, offsets, counts, G, R, H, s, q.mx,
                                sm.pages));
    MOE_CUDA(launch_ffn_wgrad_fc1_fp8(*cfg, q.d2Fq, q.d2Fsf, q.aHq, q.aHsf, counts, offsets, dW13,
                                      st, s));
    return MOE_OK;
  }
  MOE_CUDA(launch_ffn_wgrad_fc2(*cfg, dO_perm, h, counts, offsets, dW2, st, s, sm));
  MOE_CUDA(launch_ffn_wgrad_fc1(*cfg, dGU, x_perm, counts, offsets, dW13, st, s, sm));
  return MOE_OK;
}

static moe_status ffn_fwd_reordered_impl(const moe_config* cfg, const void* x_perm,
                                         const int32_t* counts, const int32_t* offsets,
                                         const int32_t* token_of, const int32_t* row_of,
                                         const float* w, const void* W13, const void* W2,
                                         void* GU, void* h, void* y_perm, void* scratch,
                                         void* stream,
    const StashMap& sm) {
  MOE_TRY(check_config(cfg));
  if (!cfg->weights_in_expert) return MOE_ERR_INVALID_ARG;
  MOE_REQUIRE(al16(x_perm) && al4(counts) && al4(offsets) && al4(token_of) && tok4(cfg, row_of));
  MOE_REQUIRE(tok4(cfg, w) && al16(W13) && al16(W2) && al16(GU) && al16(h) && al16(y_perm));
  MOE_REQUIRE(al16(scratch));
  cudaStream_t s = (cudaStream_t)stream;
  int32_t* st = status_word(scratch);
  const ReorderScratch rs = reorder_scratch(*cfg, scratch);
  MOE_CUDA(launch_row_weights(*cfg, token_of, row_of, w, offsets, rs.row_w, s));
  MOE_CUDA(launch_ffn_fc1(*cfg, x_perm, counts, offsets, W13, GU, h, st, s, rs.row_w, sm));
  MOE_CUDA(launch_ffn_fc2(*cfg, h, counts, offsets, W2, y_perm, st, s, sm));
  return MOE_OK;
}

static moe_status ffn_dgrad_reordered_impl(const moe_config* cfg, const void* dO_perm,
                                           const void* GU, void* h, const int32_t* counts,
                                           const int32_t* offsets, const int32_t* token_of,
                                           const int32_t* row_of, const float* logits,
                                           const int32_t* idx, const float* w, const float* W_r,
                                           const void* W13, const void* W2, void* dGU,
                                           void* dX_perm, float* dw, float* dlogits,
                                           void* scratch, void* stream,
    const StashMap& sm) {
  MOE_TRY(check_config(cfg));
  if (!cfg->weights_in_expert) return MOE_ERR_INVALID_ARG;
  MOE_REQUIRE(al16(dO_perm) && al16(GU) && al4(counts) && al4(offsets) && al4(token_of));
  MOE_REQUIRE(tok4(cfg, row_of) && tok4(cfg, logits) && tok4(cfg, idx) && tok4(cfg, w));
  MOE_REQUIRE(al16(W_r) && al16(W13) && al16(W2) && al16(dGU) && al16(dX_perm));
  MOE_REQUIRE(tok4(cfg, dw) && tok4(cfg, dlogits) && al16(scratch));
  MOE_REQUIRE(h == nullptr || al16(h));
  cudaStream_t s = (cudaStream_t)stream;
  int32_t* st = status_word(scratch);
  const ReorderScratch rs = reorder_scratch(*cfg, scratch);
  MOE_CUDA(launch_ffn_fc2_dgrad(*cfg, dO_perm, counts, offsets, W2, GU, dGU, st, s, rs.row_w,
                                rs.dw_part, h, sm));
  if (cfg->T > 0) {
    MOE_CUDA(launch_dw_reduce(*cfg, rs.dw_part, row_of, dw, s));
    MOE_CUDA(launch_route_bwd(*cfg, logits, idx, w, dw, dlogits, s));
  }
  MOE_CUDA(launch_ffn_fc1_dgrad(*cfg, dGU, counts, offsets, W13, token_of, dlogits, W_r, dX_perm,
                                st, s));
  return MOE_OK;
}

extern "C" {

moe_status moe_query_sizes(const moe_config* cfg, moe_sizes* out) {
  MOE_TRY(check_config(cfg));
  MOE_REQUIRE(out);
  out->rows_max = rows_max(*cfg);
  out->groups = cfg->E + cfg->n_shared;
  out->capacity = capacity_rows(*cfg);
  out->scratch_bytes = scratch_bytes(*cfg);
  out->stash_table_len = rows_max(*cfg) / 128 + 2;
  return MOE_OK;
}

moe_status moe_route(const moe_config* cfg, const void* x, const float* W_r, const float* bias,
                     float* logits, int32_t* idx, float* w, void* scratch, void* stream) {
  MOE_TRY(check_config(cfg));
  MOE_REQUIRE(tok16(cfg, x) && al16(W_r) && tok4(cfg, logits) && tok4(cfg, idx) && tok4(cfg, w));
  MOE_REQUIRE(bias == nullptr || al4(bias));
  MOE_REQUIRE(al16(scratch));
  if (cfg->T == 0) return MOE_OK;
  MOE_CUDA(launch_route(*cfg, x, W_r, bias, logits, idx, w, static_cast<uint8_t*>(scratch),
                        (cudaStream_t)stream));
  return MOE_OK;
}

moe_status moe_route_replay(const moe_config* cfg, const void* x, const float* W_r,
                            const float* bias, const int32_t* idx, float* logits, float* w,
                            void* scratch, void* stream) {
  MOE_TRY(check_config(cfg));
  MOE_REQUIRE(tok16(cfg, x) && al16(W_r) && tok4(cfg, logits) && tok4(cfg, idx) && tok4(cfg, w));
  MOE_REQUIRE(bias == nullptr || al4(bias));
  MOE_REQUIRE(al16(scratch));
  if (cfg->T == 0) return MOE_OK;
  MOE_CUDA(launch_route_replay(*cfg, x, W_r, bias, idx, logits, w,
                               static_cast<uint8_t*>(scratch), (cudaStream_t)stream));
  return MOE_OK;
}

moe_status moe_route_aux(const moe_config* cfg, const float* logits, const float* bias,
                         const int32_t* idx, float coeff, float bias_rate, int32_t* sel_counts,
                         float* p_mean, float* loss, float* bias_out, void* scratch,
                         void* stream) {
  MOE_TRY(check_config(cfg));
  MOE_REQUIRE(tok4(cfg, logits) && tok4(cfg, idx) && al4(sel_counts) && al4(p_mean) && al4(loss));
  MOE_REQUIRE((bias == nullptr || al4(bias)) && (bias_out == nullptr || al4(bias_out)));
  MOE_REQUIRE(isfinite(coeff) && isfinite(bias_rate) && al16(scratch));
  MOE_CUDA(launch_route_aux(*cfg, logits, bias, idx, coeff, bias_rate, sel_counts, p_mean, loss,
                            bias_out, static_cast<uint8_t*>(scratch), (cudaStream_t)stream));
  return MOE_OK;
}

moe_status moe_route_aux_bwd(const moe_config* cfg, const void* x, const float* logits,
                             const float* bias, const float* W_r, const int32_t* sel_counts,
                             float coeff, float dloss, float* dlogits_aux, void* dx, float* dW_r,
                             void* scratch, void* stream) {
  MOE_TRY(check_config(cfg));
  MOE_REQUIRE(tok16(cfg, x) && tok4(cfg, logits) && al16(W_r) && al4(sel_counts));
  MOE_REQUIRE(tok16(cfg, dlogits_aux) && tok16(cfg, dx) && al16(dW_r));
  MOE_REQUIRE((bias == nullptr || al4(bias)) && isfinite(coeff) && isfinite(dloss));
  MOE_REQUIRE(al16(scratch));
  MOE_CUDA(launch_route_aux_bwd(*cfg, x, logits, bias, W_r, sel_counts, coeff, dloss,
                                dlogits_aux, dx, dW_r, static_cast<uint8_t*>(scratch),
                                (cudaStream_t)stream));
  return MOE_OK;
}

moe_status moe_permute(const moe_config* cfg, const void* x, const int32_t* idx, int32_t* counts,
                       int32_t* offsets, int32_t* row_of, int32_t* token_of, int32_t* sel_offsets,
                       int32_t* sel_tokens, void* x_perm, void* scratch, void* stream) {
  MOE_TRY(own_buffers(cfg));
  return permute_impl(cfg, x, idx, counts, offsets, row_of, token_of, sel_offsets, sel_tokens,
                      x_perm, scratch, stream, nullptr);
}

moe_status moe_quantize_weights(const moe_config* cfg, const void* W13, const void* W2,
                                void* scratch, void* stream) {
  MOE_TRY(check_config(cfg));
  MOE_REQUIRE(al16(W13) && al16(W2) && al16(scratch));
  if (!is_fp8(*cfg)) return MOE_OK;
  cudaStream_t s = (cudaStream_t)stream;
  const Fp8Scratch q = fp8_scratch(*cfg, scratch);
  const int G = cfg->E + cfg->n_shared;
  if (q.mx) {
    MOE_CUDA(launch_quant_wmx(W13, q.W13q, q.W13qd, q.W13sf, q.W13sft, G, 2 * cfg->F, cfg->H, s));
    MOE_CUDA(launch_quant_wmx(W2, q.W2q, q.W2qd, q.W2sf, q.W2sft, G, cfg->H, cfg->F, s));
    return MOE_OK;
  }
  MOE_CUDA(launch_quant_tiles8(W13, q.W13q, q.W13sf, q.W13sft, G, 2 * cfg->F, cfg->H, s));
  MOE_CUDA(launch_quant_tiles8(W2, q.W2q, q.W2sf, q.W2sft, G, cfg->H, cfg->F, s));
  return MOE_OK;
}

moe_status moe_load_fp8_weights(const moe_config* cfg, const void* W13_e4m3,
                                const uint8_t* W13_scale, const void* W2_e4m3,
                                const uint8_t* W2_scale, void* scratch, void* stream) {
  MOE_TRY(check_config(cfg));
  if (cfg->dtype != MOE_DTYPE_FP8_E4M3_BLOCK) return MOE_ERR_UNSUPPORTED;
  MOE_REQUIRE(al16(W13_e4m3) && al16(W2_e4m3) && W13_scale && W2_scale && al16(scratch));
  cudaStream_t s = (cudaStream_t)stream;
  const Fp8Scratch q = fp8_scratch(*cfg, scratch);
  const int G = cfg->E + cfg->n_shared;
  const int64_t n13 = (int64_t)G * 2 * cfg->F * cfg->H, n2 = (int64_t)G * cfg->H * cfg->F;
  MOE_CUDA(cudaMemcpyAsync(q.W13q, W13_e4m3, (size_t)n13, cudaMemcpyDeviceToDevice, s));
  MOE_CUDA(cudaMemcpyAsync(q.W2q, W2_e4m3, (size_t)n2, cudaMemcpyDeviceToDevice, s));
  MOE_CUDA(launch_load_fp8_scales(W13_scale, q.W13sf, q.W13sft, G, 2 * cfg->F, cfg->H, s));
  MOE_CUDA(launch_load_fp8_scales(W2_scale, q.W2sf, q.W2sft, G, cfg->H, cfg->F, s));
  return MOE_OK;
}

moe_status moe_grouped_ffn_fwd(const moe_config* cfg, const void* x_perm, const int32_t* counts,
                               const int32_t* offsets, const void* W13, const void* W2, void* GU,
                               void* h, void* y_perm, void* scratch, void* stream) {
  MOE_TRY(own_buffers(cfg));
  return ffn_fwd_impl(cfg, x_perm, counts, offsets, W13, W2, GU, h, y_perm, scratch, stream,
                      StashMap());
}

moe_status moe_unpermute(const moe_config* cfg, const void* y_perm, const int32_t* row_of,
                         const float* w, const int32_t* offsets, void* out, void* stream) {
  MOE_TRY(own_buffers(cfg));
  return unpermute_impl(cfg, y_perm, row_of, w, offsets, out, stream, nullptr);
}

moe_status moe_unpermute_bwd(const moe_config* cfg, const void* dY, const void* y_perm,
                             const int32_t* row_of, const float* w, const int32_t* counts,
                             const int32_t* offsets, void* dO_perm, float* dw, void* scratch,
                             void* stream) {
  MOE_TRY(own_buffers(cfg));
  return unpermute_bwd_impl(cfg, dY, y_perm, row_of, w, counts, offsets, dO_perm, dw, scratch,
                            stream, nullptr);
}

moe_status moe_grouped_ffn_dgrad(const moe_config* cfg, const void* dO_perm, const void* GU,
                                 void* h, const int32_t* counts, const int32_t* offsets,
                                 const int32_t* token_of, const float* dlogits, const float* W_r,
                                 const void* W13, const void* W2, void* dGU, void* dX_perm,
                                 void* scratch, void* stream) {
  MOE_TRY(own_buffers(cfg));
  return ffn_dgrad_impl(cfg, dO_perm, GU, h, counts, offsets, token_of, dlogits, W_r, W13, W2, dGU,
                        dX_perm, scratch, stream, StashMap());
}

moe_status moe_grouped_ffn_wgrad(const moe_config* cfg, const void* dO_perm, const void* x_perm,
                                 const void* h, const void* dGU, const int32_t* counts,
                                 const int32_t* offsets, void* dW13, void* dW2, void* scratch,
                                 void* stream) {
  MOE_TRY(own_buffers(cfg));
  return ffn_wgrad_impl(cfg, dO_perm, x_perm, h, dGU, counts, offsets, dW13, dW2, scratch, stream,
                        StashMap());
}

moe_status moe_grouped_ffn_bwd(const moe_config* cfg, const void* dO_perm, const void* x_perm,
                               const void* GU, const void* h, const int32_t* counts,
                               const int32_t* offsets, const int32_t* token_of,
                               const float* dlogits, const float* W_r, const void* W13,
                               const void* W2, void* dGU, void* dX_perm, void* dW13, void* dW2,
                               void* scratch, void* stream) {
  // fine-grained recompute: the data gradient rewrites h from GU before the
  // weight gradient reads it
  MOE_TRY(moe_grouped_ffn_dgrad(cfg, dO_perm, GU, cfg->recompute_h ? const_cast<void*>(h) : nullptr,
                                counts, offsets, token_of, dlogits, W_r, W13, W2,
                                dGU, dX_perm, scratch, stream));
  MOE_TRY(moe_grouped_ffn_wgrad(cfg, dO_perm, x_perm, h, dGU, counts, offsets, dW13, dW2, scratch,
                                stream));
  return MOE_OK;
}

moe_status moe_grouped_ffn_fwd_reordered(const moe_config* cfg, const void* x_perm,
                                         const int32_t* counts, const int32_t* offsets,
                                         const int32_t* token_of, const int32_t* row_of,
                                         const float* w, const void* W13, const void* W2,
                                         void* GU, void* h, void* y_perm, void* scratch,
                                         void* stream) {
  MOE_TRY(own_buffers(cfg));
  return ffn_fwd_reordered_impl(cfg, x_perm, counts, offsets, token_of, row_of, w, W13, W2, GU, h,
                                y_perm, scratch, stream, StashMap());
}

moe_status moe_unpermute_bwd_reordered(const moe_config* cfg, const void* dY,
                                       const int32_t* row_of, const int32_t* counts,
                                       const int32_t* offsets, void* dO_perm, void* stream) {
  MOE_TRY(check_config(cfg));
  MOE_REQUIRE(tok16(cfg, dY) && tok4(cfg, row_of) && al4(counts) && al4(offsets) && al16(dO_perm));
  MOE_CUDA(launch_unpermute_bwd_copy(*cfg, dY, row_of, counts, offsets, dO_perm,
                                     (cudaStream_t)stream));
  return MOE_OK;
}

moe_status moe_grouped_ffn_dgrad_reordered(const moe_config* cfg, const void* dO_perm,
                                           const void* GU, void* h, const int32_t* counts,
                                           const int32_t* offsets, const int32_t* token_of,
                                           const int32_t* row_of, const float* logits,
                                           const int32_t* idx, const float* w, const float* W_r,
                                           const void* W13, const void* W2, void* dGU,
                                           void* dX_perm, float* dw, float* dlogits,
                                           void* scratch, void* stream) {
  MOE_TRY(own_buffers(cfg));
  return ffn_dgrad_reordered_impl(cfg, dO_perm, GU, h, counts, offsets, token_of, row_of, logits,
                                  idx, w, W_r, W13, W2, dGU, dX_perm, dw, dlogits, scratch, stream,
                                  StashMap());
}

moe_status moe_route_bwd(const moe_config* cfg, const float* logits, const int32_t* idx,
                         const float* w, const float* dw, float* dlogits, void* stream) {
  MOE_TRY(check_config(cfg));
  MOE_REQUIRE(tok4(cfg, logits) && tok4(cfg, idx) && tok4(cfg, w) && tok4(cfg, dw) && tok4(cfg, dlogits));
  if (cfg->T == 0) return MOE_OK;
  MOE_CUDA(launch_route_bwd(*cfg, logits, idx, w, dw, dlogits, (cudaStream_t)stream));
  return MOE_OK;
}

moe_status moe_permute_bwd(const moe_config* cfg, const void* dX_perm, const int32_t* row_of,
                           const int32_t* offsets, const int32_t* idx, const float* dlogits,
                           const float* W_r, void* dx, void* stream) {
  MOE_TRY(check_config(cfg));
  MOE_REQUIRE(al16(dX_perm) && tok4(cfg, row_of) && al4(offsets) && tok4(cfg, idx) && tok4(cfg, dlogits));
  MOE_REQUIRE(al16(W_r) && tok16(cfg, dx));
  MOE_CUDA(launch_permute_bwd(*cfg, dX_perm, row_of, offsets, idx, dlogits, W_r, dx,
                              (cudaStream_t)stream));
  return MOE_OK;
}

moe_status moe_router_wgrad(const moe_config* cfg, const void* x, const int32_t* sel_offsets,
                            const int32_t* sel_tokens, const float* dlogits, float* dW_r,
                            void* scratch, void* stream) {
  MOE_TRY(check_config(cfg));
  MOE_REQUIRE(tok16(cfg, x) && al4(sel_offsets) && tok4(cfg, sel_tokens) && tok16(cfg, dlogits));
  MOE_REQUIRE(al16(dW_r) && al16(scratch));
  MOE_CUDA(launch_router_wgrad(*cfg, x, sel_offsets, sel_tokens, dlogits, dW_r,
                               static_cast<uint8_t*>(scratch), (cudaStream_t)stream));
  return MOE_OK;
}

moe_status moe_layer_fwd(const moe_config* cfg, const moe_params* P, const void* x, void* out,
                         const moe_fwd_state* st, void* scratch, void* stream) {
  MOE_TRY(check_config(cfg));
  MOE_REQUIRE(P && st);
  StashMap sm;
  MOE_TRY(stash_of(cfg, st, &sm));
  const StashAlloc alloc{st->stash_table, st->stash_top, cfg->stash_pool_pages};
  // FP8 with no bf16 weights: the E4M3 weights moe_load_fp8_weights (or an
  // earlier moe_quantize_weights) left in scratch are used as they are
  if (!(is_fp8(*cfg) && !P->W13 && !P->W2))
    MOE_TRY(moe_quantize_weights(cfg, P->W13, P->W2, scratch, stream));
  MOE_TRY(moe_route(cfg, x, P->W_r, P->bias, st->logits, st->idx, st->w, scratch, stream));
  MOE_TRY(permute_impl(cfg, x, st->idx, st->counts, st->offsets, st->row_of, st->token_of,
                       st->sel_offsets, st->sel_tokens, st->x_perm, scratch, stream,
                       sm.pages ? &alloc : nullptr));
  if (cfg->weights_in_expert) {
    MOE_TRY(ffn_fwd_reordered_impl(cfg, st->x_perm, st->counts, st->offsets, st->token_of,
                                   st->row_of, st->w, P->W13, P->W2, st->GU, st->h, st->y_perm,
                                   scratch, stream, sm));
    return unpermute_impl(cfg, st->y_perm, st->row_of, nullptr, st->offsets, out, stream,
                          sm.pages);
  }
  MOE_TRY(ffn_fwd_impl(cfg, st->x_perm, st->counts, st->offsets, P->W13, P->W2, st->GU, st->h,
                       st->y_perm, scratch, stream, sm));
  MOE_TRY(unpermute_impl(cfg, st->y_perm, st->row_of, st->w, st->offsets, out, stream, sm.pages));
  return MOE_OK;
}

moe_status moe_layer_bwd(const moe_config* cfg, const moe_params* P, const void* x,
                         const void* dY, const moe_fwd_state* st, const moe_bwd_state* bs,
                         void* dx, float* dW_r, void* dW13, void* dW2, void* scratch,
                         void* stream) {
  MOE_TRY(check_config(cfg));
  MOE_REQUIRE(P && st && bs);
  StashMap sm;
  MOE_TRY(stash_of(cfg, st, &sm));
  // fine-grained recompute: the data gradient rewrites h from GU before the
  // weight gradient reads it
  void* h_out = cfg->recompute_h ? st->h : nullptr;
  if (cfg->weights_in_expert) {
    MOE_TRY(moe_unpermute_bwd_reordered(cfg, dY, st->row_of, st->counts, st->offsets,
                                        bs->dO_perm, stream));
    MOE_TRY(ffn_dgrad_reordered_impl(cfg, bs->dO_perm, st->GU, h_out, st->counts, st->offsets,
                                     st->token_of, st->row_of, st->logits, st->idx, st->w,
                                     P->W_r, P->W13, P->W2, bs->dGU, bs->dX_perm, bs->dw,
                                     bs->dlogits, scratch, stream, sm));
  } else {
    MOE_TRY(unpermute_bwd_impl(cfg, dY, st->y_perm, st->row_of, st->w, st->counts, st->offsets,
                               bs->dO_perm, bs->dw, scratch, stream, sm.pages));
    MOE_TRY(moe_route_bwd(cfg, st->logits, st->idx, st->w, bs->dw, bs->dlogits, stream));
    MOE_TRY(ffn_dgrad_impl(cfg, bs->dO_perm, st->GU, h_out, st->counts, st->offsets,
                           st->token_of, bs->dlogits, P->W_r, P->W13, P->W2, bs->dGU,
                           bs->dX_perm, scratch, stream, sm));
  }
  MOE_TRY(ffn_wgrad_impl(cfg, bs->dO_perm, st->x_perm, st->h, bs->dGU, st->counts, st->offsets,
                         dW13, dW2, scratch, stream, sm));
  MOE_TRY(moe_permute_bwd(cfg, bs->dX_perm, st->row_of, st->offsets, st->idx, bs->dlogits,
                          P->W_r, dx, stream));
  MOE_TRY(moe_router_wgrad(cfg, x, st->sel_offsets, st->sel_tokens, bs->dlogits, dW_r, scratch,
                           stream));
  if (sm.pages) MOE_TRY(moe_stash_release(cfg, st, stream));
  return MOE_OK;
}

moe_status moe_stash_release(const moe_config* cfg, const moe_fwd_state* st, void* stream) {
  MOE_TRY(check_config(cfg));
  MOE_REQUIRE(st && cfg->stash_pool_pages > 0 && al4(st->stash_table) && al4(st->stash_top));
  MOE_CUDA(launch_stash_release(*cfg, st->stash_table, st->stash_top, (cudaStream_t)stream));
  return MOE_OK;
}

moe_status moe_last_device_status(const void* scratch, int32_t* code, void* stream) {
  MOE_REQUIRE(al16(scratch) && code);
  cudaStream_t s = (cudaStream_t)stream;
  MOE_CUDA(cudaStreamSynchronize(s));
  MOE_CUDA(cudaMemcpy(code, static_cast<const uint8_t*>(scratch) + kScratchStatus,
                      sizeof(int32_t), cudaMemcpyDeviceToHost));
  return MOE_OK;
}

moe_status moe_clear_device_status(void* scratch, void* stream) {
  MOE_REQUIRE(al16(scratch));
  MOE_CUDA(cudaMemsetAsync(static_cast<uint8_t*>(scratch) + kScratchStatus, 0, sizeof(int32_t),
                           (cudaStream_t)stream));
  return MOE_OK;
}

moe_status moe_check_bounded_wait(void* scratch, int64_t budget_cycles, void* stream) {
  MOE_REQUIRE(al16(scratch) && budget_cycles > 0);
  bounded_wait_check_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(status_word(scratch),
                                                                (long long)budget_cycles);
  MOE_CUDA(cudaGetLastError());
  return MOE_OK;
}

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument (pointer, shape or alignment)";
    case MOE_ERR_UNSUPPORTED: return "configuration not supported by the library";
    case MOE_ERR_WORKSPACE: return "scratch buffer too small";
    case MOE_ERR_CUDA: return "a CUDA runtime call failed";
    case MOE_ERR_TIMEOUT: return "a device-side bounded wait ran out";
    case MOE_ERR_DEVICE_CHECK: return "a kernel found an out-of-range index";
    case MOE_ERR_STASH_FULL: return "a layer's rows did not fit its stash pool";
  }
  return "unknown status";
}

}  // extern "C"
