// Host-side launchers shared between the translation units of the library.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe_abi.h"

namespace moe {

moe_status check_config(const moe_config* c);
int64_t scratch_bytes(const moe_config& c);
int64_t capacity_rows(const moe_config& c);
int64_t rows_max(const moe_config& c);
int n_chunks(const moe_config& c);
int num_sms();

cudaError_t launch_route(const moe_config& c, const void* x, const float* W_r, const float* bias,
                         float* logits, int32_t* idx, float* w, uint8_t* scratch, cudaStream_t s);
cudaError_t launch_route_replay(const moe_config& c, const void* x, const float* W_r,
                                const float* bias, const int32_t* idx, float* logits, float* w,
                                uint8_t* scratch, cudaStream_t s);

// Where a layer keeps the rows its backward reads (x_perm, GU, h, y_perm):
// row r is row pages[r / 128] * 128 + r % 128 of pool tensors of `rows` rows
// (paged stash), or row r of the layer's own rows_max-row buffers
// (pages == nullptr, rows == 0).
struct StashMap {
  const int32_t* pages = nullptr;
  int64_t rows = 0;
};
int64_t stash_rows(const moe_config& c, const StashMap& sm);
// The paged stash's allocation, done by the dispatch once the segment
// offsets are known: the layer's page table and the pool's page counter.
struct StashAlloc {
  int32_t* table;
  int32_t* top;
  int pool_pages;
};
// Gives the layer's pages back: *top = table[rows_max / 128 + 1].
cudaError_t launch_stash_release(const moe_config& c, const int32_t* table, int32_t* top,
                                 cudaStream_t s);

struct Fp8Scratch;
// fp8 (FP8 configuration, optional): also write x_perm's 1-byte form there.
// alloc (optional): take the layer's stash pages and write x_perm into them.
cudaError_t launch_permute(const moe_config& c, const void* x, const int32_t* idx,
                           int32_t* counts, int32_t* offsets, int32_t* row_of, int32_t* token_of,
                           int32_t* sel_offsets, int32_t* sel_tokens, void* x_perm,
                           uint8_t* scratch, cudaStream_t s, const Fp8Scratch* fp8 = nullptr,
                           const StashAlloc* alloc = nullptr);

// pages (optional): y_perm is paged (StashMap).
cudaError_t launch_unpermute(const moe_config& c, const void* y_perm, const int32_t* row_of,
                             const float* w, const int32_t* offsets, void* out, cudaStream_t s,
                             const int32_t* pages = nullptr);

// dOq, dOsf (FP8 configuration, optional): also write dO_perm's 1-byte form.
// pages (optional): y_perm is paged; dO_perm is not.
cudaError_t launch_unpermute_bwd(const moe_config& c, const void* dY, const void* y_perm,
                                 const int32_t* row_of, const float* w, const int32_t* counts,
                                 const int32_t* offsets, void* dO_perm, float* dw, cudaStream_t s,
                                 uint8_t* dOq = nullptr, uint8_t* dOsf = nullptr,
                                 const int32_t* pages = nullptr);

// The layer with the routing weight inside the expert: the unweighted copy of
// dY into the expert rows (dO_perm), the routing weight of every permuted row,
// and dw from the FC2 data gradient's per-tile partial dot products.
cudaError_t launch_unpermute_bwd_copy(const moe_config& c, const void* dY, const int32_t* row_of,
                                      const int32_t* counts, const int32_t* offsets,
                                      void* dO_perm, cudaStream_t s);
cudaError_t launch_row_weights(const moe_config& c, const int32_t* token_of,
                               const int32_t* row_of, const float* w, const int32_t* offsets,
                               float* row_w, cudaStream_t s);
cudaError_t launch_dw_reduce(const moe_config& c, const float* dw_part, const int32_t* row_of,
                             float* dw, cudaStream_t s);
// Where the layer with the weight inside the expert keeps its per-row weights
// ([rows_max] fp32) and the partial dot products ([rows_max][dw_tiles] fp32).
struct ReorderScratch {
  float* row_w;
  float* dw_part;
};
ReorderScratch reorder_scratch(const moe_config& c, void* scratch);

cudaError_t launch_route_bwd(const moe_config& c, const float* logits, const int32_t* idx,
                             const float* w, const float* dw, float* dlogits, cudaStream_t s);

cudaError_t launch_permute_bwd(const moe_config& c, const void* dX_perm, const int32_t* row_of,
                               const int32_t* offsets, const int32_t* idx, const float* dlogits,
                               const float* W_r, void* dx, cudaStream_t s);

// dW_r (= or, with accumulate, +=) sum over tokens of dlogits[t,e] x[t,:]; with
// sel_offsets == sel_tokens == NULL every token counts for every expert
// (dense dlogits), else only the tokens that selected e.
cudaError_t launch_router_wgrad(const moe_config& c, const void* x, const int32_t* sel_offsets,
                                const int32_t* sel_tokens, const float* dlogits, float* dW_r,
                                uint8_t* scratch, cudaStream_t s, bool accumulate = false);

// Load-balancing loss: statistics, loss and bias update in one launch; its
// gradient into dlogits_aux, dx and dW_r.
cudaError_t launch_route_aux(const moe_config& c, const float* logits, const float* bias,
                             const int32_t* idx, float coeff, float rate, int32_t* counts,
                             float* p_mean, float* loss, float* bias_out, uint8_t* scratch,
                             cudaStream_t s);
cudaError_t launch_route_aux_bwd(const moe_config& c, const void* x, const float* logits,
                                 const float* bias, const float* W_r, const int32_t* counts,
                                 float coeff, float dloss, float* dl, void* dx, float* dW_r,
                                 uint8_t* scratch, cudaStream_t s);
int64_t aux_partial_bytes(const moe_config& c);    // the aux-loss region of scratch
int64_t aux_partial_offset(const moe_config& c);   // its byte offset in scratch

// FP8 block quantisation (E4M3 values with power-of-two block scales):
// 1-byte codes with UE8M0 scale atoms (fp8_layout.cuh) for the FP8 GEMMs --
// weights in 128x128 tiles (atoms for both orientations of the weight),
// activations in 1x128 slices along their rows -- and, for the bf16-path
// weight gradients, the dequantised values of 128x1 slices along the tokens.
cudaError_t launch_quant_tiles8(const void* W, uint8_t* Wq, uint8_t* sf_f, uint8_t* sf_d, int G,
                                int rows, int cols, cudaStream_t s);
// mx: 32-element blocks and the MX atom layout (MXFP8), else 128.
// pages (optional): X is a paged stash tensor (StashMap); the outputs are not.
cudaError_t launch_quant_cols8(const void* X, uint8_t* Xq, uint8_t* sf, const int32_t* offsets,
                               const int32_t* counts, int G, int64_t rows_max, int cols,
                               cudaStream_t s, bool mx = false, const int32_t* pages = nullptr);
// Both forms of one tensor from a single read: 1xBLK rows (Xr, sfr) and
// BLKx1 columns (Xc, sfc).
cudaError_t launch_quant_rows_cols8(const void* X, uint8_t* Xr, uint8_t* sfr, uint8_t* Xc,
                                    uint8_t* sfc, const int32_t* offsets, const int32_t* counts,
                                    int G, int64_t rows_max, int cols, cudaStream_t s,
                                    bool mx = false);
// The atoms of caller-quantised E4M3 weights from one UE8M0 code per 128x128 tile.
cudaError_t launch_load_fp8_scales(const uint8_t* scale, uint8_t* sf_f, uint8_t* sf_d, int G,
                                   int rows, int cols, cudaStream_t s);
// MXFP8 weights: forward (1x32 along cols) and data-gradient (32x1 along rows) forms.
cudaError_t launch_quant_wmx(const void* W, uint8_t* Wf, uint8_t* Wd, uint8_t* sf_f, uint8_t* sf_d,
                             int G, int rows, int cols, cudaStream_t s);

// Where the FP8 mode keeps its quantised tensors inside `scratch`.
struct Fp8Scratch {
  bool mx;          // MXFP8: 32-element blocks, MX atom layout, two weight forms
  uint8_t* W13q;    // [G,2F,H] E4M3 (forward form)
  uint8_t* W13qd;   // data-gradient form (MX), else W13q
  uint8_t* W13sf;   // atoms, N = W13 rows, K = H (forward)
  uint8_t* W13sft;  // atoms, N = H, K = W13 rows (FC1 data gradient)
  uint8_t* W2q;     // [G,H,F] E4M3 (forward form)
  uint8_t* W2qd;    // data-gradient form (MX), else W2q
  uint8_t* W2sf;    // atoms, N = H, K = F (forward)
  uint8_t* W2sft;   // atoms, N = F, K = H (FC2 data gradient)
  uint8_t* xq;      // [R,H] x_perm, 1x128 slices
  uint8_t* xsf;
  uint8_t* hq;      // [R,F] h
  uint8_t* hsf;
  uint8_t* dOq;     // [R,H] dO
  uint8_t* dOsf;
  uint8_t* dGq;     // [R,2F] dGU
  uint8_t* dGsf;
  // 128x1 slices along the tokens (weight gradients): E4M3 codes, then atoms
  // [columns / 128][row blocks / 4]
  uint8_t* cHq;     // [R,H]  dO
  uint8_t* cHsf;
  uint8_t* bFq;     // [R,F]  h
  uint8_t* bFsf;
  uint8_t* d2Fq;    // [R,2F] dGU
  uint8_t* d2Fsf;
  uint8_t* aHq;     // [R,H]  x_perm
  uint8_t* aHsf;
};
Fp8Scratch fp8_scratch(const moe_config& c, void* scratch);

// Router logits for E % 128 == 0 on the tensor cores (W3 = W_r split in three bf16 parts).
cudaError_t launch_router_logits_tc(const moe_config& c, const void* x, const void* W3,
                                    float* logits, int32_t* status, cudaStream_t s);
cudaError_t launch_router_wgrad_tc(const moe_config& c, const void* x, const void* D3,
                                   long long Tp, float* P, int chunk, int32_t* status,
                                   cudaStream_t s);
// dx [T,H] bf16 += A3 [T,K3] . B3 [H,K3]^T (bf16 operands, K-major), on the tensor cores.
cudaError_t launch_router_dx_tc(const moe_config& c, const void* A3, const void* B3, int K3,
                                void* dx, int32_t* status, cudaStream_t s);
bool router_on_tensor_cores(const moe_config& c);
// tensor-core router weight gradient: tokens per chunk (<= 271 chunks), and
// the byte offset of the chunk partial sums after the split dlogits in the
// router region of scratch
int router_wgrad_chunk(const moe_config& c);
int64_t router_wgrad_split_bytes(const moe_config& c);
int64_t router_split_bytes(const moe_config& c);   // the router region of scratch
int64_t aux_dx_split_bytes(const moe_config& c);   // the loss's split dx operands in it
int64_t router_split_offset(const moe_config& c);   // byte offset of the split in scratch
int64_t permute_scratch_bytes(const moe_config& c); // scratch the dispatch needs

// Grouped GEMMs (tcgen05). Return cudaErrorInvalidValue when a tensor map
// cannot be encoded for the given pointers. sm: where x_perm, GU, h and y_perm
// live (the other row tensors are the layer's own, at their rows).
// row_w (the routing weight inside the expert, optional): h = w_row silu(G) U.
cudaError_t launch_ffn_fc1(const moe_config& c, const void* x_perm, const int32_t* counts,
                           const int32_t* offsets, const void* W13, void* GU, void* h,
                           int32_t* status, cudaStream_t s, const float* row_w = nullptr,
                           const StashMap& sm = StashMap());
cudaError_t launch_ffn_fc2(const moe_config& c, const void* h, const int32_t* counts,
                           const int32_t* offsets, const void* W2, void* y_perm,
                           int32_t* status, cudaStream_t s, const StashMap& sm = StashMap());
// row_w, dw_part (optional): the weight inside the expert -- dh = w_row dh_s,
// and dw_part[r * dw_tiles(c) + n-tile] = the row's <dh_s, h> over that tile.
// h_out (optional): h [rows, F] rewritten from GU (fine-grained recompute).
cudaError_t launch_ffn_fc2_dgrad(const moe_config& c, const void* dO_perm, const int32_t* counts,
                                 const int32_t* offsets, const void* W2, const void* GU,
                                 void* dGU, int32_t* status, cudaStream_t s,
                                 const float* row_w = nullptr, float* dw_part = nullptr,
                                 void* h_out = nullptr, const StashMap& sm = StashMap());
int dw_tiles(const moe_config& c);
cudaError_t launch_ffn_fc1_dgrad(const moe_config& c, const void* dGU, const int32_t* counts,
                                 const int32_t* offsets, const void* W13, const int32_t* token_of,
                                 const float* dlogits, const float* W_r, void* dX_perm,
                                 int32_t* status, cudaStream_t s);
cudaError_t launch_ffn_wgrad_fc2(const moe_config& c, const void* dO_perm, const void* h,
                                 const int32_t* counts, const int32_t* offsets, void* dW2,
                                 int32_t* status, cudaStream_t s, const StashMap& sm = StashMap());
cudaError_t launch_ffn_wgrad_fc1(const moe_config& c, const void* dGU, const void* x_perm,
                                 const int32_t* counts, const int32_t* offsets, void* dW13,
                                 int32_t* status, cudaStream_t s, const StashMap& sm = StashMap());

// The FP8 configuration's forward and data-gradient GEMMs on the block-scaled
// FP8 tensor cores (tcgen05 kind::mxf8f6f4): E4M3 operands with UE8M0 scale
// atoms; the same epilogues and outputs as the bf16 launches above.
cudaError_t launch_ffn_fc1_fp8(const moe_config& c, const uint8_t* xq, const uint8_t* xsf,
                               const int32_t* counts, const int32_t* offsets, const uint8_t* W13q,
                               const uint8_t* W13sf, void* GU, void* h, uint8_t* hq, uint8_t* hsf,
                               int32_t* status, cudaStream_t s, const StashMap& sm = StashMap());
cudaError_t launch_ffn_fc2_fp8(const moe_config& c, const uint8_t* hq, const uint8_t* hsf,
                               const int32_t* counts, const int32_t* offsets, const uint8_t* W2q,
                               const uint8_t* W2sf, void* y_perm, int32_t* status,
                               cudaStream_t s, const StashMap& sm = StashMap());
cudaError_t launch_ffn_fc2_dgrad_fp8(const moe_config& c, const uint8_t* dOq, const uint8_t* dOsf,
                                     const int32_t* counts, const int32_t* offsets,
                                     const uint8_t* W2q, const uint8_t* W2sf_t, const void* GU,
                                     void* dGU, int32_t* status, cudaStream_t s,
                                     void* h_out = nullptr, const StashMap& sm = StashMap());
cudaError_t launch_ffn_fc1_dgrad_fp8(const moe_config& c, const uint8_t* dGq, const uint8_t* dGsf,
                                     const int32_t* counts, const int32_t* offsets,
                                     const uint8_t* W13q, const uint8_t* W13sf_t,
                                     const int32_t* token_of, const float* dlogits,
                                     const float* W_r, void* dX_perm, int32_t* status,
                                     cudaStream_t s);
// Weight gradients over the 128x1-slice operands (K = each group's rows):
// dW2[g] = dO^T h, dW13[g] = dGU^T x_perm (bf16; zero for empty groups).
cudaError_t launch_ffn_wgrad_fc2_fp8(const moe_config& c, const uint8_t* dOq, const uint8_t* dOsf,
                                     const uint8_t* hq, const uint8_t* hsf, const int32_t* counts,
                                     const int32_t* offsets, void* dW2, int32_t* status,
                                     cudaStream_t s);
cudaError_t launch_ffn_wgrad_fc1_fp8(const moe_config& c, const uint8_t* dGq, const uint8_t* dGsf,
                                     const uint8_t* xq, const uint8_t* xsf, const int32_t* counts,
                                     const int32_t* offsets, void* dW13, int32_t* status,
                                     cudaStream_t s);

}  // namespace moe
