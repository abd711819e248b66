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

cudaError_t launch_permute(const moe_config& c, const void* x, const int32_t* idx,
                           int32_t* counts, int32_t* offsets, int32_t* row_of, int32_t* token_of,
                           int32_t* sel_offsets, int32_t* sel_tokens, void* x_perm,
                           uint8_t* scratch, cudaStream_t s);

cudaError_t launch_unpermute(const moe_config& c, const void* y_perm, const int32_t* row_of,
                             const float* w, const int32_t* offsets, void* out, cudaStream_t s);

cudaError_t launch_unpermute_bwd(const moe_config& c, const void* dY, const void* y_perm,
                                 const int32_t* row_of, const float* w, const int32_t* counts,
                                 const int32_t* offsets, void* dO_perm, float* dw, cudaStream_t s);

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

// FP8 block quantisation (E4M3 values with power-of-two scales, stored as bf16).
cudaError_t launch_quant_tiles(const void* W, void* Wq, int G, int rows, int cols, cudaStream_t s);
cudaError_t launch_quant_rows(const void* X, void* Xq, const int32_t* offsets,
                              const int32_t* counts, int G, int64_t rows_max, int cols,
                              cudaStream_t s);
cudaError_t launch_quant_cols(const void* X, void* Xq, const int32_t* offsets,
                              const int32_t* counts, int G, int64_t rows_max, int cols,
                              cudaStream_t s);

// Where the FP8 mode keeps its quantised tensors inside `scratch`.
struct Fp8Scratch {
  void* W13q;   // [G,2F,H]
  void* W2q;    // [G,H,F]
  void* aH;     // [R,H]  x_perm rows, then x_perm columns
  void* bF;     // [R,F]  h rows, then h columns
  void* cH;     // [R,H]  dO rows, then dO columns
  void* d2F;    // [R,2F] dGU rows, then dGU columns
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
// cannot be encoded for the given pointers.
cudaError_t launch_ffn_fc1(const moe_config& c, const void* x_perm, const int32_t* counts,
                           const int32_t* offsets, const void* W13, void* GU, void* h,
                           int32_t* status, cudaStream_t s);
cudaError_t launch_ffn_fc2(const moe_config& c, const void* h, const int32_t* counts,
                           const int32_t* offsets, const void* W2, void* y_perm,
                           int32_t* status, cudaStream_t s);
cudaError_t launch_ffn_fc2_dgrad(const moe_config& c, const void* dO_perm, const int32_t* counts,
                                 const int32_t* offsets, const void* W2, const void* GU,
                                 void* dGU, int32_t* status, cudaStream_t s);
cudaError_t launch_ffn_fc1_dgrad(const moe_config& c, const void* dGU, const int32_t* counts,
                                 const int32_t* offsets, const void* W13, const int32_t* token_of,
                                 const float* dlogits, const float* W_r, void* dX_perm,
                                 int32_t* status, cudaStream_t s);
cudaError_t launch_ffn_wgrad_fc2(const moe_config& c, const void* dO_perm, const void* h,
                                 const int32_t* counts, const int32_t* offsets, void* dW2,
                                 int32_t* status, cudaStream_t s);
cudaError_t launch_ffn_wgrad_fc1(const moe_config& c, const void* dGU, const void* x_perm,
                                 const int32_t* counts, const int32_t* offsets, void* dW13,
                                 int32_t* status, cudaStream_t s);

}  // namespace moe
