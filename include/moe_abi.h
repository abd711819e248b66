/*
 * moe_abi.h -- C-ABI of a single-GPU Mixture-of-Experts layer for GB300 (sm_103a).
 *
 * The layer is the four-stage MoE layer of "Scalable Training of
 * Mixture-of-Experts Models with Megatron Core" (gist.science summaries; es:
 * "Resumen técnico" §2.1 "Arquitectura de la Capa MoE"):
 *   route    -- a router picks the k best experts of every token,
 *   dispatch -- tokens are moved to their experts (here: a permutation into
 *               per-expert contiguous rows of one buffer, since all experts
 *               live on this GPU),
 *   compute  -- every expert's SwiGLU FFN runs as one grouped GEMM,
 *   combine  -- the results return to their tokens, weighted by the router,
 * plus the backward of all four.
 *
 * Conventions shared by every call:
 *  - Pointers named x, W_*, out, ... are DEVICE pointers unless stated.
 *    cfg / params / state structs themselves live in HOST memory.
 *  - The caller owns every buffer; the library never allocates or frees
 *    device memory. Buffers are sized for the worst case with
 *    moe_query_sizes() (the Hybrid-EP article's "worst-case pre-reservation",
 *    hyper.ai, on dynamic token counts), except, with a paged stash
 *    (moe_config.stash_pool_pages), the four row tensors a layer keeps for
 *    its backward: those come from a pool of pages shared by several layers,
 *    which the layers take and give back on the device.
 *  - All calls are asynchronous on `stream` (a cudaStream_t, NULL = legacy
 *    default stream) and never synchronise the host or read device memory
 *    from the host, except moe_last_device_status(). Token counts stay on the
 *    device: kernels read them there (the sync-free, device-initiated
 *    execution of the same page, §2.3.C).
 *  - Layouts are row-major. bf16 tensors are passed as `void*` holding IEEE
 *    bfloat16. Index tensors are int32. Device buffers must be 16-byte aligned
 *    (4-byte for int32/fp32 vectors); buffers indexed by token may be NULL
 *    when T == 0.
 *  - Argument errors are returned synchronously (MOE_ERR_INVALID_ARG /
 *    MOE_ERR_UNSUPPORTED) before anything is launched. Problems detected by a
 *    kernel (an index out of range, a bounded wait that ran out) are recorded
 *    in a status word at the start of `scratch`; kernels never trap.
 *
 * Shapes: T tokens, H hidden, E routed experts, k experts per token, F FFN
 * width of one expert, S = n_shared shared experts, G = E + S groups,
 * R = rows_max (moe_query_sizes) rows in every permuted buffer.
 */
#ifndef MOE_ABI_H
#define MOE_ABI_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum moe_status {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,   /* bad pointer, shape or alignment            */
    MOE_ERR_UNSUPPORTED = 2,   /* a valid configuration the library lacks     */
    MOE_ERR_WORKSPACE = 3,     /* scratch too small                           */
    MOE_ERR_CUDA = 4,          /* a CUDA runtime call failed                  */
    MOE_ERR_TIMEOUT = 5,       /* a device-side bounded wait ran out          */
    MOE_ERR_DEVICE_CHECK = 6,  /* a kernel found an out-of-range index        */
    MOE_ERR_STASH_FULL = 7     /* a layer's rows did not fit its stash pool   */
} moe_status;

enum { MOE_SCORE_SOFTMAX = 0, MOE_SCORE_SIGMOID = 1 };
enum { MOE_GROUP_TOP2_SUM = 0, MOE_GROUP_MAX = 1 };
/* MOE_DTYPE_FP8_E4M3_BLOCK: every expert-GEMM operand is quantised to E4M3
 * with power-of-two block scales (2^ceil(log2(amax/448))): expert weights in
 * 128x128 tiles, activations in 1x128 slices along the dimension their GEMM
 * reduces, weight-gradient operands in 128x1 slices along each expert's
 * tokens. All six expert GEMMs run on the block-scaled FP8 tensor cores.
 * Router, routing weights and all outputs stay as in bf16 mode.
 * In this mode `scratch` also holds the quantised weights and activations
 * (moe_query_sizes counts them), and the scratch used by a forward must be
 * passed unchanged to its backward. Shared experts are not supported in this
 * mode (n_shared must be 0), and H and F must be multiples of 256
 * (MOE_ERR_UNSUPPORTED otherwise).
 * MOE_DTYPE_MXFP8: the same with the MX formats' 32-element blocks (the MXFP8
 * recipe the es summary §2.4 names for Blackwell): activations in 1x32 slices
 * along the reduced dimension, weight-gradient operands in 32x1 slices along
 * the tokens, and each expert weight quantised twice -- 1x32 along its input
 * dimension for the forward GEMMs and 32x1 along its output dimension for the
 * data gradients (scratch holds both forms). Same restrictions. */
enum { MOE_DTYPE_BF16 = 0, MOE_DTYPE_FP8_E4M3_BLOCK = 1, MOE_DTYPE_MXFP8 = 2 };

/* One layer configuration. */
typedef struct moe_config {
    int32_t T, H, E, k, F;
    int32_t n_shared;        /* shared experts (weight 1, every token), 0..4    */
    int32_t score_fn;        /* MOE_SCORE_SOFTMAX | MOE_SCORE_SIGMOID           */
    int32_t n_groups;        /* expert groups for group-limited top-k (1 = off) */
    int32_t topk_groups;     /* groups kept per token                           */
    int32_t group_score;     /* MOE_GROUP_TOP2_SUM | MOE_GROUP_MAX              */
    float route_scale;       /* sigmoid weights: route_scale * s_j / sum s      */
    int32_t dtype;           /* MOE_DTYPE_BF16 | _FP8_E4M3_BLOCK | _MXFP8         */
    float capacity_factor;   /* 0 = dropless; else C = ceil(cf*T*k/E) rows      */
    int32_t row_align;       /* every expert segment is a multiple of this (128)*/
    int32_t weights_in_expert; /* 1: the routing weight scales h inside the
                                * expert before FC2 (see moe_grouped_ffn_fwd_
                                * reordered); bf16 mode only. 0: it scales the
                                * expert output in the combine.              */
    int32_t recompute_h;     /* 1: the backward rewrites h from GU (the
                              * fine-grained recompute of the activation
                              * function, es summary §2.3.A): moe_layer_bwd and
                              * moe_grouped_ffn_bwd pass h to the data gradient,
                              * so the h the forward wrote need not survive
                              * until the backward. 0: h is read as stored.  */
    int32_t stash_pool_pages; /* 0: x_perm, GU, h and y_perm of moe_fwd_state
                               * are this layer's own R-row buffers. P > 0:
                               * they are the tensors of a stash pool of P
                               * pages of 128 rows (plus one spill page:
                               * (P + 1) * 128 rows each), shared by every layer
                               * of a step; moe_layer_fwd takes the pages its
                               * rows need on the device (paged stashing inside
                               * a CUDA graph instead of worst-case buffers,
                               * es summary §2.3.C), moe_layer_bwd gives them
                               * back. See moe_fwd_state.stash_table.       */
} moe_config;

/* Worst-case sizes of the caller-owned buffers for one configuration. */
typedef struct moe_sizes {
    int64_t rows_max;        /* R: rows of x_perm, GU, h, y_perm, dO, dGU, dX   */
    int64_t groups;          /* G = E + n_shared                                */
    int64_t capacity;        /* C rows per expert (0 = dropless)                */
    int64_t scratch_bytes;   /* bytes of `scratch` (zero-fill it once)          */
    int64_t stash_table_len; /* int32 entries of moe_fwd_state.stash_table:
                              * R / 128 + 2                                     */
} moe_sizes;

/* Layer parameters (device pointers).
 * W_r [E,H] fp32 router weight; bias [E] fp32 or NULL (softmax: added to the
 * logits; sigmoid: added to the scores for selection only);
 * W13 [G,2F,H] bf16 (rows 0..F-1 gate, F..2F-1 up); W2 [G,H,F] bf16. Shared
 * experts are the last S groups. */
typedef struct moe_params {
    const float* W_r;
    const float* bias;
    const void* W13;
    const void* W2;
} moe_params;

/* Forward state, kept for the backward (device pointers, caller-owned). */
typedef struct moe_fwd_state {
    float* logits;           /* [T,E]   fp32 router logits (before bias)        */
    int32_t* idx;            /* [T,k]   selected experts, best first            */
    float* w;                /* [T,k]   routing weights                         */
    int32_t* counts;         /* [G]     rows kept per group                     */
    int32_t* offsets;        /* [G+1]   first row of every group segment        */
    int32_t* row_of;         /* [T,k]   row of assignment (t,j); -1 = dropped   */
    int32_t* token_of;       /* [R]     token of row r; -1 = padding            */
    int32_t* sel_offsets;    /* [E+1]   per expert: start in sel_tokens         */
    int32_t* sel_tokens;     /* [T*k]   per expert, every selecting token, in t */
    void* x_perm;            /* [R,H]   bf16 dispatched tokens (padding = 0)    */
    void* GU;                /* [R,2F]  bf16 gate|up pre-activations            */
    void* h;                 /* [R,F]   bf16 SwiGLU output                      */
    void* y_perm;            /* [R,H]   bf16 expert outputs                     */
    /* Paged stash (cfg->stash_pool_pages = P > 0; both NULL otherwise).
     * The four row tensors above then hold (P + 1) * 128 rows and are shared
     * by the layers of a pool; row r of this layer (r as in row_of, token_of,
     * offsets) is row stash_table[r / 128] * 128 + r % 128 of them.
     * moe_layer_fwd writes the table on the device: the 128-row blocks that
     * hold the layer's kept rows (ceil(counts[g] / 128) blocks of group g, at
     * offsets[g] / 128 ...) get consecutive pages from *stash_top on, every
     * other block gets the spill page P; entry R/128 + 1 holds the first page
     * taken. When the blocks do not fit (*stash_top + blocks > P) no page is
     * taken, every block gets page P, MOE_ERR_STASH_FULL is recorded in the
     * status word and the step's results are invalid (all writes stay inside
     * the pool). moe_layer_bwd (or moe_stash_release) resets *stash_top to
     * that first page, so the layers of a pool must run their backward in the
     * reverse order of their forward. */
    int32_t* stash_table;    /* [R/128 + 2] int32, caller-owned, per layer       */
    int32_t* stash_top;      /* [1] int32: pages in use, shared by the pool's
                              * layers; zero it once before the first forward   */
} moe_fwd_state;
/* The per-stage entry points below (moe_permute, moe_grouped_ffn_*,
 * moe_unpermute*, their _reordered forms) take the layer's own R-row buffers:
 * with cfg->stash_pool_pages > 0 they return MOE_ERR_UNSUPPORTED, and paged
 * stashing runs through moe_layer_fwd / moe_layer_bwd. */

/* Backward temporaries (device pointers, caller-owned). */
typedef struct moe_bwd_state {
    void* dO_perm;           /* [R,H]   bf16 gradient at the expert outputs     */
    float* dw;               /* [T,k]   gradient of the routing weights         */
    float* dlogits;          /* [T,E]   gradient of the logits                  */
    void* dGU;               /* [R,2F]  bf16 gradient of gate|up                */
    void* dX_perm;           /* [R,H]   bf16 gradient of the dispatched tokens  */
} moe_bwd_state;

/* Worst-case buffer sizes. Returns MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED
 * for configurations the library rejects: H and F must be multiples of 128,
 * 1 <= k <= E <= 256, E % n_groups == 0, topk_groups*(E/n_groups) >= k,
 * row_align a multiple of 128. Host only. */
MOE_API moe_status moe_query_sizes(const moe_config* cfg, moe_sizes* out);

/* Stage 1, route (es summary §2.1 step 1; router in fp32, §2.4).
 * logits = x W_r^T (fp32 accumulation); selection of the k best experts with
 * ties to the lower index -- softmax: on the fp32 value logits + bias;
 * sigmoid: on sigmoid(logits) + bias evaluated in fp64, optionally limited to
 * the topk_groups best groups (group score: sum of the two best, or the best,
 * selection scores of the group). Weights: softmax over the k selected
 * (renormalised), or route_scale * s_j / sum_sel s.
 * x [T,H] bf16, W_r [E,H] f32, bias [E] f32 or NULL -> logits [T,E] f32,
 * idx [T,k] i32, w [T,k] f32. For E a multiple of 128 the logits run on the
 * tensor cores from an exact three-way bf16 split of W_r kept in `scratch`. */
MOE_API moe_status moe_route(const moe_config* cfg, const void* x, const float* W_r, const float* bias,
                     float* logits, int32_t* idx, float* w, void* scratch, void* stream);

/* Router Replay (es summary §2, RL support: routing decisions recorded by
 * inference replayed in training): stage 1 with the experts given instead of
 * selected. logits as moe_route; idx [T,k] i32 is an input (each entry in
 * [0, E)); w [T,k] f32 = the router's weights for those experts in that order
 * -- softmax over their logits + bias, or route_scale * s_j / sum s -- with
 * moe_route's own arithmetic, so replaying moe_route's idx gives its w (the
 * sigmoid router's exact-path tokens, whose selection needed fp64 keys, can
 * differ by a few fp32 ulp). An index outside [0, E), or one that repeats an
 * earlier slot of the same token, records MOE_ERR_DEVICE_CHECK in the status
 * word and gets weight 0 (moe_permute drops the same entries). The rest of the
 * layer (moe_permute on the same idx, ..., the backward) is unchanged. */
MOE_API moe_status moe_route_replay(const moe_config* cfg, const void* x, const float* W_r,
                            const float* bias, const int32_t* idx, float* logits, float* w,
                            void* scratch, void* stream);

/* Load-balancing auxiliary loss of one batch, and the auxiliary-loss-free
 * update of the selection bias, in one kernel launch after moe_route (es
 * summary §2.3.C, "Fusión de Kernels": routing, permutation and the
 * auxiliary-loss computation fused to save launches; the pages give no
 * formula, so the loss is the switch-style balance loss):
 *   sel_counts[e] = tokens whose idx row holds e (the router's selection,
 *                   before any capacity drop), f_e = sel_counts[e] / (T k),
 *   p_mean[e]     = P_e, the mean over tokens of the router's probability of
 *                   e over all E experts (softmax of logits + bias; sigmoid
 *                   router: sigmoid(logit) normalised over all E),
 *   *loss         = coeff * E * sum_e f_e P_e (uniform routing gives coeff).
 * bias_out (nullable; may equal bias): bias[e] + bias_rate * sign(T k / E -
 * sel_counts[e]) (bias NULL counts as 0), the sign step that moves every
 * expert's selection bias towards the mean load.
 * logits [T,E] fp32 and idx [T,k] int32 as written by moe_route; sel_counts
 * [E] int32, p_mean [E] fp32, loss [1] fp32, bias_out [E] fp32: device.
 * Deterministic (fixed summation order). An index outside [0, E) records
 * MOE_ERR_DEVICE_CHECK and is not counted. T == 0 gives zeros (bias_out =
 * bias). scratch: moe_sizes.scratch_bytes bytes, zero-filled once (the
 * launch keeps an arrival counter in it and leaves it zero). Returns
 * MOE_ERR_INVALID_ARG for a NULL or misaligned pointer (logits and idx may be
 * NULL when T == 0) or a non-finite coeff or bias_rate. */
MOE_API moe_status moe_route_aux(const moe_config* cfg, const float* logits, const float* bias,
                                 const int32_t* idx, float coeff, float bias_rate,
                                 int32_t* sel_counts, float* p_mean, float* loss,
                                 float* bias_out, void* scratch, void* stream);

/* Backward of moe_route_aux's loss, scaled by dloss (host scalar, the
 * gradient of the training loss w.r.t. *loss), with sel_counts held fixed:
 *   dlogits_aux[t,e] = dloss * d loss / d logits[t,e]   ([T,E] fp32, written;
 *       softmax p (g_e - sum_j p_j g_j), sigmoid s(1-s)/S (g_e - sum_j p_j g_j),
 *       g_e = coeff E sel_counts[e] / (T^2 k)),
 *   dx   [T,H] bf16  += dlogits_aux . W_r   (fp32 sum over e, one rounding),
 *   dW_r [E,H] fp32  += dlogits_aux^T . x   (every token, every expert).
 * Call it after moe_layer_bwd (or moe_permute_bwd and moe_router_wgrad) with
 * the same dx and dW_r: the loss's gradient reaches x and W_r through the
 * logits like the layer's own. x, logits and bias as given to moe_route.
 * For E a multiple of 128 the dx product runs on the tensor cores from the
 * hi + mid bf16 parts of dlogits_aux and W_r (three cross products; what they
 * leave out is about 2^-16 of sum |dl| |W_r|, far below dx's bf16 rounding),
 * otherwise on the CUDA cores in fp32. dlogits_aux and dx 16-byte aligned;
 * scratch: moe_sizes.scratch_bytes bytes (the split operands use its router
 * region). Returns MOE_ERR_INVALID_ARG for a NULL or misaligned pointer or a
 * non-finite coeff or dloss; T == 0 launches nothing. */
MOE_API moe_status moe_route_aux_bwd(const moe_config* cfg, const void* x, const float* logits,
                                     const float* bias, const float* W_r,
                                     const int32_t* sel_counts, float coeff, float dloss,
                                     float* dlogits_aux, void* dx, float* dW_r, void* scratch,
                                     void* stream);

/* Stage 2, dispatch (es summary §2.1 step 2, done locally). A stable counting
 * sort of the (token, slot) assignments by (expert, token): expert e's kept
 * tokens occupy rows offsets[e] .. offsets[e]+counts[e]-1 in increasing token
 * order; segments are padded to row_align rows (or are C rows in capacity
 * mode, where the first C tokens of an expert are kept); shared experts
 * follow, one row per token. Writes the maps and x_perm: the padding rows in
 * the last 128-row block of a segment (the rows the grouped GEMMs read) are
 * zero; rows of a segment past that block (capacity mode, row_align > 128)
 * are not written. token_of is -1 on every padding row.
 * An idx entry outside [0, E), or one that repeats an earlier slot of the
 * same token (only a caller-given idx can), records MOE_ERR_DEVICE_CHECK in
 * the status word and is dropped: row_of = -1, not counted, no row.
 * FP8 mode: every row is also written in its 1-byte form (E4M3 codes of its
 * 1x128 slices, UE8M0 scales) into `scratch`, where moe_grouped_ffn_fwd reads
 * it: pass the same scratch to both.
 * scratch: moe_sizes.scratch_bytes bytes. */
MOE_API moe_status moe_permute(const moe_config* cfg, const void* x, const int32_t* idx,
                       int32_t* counts, int32_t* offsets, int32_t* row_of, int32_t* token_of,
                       int32_t* sel_offsets, int32_t* sel_tokens, void* x_perm,
                       void* scratch, void* stream);

/* moe_permute without the `scratch` argument: it allocates nothing.
 * The pages have no counterpart; this entry point exists for callers that
 * cannot provide device scratch memory (code inside a framework that owns all
 * device memory, or on a path where cudaMalloc may not be called). Its scratch
 * is a fixed 512 KiB array inside the library, resident on every GPU that
 * loads the library until the process exits.
 *  - Limit: configurations whose dispatch scratch (4096 + 4*E*ceil(T/256) +
 *    256 bytes, rounded up to 256) exceeds 512 KiB return MOE_ERR_WORKSPACE
 *    without launching anything.
 *  - Every call looks up the array's device address in the current context
 *    (the first lookup on a device may load the library's device code, so
 *    make the first call on each device before any stream capture).
 *  - All calls share the one array, which keeps the last call's contents:
 *    calls whose kernels overlap on the GPU (e.g. on two streams) race. Each
 *    call clears the array's status word; index problems a kernel finds are
 *    recorded there and are not reported by this call.
 *  - bf16 configurations only (MOE_ERR_UNSUPPORTED otherwise): in the FP8
 *    configuration the dispatch also writes x_perm's E4M3 form into the
 *    caller's scratch, which this entry point does not take.
 * Other arguments, layouts and results are those of moe_permute. */
MOE_API moe_status moe_permute_noalloc(const moe_config* cfg, const void* x, const int32_t* idx,
                                       int32_t* counts, int32_t* offsets, int32_t* row_of,
                                       int32_t* token_of, int32_t* sel_offsets,
                                       int32_t* sel_tokens, void* x_perm, void* stream);

/* The status word of the no-scratch dispatch's array: synchronises `stream`,
 * then copies to *code (host) what the last moe_permute_noalloc call on the
 * current device recorded -- 0, or MOE_ERR_DEVICE_CHECK for an idx entry
 * outside [0, E) or repeated within a token. Allocates nothing. */
MOE_API moe_status moe_permute_noalloc_status(int32_t* code, void* stream);

/* FP8 mode only (es summary §2.4: expert GEMMs in FP8, MXFP8 -- power-of-two
 * block scales -- on Blackwell): quantises the expert weights W13 [G,2F,H] and
 * W2 [G,H,F] (bf16) into E4M3 codes with one UE8M0 scale per 128x128 tile,
 * kept in `scratch` for the FP8 grouped GEMMs (both orientations of every
 * weight: forward and data gradient). Call it after every change of the
 * weights and before moe_grouped_ffn_fwd / moe_grouped_ffn_dgrad on the same
 * scratch (moe_layer_fwd calls it itself). A tile whose largest magnitude is
 * below 448 * 2^-128 is scaled by 2^-127, the smallest UE8M0 scale. In bf16
 * mode it launches nothing and returns MOE_OK. */
MOE_API moe_status moe_quantize_weights(const moe_config* cfg, const void* W13, const void* W2,
                                        void* scratch, void* stream);

/* FP8 block recipe (MOE_DTYPE_FP8_E4M3_BLOCK; MOE_ERR_UNSUPPORTED otherwise):
 * expert weights the caller quantised itself, in place of moe_quantize_weights.
 * W13_e4m3 [G,2F,H] and W2_e4m3 [G,H,F]: E4M3 codes (1 byte each, 16-byte
 * aligned); W13_scale [G, 2F/128, H/128] and W2_scale [G, H/128, F/128]: one
 * UE8M0 code per 128x128 tile (the tile's weights are code value x
 * 2^(scale - 127)). The codes are copied into `scratch` and the scales laid
 * out as the GEMMs read them, for both orientations. moe_layer_fwd skips its
 * own weight quantisation when params->W13 and params->W2 are both NULL in
 * an FP8 mode and uses what scratch holds (so E4M3 weights kept across several
 * steps are loaded once); the FP8 backward never reads the bf16 weights. */
MOE_API moe_status moe_load_fp8_weights(const moe_config* cfg, const void* W13_e4m3,
                                        const uint8_t* W13_scale, const void* W2_e4m3,
                                        const uint8_t* W2_scale, void* scratch, void* stream);

/* Stage 3, compute (es summary §2.1 step 3; grouped GEMM, §2.3.C): for every
 * group g, on its rows X: [G|U] = X W13[g]^T (GU, bf16), h = bf16(silu(G) U),
 * y_perm = bf16(h W2[g]^T). tcgen05 grouped GEMMs that read counts/offsets on
 * the device. FP8 mode: both GEMMs run on the block-scaled FP8 tensor cores
 * (tcgen05 kind::mxf8f6f4) with the weights moe_quantize_weights left in
 * scratch and the 1-byte x_perm that moe_permute left there (W13, W2 and
 * x_perm are then not read); h is quantised in 1x128 slices (E4M3 + UE8M0,
 * kept in scratch) for FC2. */
MOE_API moe_status moe_grouped_ffn_fwd(const moe_config* cfg, const void* x_perm, const int32_t* counts,
                               const int32_t* offsets, const void* W13, const void* W2,
                               void* GU, void* h, void* y_perm, void* scratch, void* stream);

/* Stage 4, combine (es summary §2.1 step 4, done locally):
 * out[t] = bf16( sum_j w[t,j] y_perm[row_of[t,j]] + sum_s y_perm[offsets[E+s]+t] ),
 * fp32 accumulation; dropped assignments contribute 0. w may be NULL: unit
 * weights (the layer with the weight inside the expert, whose y_perm rows
 * already carry it). */
MOE_API moe_status moe_unpermute(const moe_config* cfg, const void* y_perm, const int32_t* row_of,
                         const float* w, const int32_t* offsets, void* out, void* stream);

/* Backward of stage 4: dO_perm[row_of[t,j]] = bf16(w[t,j] dY[t]),
 * dw[t,j] = <dY[t], y_perm[row_of[t,j]]> (0 if dropped); shared rows get dY;
 * padding rows of dO_perm are zeroed as moe_permute zeroes those of x_perm
 * (the ones in the last 128-row block of a segment). FP8 mode: every row is
 * also written in its 1-byte form (E4M3 codes of its 1x128 slices, UE8M0
 * scales) into `scratch`, where moe_grouped_ffn_dgrad reads it: pass the same
 * scratch to both. scratch: moe_sizes.scratch_bytes bytes. */
MOE_API moe_status moe_unpermute_bwd(const moe_config* cfg, const void* dY, const void* y_perm,
                             const int32_t* row_of, const float* w, const int32_t* counts,
                             const int32_t* offsets, void* dO_perm, float* dw, void* scratch,
                             void* stream);

/* Data-gradient half of moe_grouped_ffn_bwd (the W/D split of es summary
 * §2.3.B): dGU and dX_perm exactly as moe_grouped_ffn_bwd writes them. FP8
 * mode: both GEMMs run on the block-scaled FP8 tensor cores with the weights
 * moe_quantize_weights left in scratch and the 1-byte dO that
 * moe_unpermute_bwd left there (W13, W2 are then not read, dO_perm only by the
 * weight gradients); dGU is quantised in 1x128 slices for FC1's and, in the
 * same pass, in 128x1 slices for moe_grouped_ffn_wgrad.
 * h: NULL, or h [R,F] bf16 to rewrite from GU in the FC2 data-gradient
 * epilogue (bit for bit the forward's h: the fine-grained recompute of the
 * activation function), so that the weight gradient can run after the forward's
 * h was discarded. */
MOE_API moe_status moe_grouped_ffn_dgrad(const moe_config* cfg, const void* dO_perm,
                                         const void* GU, void* h, const int32_t* counts,
                                         const int32_t* offsets, const int32_t* token_of,
                                         const float* dlogits, const float* W_r, const void* W13,
                                         const void* W2, void* dGU, void* dX_perm, void* scratch,
                                         void* stream);

/* Weight-gradient half of moe_grouped_ffn_bwd: dW2[g] = dO^T h and
 * dW13[g] = dGU^T x_perm over the group's rows (bf16, zero for empty groups),
 * after moe_grouped_ffn_dgrad has written dGU. FP8 mode: both operands are
 * quantised to E4M3 in 128x1 slices along the group's tokens (into scratch)
 * and multiplied on the block-scaled FP8 tensor cores; dGU's E4M3 form is the
 * one moe_grouped_ffn_dgrad left in scratch (the dGU argument is not read), so
 * pass the scratch of that call. */
MOE_API moe_status moe_grouped_ffn_wgrad(const moe_config* cfg, const void* dO_perm,
                                         const void* x_perm, const void* h, const void* dGU,
                                         const int32_t* counts, const int32_t* offsets,
                                         void* dW13, void* dW2, void* scratch, void* stream);

/* Backward of stage 3 (the W/D split of es summary §2.3.B: separate data- and
 * weight-gradient GEMMs; moe_grouped_ffn_dgrad then moe_grouped_ffn_wgrad):
 * dh = dO W2[g] (fp32, not stored); SwiGLU backward
 * with the stored GU -> dGU (bf16); dW2[g] = dO^T h; dW13[g] = dGU^T x_perm
 * (weight gradients in bf16, zero for empty groups);
 * dX_perm[r] = bf16( dGU[r] W13[g] + dlogits[token_of[r], g] W_r[g] ) for the
 * rows r of a routed expert g (< E), bf16(dGU[r] W13[g]) for shared experts.
 * The second term is the router-logit gradient of the row's assignment: the
 * part of dx that flows through logit (t, g). It is added in the GEMM's fp32
 * epilogue, where W_r[g] is one row for a whole tile, instead of in
 * moe_permute_bwd, which would read k rows of W_r for every token.
 * token_of [rows_max] i32 and dlogits [T,E] f32 come from moe_permute and
 * moe_route_bwd; W_r [E,H] f32. */
MOE_API moe_status moe_grouped_ffn_bwd(const moe_config* cfg, const void* dO_perm, const void* x_perm,
                               const void* GU, const void* h, const int32_t* counts,
                               const int32_t* offsets, const int32_t* token_of,
                               const float* dlogits, const float* W_r, const void* W13,
                               const void* W2, void* dGU, void* dX_perm, void* dW13, void* dW2,
                               void* scratch, void* stream);

/* The layer with the routing weight inside the expert (cfg->weights_in_expert
 * = 1; the memory-efficient permutation of es summary §2.3.A: an algebraic
 * reordering of the routing weights, so that the permuted expert outputs are
 * not needed by the backward). Since y = h W2^T is linear in h, the weight
 * moves before FC2:
 *   forward:  h[r] = bf16(w_row silu(G) U) (GU as in moe_grouped_ffn_fwd),
 *             y_perm = bf16(h W2^T), then moe_unpermute with w = NULL;
 *   backward: dO_perm rows = dY[t] unweighted (moe_unpermute_bwd_reordered),
 *             dh_s = dO W2 (fp32), dw[t,j] = <dh_s, silu(G) U> of the row,
 *             dh = w_row dh_s into the SwiGLU backward -> dGU, then dlogits
 *             from dw (as moe_route_bwd), then dX_perm as moe_grouped_ffn_bwd
 *             with that dlogits; moe_grouped_ffn_wgrad gives dW2 = dO^T h.
 * y_perm is read only by the combine: its buffer need not survive from the
 * forward to the backward. w_row is w[t,j] of the row's assignment (1 for a
 * shared expert's row, 0 for padding), kept in `scratch` by the forward: pass
 * the forward's scratch to the backward. bf16 mode only.
 * moe_grouped_ffn_fwd_reordered: x_perm, counts, offsets, token_of, row_of
 * from moe_permute and w from moe_route; writes GU, h (the weighted h_s) and
 * y_perm. Returns MOE_ERR_INVALID_ARG unless cfg->weights_in_expert = 1. */
MOE_API moe_status moe_grouped_ffn_fwd_reordered(const moe_config* cfg, const void* x_perm,
                                                 const int32_t* counts, const int32_t* offsets,
                                                 const int32_t* token_of, const int32_t* row_of,
                                                 const float* w, const void* W13, const void* W2,
                                                 void* GU, void* h, void* y_perm, void* scratch,
                                                 void* stream);

/* dO_perm[row_of[t,j]] = dY[t] for kept assignments, shared rows get dY,
 * padding rows zero as in moe_unpermute_bwd (no weighting, y_perm not read,
 * no dw). */
MOE_API moe_status moe_unpermute_bwd_reordered(const moe_config* cfg, const void* dY,
                                               const int32_t* row_of, const int32_t* counts,
                                               const int32_t* offsets, void* dO_perm,
                                               void* stream);

/* The data gradients of the layer with the weight inside the expert, with the
 * routing weights' gradient: writes dGU, dw [T,k] (fp32; 0 for dropped
 * assignments), dlogits [T,E] (as moe_route_bwd from dw) and dX_perm (as
 * moe_grouped_ffn_bwd, router term from this dlogits). logits, idx, w from
 * moe_route; the scratch of the forward. Deterministic: dw sums the FC2 data
 * gradient's per-tile partial dot products in tile order. h: NULL, or h_s
 * [R,F] to rewrite from GU and the rows' weights (as moe_grouped_ffn_dgrad). */
MOE_API moe_status moe_grouped_ffn_dgrad_reordered(const moe_config* cfg, const void* dO_perm,
                                                   const void* GU, void* h,
                                                   const int32_t* counts,
                                                   const int32_t* offsets,
                                                   const int32_t* token_of,
                                                   const int32_t* row_of, const float* logits,
                                                   const int32_t* idx, const float* w,
                                                   const float* W_r, const void* W13,
                                                   const void* W2, void* dGU, void* dX_perm,
                                                   float* dw, float* dlogits, void* scratch,
                                                   void* stream);

/* Backward of the routing weights to the logits (dense [T,E], zero outside the
 * selected experts). softmax: dl_j = w_j (dw_j - sum_i w_i dw_i); sigmoid:
 * ds_j = (r/S)(dw_j - sum_i (s_i/S) dw_i), dl_j = ds_j s_j (1 - s_j). */
MOE_API moe_status moe_route_bwd(const moe_config* cfg, const float* logits, const int32_t* idx,
                         const float* w, const float* dw, float* dlogits, void* stream);

/* Backward of stage 2 plus the rest of the router's input gradient:
 * dx[t] = bf16( sum_j dX_perm[row_of[t,j]] + sum_s dX_perm[offsets[E+s]+t]
 *               + sum_{j: row_of[t,j] = -1} dlogits[t, idx[t,j]] W_r[idx[t,j]] ).
 * dX_perm as moe_grouped_ffn_bwd writes it, which already holds the router
 * term of every kept assignment; only assignments dropped by the capacity
 * limit add theirs here. Together: dx[t] = sum over t's rows of the expert
 * input gradients + dlogits[t,:] W_r. */
MOE_API moe_status moe_permute_bwd(const moe_config* cfg, const void* dX_perm, const int32_t* row_of,
                           const int32_t* offsets, const int32_t* idx, const float* dlogits,
                           const float* W_r, void* dx, void* stream);

/* Router weight gradient: dW_r[e] = sum over tokens t that selected e of
 * dlogits[t,e] x[t] (fp32 [E,H]; dlogits is zero outside the selected experts,
 * as moe_route_bwd writes it, so this is dlogits^T x). For E a multiple of 128
 * on the tensor cores: dlogits split exactly into three bf16 parts, each chunk
 * of at most max(1024, ~T/256) tokens summed by the tensor cores (fp32
 * accumulation), the chunks added in order in fp32; otherwise one block per
 * (expert, column slab) summing the expert's selecting tokens (sel_offsets /
 * sel_tokens from moe_permute) in token order. Either way the summation order
 * is fixed: the result is bitwise reproducible. scratch: as moe_query_sizes
 * sizes it (the tensor-core path keeps the split dlogits and the chunk sums
 * there). */
MOE_API moe_status moe_router_wgrad(const moe_config* cfg, const void* x, const int32_t* sel_offsets,
                            const int32_t* sel_tokens, const float* dlogits, float* dW_r,
                            void* scratch, void* stream);

/* The whole layer forward: (FP8 mode: moe_quantize_weights,) route, permute,
 * grouped FFN, unpermute (with weights_in_expert = 1: the reordered grouped
 * FFN and the unweighted combine). */
MOE_API moe_status moe_layer_fwd(const moe_config* cfg, const moe_params* params, const void* x,
                         void* out, const moe_fwd_state* st, void* scratch, void* stream);

/* The whole layer backward from the forward state: dx (bf16), dW_r (fp32),
 * dW13, dW2 (bf16). With a paged stash it ends with moe_stash_release. */
MOE_API moe_status moe_layer_bwd(const moe_config* cfg, const moe_params* params, const void* x,
                         const void* dY, const moe_fwd_state* st, const moe_bwd_state* bs,
                         void* dx, float* dW_r, void* dW13, void* dW2, void* scratch,
                         void* stream);

/* Gives back the stash pages the layer's forward took (cfg->stash_pool_pages
 * > 0): *stash_top = the layer's first page, on the device. moe_layer_bwd calls
 * it; a forward that is not followed by a backward (evaluation) calls it
 * itself. Returns MOE_ERR_INVALID_ARG without a pool or for NULL pointers. */
MOE_API moe_status moe_stash_release(const moe_config* cfg, const moe_fwd_state* st, void* stream);

/* Synchronises `stream`, then copies the device status word from scratch to
 * *code (0 = no problem recorded). */
MOE_API moe_status moe_last_device_status(const void* scratch, int32_t* code, void* stream);

/* Resets the device status word (async on stream). */
MOE_API moe_status moe_clear_device_status(void* scratch, void* stream);

/* Health check of the device-side failure detection: launches one kernel that
 * waits, through the same bounded mbarrier wait every grouped-GEMM role uses,
 * on a barrier that nothing completes. After about `budget_cycles` SM clock
 * cycles the wait gives up and MOE_ERR_TIMEOUT is recorded in the status word
 * of `scratch` (read it with moe_last_device_status); the kernel then exits
 * normally and the context stays usable. */
MOE_API moe_status moe_check_bounded_wait(void* scratch, int64_t budget_cycles, void* stream);

/* Static text for a status code. */
MOE_API const char* moe_status_string(moe_status s);

#ifdef __cplusplus
}
#endif

#endif /* MOE_ABI_H */
