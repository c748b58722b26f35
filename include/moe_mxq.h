/*
 * moe_mxq.h -- C ABI of the MoE expert layer for GB300 (sm_103a).
 *
 * The layer (MegaMoE (study notes), "Baseline implementation" and the data-flow
 * figure after "Combine"; Counting Sort / Bucketization in DeepGEMM Mega MoE,
 * sections 2 and 5):
 *
 *   x bf16 [T,H] --mxq_quantize_act--> xq e4m3 [T,H] + xs ue8m0 [T,H/32]
 *   logits f32 [T,E] --moe_route_topk--> topk_idx i32 [T,k], topk_w f32 [T,k]
 *   topk_idx --moe_permute--> counts [E], offsets [E+1], perm [P], inv_perm [P]
 *   moe_expert_forward: GEMM1 (W1|W3) + SwiGLU (.) topk_w + FP8 requant,
 *                       GEMM2 (W2) -> y_pairs bf16 [k,T,H]
 *   moe_combine: y[t] = bf16( sum_j y_pairs[j,t] ) -> y bf16 [T,H]
 *   moe_forward: all of the above in one call.
 *
 * Conventions shared by every entry point
 *   - Tensor arguments are DEVICE pointers owned by the caller.  The library
 *     never allocates, frees or synchronises (except moe_get_device_status,
 *     which synchronises the given stream).
 *   - Work is enqueued on the given stream; the return value is a status
 *     (enum moe_status).  When the host detects an error nothing is enqueued.
 *   - BF16 is passed as uint16_t bit patterns; FP8 E4M3 codes and UE8M0 scale
 *     bytes as uint8_t; FP4 E2M1 codes are packed two per byte, the even K
 *     index in the low nibble.  Indices are int32_t.
 *   - UE8M0 byte b means 2^(b-127); the scale of a 32-group is
 *     2^ceil(log2(amax/Q)), Q = 448 (E4M3) or 6 (E2M1), clamped to bytes
 *     [0,254]; amax = 0 gives byte 0.  Codes round to nearest, ties to even;
 *     the sign of values that round to zero is kept.
 *   - Shape limits: K (= H or I) a multiple of 128; 1 <= k <= min(E, 32);
 *     1 <= E <= 1024; T >= 0 (T = 0 is a no-op); T*k < 2^31.
 *   - Pointer alignment: 16 bytes for every tensor, 32 bytes for packed FP4
 *     weights (MOE_ERR_MISALIGNED otherwise).
 */
#ifndef MOE_MXQ_H
#define MOE_MXQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

/* Same definition as the CUDA runtime's cudaStream_t. */
struct CUstream_st;
typedef struct CUstream_st *cudaStream_t;

enum moe_status {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,         /* null pointer, negative size, bad enum   */
    MOE_ERR_UNSUPPORTED_SHAPE = 2,   /* outside the shape limits above          */
    MOE_ERR_MISALIGNED = 3,          /* pointer alignment rule broken           */
    MOE_ERR_WORKSPACE_TOO_SMALL = 4, /* workspace_bytes below the stated size   */
    MOE_ERR_CUDA = 5,                /* a CUDA launch or driver call failed     */
    MOE_ERR_TIMEOUT = 6,             /* a device-side wait gave up (status word)*/
    MOE_ERR_DEVICE_INDEX = 7         /* device found an index out of range      */
};

/* Layouts of quantised weights (mxq_quantize_weight).
 *
 * MXQ_LAYOUT_CANONICAL: codes [G][N][K/2] (row n, packed along K),
 *   scales [G][N][K/32].
 * MXQ_LAYOUT_MMA_L1 (GEMM1 weights, N = 2I with gate rows [0,I) and up rows
 *   [I,2I) in the input): rows are interleaved in groups of 8, gate then up
 *   (MegaMoE (study notes), "_interleave_l1_weights (gran = 8)"): stored row
 *   r = 16b + c holds input row 8b + c when c < 8 and row I + 8b + c - 8
 *   otherwise.  Codes are stored in tile-contiguous blocks
 *   [G][N/128][K/128][128][64]: block (g, nt, kb) holds stored rows
 *   128*nt .. 128*nt+127, K values 128*kb .. 128*kb+127, each row packed in
 *   64 bytes, so one 128 x 128 weight tile is 8 KB in one piece.  Scales are
 *   in MMA chunk order: [G][N/128][K/128][512], where byte
 *   (r%32)*16 + (r/32)*4 + kk of chunk (g, nt, kb) is the scale of stored row
 *   128*nt + r, K-group 4*kb + kk.  N must be a multiple of 128.
 * MXQ_LAYOUT_MMA_L2 (GEMM2 weights): rows in input order, codes and scales
 *   in the same tile-contiguous / chunk orders.
 */
enum mxq_layout { MXQ_LAYOUT_CANONICAL = 0, MXQ_LAYOUT_MMA_L1 = 1, MXQ_LAYOUT_MMA_L2 = 2 };

/* Activation cast BF16 -> FP8 E4M3 + UE8M0 per 32 along K.
 * MegaMoE (study notes), "Dispatch" section (per-token cast, gran_k = 32).
 * x [rows][K] bf16; q [rows][K] e4m3; s [rows][K/32] ue8m0.  rows >= 0. */
MOE_API int mxq_quantize_act(const uint16_t *x, int64_t rows, int64_t K,
                     uint8_t *q, uint8_t *s, cudaStream_t stream);

/* Weight cast BF16 [G][N][K] -> FP4 E2M1 packed + UE8M0 per 32 along K, no
 * grouping along N.  MegaMoE (study notes), "Expert weight quantisation";
 * the MMA layouts are described at enum mxq_layout.
 * q: G*N*K/2 bytes; s: G*N*K/32 bytes. */
MOE_API int mxq_quantize_weight(const uint16_t *w, int64_t G, int64_t N, int64_t K, int layout,
                        uint8_t *q, uint8_t *s, cudaStream_t stream);

/* Routing modes: the score (low two bits) and MOE_ROUTE_NO_RENORM.  0 is
 * the default, softmax renormalised over the k chosen.  Raw scores are never
 * renormalised (MOE_ROUTE_RAW with or without the flag). */
enum moe_route_mode {
    MOE_ROUTE_SOFTMAX = 0,       /* softmax over the E logits                  */
    MOE_ROUTE_SIGMOID = 1,       /* s = 1 / (1 + exp(-l)) per expert           */
    MOE_ROUTE_RAW = 2,           /* the logits themselves (MegaMoE test)       */
    MOE_ROUTE_NO_RENORM = 4      /* flag: keep the scores of the k chosen as is */
};

/* Router: per token, the k largest logits (equal logits: lower expert index
 * first; -0.0 equals +0.0), in descending order, and their weights.  Every
 * score is an increasing function of the logit, so ranking the logits
 * selects the k best scores.  With l_max the top logit and S the k chosen:
 *   softmax:              w_j = exp(l_j - l_max) / sum_{i in S} exp(l_i - l_max)
 *   softmax | NO_RENORM:  w_j = exp(l_j - l_max) / sum_{all e} exp(l_e - l_max)
 *   sigmoid:              w_j = s_j / sum_{i in S} s_i
 *   sigmoid | NO_RENORM:  w_j = s_j
 *   raw:                  w_j = l_j
 * MonoMoe kernel -- design, section 1 (phase 1: softmax or sigmoid top-K with
 * optional renormalisation); raw scores as the MegaMoE test's topk of randn
 * scores (Counting Sort / Bucketization in DeepGEMM Mega MoE, section 7.1).
 * logits [T][E] f32 (finite); topk_idx [T][k] i32; topk_w [T][k] f32.
 * 1 <= k <= min(E, 32), E <= 1024; an unknown mode is MOE_ERR_INVALID_ARG.
 * moe_route_topk is moe_route_topk_ex with mode MOE_ROUTE_SOFTMAX. */
MOE_API int moe_route_topk(const float *logits, int64_t T, int32_t E, int32_t k,
                   int32_t *topk_idx, float *topk_w, cudaStream_t stream);
MOE_API int moe_route_topk_ex(const float *logits, int64_t T, int32_t E, int32_t k, int32_t mode,
                   int32_t *topk_idx, float *topk_w, cudaStream_t stream);

/* Counting-sort permute of the P = T*k (token, slot) pairs, pair id
 * p = t*k + j.  Counting Sort / Bucketization in DeepGEMM Mega MoE,
 * sections 2.1 (count), 2.2 (prefix sum), 2.3 (scatter), 8.2 (pair id).
 *   counts[e]  = number of pairs with topk_idx == e             [E]
 *   offsets[e] = sum of counts[e'] for e' < e; offsets[E] = total [E+1]
 *   perm[offsets[e] + r] = the r-th smallest pair id routed to e  [P]
 *                          (stable: token-ascending; entries past offsets[E] untouched)
 *   inv_perm[p] = position of p in perm, or -1 for a dropped pair  [P]
 * topk_idx < 0 marks a dropped pair; topk_idx >= E is reported through the
 * device status word (MOE_ERR_DEVICE_INDEX) of the workspace and the pair is
 * treated as dropped.  Deterministic: no result depends on thread timing.
 * workspace: at least moe_permute_workspace_size(T, E, k) bytes, 256-byte
 * aligned; its status word is reset by the call. */
MOE_API size_t moe_permute_workspace_size(int64_t T, int32_t E, int32_t k);
MOE_API int moe_permute(const int32_t *topk_idx, int64_t T, int32_t E, int32_t k,
                int32_t *counts, int32_t *offsets, int32_t *perm, int32_t *inv_perm,
                void *workspace, size_t workspace_bytes, cudaStream_t stream);

/* moe_permute for callers that cannot allocate device memory (no counterpart
 * on the pages).  Some callers have no workspace to give: plugins inside a
 * host framework that owns every device allocation, or serving loops that
 * must not call cudaMalloc while they run.  Same inputs, outputs and results
 * as moe_permute, but the scratch (status words and the per-block expert
 * histogram) is a file-scope device array of the library: 256 bytes plus
 * MOE_PERMUTE_NOALLOC_MAX_HIST_BYTES, held by every GPU that loads the
 * library until the process exits.  Nothing is allocated or freed.
 *   device_status: optional caller-owned device int32 (NULL = not reported);
 *     set to 0 by the call, then to MOE_ERR_DEVICE_INDEX if an index >= E
 *     was seen.
 * Errors: MOE_ERR_UNSUPPORTED_SHAPE when the histogram would exceed the
 * array (moe_permute_workspace_size(T,E,k) - 256 > the maximum, e.g. E = 1024
 * with more than 32768 pairs); MOE_ERR_CUDA if the array's device address
 * cannot be looked up.
 * The first call on each device looks up the array's address (once per
 * device and context, with that device current; a device reset replaces the
 * context and the next call looks it up again); make that first call before
 * any stream capture.
 * All calls on a device share the array, which keeps the last call's
 * contents: calls that overlap on the GPU race. */
#define MOE_PERMUTE_NOALLOC_MAX_HIST_BYTES 65536
MOE_API int moe_permute_noalloc(const int32_t *topk_idx, int64_t T, int32_t E, int32_t k,
                                int32_t *counts, int32_t *offsets, int32_t *perm, int32_t *inv_perm,
                                int32_t *device_status, cudaStream_t stream);

/* Grouped expert GEMMs: GEMM1 (FP8 x FP4 W1|W3, FP32 accumulate) with the
 * fused epilogue h = silu(gate) * up * topk_w, requantised to E4M3 + UE8M0
 * per 32 along I; then GEMM2 (FP8 h x FP4 W2) cast to BF16 per pair.
 * MegaMoE (study notes), "L1 epilogue", "L2 epilogue"; Warp Specialization:
 * DeepEP vs Mega MoE, epilogue listings.
 *   xq/xs: activations [T][H] / [T][H/32] (mxq_quantize_act)
 *   w1q/w1s: GEMM1 weights [E][2I][H] in MXQ_LAYOUT_MMA_L1
 *   w2q/w2s: GEMM2 weights [E][H][I] in MXQ_LAYOUT_MMA_L2
 *   topk_idx/topk_w [T][k]; counts/offsets/perm from moe_permute
 *   y_pairs: output, bf16 [k][T][H]; row (j, t) holds pair p = t*k + j.
 *            Rows of dropped pairs are not written.
 *   hq/hs: optional outputs (NULL = not written): the requantised h in pool
 *          order, hq [P][I] e4m3 and hs [P][I/32] ue8m0, row s = pair perm[s].
 *   tile_n: token tile (16, 32, 64, 128, 208, 224) or 0 to let the library
 *          choose.  208 and 224 both mean the large tile: 208 tokens with the
 *          GEMMs on CTA pairs where both GEMMs' 128-row weight tiles pair up
 *          (2I/128 and H/128 even), 224 tokens on single CTAs otherwise.
 *   phases: 0 for the whole layer, or a mask of enum moe_phase to run steps
 *          separately on the same workspace (same tile_n in every call):
 *          TOKEN_SCALES gathers GEMM1's token scales into the workspace;
 *          GEMM1 writes h (to hq if given, else to the workspace) and GEMM2's
 *          scale chunks; GEMM2 reads them; H_SCALES instead builds GEMM2's
 *          scale chunks from a caller-provided h (hq and hs required, pool
 *          order), so that GEMM2 can run on an h computed elsewhere.
 *   workspace: at least moe_expert_workspace_size(...) bytes, 256-byte aligned.
 */
enum moe_phase {
    MOE_PHASE_TOKEN_SCALES = 1,
    MOE_PHASE_GEMM1 = 2,
    MOE_PHASE_GEMM2 = 4,
    MOE_PHASE_H_SCALES = 8,
    MOE_PHASE_RESET = 16      /* moe_forward only: zero the status words and arrival counters */
};

typedef struct moe_expert_args {
    uint32_t struct_size;   /* sizeof(moe_expert_args) */
    int64_t T, H, I;
    int32_t E, k;
    const uint8_t *xq, *xs;
    const uint8_t *w1q, *w1s, *w2q, *w2s;
    const int32_t *topk_idx;
    const float *topk_w;
    const int32_t *counts, *offsets, *perm;
    uint16_t *y_pairs;
    uint8_t *hq, *hs;
    int32_t tile_n;
    int32_t phases;
    void *workspace;
    size_t workspace_bytes;
} moe_expert_args;

MOE_API size_t moe_expert_workspace_size(int64_t T, int64_t H, int64_t I, int32_t E, int32_t k);
MOE_API int moe_expert_forward(const moe_expert_args *args, cudaStream_t stream);

/* Top-k combine: y[t][n] = bf16( sum over slots j with topk_idx[t][j] >= 0 of
 * y_pairs[j][t][n] ), summed in FP32 in slot order.  The top-k weight was
 * applied before GEMM2, so the sum is unweighted.  MegaMoE (study notes),
 * "Combine" and "L2 epilogue"; Warp Specialization: DeepEP vs Mega MoE,
 * combine listing.  y_pairs [k][T][H]; y [T][H]. */
MOE_API int moe_combine(const uint16_t *y_pairs, const int32_t *topk_idx, int64_t T, int32_t k,
                int64_t H, uint16_t *y, cudaStream_t stream);

/* The whole layer in one call (quantise, route, permute, GEMM1+epilogue,
 * GEMM2, combine).  Inputs: x bf16 [T][H], logits f32 [T][E], weights as for
 * moe_expert_forward.  Output y bf16 [T][H].  Optional outputs (NULL = not
 * written): topk_idx/topk_w [T][k], counts [E], offsets [E+1], perm [P].
 * workspace: at least moe_workspace_size(T, H, I, E, k) bytes, 256-byte
 * aligned; the call resets what it needs, callers do not zero it. */
typedef struct moe_forward_args {
    uint32_t struct_size;   /* sizeof(moe_forward_args) */
    int64_t T, H, I;
    int32_t E, k;
    const uint16_t *x;
    const float *logits;
    const uint8_t *w1q, *w1s, *w2q, *w2s;
    uint16_t *y;
    int32_t *topk_idx_out;
    float *topk_w_out;
    int32_t *counts_out, *offsets_out, *perm_out;
    int32_t tile_n;
    void *workspace;
    size_t workspace_bytes;
    int32_t route_mode;     /* enum moe_route_mode; 0 = softmax, renormalised */
    /* 0: the whole layer.  Otherwise a mask of enum moe_phase, for timing the
     * expert GEMMs alone on the state that an earlier whole-layer call with
     * the same arguments left in the workspace:
     *   MOE_PHASE_RESET zeroes the status words and arrival counters (the
     *     first thing a whole-layer call does);
     *   MOE_PHASE_GEMM1 / MOE_PHASE_GEMM2 re-run the layer's GEMM launches
     *     (the same kernels and launch shapes as the whole-layer call); where
     *     the layer runs GEMM1, GEMM2 and the combine in one launch, both bits
     *     are required together, that launch also writes y, and its arrival
     *     counters must have been zeroed (RESET, in this call or an earlier one).
     * RESET runs before the GEMMs when combined.  Routing, permute and the
     * activation cast are not re-run.  Other bits: MOE_ERR_INVALID_ARG. */
    int32_t phases;
    /* enum moe_schedule: how large problems whose GEMMs run on CTA pairs
     * (208-token tiles, see tile_n) schedule GEMM1, GEMM2 and the combine.
     * Ignored elsewhere.  Other values: MOE_ERR_INVALID_ARG. */
    int32_t schedule;
} moe_forward_args;

enum moe_schedule {
    /* the library's choice: currently MOE_SCHEDULE_SEPARATE (measured faster) */
    MOE_SCHEDULE_DEFAULT = 0,
    /* GEMM1, GEMM2 and the combine as three launches */
    MOE_SCHEDULE_SEPARATE = 1,
    /* one persistent launch that walks expert waves: GEMM1 items of a wave of
     * token tiles, then (one wave later) its GEMM2 items, which wait on per-
     * tile arrival counters, then the combine (MegaMoE (study notes), "Wave",
     * "Scheduler"; MegaMoE overview, "3. Wave-Based Expert Processing").
     * Every CTA of the launch must be resident at once (one per SM); if the
     * GPU is shared so that some cannot be, the waits give up with
     * MOE_ERR_TIMEOUT instead of hanging. */
    MOE_SCHEDULE_EXPERT_WAVES = 2
};

MOE_API size_t moe_workspace_size(int64_t T, int64_t H, int64_t I, int32_t E, int32_t k);
MOE_API int moe_forward(const moe_forward_args *args, cudaStream_t stream);

/* Reads the device status word that kernels write into a workspace (first
 * 4 bytes of any workspace above): MOE_OK, MOE_ERR_TIMEOUT (a bounded
 * device-side wait gave up) or MOE_ERR_DEVICE_INDEX.  Synchronises `stream`.
 * The int32 words after it: [1] abort flag (raised by the first timeout;
 * every other wait of the launch then gives up at once), [2] site of the
 * wait that timed out (1 producer/empty stage, 2 MMA/free accumulator,
 * 3 MMA/full stage, 4 epilogue/full accumulator, 5 producer drain, 6 MMA
 * drain, 7 debug wait), [3] its CTA, [4] its loop position.  All are
 * cleared by each moe_forward / moe_expert_forward call.
 *
 * Debug hook for failure-detection tests: with the environment variable
 * MOE_MXQ_DEBUG_INJECT_WAIT=1 set when a GEMM is launched, the MMA warp of
 * every CTA with work first waits on a barrier that nothing completes; the
 * wait gives up after ~10 ms and the launch ends with MOE_ERR_TIMEOUT, site
 * 7, without faulting and with the context still usable. */
MOE_API int moe_get_device_status(const void *workspace, cudaStream_t stream, int *out);

/* Human-readable text of a status code (static storage). */
MOE_API const char *moe_status_string(int status);

/* Library version string (static storage). */
MOE_API const char *moe_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_MXQ_H */
