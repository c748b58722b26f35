/*
 * moe_bfp8.h -- C ABI of the block-FP8 variant of the MoE expert layer for
 * GB300 (sm_103a).
 *
 * The variant is the single-kernel top-k MoE of the MonoMoe kernel design
 * page ("Fixed shape": E = 256 experts, hidden K = 2048, N = 512 rows each for
 * gate and up, at most 8 tokens, block-FP8 (128 x 128) weights; section 1,
 * "Five-phase pipeline": routing, BF16 -> FP8 cast of the input, up-projection
 * + SiLU with an FP8 write-back, down-projection with FP32 partials summed
 * per token, BF16 cast).  Any shape within the limits below is accepted.
 *
 *   x bf16 [T,H] --bfp8_quantize_act--> xq e4m3 [T,H] + xs f32 [T,H/128]
 *   routing and the counting-sort permute as in moe_mxq.h
 *   GEMM1: acc[j] = sum_kb w1s[e][j/128][kb] * xs[t][kb] * <xq[t], w1q[e][j]>_kb
 *          h = silu(acc[0..I)) * acc[I..2I)  -> hq e4m3 + hs f32 per 128 along I
 *   GEMM2: y_pair[n] = sum_kb w2s[e][n/128][kb] * hs[p][kb] * <hq[p], w2q[e][n]>_kb
 *   y[t] = bf16( sum over the token's valid slots j of topk_w[t][j] * y_pair )
 *
 * Formats (all in this file):
 *   - E4M3 codes are uint8_t (OCP FP8 "FN": max 448, no infinities).
 *   - A scale is a float32: scale = amax / 448 over its group (128 values of
 *     one row along K for activations and h; one 128 x 128 block for weights),
 *     computed in float32 with round-to-nearest; codes are the E4M3
 *     round-to-nearest-even of value / scale computed in float32, saturating
 *     at +-448; the sign of values that round to zero is kept.  A group whose
 *     amax is 0 has scale 0 and all codes 0.
 *   - Weights: l1 [E][2I][H] (gate rows [0,I), up rows [I,2I)) with scales
 *     [E][2I/128][H/128]; l2 [E][H][I] with scales [E][H/128][I/128].  The
 *     scales are always in that order; the codes are stored in one of two
 *     layouts (enum bfp8_layout):
 *       BFP8_LAYOUT_CANONICAL: row-major [G][N][K];
 *       BFP8_LAYOUT_TILED: tile-contiguous [G][N/128][K/128][128][128] --
 *         each 128 x 128 block is 16 KB in one piece (rows of 128 codes), so
 *         that a GEMM streams whole DRAM pages instead of 128-byte pieces of
 *         rows 2 KB apart.
 *
 * Conventions are those of moe_mxq.h: device pointers owned by the caller,
 * no allocation, no synchronisation, work enqueued on `stream`, a moe_status
 * returned (nothing enqueued when the host detects an error), device status
 * in the first bytes of the workspace (moe_get_device_status).
 * Shape limits: H and I multiples of 128; 1 <= E <= 1024; 1 <= k <= min(E, 32);
 * T >= 0 (T = 0 is a no-op); T*k < 2^31.  Alignment: 16 bytes for every
 * tensor except the float32 scale arrays (w1s, w2s, s, hs_out), which need
 * 4 bytes, so that one expert's slice of a stacked array can be passed.
 */
#ifndef MOE_BFP8_H
#define MOE_BFP8_H

#include "moe_mxq.h"

#ifdef __cplusplus
extern "C" {
#endif

/* BF16 [rows, K] -> E4M3 codes [rows, K] and float32 scales [rows, K/128],
 * one scale per 128 consecutive values of a row (MonoMoe kernel design,
 * section 1, phase 2).  K must be a multiple of 128.  Out of range sizes:
 * MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED_SHAPE. */
MOE_API int bfp8_quantize_act(const uint16_t *x, int64_t rows, int64_t K, uint8_t *q, float *s,
                              cudaStream_t stream);

enum bfp8_layout { BFP8_LAYOUT_CANONICAL = 0, BFP8_LAYOUT_TILED = 1 };

/* BF16 [G, N, K] -> E4M3 codes (layout: enum bfp8_layout) and float32 scales
 * [G, N/128, K/128], one per 128 x 128 block (MonoMoe kernel design, "Fixed
 * shape").  N and K must be multiples of 128; another layout value:
 * MOE_ERR_INVALID_ARG. */
MOE_API int bfp8_quantize_weight(const uint16_t *w, int64_t G, int64_t N, int64_t K, int layout, uint8_t *q,
                                 float *s, cudaStream_t stream);

typedef struct moe_bfp8_args {
    uint32_t struct_size;      /* sizeof(moe_bfp8_args) */
    int64_t T, H, I;
    int32_t E, k;
    int32_t route_mode;        /* enum moe_route_mode; 0 = softmax, renormalised */
    const uint16_t *x;         /* [T, H] bf16 */
    const float *logits;       /* [T, E] */
    const uint8_t *w1q;        /* [E, 2I, H] e4m3 */
    const float *w1s;          /* [E, 2I/128, H/128] */
    const uint8_t *w2q;        /* [E, H, I] e4m3 */
    const float *w2s;          /* [E, H/128, I/128] */
    uint16_t *y;               /* out [T, H] bf16 */
    /* optional outputs (NULL = not written): the routing, the permute and the
     * requantised h in pool order (pool row s holds pair perm[s]) */
    int32_t *topk_idx_out;     /* [T, k] */
    float *topk_w_out;         /* [T, k] */
    int32_t *counts_out;       /* [E] */
    int32_t *offsets_out;      /* [E + 1] */
    int32_t *perm_out;         /* [T*k] */
    uint8_t *hq_out;           /* [T*k, I] */
    float *hs_out;             /* [T*k, I/128] */
    void *workspace;           /* moe_bfp8_workspace_size bytes, 256-byte aligned */
    size_t workspace_bytes;
    int32_t weight_layout;     /* enum bfp8_layout of w1q and w2q */
    /* 0: the whole layer.  MOE_PHASE_GEMM1 and/or MOE_PHASE_GEMM2: only those
     * GEMM launches, on the routing, permute, pool rows and h that an earlier
     * whole-layer call with the same arguments left in the workspace (and in
     * the optional outputs); y and the routing are not touched.  Used to time
     * one GEMM.  Other bits: MOE_ERR_INVALID_ARG. */
    int32_t phases;
} moe_bfp8_args;

/* Workspace bytes moe_forward_bfp8 needs for this shape (0 for invalid sizes). */
MOE_API size_t moe_bfp8_workspace_size(int64_t T, int64_t H, int64_t I, int32_t E, int32_t k);

/* The whole block-FP8 layer: routing, permute, cast of x into pool rows,
 * GEMM1 + SiLU(gate)*up + FP8 write-back, GEMM2, weighted combine.  Device
 * waits are bounded (MOE_ERR_TIMEOUT in the workspace status words, read with
 * moe_get_device_status); the debug hook MOE_MXQ_DEBUG_INJECT_WAIT described
 * in moe_mxq.h applies to these GEMM launches too. */
MOE_API int moe_forward_bfp8(const moe_bfp8_args *args, cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_BFP8_H */
