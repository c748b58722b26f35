// gemm_common.cuh -- pieces shared by the expert-GEMM kernels (gemm.cu: one
// CTA per tile; gemm2sm.cu: a CTA pair per tile): tile constants, work-item
// decoding, and the per-chunk GEMM1 / GEMM2 epilogues.
#pragma once
#include <cuda_bf16.h>

#include <cstdint>

#include "ptx.cuh"

namespace mxq {

constexpr int kBM = 128;
constexpr int kBK = 128;
constexpr int kChunk = 16;                    // accumulator columns per epilogue step
constexpr long long kWaitLimit = 2000000000LL;
constexpr long long kInjectedWaitLimit = 20000000LL;   // ~10 ms: the debug wait's budget
constexpr int kMaxE = 1024;
constexpr int kWTileBytes = kBM * kBK / 2;    // one packed FP4 weight tile in HBM (8 KB)
constexpr int kPrefetchAhead = 2;             // K blocks between an L2 prefetch and its TMA load

struct TileInfo {
  int e, mt, g, s0, valid;
};

// counts/offsets -> shared memory with independent loads by every thread of
// the block (no chain of dependent global loads in the prologue).
__device__ __forceinline__ void load_expert_table(const int32_t *counts, const int32_t *offsets, int E,
                                                  int *cnt_sm, int *off_sm, bool from_l2 = false) {
  for (int e = threadIdx.x; e <= E; e += blockDim.x) {
    if (from_l2) {
      if (e < E) cnt_sm[e] = __ldcg(counts + e);
      off_sm[e] = __ldcg(offsets + e);
    } else {
      if (e < E) cnt_sm[e] = __ldg(counts + e);
      off_sm[e] = __ldg(offsets + e);
    }
  }
}

template <int BN>
__device__ __forceinline__ TileInfo decode_work(int w, int MT, int E, const int *tile_off, const int *cnt_sm,
                                                const int *off_sm) {
  const int tq = w / MT;
  int lo = 0, hi = E;                // find e with tile_off[e] <= tq < tile_off[e+1]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tile_off[mid] <= tq) lo = mid; else hi = mid;
  }
  TileInfo ti;
  ti.e = lo;
  const int nte = tile_off[lo + 1] - tile_off[lo];
  const int local = w - tile_off[lo] * MT;
  ti.mt = local / nte;
  const int nt = local - ti.mt * nte;
  ti.g = tile_off[lo] + nt;
  ti.s0 = off_sm[lo] + nt * BN;
  const int rem = cnt_sm[lo] - nt * BN;
  ti.valid = rem < BN ? rem : BN;
  return ti;
}

// Optional wait-time accounting (build with -DMOE_MXQ_WAIT_STATS): each role
// adds the clock cycles it spent in bounded waits, and its total, to 64-bit
// counters at byte 64 of the status area: [0] producer on empty stages,
// [1] MMA on full stages, [2] MMA on free accumulators, [3] epilogue on full
// accumulators, [4] kernel cycles of warp 0, [5] kernel cycles of warp 1,
// [6] kernel cycles of warp 2, [7] work items.
#ifdef MOE_MXQ_WAIT_STATS
#define MXQ_TIMED_WAIT(slot, expr)                                   \
  ([&]() {                                                           \
    const long long _t0 = clock64();                                 \
    const bool _r = (expr);                                          \
    if (lane == 0) wait_acc[slot] += clock64() - _t0;                \
    return _r;                                                       \
  }())
#else
#define MXQ_TIMED_WAIT(slot, expr) (expr)
#endif

// y_pairs row (slot * T + token) of pair p = token * k + slot.
__device__ __forceinline__ int pair_row(int p, int k, int T) {
  const int t = p / k;
  return (p - t * k) * T + t;
}

// GEMM1 epilogue of one 16-column accumulator chunk (MegaMoE (study notes),
// "L1 epilogue"; Warp Specialization: DeepEP vs Mega MoE, L1 epilogue
// listing): h = silu(gate) * up * topk_w, requantised to E4M3 + UE8M0 per 32
// features, written to hq (pool order) and to GEMM2's token-scale chunks
// (`tok_chunk` bytes per (token tile, K block)), optionally to hs_out.
// Called by the four warps of one epilogue half (named barrier `bar_half`,
// 128 threads); v holds TMEM lane 32q + lane, columns c0 .. c0 + 15; row_w is
// the top-k weight of each token column; ebuf_f this half's 4 KB staging.
__device__ __forceinline__ void epilogue_gemm1_chunk(const uint32_t (&v)[16], int c0, int q, int lane,
                                                     const TileInfo &ti, const float *row_w, float *ebuf_f,
                                                     uint32_t bar_half, int I, int tok_chunk, uint8_t *hq,
                                                     uint8_t *sfb2, uint8_t *hs_out) {
  // lane l of quadrant q holds stored row 32q+l: gate when (l & 8) == 0,
  // the matching up row sits 8 lanes away (8-row gate/up interleave).
  const bool is_gate = (lane & 8) == 0;
  const int feat = 16 * q + 8 * (lane >> 4) + (lane & 7);   // tile-local feature 0..63
  const int jbase = is_gate ? 0 : 8;                         // columns this lane evaluates
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float mine = __uint_as_float(v[j]);
    const float other = __shfl_xor_sync(0xffffffffu, mine, 8);
    // columns past the tile's tokens hold no pair and are never stored
    if (j >= jbase && j < jbase + 8 && c0 + j < ti.valid) {
      const float g = is_gate ? mine : other;
      const float u = is_gate ? other : mine;
      // silu(g) = g / (1 + e^-g); the approximate divide (2 ulp, no
      // slow path) is far inside the FP8 step of the requantisation
      const float h = __fdividef(g, 1.0f + __expf(-g)) * u * row_w[c0 + j];
      ebuf_f[j * 64 + feat] = h;
    }
  }
  named_bar_sync(bar_half, 128);
  // requantise: 16 columns x 2 groups of 32 features = 32 items; an
  // 8-lane group takes one item, 4 features per lane (one 16-byte
  // read, a 3-step xor max, one 4-byte store), 4 items per warp pass
#pragma unroll
  for (int pass = 0; pass < 2; ++pass) {
    const int it = q * 8 + pass * 4 + (lane >> 3);
    const int col = it >> 1, grp = it & 1;
    const int c = c0 + col;
    const int f4 = (lane & 7) * 4;                            // this lane's first feature in the group
    const float4 hv = *reinterpret_cast<const float4 *>(ebuf_f + col * 64 + grp * 32 + f4);
    float amax = fmaxf(fmaxf(fabsf(hv.x), fabsf(hv.y)), fmaxf(fabsf(hv.z), fabsf(hv.w)));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
    if (c >= ti.valid) continue;                              // uniform in the 8-lane group
    const int e = ue8m0_exponent<true>(amax);
    const float inv = pow2_neg(e);
    const uint32_t codes = (uint32_t)cvt_e4m3x2(hv.x * inv, hv.y * inv) |
                           ((uint32_t)cvt_e4m3x2(hv.z * inv, hv.w * inv) << 16);
    const size_t s = (size_t)(ti.s0 + c);
    const int fcol = ti.mt * 64 + grp * 32;                  // first feature of the group
    *reinterpret_cast<uint32_t *>(hq + s * I + fcol + f4) = codes;
    if ((lane & 7) == 0) {
      const int fg = fcol >> 5;                               // 32-group index along I
      const size_t chunk = (size_t)ti.g * (I / 128) + (fg >> 2);
      const int cr = c & 127;
      sfb2[chunk * tok_chunk + (c >> 7) * 512 + (cr & 31) * 16 + (cr >> 5) * 4 + (fg & 3)] =
          (uint8_t)(e + 127);
      if (hs_out) hs_out[s * (I / 32) + fg] = (uint8_t)(e + 127);
    }
  }
  named_bar_sync(bar_half, 128);
}

// GEMM2 epilogue of one 16-column chunk (MegaMoE (study notes), "L2
// epilogue"): FP32 accumulators -> BF16, staged in shared memory, stored as
// 256-byte rows of y_pairs[slot][token]; row_dst[c] = slot * T + token of
// token column c (filled with the item's row info).
__device__ __forceinline__ void epilogue_gemm2_chunk(const uint32_t (&v)[16], int c0, int q, int lane,
                                                     const TileInfo &ti, const int32_t *row_dst, uint16_t *ebuf_h,
                                                     uint32_t bar_half, int H, uint16_t *y_pairs) {
  const int row = 32 * q + lane;                             // output feature inside the tile
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const __nv_bfloat16 b = __float2bfloat16_rn(__uint_as_float(v[j]));
    ebuf_h[j * 128 + row] = *reinterpret_cast<const uint16_t *>(&b);
  }
  named_bar_sync(bar_half, 128);
#pragma unroll
  for (int it = 0; it < 2; ++it) {
    const int col = q + 4 * (2 * it + (lane >> 4));
    const int c = c0 + col;
    if (c < ti.valid) {
      const int l16 = lane & 15;
      uint16_t *dst = y_pairs + (size_t)row_dst[c] * H + (size_t)ti.mt * kBM + l16 * 8;
      *reinterpret_cast<uint4 *>(dst) = *reinterpret_cast<const uint4 *>(ebuf_h + col * 128 + l16 * 8);
    }
  }
  named_bar_sync(bar_half, 128);
}

// Combine (MegaMoE (study notes), "Combine"): y[t] = bf16( sum over slots j
// with topk_idx[t][j] >= 0 of y_pairs[j][t] ), in FP32 in slot order, for the
// (token, 8-value chunk) items first, first + stride, ... of T * H/8.
// y_pairs is read through L2 (written by other CTAs of the same launch).
__device__ __forceinline__ void combine_share(const uint16_t *y_pairs, const int32_t *topk_idx, int T, int k, int H,
                                              uint4 *y, int first, int stride) {
  const int H8 = H / 8;
  const int items = T * H8;
  const uint4 *yp = reinterpret_cast<const uint4 *>(y_pairs);
  for (int i = first; i < items; i += stride) {
    const int t = i / H8;
    float acc8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int j0 = 0; j0 < k; j0 += 8) {
      bool use[8];
      uint4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) use[u] = j0 + u < k && __ldg(topk_idx + t * k + j0 + u) >= 0;
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (use[u]) v[u] = __ldcg(yp + (size_t)(j0 + u) * items + i);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (!use[u]) continue;
        const uint32_t wv[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
        for (int q2 = 0; q2 < 4; ++q2) {
          acc8[2 * q2] += bf16_bits_to_float(wv[q2] & 0xFFFFu);
          acc8[2 * q2 + 1] += bf16_bits_to_float(wv[q2] >> 16);
        }
      }
    }
    uint32_t o[4];
#pragma unroll
    for (int q2 = 0; q2 < 4; ++q2) {
      const __nv_bfloat162 b2 = __floats2bfloat162_rn(acc8[2 * q2], acc8[2 * q2 + 1]);
      o[q2] = *reinterpret_cast<const uint32_t *>(&b2);
    }
    y[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

}  // namespace mxq
