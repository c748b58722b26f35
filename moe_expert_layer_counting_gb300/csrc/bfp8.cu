// bfp8.cu -- the block-FP8 variant of the MoE expert layer on sm_103a.
//
// Format (MonoMoe kernel -- design, "Fixed shape"): E4M3 weights with one
// float32 scale per 128 x 128 block (codes row-major or tile-contiguous, one
// 16 KB piece per block), E4M3 activations with one float32 scale per 128
// values of a row along K.  Pipeline (same page, section 1): routing and the
// counting-sort permute, the BF16 -> FP8 cast of x into expert-major pool
// rows, GEMM1 (gate and up) with SiLU(gate) * up and an FP8 write-back of h,
// GEMM2, and a combine that sums the k weighted FP32 partials of each token
// and casts once to BF16.  Small problems (T <= 64, E <= 256) run it as two
// launches: bfp8_front_kernel (routing + permute + cast) and one resident
// launch of GEMM1 + GEMM2 + combine; larger ones as the layer's routing and
// permute kernels, the pool cast, GEMM1, GEMM2 and the combine.
//
// The scales are plain float32 values, so the block-scaled MMA (power-of-two
// scales per 32) cannot carry them.  Each 128-wide K block is instead one
// group of plain tcgen05.mma kind::f8f6f4 instructions (E4M3 x E4M3, K = 32
// each) into its own TMEM slot; the epilogue warps read the slot back and
// fold it into register accumulators with the block's two scales
// (acc += s_w * s_x * partial), while the MMA warp fills the next slots.
// What the page's Hopper kernel keeps in registers between WGMMA groups, this
// kernel keeps in a ring of TMEM slots.
//
// GEMM1 work item: one expert, 128 output features j and one 16-token tile;
// the gate tile (rows j) and the up tile (rows I + j) of a K block land in
// the two halves of one slot, so every epilogue thread holds gate and up of
// its own feature, and the 128 features of a token's h form exactly one
// 128-value group of the FP8 write-back (per-token amax over the CTA's 128
// TMEM lanes).  GEMM2 work item: one expert, 128 output columns, one token
// tile; the epilogue multiplies by the pair's top-k weight and stores FP32
// rows y_pair[slot][token], which the combine sums in slot order.
#include <cuda_bf16.h>

#include <algorithm>
#include <cstdlib>

#include "../../include/moe_bfp8.h"
#include "host_common.h"
#include "layer_blocks.cuh"
#include "ptx.cuh"

namespace mxq {
namespace {

constexpr int kCastThreads = 256;
constexpr float kE4M3Max = 448.0f;

__device__ __forceinline__ void unpack_bf16x8(const uint4 &v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// value / scale in float32 (round to nearest) -> E4M3 (nearest even,
// saturating); scale 0 marks an all-zero group, whose codes are 0.
__device__ __forceinline__ uint32_t e4m3x4_scaled(float a, float b, float c, float d, float s) {
  if (s == 0.0f) return 0u;
  const uint32_t lo = cvt_e4m3x2(__fdiv_rn(a, s), __fdiv_rn(b, s));
  const uint32_t hi = cvt_e4m3x2(__fdiv_rn(c, s), __fdiv_rn(d, s));
  return lo | (hi << 16);
}

// Activation cast, 16 threads per 128-value group (8 values each).  Output
// row r reads input row r itself, or, for pool rows, the token of pair
// perm[r] (perm[r] / k); src_rows is the input's row count.
__global__ void __launch_bounds__(kCastThreads) bfp8_cast_kernel(const uint4 *__restrict__ x, int64_t rows,
                                                                 int64_t K, const int32_t *__restrict__ perm,
                                                                 int k, int64_t src_rows, uint2 *__restrict__ q,
                                                                 float *__restrict__ s) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t groups_per_row = K / 128;
  const int64_t items = rows * groups_per_row * 16;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t base = (int64_t)blockIdx.x * blockDim.x; base < items; base += stride) {
    const int64_t i = base + threadIdx.x;
    const bool valid = i < items;       // items % 16 == 0: a 16-lane group is all valid or all not
    const int64_t grp = i >> 4;
    const int sub = (int)(i & 15);
    const int64_t r = valid ? grp / groups_per_row : 0;
    const int64_t g = grp - r * groups_per_row;
    float f[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (valid) {
      // a pool row whose pair lies outside [0, T * k) reads zeros
      const int64_t src = perm ? (int64_t)__ldg(perm + r) / k : r;
      if (src >= 0 && src < src_rows) unpack_bf16x8(__ldg(x + (src * K + g * 128) / 8 + sub), f);
    }
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
#pragma unroll
    for (int m = 1; m < 16; m <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
    if (!valid) continue;
    const float sc = __fdiv_rn(amax, kE4M3Max);
    uint2 out;
    out.x = e4m3x4_scaled(f[0], f[1], f[2], f[3], sc);
    out.y = e4m3x4_scaled(f[4], f[5], f[6], f[7], sc);
    q[(r * K + g * 128) / 8 + sub] = out;
    if (sub == 0) s[r * groups_per_row + g] = sc;
  }
}

// Weight cast: one CTA per 128 x 128 block (grid-stride), 256 threads, each
// thread 64 values of one row (half a block row).  Codes row-major, or
// tile-contiguous (tiled: block b's 16 KB at b * 16 KB, rows of 128 codes).
constexpr int kWqThreads = 256;
__global__ void __launch_bounds__(kWqThreads) bfp8_weight_kernel(const uint4 *__restrict__ w, int64_t G, int64_t N,
                                                                 int64_t K, int tiled, uint4 *__restrict__ q,
                                                                 float *__restrict__ s) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ float warp_max[kWqThreads / 32];
  __shared__ float block_scale;
  const int64_t NB = N / 128, KB = K / 128;
  const int64_t nblocks = G * NB * KB;
  const int r = threadIdx.x >> 1, half = threadIdx.x & 1;
  for (int64_t b = blockIdx.x; b < nblocks; b += gridDim.x) {
    const int64_t g = b / (NB * KB);
    const int64_t nb = (b / KB) % NB;
    const int64_t kb = b % KB;
    const int64_t elem0 = (g * N + nb * 128 + r) * K + kb * 128 + half * 64;   // first of this thread's 64
    uint4 raw[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) raw[i] = __ldg(w + elem0 / 8 + i);
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float f[8];
      unpack_bf16x8(raw[i], f);
#pragma unroll
      for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
    }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
    if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = amax;
    __syncthreads();
    if (threadIdx.x == 0) {
      float m = 0.f;
      for (int i = 0; i < kWqThreads / 32; ++i) m = fmaxf(m, warp_max[i]);
      block_scale = __fdiv_rn(m, kE4M3Max);
      s[b] = block_scale;                 // b = (g * NB + nb) * KB + kb
    }
    __syncthreads();
    const float sc = block_scale;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float f[8], h[8];
      unpack_bf16x8(raw[2 * i], f);
      unpack_bf16x8(raw[2 * i + 1], h);
      uint4 out;
      out.x = e4m3x4_scaled(f[0], f[1], f[2], f[3], sc);
      out.y = e4m3x4_scaled(f[4], f[5], f[6], f[7], sc);
      out.z = e4m3x4_scaled(h[0], h[1], h[2], h[3], sc);
      out.w = e4m3x4_scaled(h[4], h[5], h[6], h[7], sc);
      const int64_t dst = tiled ? (b * 16384 + r * 128 + half * 64) / 16 : elem0 / 16;
      q[dst + i] = out;
    }
    __syncthreads();                      // warp_max / block_scale reused by the next block
  }
}

// Small problems (T <= 64, E <= 256): routing, the counting-sort permute and
// the pool cast in one launch.  One CTA per 128-column group of x: every CTA
// routes all tokens (one warp per token) and ranks all pairs -- the same
// result in every CTA, CTA 0 writes the routing and permute outputs -- then
// casts its column group of every pool row (16 threads per row).
constexpr int kBFrontThreads = 256;
constexpr int kBFrontMaxT = 64, kBFrontMaxE = 256;

__global__ void __launch_bounds__(kBFrontThreads) bfp8_front_kernel(
    const float *__restrict__ logits, const uint4 *__restrict__ x, int T, int E, int k, int H, int mode,
    int32_t *__restrict__ idx_out, float *__restrict__ w_out, int32_t *__restrict__ counts_out,
    int32_t *__restrict__ offsets_out, int32_t *__restrict__ perm_out, uint2 *__restrict__ xq,
    float *__restrict__ xs) {
  constexpr int kW = kBFrontThreads / 32;
  extern __shared__ __align__(16) unsigned char fsm[];
  const int P = T * k, g = blockIdx.x, KB = H / 128, H8 = H / 8;
  uint4 *xsm = reinterpret_cast<uint4 *>(fsm);                          // [T][16]: this CTA's columns
  int *idx_sm = reinterpret_cast<int *>(xsm + (size_t)T * 16);          // [P]
  int *perm_sm = idx_sm + P;                                            // [P]
  int *cnt = perm_sm + P;                                               // [E + 1]
  int *base = cnt + (E + 1);                                            // [E]
  int *warp_sums = base + E;                                            // [kW]
  int *total = warp_sums + kW;                                          // [1]
  uint16_t *wc = reinterpret_cast<uint16_t *>(total + 4);               // [kW][E]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool writer = blockIdx.x == 0;
  pdl_launch_dependents();
  pdl_wait();
  // 0. this CTA's 128 columns of every token; the first 16 bytes per thread
  // wait in a register while the logits load
  const int nx = T * 16;
  uint4 xv = make_uint4(0, 0, 0, 0);
  if (tid < nx) xv = __ldg(x + (size_t)(tid >> 4) * H8 + g * 16 + (tid & 15));
  for (int i = tid + kBFrontThreads; i < nx; i += kBFrontThreads)
    xsm[i] = __ldg(x + (size_t)(i >> 4) * H8 + g * 16 + (i & 15));
  // 1. routing, one warp per token
  for (int t = warp; t < T; t += kW) {
    int my_idx;
    float my_w;
    warp_route_token<kBFrontMaxE / 32>(logits + (size_t)t * E, E, k, lane, mode, &my_idx, &my_w);
    if (lane < k) {
      idx_sm[t * k + lane] = my_idx;
      if (writer) {
        idx_out[t * k + lane] = my_idx;
        w_out[t * k + lane] = my_w;
      }
    }
    __syncwarp();
  }
  if (tid < nx) xsm[tid] = xv;
  for (int e = tid; e <= E; e += kBFrontThreads) cnt[e] = 0;
  __syncthreads();
  // 2. count -> exclusive prefix -> stable ranks
  for (int p = tid; p < P; p += kBFrontThreads) atomicAdd(&cnt[idx_sm[p]], 1);
  __syncthreads();
  const int o = block_exclusive_scan<kBFrontThreads>(tid < E ? cnt[tid] : 0, warp_sums, total);
  if (tid < E) {
    base[tid] = o;
    if (writer) {
      counts_out[tid] = cnt[tid];
      offsets_out[tid] = o;
    }
  }
  if (tid == 0 && writer) offsets_out[E] = *total;
  __syncthreads();
  block_stable_ranks<kBFrontThreads>([&](int64_t p) { return idx_sm[p]; }, 0, P, E, base, wc,
                                     writer ? perm_out : nullptr, nullptr, perm_sm);
  // 3. this CTA's 128-value group of every pool row
  for (int b0 = 0; b0 < P * 16; b0 += kBFrontThreads) {
    const int i = b0 + tid;
    const bool valid = i < P * 16;      // P * 16 is a multiple of 16: 16-lane groups stay whole
    const int sr = i >> 4, sub = i & 15;
    float f[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (valid) unpack_bf16x8(xsm[(perm_sm[sr] / k) * 16 + sub], f);
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
#pragma unroll
    for (int m = 1; m < 16; m <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
    if (!valid) continue;
    const float sc = __fdiv_rn(amax, kE4M3Max);
    uint2 out;
    out.x = e4m3x4_scaled(f[0], f[1], f[2], f[3], sc);
    out.y = e4m3x4_scaled(f[4], f[5], f[6], f[7], sc);
    xq[(size_t)sr * H8 + g * 16 + sub] = out;
    if (sub == 0) xs[(size_t)sr * KB + g] = sc;
  }
}

size_t bfp8_front_smem(int T, int E, int k) {
  const int P = T * k;
  return (size_t)T * 256 + (size_t)2 * P * 4 + (size_t)(2 * E + 1) * 4 + (kBFrontThreads / 32) * 4 + 16 +
         (size_t)(kBFrontThreads / 32) * E * 2;
}

bool bfp8_front_eligible(int64_t T, int64_t H, int E, int k) {
  return T >= 1 && T <= kBFrontMaxT && E <= kBFrontMaxE && T * k * H <= (int64_t(4) << 20);
}

// ---------------------------------------------------------------- expert GEMMs
// One stage = one 128 x 128 E4M3 weight tile (16 KB) + one 16-token tile of
// E4M3 rows (2 KB), both 128-byte swizzled.  GEMM1 spends two stages per K
// block (gate tile, up tile; the token tile is loaded with each), GEMM2 one.
// Two CTAs per SM: 192 threads (warp 0 TMA producer, warp 1 TMEM allocator +
// MMA issuer, warps 2-5 epilogue, one TMEM lane quadrant each).
constexpr int kGBN = 16;                          // tokens per tile (MMA N)
constexpr int kGTileA = 128 * 128;
constexpr int kGTileB = kGBN * 128;
constexpr int kGStages = 5;
constexpr int kGThreads = 192;
constexpr int kGCtasPerSm = 2;
constexpr uint32_t kGTmemCols = 128;
constexpr long long kGWaitLimit = 2000000000LL;
constexpr long long kGInjectedWaitLimit = 20000000LL;  // ~10 ms: the debug wait's budget
constexpr int kGOffA = 0;
constexpr int kGOffB = kGOffA + kGStages * kGTileA;
constexpr int kGOffBar = kGOffB + kGStages * kGTileB;
constexpr int kGNumBars = 2 * kGStages + 2 * 8 + 2;   // full/empty stages, full/empty slots (<= 8), MMAs done, debug
constexpr int kGOffMisc = kGOffBar + 256;             // tmem ptr, votes, column maxima, row info
constexpr int kGOffScan = kGOffMisc + 512;
constexpr int kGOffSc = kGOffScan + 64;               // scales: weights [2][KB], tokens [KB][16]
static_assert(kGNumBars * 8 <= 256, "barrier area");
static_assert(kGTmemCols * kGCtasPerSm <= 512, "co-resident CTAs share the SM's TMEM");

// PHASE 1: GEMM1 (+ SiLU(gate) * up + FP8 write-back of h); 2: GEMM2 (+ the
// top-k weight, FP32 pair rows); 3: both and the combine in one launch (small
// problems, every CTA resident): GEMM1 items first, then GEMM2 items, each
// waiting on the arrival counter of its token tile that the GEMM1 epilogues
// raise, then the combine, after the counter of finished GEMM2 items -- the
// pages' arrival mask between the two GEMMs, as bounded waits.
template <int PHASE>
struct GCfg {
  // TMEM columns of one K block's partial: gate and up halves for GEMM1 items
  static constexpr int kSlotCols = PHASE == 2 ? kGBN : 2 * kGBN;
  static constexpr int kSlots = (int)kGTmemCols / kSlotCols;   // 4 (GEMM1 items) or 8
};

__host__ __device__ inline size_t gemm_sc_bytes(int KB) { return ((size_t)KB * (2 + kGBN) * 4 + 15) / 16 * 16; }
inline size_t gemm_smem_bytes(int KB, int E) {
  return 1024 + kGOffSc + gemm_sc_bytes(KB) + (size_t)3 * (E + 1) * 4;
}

struct BGemmArgs {
  int E, k, T, H, I;
  int KB, MT;                      // the launch's (first) GEMM: K blocks, 128-row output tiles per expert
  int KB2, MT2;                    // PHASE 3: GEMM2's
  int P;                           // pool rows (T * k, dropped pairs excluded from the tiles)
  int tiled;                       // weight codes tile-contiguous (else row-major)
  int inject_wait;                 // debug: 1 = the MMA warp first waits on a barrier nothing completes
  const int32_t *counts, *offsets, *perm;
  const float *topk_w;             // [T*k] by pair id
  const float *w_scales;           // GEMM1: [E][2I/128][KB]; GEMM2: [E][H/128][KB]
  const float *x_scales;           // token scales of the pool rows [P][KB]
  const float *w_scales2;          // PHASE 3: GEMM2's weight-block scales
  const float *x_scales2;          // PHASE 3: hs
  uint8_t *hq;                     // GEMM1 out [P][I]
  float *hs;                       // GEMM1 out [P][I/128]
  float *y_pairs;                  // GEMM2 out [k][T][H]
  int *status;
  int *sync;                       // PHASE 3: [0] GEMM2 items done, [1 + g] GEMM1 items of token tile g done
  const int32_t *topk_idx;         // PHASE 3: combine (dropped slots skipped)
  uint4 *y;                        // PHASE 3: combine output [T][H] bf16
};

__device__ __forceinline__ void mma_f8f6f4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t"
      "}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Instruction descriptor of kind::f8f6f4 without block scaling: FP32
// accumulator, A and B E4M3, both K-major, M = 128, N = n.
__device__ __forceinline__ uint32_t idesc_e4m3_f32(uint32_t n) {
  uint32_t d = 0;
  d |= 1u << 4;                    // D format: F32
  d |= 0u << 7;                    // A format: E4M3
  d |= 0u << 10;                   // B format: E4M3
  d |= ((n >> 3) & 0x3Fu) << 17;
  d |= ((128u >> 4) & 0x1Fu) << 24;
  return d;
}

struct BTile {
  int e, mt, g, s0, valid;         // expert, output tile, global token tile, first pool row, valid tokens
};

// Work item w -> its tile; items are expert-major, then output tile, then
// token tile.
__device__ __forceinline__ BTile decode_item(int w, int MT, int E, const int *tile_off, const int *cnt,
                                             const int *off) {
  const int tq = w / MT;
  int lo = 0, hi = E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tile_off[mid] <= tq) lo = mid; else hi = mid;
  }
  BTile ti;
  ti.e = lo;
  const int nte = tile_off[lo + 1] - tile_off[lo];
  const int local = w - tile_off[lo] * MT;
  ti.mt = local / nte;
  const int nt = local - ti.mt * nte;
  ti.g = tile_off[lo] + nt;
  ti.s0 = off[lo] + nt * kGBN;
  const int rem = cnt[lo] - nt * kGBN;
  ti.valid = rem < kGBN ? rem : kGBN;
  return ti;
}

// Output items [first, n) step `stride` of the combine: y[t] (8 values per
// item) = bf16( sum over valid slots j, in slot order, of y_pairs[j][t] ).
// from_l2: the pair rows were written by other CTAs of the same launch.
__device__ __forceinline__ void combine_items(int64_t first, int64_t stride, const float4 *y_pairs,
                                              const int32_t *idx, int64_t T, int k, int64_t H, uint4 *y,
                                              bool from_l2) {
  const int64_t H8 = H / 8;
  for (int64_t i = first; i < T * H8; i += stride) {
    const int64_t t = i / H8, c = i - t * H8;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int j = 0; j < k; ++j) {
      if (__ldg(idx + t * k + j) < 0) continue;
      const float4 *row = y_pairs + (((int64_t)j * T + t) * H) / 4 + 2 * c;
      const float4 a = from_l2 ? __ldcg(row) : __ldg(row);
      const float4 b = from_l2 ? __ldcg(row + 1) : __ldg(row + 1);
      acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
      acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
    }
    uint32_t packed[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * p]));
      const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * p + 1]));
      packed[p] = lo | (hi << 16);
    }
    y[i] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  }
}

// The combine as its own launch (larger problems): the pairs' rows already
// carry their top-k weight.
__global__ void __launch_bounds__(kCastThreads) bfp8_combine_kernel(const float4 *__restrict__ y_pairs,
                                                                    const int32_t *__restrict__ idx, int64_t T,
                                                                    int k, int64_t H, uint4 *__restrict__ y) {
  pdl_launch_dependents();
  pdl_wait();
  combine_items((int64_t)blockIdx.x * blockDim.x + threadIdx.x, (int64_t)gridDim.x * blockDim.x, y_pairs, idx, T,
                k, H, y, false);
}

// Optional wait-time accounting (build with -DMOE_MXQ_WAIT_STATS): each role
// adds the clock cycles it spent in bounded waits, and its total, to 64-bit
// counters at byte 64 of the status area: [0] producer on empty stages,
// [1] MMA on full stages, [2] MMA on free TMEM slots, [3] epilogue on full
// slots, [4] kernel cycles of warp 0, [5] of warp 1, [6] of warp 2, [7] work
// items.
#ifdef MOE_MXQ_WAIT_STATS
#define BFP8_TIMED_WAIT(slot, expr)                                  \
  ([&]() {                                                           \
    const long long _t0 = clock64();                                 \
    const bool _r = (expr);                                          \
    if (lane == 0) wait_acc[slot] += clock64() - _t0;                \
    return _r;                                                       \
  }())
#else
#define BFP8_TIMED_WAIT(slot, expr) (expr)
#endif

template <int PHASE>
__global__ void __launch_bounds__(kGThreads, kGCtasPerSm)
    bfp8_gemm_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_b,
                     const __grid_constant__ CUtensorMap tmap_w2, const __grid_constant__ CUtensorMap tmap_b2,
                     const BGemmArgs args) {
  using C = GCfg<PHASE>;
  constexpr bool kFused = PHASE == 3;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                          ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kGOffBar);
  uint64_t *full = bars;
  uint64_t *empty = bars + kGStages;
  uint64_t *slot_full = bars + 2 * kGStages;
  uint64_t *slot_empty = slot_full + 8;
  uint64_t *mma_done = slot_empty + 8;
  uint64_t *never = mma_done + 1;           // debug wait target: initialised, never arrived on
  uint32_t *tmem_ptr = reinterpret_cast<uint32_t *>(smem + kGOffMisc);
  int *flag = reinterpret_cast<int *>(smem + kGOffMisc + 8);            // combine go-ahead
  int *vote = reinterpret_cast<int *>(smem + kGOffMisc + 16);           // [4]
  float *colmax = reinterpret_cast<float *>(smem + kGOffMisc + 64);     // [4][16]
  int *row_pair = reinterpret_cast<int *>(smem + kGOffMisc + 320);      // [16]
  float *row_w = reinterpret_cast<float *>(smem + kGOffMisc + 384);     // [16]
  int *scan_ws = reinterpret_cast<int *>(smem + kGOffScan);
  const int kb_max = kFused ? max(args.KB, args.KB2) : args.KB;
  float *sw = reinterpret_cast<float *>(smem + kGOffSc);                // [halves][KB]
  float *sx = sw + 2 * kb_max;                                          // [KB][16]
  int *tile_off = reinterpret_cast<int *>(smem + kGOffSc + gemm_sc_bytes(kb_max));
  int *cnt_sm = tile_off + (args.E + 1);
  int *off_sm = cnt_sm + (args.E + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int *status = args.status;
#ifdef MOE_MXQ_WAIT_STATS
  long long wait_acc[4] = {0, 0, 0, 0};
  const long long k_t0 = clock64();
#endif

  pdl_launch_dependents();
  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tmap_w);
      tma_prefetch_desc(&tmap_b);
      if (kFused) {
        tma_prefetch_desc(&tmap_w2);
        tma_prefetch_desc(&tmap_b2);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      for (int s = 0; s < kGStages; ++s) {
        mbar_init(&full[s], 1);
        mbar_init(&empty[s], 1);
      }
      for (int s = 0; s < C::kSlots; ++s) {
        mbar_init(&slot_full[s], 1);
        mbar_init(&slot_empty[s], 4);
      }
      mbar_init(mma_done, 1);
      mbar_init(never, 1);
      fence_mbar_init();
    }
    __syncwarp();
    tmem_alloc(tmem_ptr, kGTmemCols);
    tmem_relinquish();
  }
  // the routing, permute, pool rows (and, for GEMM2, h) come from earlier kernels
  pdl_wait();
  for (int e = threadIdx.x; e <= args.E; e += blockDim.x) {
    if (e < args.E) cnt_sm[e] = __ldg(args.counts + e);
    off_sm[e] = __ldg(args.offsets + e);
  }
  __syncthreads();
  block_tile_map<kGThreads>(cnt_sm, args.E, kGBN, tile_off, scan_ws, scan_ws + 15);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_ptr;
  const int n1 = tile_off[args.E] * args.MT;
  const int n2 = kFused ? tile_off[args.E] * args.MT2 : 0;
  const int total = n1 + n2;
  struct Item {
    BTile ti;
    bool l1, second;                 // a GEMM1 item; the single launch's GEMM2 item
    int KB, MT, halves;
  };
  auto get_item = [&](int w) {
    Item it;
    it.second = kFused && w >= n1;
    it.l1 = PHASE == 1 || (kFused && !it.second);
    it.KB = it.second ? args.KB2 : args.KB;
    it.MT = it.second ? args.MT2 : args.MT;
    it.halves = it.l1 ? 2 : 1;
    it.ti = decode_item(it.second ? w - n1 : w, it.MT, args.E, tile_off, cnt_sm, off_sm);
    return it;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    int stage = 0;
    uint32_t phase = 0, issued_mask = 0, issued_phase = 0;
    bool ok = true;
    auto record = [&](int st, uint32_t ph) {
      issued_mask |= 1u << st;
      issued_phase = (issued_phase & ~(1u << st)) | (ph << st);
    };
    for (int w = blockIdx.x; w < total && ok; w += gridDim.x) {
      const Item it = get_item(w);
      const CUtensorMap *tw = it.second ? &tmap_w2 : &tmap_w;
      const CUtensorMap *tb = it.second ? &tmap_b2 : &tmap_b;
      // weight rows of this item's tile(s) in the [E * rows][K] weight tensor
      const int row0 = it.ti.e * (it.l1 ? 2 * args.I : args.H) + it.ti.mt * 128;
      const int nst = it.KB * it.halves;                    // stages of this item
      // stage a: K block a / halves, half (gate, up) a % halves; row-major codes:
      // the box at (K offset, row); tiled: block (row / 128, kb) is rows
      // [(row / 128 * KB + kb) * 128, +128) of a 128-byte-wide tensor
      auto issue_w = [&](int st, int a) {
        const int kb = a / it.halves, wrow = row0 + (a - kb * it.halves) * args.I;
        mbar_arrive_expect_tx(&full[st], (uint32_t)(kGTileA + kGTileB));
        if (args.tiled)
          tma_load_2d(smem + kGOffA + st * kGTileA, tw, &full[st], 0, ((wrow >> 7) * it.KB + kb) * 128);
        else
          tma_load_2d(smem + kGOffA + st * kGTileA, tw, &full[st], kb * 128, wrow);
      };
      auto issue_b = [&](int st, int a) {
        tma_load_2d(smem + kGOffB + st * kGTileB, tb, &full[st], (a / it.halves) * 128, it.ti.s0);
      };
      int a0 = 0;
      if (it.second) {
        // the weight parts of the first stages now, then the wait for the h
        // rows of the token tile (all its GEMM1 items), then their token
        // parts -- issued even after a failed wait, so that every armed
        // barrier completes (the status word says why)
        const int npre = min(nst, kGStages);
        const int st0 = stage;
        const uint32_t ph0 = phase;
        int armed = 0;
        for (; armed < npre; ++armed) {
          if (!__all_sync(0xffffffffu, BFP8_TIMED_WAIT(0, mbar_wait(&empty[stage], phase ^ 1, status, kGWaitLimit, kWaitProducerEmpty, armed))))
            break;
          if (lane == 0) issue_w(stage, armed);
          __syncwarp();
          if (++stage == kGStages) { stage = 0; phase ^= 1; }
        }
        bool dep_ok = true;
        if (lane == 0) {
          dep_ok = wait_counter(args.sync + 1 + it.ti.g, args.MT, status, kGWaitLimit, w);
          fence_proxy_async_global();
        }
        dep_ok = __shfl_sync(0xffffffffu, dep_ok ? 1 : 0, 0) != 0;
        for (int a = 0; a < armed; ++a) {
          // armed <= kGStages: the ring wraps at most once inside one item
          const int st = (st0 + a) % kGStages;
          if (lane == 0) issue_b(st, a);
          record(st, ph0 ^ (uint32_t)((st0 + a) / kGStages));
        }
        __syncwarp();
        if (armed < npre || !dep_ok) {
          ok = false;
          break;
        }
        a0 = npre;
      }
      for (int a = a0; a < nst; ++a) {
        if (!__all_sync(0xffffffffu, BFP8_TIMED_WAIT(0, mbar_wait(&empty[stage], phase ^ 1, status, kGWaitLimit, kWaitProducerEmpty, a)))) {
          ok = false;
          break;
        }
        if (lane == 0) {
          issue_w(stage, a);
          issue_b(stage, a);
        }
        __syncwarp();
        record(stage, phase);
        if (++stage == kGStages) { stage = 0; phase ^= 1; }
      }
    }
    // never leave with copies in flight
    for (int s = 0; s < kGStages; ++s)
      if (issued_mask & (1u << s))
        mbar_wait(&full[s], (issued_phase >> s) & 1u, status, kGWaitLimit, kWaitProducerDrain, s, false);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    int stage = 0, slot = 0;
    uint32_t phase = 0, slot_phase = 0;
    bool ok = true;
    const uint32_t idesc = idesc_e4m3_f32(kGBN);
    for (int w = blockIdx.x; w < total && ok; w += gridDim.x) {
      const Item it = get_item(w);
      // failure-detection test hook: a wait that can only end by its timeout
      if (args.inject_wait == 1 && w == (int)blockIdx.x &&
          !__all_sync(0xffffffffu, mbar_wait(never, 0, status, kGInjectedWaitLimit, kWaitInjected, w)))
        break;
      for (int kb = 0; kb < it.KB; ++kb) {
        if (!__all_sync(0xffffffffu, BFP8_TIMED_WAIT(2, mbar_wait(&slot_empty[slot], slot_phase ^ 1, status, kGWaitLimit, kWaitMmaTmemEmpty, kb)))) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int hf = 0; hf < it.halves && ok; ++hf) {
          if (!__all_sync(0xffffffffu, BFP8_TIMED_WAIT(1, mbar_wait(&full[stage], phase, status, kGWaitLimit, kWaitMmaFull, kb)))) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (lane == 0) {
            const uint32_t a_base = smem_u32(smem + kGOffA + stage * kGTileA);
            const uint32_t b_base = smem_u32(smem + kGOffB + stage * kGTileB);
            const uint32_t d = tmem_base + (uint32_t)(slot * C::kSlotCols + hf * kGBN);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_f8f6f4(d, make_smem_desc(a_base + kk * 32, 16, 1024, kSwizzle128B),
                         make_smem_desc(b_base + kk * 32, 16, 1024, kSwizzle128B), idesc, kk != 0 ? 1u : 0u);
            tc_commit(&empty[stage]);
          }
          __syncwarp();
          if (++stage == kGStages) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        if (lane == 0) tc_commit(&slot_full[slot]);
        __syncwarp();
        if (++slot == C::kSlots) { slot = 0; slot_phase ^= 1; }
      }
    }
    // every MMA of this thread completes before TMEM is released
    if (lane == 0) tc_commit(mma_done);
    __syncwarp();
    mbar_wait(mma_done, 0, status, kGWaitLimit, kWaitMmaDone, 0, false);
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                     // TMEM lane quadrant of this warp
    const int et = threadIdx.x - 64;            // 0 .. 127
    const int r = 32 * q + lane;                // output row of the tile held by this thread
    int slot = 0;
    uint32_t slot_phase = 0;
    for (int w = blockIdx.x; w < total; w += gridDim.x) {
      const Item it = get_item(w);
      const BTile &ti = it.ti;
      const int KB = it.KB;
      named_bar_sync(1, 128);                   // the previous item's scales and row info are read
      bool ok = true;
      if (it.second && lane == 0) ok = wait_counter(args.sync + 1 + ti.g, args.MT, status, kGWaitLimit, w);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      __syncwarp();                             // the other lanes' h-scale reads come after lane 0's acquire
      // this item's scales: the weight blocks of its tile(s) and the token rows
      // (h scales of the single launch: written by other CTAs, read from L2)
      const float *wsc = it.second ? args.w_scales2 : args.w_scales;
      const float *xsc = it.second ? args.x_scales2 : args.x_scales;
      for (int i = et; i < it.halves * KB; i += 128) {
        const int hf = i / KB, kb = i - hf * KB;
        const int wrow = it.l1 ? ti.e * (2 * args.I / 128) + hf * (args.I / 128) + ti.mt
                               : ti.e * (args.H / 128) + ti.mt;
        sw[i] = __ldg(wsc + (size_t)wrow * KB + kb);
      }
      for (int i = et; i < KB * kGBN; i += 128) {
        const int kb = i / kGBN, c = i - kb * kGBN;
        const float *src = xsc + (size_t)(ti.s0 + c) * KB + kb;
        sx[i] = c < ti.valid ? (it.second ? __ldcg(src) : __ldg(src)) : 0.f;
      }
      if (!it.l1 && et < ti.valid) {
        const int p = __ldg(args.perm + ti.s0 + et);
        row_pair[et] = p;
        row_w[et] = __ldg(args.topk_w + p);
      }
      named_bar_sync(1, 128);
      float accg[kGBN], accu[kGBN];
#pragma unroll
      for (int c = 0; c < kGBN; ++c) {
        accg[c] = 0.f;
        accu[c] = 0.f;
      }
      for (int kb = 0; kb < KB && ok; ++kb) {
        if (!__all_sync(0xffffffffu, BFP8_TIMED_WAIT(3, mbar_wait(&slot_full[slot], slot_phase, status, kGWaitLimit, kWaitEpiTmemFull, kb)))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(slot * C::kSlotCols);
        uint32_t vg[kGBN], vu[kGBN];
        tmem_ld_32x32b_x16(taddr, vg);
        if (PHASE != 2 && it.l1) tmem_ld_32x32b_x16(taddr + kGBN, vu);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&slot_empty[slot]);
        if (++slot == C::kSlots) { slot = 0; slot_phase ^= 1; }
        // promotion: acc += (weight-block scale * token scale) * K-block partial
        const float sg = sw[kb];
#pragma unroll
        for (int c = 0; c < kGBN; ++c) accg[c] = fmaf(sg * sx[kb * kGBN + c], __uint_as_float(vg[c]), accg[c]);
        if (PHASE != 2 && it.l1) {
          const float su = sw[KB + kb];
#pragma unroll
          for (int c = 0; c < kGBN; ++c) accu[c] = fmaf(su * sx[kb * kGBN + c], __uint_as_float(vu[c]), accu[c]);
        }
      }
      // the four warps agree on the outcome of their bounded waits before the
      // next named barrier
      if (lane == 0) vote[warp - 2] = ok ? 1 : 0;
      named_bar_sync(1, 128);
      if (!(vote[0] && vote[1] && vote[2] && vote[3])) break;
      if (PHASE != 2 && it.l1) {
        // h = silu(gate) * up for feature mt*128 + r of every token column,
        // then the token's 128 features -> one E4M3 group (amax over the
        // 128 TMEM lanes: warp shuffles, then the four quadrants)
        float h[kGBN];
#pragma unroll
        for (int c = 0; c < kGBN; ++c) {
          // silu(g) = g / (1 + e^-g); the approximate divide (2 ulp, no slow
          // path) is far inside the FP8 step of the write-back
          h[c] = c < ti.valid ? __fdividef(accg[c], 1.0f + __expf(-accg[c])) * accu[c] : 0.f;
          float m = fabsf(h[c]);
#pragma unroll
          for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
          if (lane == 0) colmax[q * kGBN + c] = m;
        }
        named_bar_sync(1, 128);
        const int I = args.I;
#pragma unroll
        for (int c = 0; c < kGBN; ++c) {
          if (c < ti.valid) {
            const float amax = fmaxf(fmaxf(colmax[c], colmax[kGBN + c]), fmaxf(colmax[2 * kGBN + c], colmax[3 * kGBN + c]));
            const float sc = __fdiv_rn(amax, kE4M3Max);
            const uint8_t code = sc == 0.0f ? (uint8_t)0 : (uint8_t)(cvt_e4m3x2(__fdiv_rn(h[c], sc), 0.0f) & 0xFFu);
            args.hq[(size_t)(ti.s0 + c) * I + ti.mt * 128 + r] = code;
            if (et == c) args.hs[(size_t)(ti.s0 + c) * (I / 128) + ti.mt] = sc;
          }
        }
        if (kFused) {
          // release this item's h rows to the GEMM2 items of its token tile
          // (their h tiles are read by TMA: async proxy)
          fence_proxy_async_global();
          named_bar_sync(1, 128);
          if (et == 0) {
            __threadfence();
            atomicAdd(args.sync + 1 + ti.g, 1);
          }
        }
      } else {
        // FP32 row of each pair, times its top-k weight, into y_pairs[slot][token]
#pragma unroll
        for (int c = 0; c < kGBN; ++c) {
          if (c < ti.valid) {
            const int p = row_pair[c];
            const int t = p / args.k, j = p - t * args.k;
            args.y_pairs[((size_t)j * args.T + t) * args.H + ti.mt * 128 + r] = accg[c] * row_w[c];
          }
        }
        if (kFused) {
          named_bar_sync(1, 128);
          if (et == 0) {
            __threadfence();
            atomicAdd(args.sync, 1);
          }
        }
      }
    }
  }
  if (kFused) {
    // the combine, once every CTA's GEMM2 items are done (bounded wait; a
    // failed wait leaves y unwritten and the status word set)
    __syncthreads();
    if (threadIdx.x == 0) *flag = wait_counter(args.sync, n2, status, kGWaitLimit, -1) ? 1 : 0;
    __syncthreads();
    if (*flag)
      combine_items((int64_t)blockIdx.x * blockDim.x + threadIdx.x, (int64_t)gridDim.x * blockDim.x,
                    reinterpret_cast<const float4 *>(args.y_pairs), args.topk_idx, args.T, args.k, args.H, args.y,
                    true);
  }
#ifdef MOE_MXQ_WAIT_STATS
  if (lane == 0) {
    unsigned long long *acc64 = reinterpret_cast<unsigned long long *>(reinterpret_cast<char *>(status) + 64);
    for (int i = 0; i < 4; ++i)
      if (wait_acc[i]) atomicAdd(acc64 + i, (unsigned long long)wait_acc[i]);
    if (warp <= 2) atomicAdd(acc64 + 4 + warp, (unsigned long long)(clock64() - k_t0));
    if (warp == 0) {
      int n_items = 0;
      for (int w = blockIdx.x; w < total; w += gridDim.x) ++n_items;
      atomicAdd(acc64 + 7, (unsigned long long)n_items);
    }
  }
#endif
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kGTmemCols);
  }
}

int cast_grid(int64_t threads) {
  const int64_t blocks = ceil_div(threads, kCastThreads);
  const int64_t cap = (int64_t)num_sms() * 8;
  return (int)(blocks < 1 ? 1 : (blocks < cap ? blocks : cap));
}

// CTAs per SM of a GEMM launch with `smem` bytes of dynamic shared memory (two
// where shared memory allows, 1 KB reserved per CTA), 0 if it does not fit.
int gemm_ctas_per_sm(size_t smem) {
  int dev = 0, optin = 0, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess)
    return 0;
  if (smem > (size_t)optin) return 0;
  return (size_t)kGCtasPerSm * (smem + 1024) <= (size_t)per_sm ? kGCtasPerSm : 1;
}

template <int PHASE>
int launch_bfp8_gemm(const CUtensorMap &tw, const CUtensorMap &tb, const CUtensorMap &tw2, const CUtensorMap &tb2,
                     const BGemmArgs &ga, cudaStream_t st) {
  const size_t smem = gemm_smem_bytes(PHASE == 3 ? std::max(ga.KB, ga.KB2) : ga.KB, ga.E);
  const int per = gemm_ctas_per_sm(smem);
  if (per == 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  // the largest shared-memory carve-out, so that the CTAs per SM counted above are resident
  if (cudaFuncSetAttribute(bfp8_gemm_kernel<PHASE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
          cudaSuccess ||
      cudaFuncSetAttribute(bfp8_gemm_kernel<PHASE>, cudaFuncAttributePreferredSharedMemoryCarveout, 100) !=
          cudaSuccess)
    return MOE_ERR_CUDA;
  BGemmArgs g = ga;
  // debug hook of the failure-detection tests (see moe_get_device_status)
  if (const char *env = getenv("MOE_MXQ_DEBUG_INJECT_WAIT")) g.inject_wait = atoi(env);
  return launch_pdl(bfp8_gemm_kernel<PHASE>, dim3(num_sms() * per), dim3(kGThreads), smem, st, tw, tb, tw2, tb2, g);
}

struct BWs {
  size_t sync_end;   // status words, then the single launch's arrival counters (zeroed per call)
  size_t idx, w, counts, offsets, perm, inv_perm, perm_scratch, xq, xs, hq, hs, y_pairs, total;
};

// arrival counters of the single launch: GEMM2 items done, then one per token tile
int64_t bfp8_sync_ints(int64_t T, int64_t E, int64_t k) { return 1 + max_token_tiles(T * k, E, kGBN); }

BWs bfp8_ws_layout(int64_t T, int64_t H, int64_t I, int64_t E, int64_t k) {
  const int64_t P = T * k;
  BWs l;
  size_t off = kStatusBytes;
  off += round_up((size_t)bfp8_sync_ints(T, E, k) * 4, 256);
  l.sync_end = off;
  l.idx = off;          off += round_up((size_t)P * 4, 256);
  l.w = off;            off += round_up((size_t)P * 4, 256);
  l.counts = off;       off += round_up((size_t)E * 4, 256);
  l.offsets = off;      off += round_up((size_t)(E + 1) * 4, 256);
  l.perm = off;         off += round_up((size_t)P * 4, 256);
  l.inv_perm = off;     off += round_up((size_t)P * 4, 256);
  l.perm_scratch = off; off += round_up(permute_scratch_bytes(T, (int)E, (int)k), 256);
  l.xq = off;           off += round_up((size_t)P * H, 256);
  l.xs = off;           off += round_up((size_t)P * (H / 128) * 4, 256);
  l.hq = off;           off += round_up((size_t)P * I, 256);
  l.hs = off;           off += round_up((size_t)P * (I / 128) * 4, 256);
  l.y_pairs = off;      off += round_up((size_t)P * H * 4, 256);
  l.total = off;
  return l;
}

bool bfp8_shape_ok(int64_t T, int64_t H, int64_t I, int64_t E, int64_t k) {
  if (H % 128 != 0 || I % 128 != 0) return false;
  if (E > 1024 || k > 32 || k > E) return false;
  if (T * k >= (int64_t(1) << 31)) return false;
  // tensor-map row counts and the GEMMs' int arithmetic (tiled rows: rows * K / 128)
  if (E * 2 * I * (H / 128) >= (int64_t(1) << 31) || E * H * (I / 128) >= (int64_t(1) << 31)) return false;
  return true;
}

}  // namespace
}  // namespace mxq

using namespace mxq;

extern "C" int bfp8_quantize_act(const uint16_t *x, int64_t rows, int64_t K, uint8_t *q, float *s,
                                 cudaStream_t stream) {
  if (rows < 0 || K <= 0) return MOE_ERR_INVALID_ARG;
  if (K % 128 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (rows == 0) return MOE_OK;
  if (!x || !q || !s) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(q, 16) || !aligned(s, 4)) return MOE_ERR_MISALIGNED;
  return launch_pdl(bfp8_cast_kernel, dim3(cast_grid(rows * (K / 128) * 16)), dim3(kCastThreads), 0, stream,
                    reinterpret_cast<const uint4 *>(x), rows, K, static_cast<const int32_t *>(nullptr), 1, rows,
                    reinterpret_cast<uint2 *>(q), s);
}

extern "C" int bfp8_quantize_weight(const uint16_t *w, int64_t G, int64_t N, int64_t K, int layout, uint8_t *q,
                                    float *s, cudaStream_t stream) {
  if (G < 0 || N <= 0 || K <= 0) return MOE_ERR_INVALID_ARG;
  if (layout != BFP8_LAYOUT_CANONICAL && layout != BFP8_LAYOUT_TILED) return MOE_ERR_INVALID_ARG;
  if (N % 128 != 0 || K % 128 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (G == 0) return MOE_OK;
  if (!w || !q || !s) return MOE_ERR_INVALID_ARG;
  if (!aligned(w, 16) || !aligned(q, 16) || !aligned(s, 4)) return MOE_ERR_MISALIGNED;
  const int64_t blocks = G * (N / 128) * (K / 128);
  const int64_t cap = (int64_t)num_sms() * 8;
  return launch_pdl(bfp8_weight_kernel, dim3((unsigned)(blocks < cap ? blocks : cap)), dim3(kWqThreads), 0, stream,
                    reinterpret_cast<const uint4 *>(w), G, N, K, layout == BFP8_LAYOUT_TILED ? 1 : 0,
                    reinterpret_cast<uint4 *>(q), s);
}

extern "C" size_t moe_bfp8_workspace_size(int64_t T, int64_t H, int64_t I, int32_t E, int32_t k) {
  if (T < 0 || H <= 0 || I <= 0 || E <= 0 || k <= 0) return 0;
  return bfp8_ws_layout(T, H, I, E, k).total;
}

extern "C" int moe_forward_bfp8(const moe_bfp8_args *a, cudaStream_t st) {
  if (!a || a->struct_size != sizeof(moe_bfp8_args)) return MOE_ERR_INVALID_ARG;
  if (a->T < 0 || a->H <= 0 || a->I <= 0 || a->E <= 0 || a->k <= 0) return MOE_ERR_INVALID_ARG;
  if (!route_mode_valid(a->route_mode)) return MOE_ERR_INVALID_ARG;
  if (a->phases & ~(MOE_PHASE_GEMM1 | MOE_PHASE_GEMM2)) return MOE_ERR_INVALID_ARG;
  if (a->weight_layout != BFP8_LAYOUT_CANONICAL && a->weight_layout != BFP8_LAYOUT_TILED) return MOE_ERR_INVALID_ARG;
  if (!bfp8_shape_ok(a->T, a->H, a->I, a->E, a->k)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!a->workspace) return MOE_ERR_INVALID_ARG;
  if (!aligned(a->workspace, 256)) return MOE_ERR_MISALIGNED;
  const BWs lay = bfp8_ws_layout(a->T, a->H, a->I, a->E, a->k);
  if (a->workspace_bytes < lay.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (a->T > 0) {
    if (!a->x || !a->logits || !a->y || !a->w1q || !a->w1s || !a->w2q || !a->w2s) return MOE_ERR_INVALID_ARG;
    const void *ptrs[] = {a->x, a->logits, a->y, a->w1q, a->w2q};
    for (const void *p : ptrs)
      if (!aligned(p, 16)) return MOE_ERR_MISALIGNED;
    if (!aligned(a->w1s, 4) || !aligned(a->w2s, 4) || (a->hs_out && !aligned(a->hs_out, 4)))
      return MOE_ERR_MISALIGNED;
    const void *opt[] = {a->topk_idx_out, a->topk_w_out, a->counts_out, a->offsets_out, a->perm_out, a->hq_out};
    for (const void *p : opt)
      if (p && !aligned(p, 16)) return MOE_ERR_MISALIGNED;
  }
  char *ws = reinterpret_cast<char *>(a->workspace);
  int *status = reinterpret_cast<int *>(ws);
  if (cudaMemsetAsync(ws, 0, lay.sync_end, st) != cudaSuccess) return MOE_ERR_CUDA;
  if (a->T == 0) {
    if (a->counts_out && cudaMemsetAsync(a->counts_out, 0, (size_t)a->E * 4, st) != cudaSuccess) return MOE_ERR_CUDA;
    if (a->offsets_out && cudaMemsetAsync(a->offsets_out, 0, (size_t)(a->E + 1) * 4, st) != cudaSuccess)
      return MOE_ERR_CUDA;
    return MOE_OK;
  }
  const int64_t T = a->T, H = a->H, I = a->I, P = a->T * a->k;
  const int E = a->E, k = a->k;
  int32_t *idx = a->topk_idx_out ? a->topk_idx_out : reinterpret_cast<int32_t *>(ws + lay.idx);
  float *wts = a->topk_w_out ? a->topk_w_out : reinterpret_cast<float *>(ws + lay.w);
  int32_t *counts = a->counts_out ? a->counts_out : reinterpret_cast<int32_t *>(ws + lay.counts);
  int32_t *offsets = a->offsets_out ? a->offsets_out : reinterpret_cast<int32_t *>(ws + lay.offsets);
  int32_t *perm = a->perm_out ? a->perm_out : reinterpret_cast<int32_t *>(ws + lay.perm);
  int32_t *inv_perm = reinterpret_cast<int32_t *>(ws + lay.inv_perm);
  uint8_t *xq = reinterpret_cast<uint8_t *>(ws + lay.xq);
  float *xs = reinterpret_cast<float *>(ws + lay.xs);
  uint8_t *hq = a->hq_out ? a->hq_out : reinterpret_cast<uint8_t *>(ws + lay.hq);
  float *hs = a->hs_out ? a->hs_out : reinterpret_cast<float *>(ws + lay.hs);
  float *y_pairs = reinterpret_cast<float *>(ws + lay.y_pairs);

  // weights: [rows][K] row-major, or tiled as [rows * K / 128][128]
  const bool tiled = a->weight_layout == BFP8_LAYOUT_TILED;
  const uint64_t w1_cols = tiled ? 128 : (uint64_t)H, w1_rows = (uint64_t)E * 2 * I * (tiled ? H / 128 : 1);
  const uint64_t w2_cols = tiled ? 128 : (uint64_t)I, w2_rows = (uint64_t)E * H * (tiled ? I / 128 : 1);
  CUtensorMap tw1, tx, tw2, th;
  if (!encode_tmap_2d(&tw1, CU_TENSOR_MAP_DATA_TYPE_UINT8, const_cast<uint8_t *>(a->w1q), w1_cols, w1_rows, w1_cols,
                      128, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tmap_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_UINT8, xq, (uint64_t)H, (uint64_t)P, (uint64_t)H, 128, kGBN,
                      CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tmap_2d(&tw2, CU_TENSOR_MAP_DATA_TYPE_UINT8, const_cast<uint8_t *>(a->w2q), w2_cols, w2_rows, w2_cols,
                      128, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tmap_2d(&th, CU_TENSOR_MAP_DATA_TYPE_UINT8, hq, (uint64_t)I, (uint64_t)P, (uint64_t)I, 128, kGBN,
                      CU_TENSOR_MAP_SWIZZLE_128B))
    return MOE_ERR_CUDA;

  const bool whole = a->phases == 0;
  const bool small = bfp8_front_eligible(T, H, E, k);
  int rc = MOE_OK;
  if (whole && small) {
    rc = launch_pdl(bfp8_front_kernel, dim3((unsigned)(H / 128)), dim3(kBFrontThreads), bfp8_front_smem((int)T, E, k),
                    st, a->logits, reinterpret_cast<const uint4 *>(a->x), (int)T, E, k, (int)H, a->route_mode, idx, wts,
                    counts, offsets, perm, reinterpret_cast<uint2 *>(xq), xs);
    if (rc != MOE_OK) return rc;
  } else if (whole) {
    rc = launch_route(a->logits, T, E, k, a->route_mode, idx, wts, st);
    if (rc != MOE_OK) return rc;
    rc = launch_permute(idx, T, E, k, counts, offsets, perm, inv_perm, status, ws + lay.perm_scratch, st);
    if (rc != MOE_OK) return rc;
    rc = launch_pdl(bfp8_cast_kernel, dim3(cast_grid(P * (H / 128) * 16)), dim3(kCastThreads), 0, st,
                    reinterpret_cast<const uint4 *>(a->x), P, H, static_cast<const int32_t *>(perm), k, T,
                    reinterpret_cast<uint2 *>(xq), xs);
    if (rc != MOE_OK) return rc;
  }

  BGemmArgs g{};
  g.E = E; g.k = k; g.T = (int)T; g.H = (int)H; g.I = (int)I; g.P = (int)P;
  g.counts = counts; g.offsets = offsets; g.perm = perm; g.topk_w = wts; g.status = status;
  g.tiled = tiled ? 1 : 0;
  g.KB = (int)(H / 128); g.MT = (int)(I / 128);
  g.w_scales = a->w1s; g.x_scales = xs; g.hq = hq; g.hs = hs; g.y_pairs = y_pairs;
  if (whole && small) {
    // GEMM1, GEMM2 and the combine in one launch (every CTA resident)
    g.KB2 = (int)(I / 128); g.MT2 = (int)(H / 128);
    g.w_scales2 = a->w2s; g.x_scales2 = hs;
    g.sync = status + kStatusBytes / 4; g.topk_idx = idx; g.y = reinterpret_cast<uint4 *>(a->y);
    return launch_bfp8_gemm<3>(tw1, tx, tw2, th, g, st);
  }
  if (whole || (a->phases & MOE_PHASE_GEMM1)) {
    rc = launch_bfp8_gemm<1>(tw1, tx, tw1, tx, g, st);
    if (rc != MOE_OK) return rc;
  }
  g.KB = (int)(I / 128); g.MT = (int)(H / 128);
  g.w_scales = a->w2s; g.x_scales = hs;
  if (whole || (a->phases & MOE_PHASE_GEMM2)) {
    rc = launch_bfp8_gemm<2>(tw2, th, tw2, th, g, st);
    if (rc != MOE_OK) return rc;
  }
  if (!whole) return MOE_OK;
  return launch_pdl(bfp8_combine_kernel, dim3(cast_grid(T * (H / 8))), dim3(kCastThreads), 0, st,
                    reinterpret_cast<const float4 *>(y_pairs), static_cast<const int32_t *>(idx), T, k, H,
                    reinterpret_cast<uint4 *>(a->y));
}
