// quant.cu -- BF16 -> FP8 E4M3 (activations) and BF16 -> FP4 E2M1 (weights),
// one UE8M0 scale per 32 values along K.
//
// MegaMoE (study notes), "Dispatch" (tokens cast per 32 along hidden) and
// "Expert weight quantisation" (BF16 [G, n, k] -> FP4 + UE8M0 [G, n, k/32]).
// Both kernels stream: one thread owns 8 consecutive BF16 values (one 16-byte
// load), four neighbouring lanes form a 32-group and agree on its amax with
// two xor-shuffles.  Pure HBM streaming: 2 B read, 1 B (E4M3) or 0.5 B (E2M1)
// written per element plus 1/32 B of scale.
#include "host_common.h"
#include "ptx.cuh"

namespace mxq {

namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ void unpack8(const uint4 &v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = bf16_bits_to_float(w[i] & 0xFFFFu);
    f[2 * i + 1] = bf16_bits_to_float(w[i] >> 16);
  }
}

__device__ __forceinline__ float group4_amax(float a) {
  a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
  a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
  return a;
}

// items = rows * K / 8; item i covers elements [8i, 8i+8) of the flattened
// [rows][K] array, so the 32-group of item i is i / 4.
__global__ void __launch_bounds__(kThreads) quant_act_kernel(const uint4 *__restrict__ x, int64_t items,
                                                             uint2 *__restrict__ q, uint8_t *__restrict__ s) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t base = (int64_t)blockIdx.x * blockDim.x; base < items; base += stride) {
    const int64_t i = base + threadIdx.x;
    const bool valid = i < items;
    uint8_t sb;
    const uint2 codes = cast8_e4m3(valid ? __ldg(x + i) : make_uint4(0, 0, 0, 0), valid, &sb);
    if (!valid) continue;
    q[i] = codes;
    if ((i & 3) == 0) s[i >> 2] = sb;
  }
}

// Weight quantisation.  Row n of group g in the input (K values) is written
// to stored row r (the gate/up interleave for MMA_L1).  Canonical: codes
// row-major [G][N][K/2], scales [G][N][K/32].  MMA layouts: codes in
// tile-contiguous blocks [G][N/128][K/128][128 rows][64 bytes] (one 128 x 128
// tile = 8 KB in one piece) and scales in chunks [G][N/128][K/128][512] with
// byte (r%32)*16 + (r/32)*4 + kk.
__global__ void __launch_bounds__(kThreads) quant_weight_kernel(const uint4 *__restrict__ w, int64_t G,
                                                                int64_t N, int64_t K, int layout,
                                                                uint32_t *__restrict__ q,
                                                                uint8_t *__restrict__ s) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t items = G * N * K / 8;
  const int64_t items_per_row = K / 8;
  const int64_t half = N / 2;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t base = (int64_t)blockIdx.x * blockDim.x; base < items; base += stride) {
    const int64_t i = base + threadIdx.x;
    const bool valid = i < items;
    float f[8];
    float amax = 0.f;
    if (valid) {
      unpack8(__ldg(w + i), f);
#pragma unroll
      for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
    }
    amax = group4_amax(amax);
    if (!valid) continue;
    const int e = ue8m0_exponent<false>(amax);
    const float inv = pow2_neg(e);
    uint32_t packed = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) packed |= cvt_e2m1x2(f[2 * j] * inv, f[2 * j + 1] * inv) << (8 * j);

    const int64_t row = i / items_per_row;        // g * N + n
    const int64_t col_item = i - row * items_per_row;
    const int64_t g = row / N;
    const int64_t n = row - g * N;
    int64_t r = n;                                 // stored row inside group g
    if (layout == MXQ_LAYOUT_MMA_L1) {
      const int64_t up = n >= half;
      const int64_t f_idx = up ? n - half : n;
      r = (f_idx >> 3) * 16 + (up ? 8 : 0) + (f_idx & 7);
    }
    if (layout == MXQ_LAYOUT_CANONICAL) {
      q[(g * N + r) * items_per_row + col_item] = packed;
    } else {
      // tile-contiguous: [g][r/128][k/128][r%128][64 bytes]; 16 words of 4 bytes per tile row
      const int64_t nt = r >> 7, rr = r & 127, kb = col_item >> 4, w16 = col_item & 15;
      q[(((g * (N / 128) + nt) * (K / 128) + kb) * 128 + rr) * 16 + w16] = packed;
    }
    if ((col_item & 3) == 0) {
      const int64_t kg = col_item >> 2;           // 32-group along K
      int64_t off;
      if (layout == MXQ_LAYOUT_CANONICAL) {
        off = (g * N + r) * (K / 32) + kg;
      } else {
        const int64_t nt = r >> 7, rr = r & 127, kb = kg >> 2, kk = kg & 3;
        off = ((g * (N / 128) + nt) * (K / 128) + kb) * 512 + (rr & 31) * 16 + (rr >> 5) * 4 + kk;
      }
      s[off] = (uint8_t)(e + 127);
    }
  }
}

int grid_for(int64_t items) {
  const int64_t blocks = ceil_div(items, kThreads);
  const int64_t cap = (int64_t)num_sms() * 8;
  return (int)(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

}  // namespace

int launch_quant_act(const uint16_t *x, int64_t rows, int64_t K, uint8_t *q, uint8_t *s, cudaStream_t st) {
  const int64_t items = rows * K / 8;
  if (items == 0) return MOE_OK;
  return launch_pdl(quant_act_kernel, dim3(grid_for(items)), dim3(kThreads), 0, st,
                    reinterpret_cast<const uint4 *>(x), items, reinterpret_cast<uint2 *>(q), s);
}

}  // namespace mxq

using namespace mxq;

extern "C" int mxq_quantize_act(const uint16_t *x, int64_t rows, int64_t K, uint8_t *q, uint8_t *s,
                                cudaStream_t stream) {
  if (rows < 0 || K <= 0) return MOE_ERR_INVALID_ARG;
  if (K % 32 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (rows == 0) return MOE_OK;
  if (!x || !q || !s) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(q, 16)) return MOE_ERR_MISALIGNED;
  return launch_quant_act(x, rows, K, q, s, stream);
}

extern "C" int mxq_quantize_weight(const uint16_t *w, int64_t G, int64_t N, int64_t K, int layout,
                                   uint8_t *q, uint8_t *s, cudaStream_t stream) {
  if (G < 0 || N <= 0 || K <= 0) return MOE_ERR_INVALID_ARG;
  if (layout != MXQ_LAYOUT_CANONICAL && layout != MXQ_LAYOUT_MMA_L1 && layout != MXQ_LAYOUT_MMA_L2)
    return MOE_ERR_INVALID_ARG;
  if (K % 32 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (layout != MXQ_LAYOUT_CANONICAL && (K % 128 != 0 || N % 128 != 0)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (layout == MXQ_LAYOUT_MMA_L1 && N % 16 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (G == 0) return MOE_OK;
  if (!w || !q || !s) return MOE_ERR_INVALID_ARG;
  if (!aligned(w, 16) || !aligned(q, 16)) return MOE_ERR_MISALIGNED;
  const int64_t items = G * N * K / 8;
  return launch_pdl(quant_weight_kernel, dim3(grid_for(items)), dim3(kThreads), 0, stream,
                    reinterpret_cast<const uint4 *>(w), G, N, K, layout, reinterpret_cast<uint32_t *>(q), s);
}
