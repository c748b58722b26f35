// combine.cu -- top-k combine back to token order.
//
// MegaMoE (study notes), "Combine" and "L2 epilogue"; Warp Specialization:
// DeepEP vs Mega MoE, combine listing: the k BF16 copies of a token are
// summed in FP32 and cast to BF16 once.  The top-k weight already scaled h
// before GEMM2, so the sum is unweighted.  Dropped slots (index < 0) are
// skipped.  One thread owns 8 output values (16-byte loads and stores).
// The slot indices, then the slots' rows, are loaded eight at a time as
// independent loads (one memory round trip each, not one per slot); the sum
// still runs in slot order, so the result is deterministic.
#include <cuda_bf16.h>

#include "host_common.h"
#include "ptx.cuh"

namespace mxq {

namespace {

constexpr int kThreads = 256;
constexpr int kSlotBatch = 8;              // slots whose loads are in flight together

__global__ void __launch_bounds__(kThreads) combine_kernel(const uint4 *__restrict__ yp,
                                                           const int32_t *__restrict__ idx, int64_t T, int k,
                                                           int64_t H8, uint4 *__restrict__ y) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t items = T * H8;
  const int64_t slot_stride = T * H8;        // uint4 elements between slots
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < items;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / H8;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int j0 = 0; j0 < k; j0 += kSlotBatch) {
      bool use[kSlotBatch];
      uint4 v[kSlotBatch];
#pragma unroll
      for (int u = 0; u < kSlotBatch; ++u) use[u] = j0 + u < k && __ldg(idx + t * k + j0 + u) >= 0;
#pragma unroll
      for (int u = 0; u < kSlotBatch; ++u)
        if (use[u]) v[u] = __ldg(yp + (j0 + u) * slot_stride + i);
#pragma unroll
      for (int u = 0; u < kSlotBatch; ++u) {
        if (!use[u]) continue;
        const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          acc[2 * q] += bf16_bits_to_float(w[q] & 0xFFFFu);
          acc[2 * q + 1] += bf16_bits_to_float(w[q] >> 16);
        }
      }
    }
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * q], acc[2 * q + 1]);
      o[q] = *reinterpret_cast<const uint32_t *>(&b);
    }
    y[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

}  // namespace

int launch_combine(const uint16_t *y_pairs, const int32_t *idx, int64_t T, int k, int64_t H, uint16_t *y,
                   cudaStream_t st) {
  if (T == 0) return MOE_OK;
  const int64_t items = T * (H / 8);
  const int64_t blocks = ceil_div(items, kThreads);
  const int64_t cap = (int64_t)num_sms() * 8;
  return launch_pdl(combine_kernel, dim3((int)(blocks < cap ? blocks : cap)), dim3(kThreads), 0, st,
                    reinterpret_cast<const uint4 *>(y_pairs), idx, T, k, H / 8, reinterpret_cast<uint4 *>(y));
}

}  // namespace mxq

using namespace mxq;

extern "C" int moe_combine(const uint16_t *y_pairs, const int32_t *topk_idx, int64_t T, int32_t k, int64_t H,
                           uint16_t *y, cudaStream_t stream) {
  if (T < 0 || k <= 0 || H <= 0) return MOE_ERR_INVALID_ARG;
  if (k > 32 || H % 8 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (T == 0) return MOE_OK;
  if (!y_pairs || !topk_idx || !y) return MOE_ERR_INVALID_ARG;
  if (!aligned(y_pairs, 16) || !aligned(y, 16)) return MOE_ERR_MISALIGNED;
  return launch_combine(y_pairs, topk_idx, T, k, H, y, stream);
}
