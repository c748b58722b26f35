// route.cu -- softmax top-k routing with renormalisation, one warp per token.
//
// MonoMoe kernel -- design, section 1 (phase 1: softmax top-K with optional
// renormalisation); the MegaMoE test routes with torch.topk over randn
// scores (Counting Sort / Bucketization in DeepGEMM Mega MoE, section 7.1).
// Selection ranks raw logits (same set as ranking softmax probabilities);
// equal logits go to the lower expert index.  Weights are
// exp(l_j - l_max) / sum over the chosen k -- the full softmax denominator
// cancels in the renormalisation.
#include "host_common.h"
#include "layer_blocks.cuh"
#include "ptx.cuh"

namespace mxq {

namespace {

constexpr int kWarps = 8;
constexpr int kMaxE = 1024;

__global__ void __launch_bounds__(kWarps * 32) route_kernel(const float *__restrict__ logits, int64_t T, int E,
                                                            int k, int mode, int32_t *__restrict__ idx,
                                                            float *__restrict__ w, int *__restrict__ zero_words,
                                                            int n_zero) {
  pdl_launch_dependents();
  pdl_wait();
  // moe_forward: the call's status words and arrival counters (read by the
  // launches after this one, which wait for its completion)
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < n_zero; i += blockDim.x) zero_words[i] = 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int64_t t = (int64_t)blockIdx.x * kWarps + warp; t < T; t += (int64_t)gridDim.x * kWarps) {
    int my_idx;
    float my_w;
    if (E <= 256) warp_route_token<8>(logits + t * E, E, k, lane, mode, &my_idx, &my_w);
    else warp_route_token<kMaxE / 32>(logits + t * E, E, k, lane, mode, &my_idx, &my_w);
    if (lane < k) {
      idx[t * k + lane] = my_idx;
      w[t * k + lane] = my_w;
    }
    __syncwarp();
  }
}

}  // namespace

int launch_route(const float *logits, int64_t T, int E, int k, int mode, int32_t *idx, float *w, cudaStream_t st,
                 int *zero_words, int n_zero) {
  if (T == 0) return MOE_OK;
  const int64_t blocks = ceil_div(T, kWarps);
  const int64_t cap = (int64_t)num_sms() * 8;
  const int grid = (int)(blocks < cap ? blocks : cap);
  return launch_pdl(route_kernel, dim3(grid), dim3(kWarps * 32), 0, st, logits, T, E, k, mode, idx, w, zero_words,
                    n_zero);
}

bool route_mode_valid(int mode) {
  return mode >= 0 && mode <= (kRouteNoRenorm | 3) && (mode & 3) != 3;
}

}  // namespace mxq

using namespace mxq;

extern "C" int moe_route_topk_ex(const float *logits, int64_t T, int32_t E, int32_t k, int32_t mode,
                                 int32_t *topk_idx, float *topk_w, cudaStream_t stream) {
  if (T < 0 || E <= 0 || k <= 0 || !route_mode_valid(mode)) return MOE_ERR_INVALID_ARG;
  if (E > kMaxE || k > E || k > 32) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (T == 0) return MOE_OK;
  if (!logits || !topk_idx || !topk_w) return MOE_ERR_INVALID_ARG;
  if (!aligned(logits, 16) || !aligned(topk_idx, 16) || !aligned(topk_w, 16)) return MOE_ERR_MISALIGNED;
  return launch_route(logits, T, E, k, mode, topk_idx, topk_w, stream);
}

extern "C" int moe_route_topk(const float *logits, int64_t T, int32_t E, int32_t k, int32_t *topk_idx,
                              float *topk_w, cudaStream_t stream) {
  return moe_route_topk_ex(logits, T, E, k, MOE_ROUTE_SOFTMAX, topk_idx, topk_w, stream);
}
