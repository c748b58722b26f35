// permute.cu -- deterministic counting-sort permute of (token, slot) pairs.
//
// Counting Sort / Bucketization in DeepGEMM Mega MoE: section 2.1 COUNT
// (per-SM shared-memory histogram), 2.2 PREFIX SUM (a second level across
// SMs), 2.3 SCATTER (each pair takes a slot inside its expert's bucket),
// 5.2 (expert-contiguous pool), 8.2 (pair id = token * num_topk + slot).
//
// The pages take the cross-SM level and the slot inside a bucket from atomic
// counters, so the order inside an expert depends on timing.  Here both
// levels are exclusive scans in block order and the slot is the pair's rank
// among the same-expert pairs before it, so the result is the stable
// (token-ascending) permutation and is bit-reproducible:
//   count kernel   : block b histograms pairs [b*C, (b+1)*C) -> hist[b][e]
//   scatter kernel : block b sums hist of blocks < b (its base inside every
//                    bucket) and of all blocks (the totals), scans the totals
//                    into offsets, then ranks its pairs 1024 at a time with
//                    warp match_any + a per-warp count table in shared memory.
// With a single block the scatter kernel counts for itself (one launch).
#include "host_common.h"
#include "layer_blocks.cuh"
#include "ptx.cuh"

namespace mxq {

namespace {

constexpr int kThreads = 1024;
constexpr int kMaxE = 1024;
constexpr int kMaxBlocks = 64;

struct PermPlan {
  int64_t P, chunk;
  int nb;
};

PermPlan plan(int64_t T, int k) {
  PermPlan p;
  p.P = T * k;
  const int64_t per = round_up((size_t)ceil_div(p.P, kMaxBlocks), 1024);
  p.chunk = per > 2048 ? per : 2048;
  p.nb = (int)(p.P > 0 ? ceil_div(p.P, p.chunk) : 0);
  return p;
}

__global__ void __launch_bounds__(kThreads) perm_count_kernel(const int32_t *__restrict__ idx, int64_t P,
                                                              int E, int64_t chunk, int32_t *__restrict__ hist,
                                                              int *ws_status) {
  extern __shared__ int cnt[];
  pdl_launch_dependents();
  pdl_wait();
  for (int e = threadIdx.x; e < E; e += kThreads) cnt[e] = 0;
  __syncthreads();
  const int64_t lo = (int64_t)blockIdx.x * chunk;
  const int64_t hi = lo + chunk < P ? lo + chunk : P;
  for (int64_t p = lo + threadIdx.x; p < hi; p += kThreads) {
    const int e = __ldg(idx + p);
    if (e >= E) report_status(ws_status, kStatusBadIndex);
    else if (e >= 0) atomicAdd(&cnt[e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kThreads) hist[(int64_t)blockIdx.x * E + e] = cnt[e];
}

__global__ void __launch_bounds__(kThreads) perm_scatter_kernel(
    const int32_t *__restrict__ idx, int64_t P, int E, int64_t chunk, int nb,
    const int32_t *__restrict__ hist, int32_t *__restrict__ counts, int32_t *__restrict__ offsets,
    int32_t *__restrict__ perm, int32_t *__restrict__ inv_perm, int *ws_status) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  int *base = reinterpret_cast<int *>(smem_raw);                    // [E]
  int *self_cnt = base + kMaxE;                                     // [E] (single-block mode)
  int *warp_sums = self_cnt + kMaxE;                                // [32]
  int *total_sh = warp_sums + 32;                                   // [1]
  uint16_t *wc = reinterpret_cast<uint16_t *>(total_sh + 4);        // [32][E]

  const int tid = threadIdx.x;
  const int64_t lo = (int64_t)blockIdx.x * chunk;
  const int64_t hi = lo + chunk < P ? lo + chunk : P;
  pdl_launch_dependents();
  pdl_wait();

  // 1. totals and this block's base inside every bucket
  int tot = 0, pre = 0;
  if (nb == 1) {
    if (tid < E) self_cnt[tid] = 0;
    __syncthreads();
    for (int64_t p = tid; p < P; p += kThreads) {
      const int e = __ldg(idx + p);
      if (e >= E) report_status(ws_status, kStatusBadIndex);
      else if (e >= 0) atomicAdd(&self_cnt[e], 1);
    }
    __syncthreads();
    if (tid < E) tot = self_cnt[tid];
  } else if (tid < E) {
    for (int b = 0; b < nb; ++b) {
      const int h = __ldg(hist + (int64_t)b * E + tid);
      if (b < (int)blockIdx.x) pre += h;
      tot += h;
    }
  }
  // 2. offsets = exclusive scan of the totals
  const int off = block_exclusive_scan<kThreads>(tid < E ? tot : 0, warp_sums, total_sh);
  if (tid < E) base[tid] = off + pre;
  if (blockIdx.x == 0) {
    if (tid < E) {
      counts[tid] = tot;
      offsets[tid] = off;
    }
    if (tid == 0) offsets[E] = *total_sh;
  }
  __syncthreads();

  // 3. stable ranks, 1024 pairs at a time
  block_stable_ranks<kThreads>([&](int64_t p) { return (int)__ldg(idx + p); }, lo, hi, E, base, wc, perm, inv_perm);
}

size_t scatter_smem(int E) { return (size_t)(2 * kMaxE + 32 + 4) * 4 + (size_t)32 * E * 2; }

}  // namespace

size_t permute_scratch_bytes(int64_t T, int E, int k) {
  const PermPlan pl = plan(T, k);
  return round_up((size_t)pl.nb * E * 4, 256);
}

int launch_permute(const int32_t *idx, int64_t T, int E, int k, int32_t *counts, int32_t *offsets,
                   int32_t *perm, int32_t *inv_perm, int *status, void *scratch, cudaStream_t st) {
  const PermPlan pl = plan(T, k);
  int32_t *hist = reinterpret_cast<int32_t *>(scratch);
  if (pl.P == 0) {
    if (cudaMemsetAsync(counts, 0, (size_t)E * 4, st) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaMemsetAsync(offsets, 0, (size_t)(E + 1) * 4, st) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
  }
  const size_t sm = scatter_smem(E);
  if (sm > 48 * 1024 &&
      cudaFuncSetAttribute(perm_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm) !=
          cudaSuccess)
    return MOE_ERR_CUDA;
  if (pl.nb > 1) {
    if (launch_pdl(perm_count_kernel, dim3(pl.nb), dim3(kThreads), (size_t)E * 4, st, idx, pl.P, E, pl.chunk, hist,
                   status) != MOE_OK)
      return MOE_ERR_CUDA;
  }
  return launch_pdl(perm_scatter_kernel, dim3(pl.nb), dim3(kThreads), sm, st, idx, pl.P, E, pl.chunk, pl.nb,
                    (const int32_t *)hist, counts, offsets, perm, inv_perm, status);
}

}  // namespace mxq

using namespace mxq;

extern "C" size_t moe_permute_workspace_size(int64_t T, int32_t E, int32_t k) {
  if (T < 0 || E <= 0 || k <= 0) return 0;
  return kStatusBytes + permute_scratch_bytes(T, E, k);
}

extern "C" int moe_permute(const int32_t *topk_idx, int64_t T, int32_t E, int32_t k, int32_t *counts,
                           int32_t *offsets, int32_t *perm, int32_t *inv_perm, void *workspace,
                           size_t workspace_bytes, cudaStream_t stream) {
  if (T < 0 || E <= 0 || k <= 0) return MOE_ERR_INVALID_ARG;
  if (E > kMaxE || k > E || k > 32 || T * (int64_t)k >= ((int64_t)1 << 31)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!counts || !offsets || !workspace) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!topk_idx || !perm || !inv_perm)) return MOE_ERR_INVALID_ARG;
  if (!aligned(workspace, 256)) return MOE_ERR_MISALIGNED;
  if (workspace_bytes < kStatusBytes + permute_scratch_bytes(T, E, k)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (cudaMemsetAsync(workspace, 0, 32, stream) != cudaSuccess) return MOE_ERR_CUDA;
  return launch_permute(topk_idx, T, E, k, counts, offsets, perm, inv_perm, reinterpret_cast<int *>(workspace),
                        reinterpret_cast<char *>(workspace) + kStatusBytes, stream);
}
