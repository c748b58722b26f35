// layer_blocks.cuh -- device routines shared by the standalone routing /
// permute kernels and by the fused small-problem front kernel.
#pragma once
#include <cstdint>

#include "ptx.cuh"

namespace mxq {

__device__ __forceinline__ bool route_better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

// Softmax top-k routing of one token by one warp (MonoMoe kernel -- design,
// section 1).  `row` is the token's E logits in this warp's shared memory (it
// is consumed: chosen entries are overwritten).  Selection ranks the raw
// logits, equal logits go to the lower expert index, output in descending
// order; w_j = exp(l_j - l_max) / sum over the k chosen.  Lane j < k returns
// the j-th choice in *idx_out / *w_out.
__device__ __forceinline__ void warp_route_token(float *row, int E, int k, int lane, int *idx_out, float *w_out) {
  float my_val = 0.f;
  int my_idx = 0;
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int e = lane; e < E; e += 32) {
      const float v = row[e];
      if (route_better(v, e, bv, bi)) { bv = v; bi = e; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (route_better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
    }
    if (lane == j) { my_val = bv; my_idx = bi; }
    if (lane == (bi & 31)) row[bi] = -INFINITY;     // taken (logits are finite)
    __syncwarp();
  }
  const float lmax = __shfl_sync(0xffffffffu, my_val, 0);
  const float ex = lane < k ? expf(my_val - lmax) : 0.f;
  float sum = ex;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  *idx_out = my_idx;
  *w_out = __fdiv_rn(ex, sum);
}

// Exclusive scan of one value per thread over a block of NT threads; returns
// the prefix and writes the block total to *total.  warp_sums: NT/32 ints.
template <int NT>
__device__ __forceinline__ int block_exclusive_scan(int v, int *warp_sums, int *total) {
  constexpr int kWarps = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += n;
  }
  if (lane == 31) warp_sums[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const int s = lane < kWarps ? warp_sums[lane] : 0;
    int si = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, si, o);
      if (lane >= o) si += n;
    }
    if (lane < kWarps) warp_sums[lane] = si - s;   // exclusive prefix of warp sums
    if (lane == 31) *total = si;
  }
  __syncthreads();
  return inc - v + warp_sums[warp];
}

// Stable ranks of pairs [lo, hi) inside their experts, NT pairs at a time
// (Counting Sort / Bucketization in DeepGEMM Mega MoE, section 2.3, with the
// slot taken as the rank among earlier same-expert pairs instead of an atomic
// counter).  expert_of(p) gives the expert of pair p (negative or >= E:
// dropped).  base[e] enters as the position of the block's first pair of e in
// perm and is advanced.  wc: (NT/32) * E uint16 scratch.  All NT threads call.
template <int NT, typename ExpertOf>
__device__ __forceinline__ void block_stable_ranks(ExpertOf expert_of, int64_t lo, int64_t hi, int E, int *base,
                                                   uint16_t *wc, int32_t *perm, int32_t *inv_perm,
                                                   int32_t *perm_smem = nullptr) {
  constexpr int kWarps = NT / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t lt_mask = (1u << lane) - 1u;
  for (int64_t start = lo; start < hi; start += NT) {
    uint32_t *wc32 = reinterpret_cast<uint32_t *>(wc);
    for (int i = tid; i < kWarps * E / 2; i += NT) wc32[i] = 0u;
    const int64_t p = start + tid;
    int e = -1;
    if (p < hi) {
      e = expert_of(p);
      if (e >= E) e = -1;
    }
    __syncthreads();
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    const int lrank = __popc(peers & lt_mask);
    if (e >= 0 && lrank == 0) wc[warp * E + e] = (uint16_t)__popc(peers);
    __syncthreads();
    int run[(1024 + NT - 1) / NT];
#pragma unroll
    for (int i = 0; i < (1024 + NT - 1) / NT; ++i) run[i] = 0;
#pragma unroll
    for (int i = 0; i < (1024 + NT - 1) / NT; ++i) {
      const int ee = tid + i * NT;
      if (ee < E) {
        int r = 0;
        for (int w = 0; w < kWarps; ++w) {
          const int c = wc[w * E + ee];
          wc[w * E + ee] = (uint16_t)r;
          r += c;
        }
        run[i] = r;
      }
    }
    __syncthreads();
    if (p < hi) {
      if (e >= 0) {
        const int pos = base[e] + wc[warp * E + e] + lrank;
        if (perm) perm[pos] = (int32_t)p;
        if (perm_smem) perm_smem[pos] = (int32_t)p;
        if (inv_perm) inv_perm[p] = pos;
      } else if (inv_perm) {
        inv_perm[p] = -1;
      }
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < (1024 + NT - 1) / NT; ++i) {
      const int ee = tid + i * NT;
      if (ee < E) base[ee] += run[i];
    }
    __syncthreads();
  }
}

}  // namespace mxq
