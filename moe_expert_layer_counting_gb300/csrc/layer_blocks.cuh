// layer_blocks.cuh -- device routines shared by the standalone routing /
// permute kernels and by the fused small-problem front kernel.
#pragma once
#include <cstdint>

#include "ptx.cuh"

namespace mxq {

// Order-preserving key of a finite logit (larger key = larger value); -0.0
// takes +0.0's key, so that equal values differ only by expert index.
__device__ __forceinline__ uint32_t route_key(float v) {
  const uint32_t u = __float_as_uint(v == 0.f ? 0.f : v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float route_key_value(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

// Routing modes (the ABI's MOE_ROUTE_* values): bits 0-1 the score
// (0 softmax, 1 sigmoid, 2 raw logits), bit 2 no renormalisation (raw scores
// are never renormalised).
enum : int { kRouteSoftmax = 0, kRouteSigmoid = 1, kRouteRaw = 2, kRouteNoRenorm = 4 };

// Top-k routing of one token by one warp (MonoMoe kernel -- design,
// section 1: softmax or sigmoid top-K with optional renormalisation; raw
// scores as in the MegaMoE test's topk of randn scores), straight from the
// token's E logits in global memory.  Selection ranks the raw logits (every
// score is an increasing function of them), equal logits go to the lower
// expert index, output in descending order.  Weights (l_max the top logit,
// S the k chosen):
//   softmax:   exp(l_j - l_max) / sum over S (renormalised) or over all E
//   sigmoid:   s_j = 1 / (1 + exp(-l_j)), divided by sum over S if renormalised
//   raw:       l_j
// Lane l holds the keys of experts l + 32 u (u < NV) in registers; each of
// the k rounds takes every lane's best remaining key, the warp maximum of
// those (redux) and, among the lanes that hold it, the lowest expert index
// (redux again); the owner clears that key.  Lane j < k returns the j-th
// choice in *idx_out / *w_out.  E <= 32 * NV; k <= min(E, 32).
template <int NV>
__device__ __forceinline__ void warp_route_token(const float *__restrict__ src, int E, int k, int lane, int mode,
                                                 int *idx_out, float *w_out) {
  uint32_t key[NV];
#pragma unroll
  for (int u = 0; u < NV; ++u) {
    const int e = lane + 32 * u;
    key[u] = e < E ? route_key(__ldg(src + e)) : 0u;    // 0: no expert (below every finite logit's key)
  }
  const int scoring = mode & 3;
  const bool renorm = scoring != kRouteRaw && !(mode & kRouteNoRenorm);
  float full_sum = 0.f;                      // softmax without renormalisation: sum over all E
  if (scoring == kRouteSoftmax && !renorm) {
    uint32_t lk = 0;
#pragma unroll
    for (int u = 0; u < NV; ++u) lk = key[u] > lk ? key[u] : lk;
    const float lmax = route_key_value(__reduce_max_sync(0xffffffffu, lk));
#pragma unroll
    for (int u = 0; u < NV; ++u)
      if (key[u] != 0u) full_sum += expf(route_key_value(key[u]) - lmax);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) full_sum += __shfl_xor_sync(0xffffffffu, full_sum, o);
  }
  int my_idx = 0;
  uint32_t my_key = 0;
  for (int j = 0; j < k; ++j) {
    uint32_t bk = 0;
    int bu = 0;
#pragma unroll
    for (int u = 0; u < NV; ++u)
      if (key[u] > bk) { bk = key[u]; bu = u; }           // ascending u: ties keep the lower index
    const uint32_t kmax = __reduce_max_sync(0xffffffffu, bk);
    const int e = (int)__reduce_min_sync(0xffffffffu, bk == kmax ? (uint32_t)(lane + 32 * bu) : 0xffffffffu);
    if (lane == j) { my_idx = e; my_key = kmax; }
#pragma unroll
    for (int u = 0; u < NV; ++u)
      if (lane == (e & 31) && u == (e >> 5)) key[u] = 0;
  }
  const float my_val = route_key_value(my_key);
  float score;                               // this lane's unnormalised weight (0 for lanes >= k)
  if (scoring == kRouteSoftmax) {
    const float lmax = __shfl_sync(0xffffffffu, my_val, 0);
    score = lane < k ? expf(my_val - lmax) : 0.f;
  } else if (scoring == kRouteSigmoid) {
    score = lane < k ? __fdiv_rn(1.f, 1.f + expf(-my_val)) : 0.f;
  } else {
    score = lane < k ? __ldg(src + my_idx) : 0.f;          // the logit itself (keeps the sign of a zero)
  }
  float denom = full_sum;
  if (renorm) {
    denom = score;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) denom += __shfl_xor_sync(0xffffffffu, denom, o);
  }
  *idx_out = my_idx;
  *w_out = lane >= k ? 0.f : (scoring == kRouteRaw || (scoring == kRouteSigmoid && !renorm)) ? score
                                                                                             : __fdiv_rn(score, denom);
}

// Exclusive prefix of ceil(cnt[e] / bn) over e < E into tile_off[0..E] (the
// first token tile of each expert; tile_off[E] = all tiles), by all NT
// threads of the block: each thread sums a contiguous run of experts, one
// block scan joins the runs.  warp_sums: NT/32 ints, total: 1 int.  The
// caller synchronises before reading tile_off.
template <int NT>
__device__ __forceinline__ void block_tile_map(const int *cnt, int E, int bn, int *tile_off, int *warp_sums,
                                               int *total);

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

template <int NT>
__device__ __forceinline__ void block_tile_map(const int *cnt, int E, int bn, int *tile_off, int *warp_sums,
                                               int *total) {
  const int per = (E + NT - 1) / NT;
  const int lo = min(E, (int)threadIdx.x * per), hi = min(E, lo + per);
  int sum = 0;
  for (int e = lo; e < hi; ++e) sum += (cnt[e] + bn - 1) / bn;
  int run = block_exclusive_scan<NT>(sum, warp_sums, total);
  for (int e = lo; e < hi; ++e) {
    tile_off[e] = run;
    run += (cnt[e] + bn - 1) / bn;
  }
  if (threadIdx.x == 0) tile_off[E] = *total;
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
