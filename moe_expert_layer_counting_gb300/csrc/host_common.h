// host_common.h -- host-side helpers shared by the C-ABI translation units:
// argument checks, launch-error mapping, tensor-map encoding through the
// driver entry point, and the tile-size / workspace arithmetic.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <algorithm>
#include <cstdint>
#include <utility>

#include "../../include/moe_mxq.h"

namespace mxq {

inline bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline int launch_status() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

inline size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Launches a kernel with programmatic stream serialization, so that it may
// start while the previous kernel of the stream finishes (each kernel waits
// with griddepcontrol.wait before touching global memory).  Returns a status.
template <typename... KArgs, typename... Args>
inline int launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                      Args &&...args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Number of SMs of the current device (cached per device).
int num_sms();

// Encodes a 2-D tiled tensor map (dims/strides in elements/bytes as the
// driver expects).  Returns false if the driver rejects it.
bool encode_tmap_2d(CUtensorMap *map, CUtensorMapDataType dtype, void *base, uint64_t dim0, uint64_t dim1,
                    uint64_t stride1_bytes, uint32_t box0, uint32_t box1, CUtensorMapSwizzle swz);

// ------------------------------------------------------------------ scratch of
// the expert GEMMs (offsets are multiples of 256 bytes from the region base).
struct ExpertWs {
  size_t sfb1;       // GEMM1 token-scale chunks [max_tiles][H/128][512]
  size_t sfb2;       // GEMM2 token-scale chunks [max_tiles][I/128][512]
  size_t hq;         // requantised h in pool order [P][I]
  size_t tok_pool;   // token index of each pool row [P]
  size_t w_pool;     // top-k weight of each pool row [P]
  size_t xq_pool;    // FP8 activations in pool order [P][H] (large token tiles)
  size_t total;
};

inline int64_t max_token_tiles(int64_t P, int64_t E, int64_t bn) {
  const int64_t ne = E < P ? E : P;
  return ceil_div(P, bn) + ne;
}

inline ExpertWs expert_ws_layout(int64_t T, int64_t H, int64_t I, int64_t E, int64_t k) {
  const int64_t P = T * k;
  // token-scale chunks: the most (tiles x chunk bytes) over the tile sizes
  // (16 tokens: most tiles, 512 B chunks; 208 tokens: the most 1 KB chunks)
  const int64_t chunks = std::max(max_token_tiles(P, E, 16) * 512, max_token_tiles(P, E, 208) * 1024);
  ExpertWs w;
  size_t off = 0;
  w.sfb1 = off;    off += round_up((size_t)chunks * (size_t)(H / 128), 256);
  w.sfb2 = off;    off += round_up((size_t)chunks * (size_t)(I / 128), 256);
  w.hq = off;      off += round_up((size_t)P * (size_t)I, 256);
  w.tok_pool = off; off += round_up((size_t)P * 4, 256);
  w.w_pool = off;  off += round_up((size_t)P * 4, 256);
  w.xq_pool = off; off += round_up((size_t)P * (size_t)H, 256);
  w.total = off;
  return w;
}

// Every public workspace starts with this many bytes of status words.
constexpr size_t kStatusBytes = 256;

// Token tile chosen from the mean number of pairs per routed expert: tiles up
// to 64 tokens run two CTAs per SM; above that a large tile gives each
// tcgen05 instruction more tensor work (the MMA's N follows the tile's valid
// tokens rounded up to 16, or 32 on CTA pairs): 224 here, which
// resolve_tile_n turns into 208 where the GEMMs run on CTA pairs.
inline int choose_tile_n(int64_t P, int64_t E) {
  const int64_t ne = E < P ? E : P;
  const int64_t mean = ne > 0 ? ceil_div(P, ne) : 1;
  if (mean <= 16) return 16;
  if (mean <= 32) return 32;
  if (mean <= 64) return 64;
  return 224;
}

// Internal launchers (return a moe_status).  `status` points at the two
// status words of the caller's workspace.
int launch_quant_act(const uint16_t *x, int64_t rows, int64_t K, uint8_t *q, uint8_t *s, cudaStream_t st);
// zero_words[0, n_zero) are zeroed too (moe_forward's status words and
// arrival counters, before the launches that read them)
int launch_route(const float *logits, int64_t T, int E, int k, int mode, int32_t *idx, float *w, cudaStream_t st,
                 int *zero_words = nullptr, int n_zero = 0);
bool route_mode_valid(int mode);
size_t permute_scratch_bytes(int64_t T, int E, int k);
int launch_permute(const int32_t *idx, int64_t T, int E, int k, int32_t *counts, int32_t *offsets,
                   int32_t *perm, int32_t *inv_perm, int *status, void *scratch, cudaStream_t st);
int check_expert_args(const moe_expert_args *a, bool need_ws);
int launch_expert_forward(const moe_expert_args *a, int *status, void *scratch, cudaStream_t st);
// Activation cast straight into GEMM1's pool rows and scale chunks (replaces
// mxq_quantize_act + the token-scale step inside moe_forward).
int launch_pool_cast(const moe_expert_args *a, const uint16_t *x, void *scratch, cudaStream_t st);
// Large problems: the activation cast in token order, each BF16 row read once
// and written to its k pool rows + scale chunks (inv_perm from moe_permute).
int launch_token_cast(const moe_expert_args *a, const uint16_t *x, const int32_t *inv_perm, void *scratch,
                      cudaStream_t st);
// Small problems (front_eligible): routing, counting-sort permute and the pool
// cast in one launch.  `a` supplies shapes, tile size and the counts / offsets /
// perm outputs; the kernel also zeroes zero_words[0, n_zero) (the call's status
// words and arrival counters) before the next launch reads them.
bool front_eligible(int64_t T, int64_t H, int E, int k);
// GEMM1 + GEMM2 + combine in one launch after the front kernel (16-token
// tiles, all CTAs co-resident): eligibility, the arrival counters it needs
// (zeroed before the launch), and the launch (y: [T][H] output; ews: the
// expert workspace the front kernel filled).
bool fused_eligible(int64_t T, int64_t H, int E, int k, int tile_n);
size_t fused_sync_ints(int64_t T, int E, int k);
int launch_fused_gemms(const moe_expert_args *a, uint16_t *y, int *sync, int *status, char *ews, cudaStream_t st);
int launch_front(const moe_expert_args *a, const uint16_t *x, const float *logits, int mode, int32_t *idx,
                 float *wts, int32_t *inv_perm, void *scratch, int *zero_words, int n_zero, cudaStream_t st);
// Large problems (224-token tiles): GEMM1 / GEMM2 on 2-CTA clusters sharing
// one M = 256 MMA (gemm2sm.cu).  Eligible when both GEMMs' 128-row weight
// tiles pair up (2I/128 and H/128 even) and the shared memory fits.
bool pair_eligible(int64_t H, int64_t I, int E);
// moe_forward's large problems: GEMM1 + GEMM2 + combine in one launch on CTA
// pairs (expert waves, 208-token tiles), after the pool rows and token-scale
// chunks were written into the expert workspace `ews`; `sync` as for
// launch_fused_gemms (zeroed before the launch).
int launch_pair_layer(const moe_expert_args *a, uint16_t *y, int *sync, int *status, char *ews, cudaStream_t st);
// The token tile a call uses: tile_n, or choose_tile_n's when 0; the large
// tile is 208 tokens on CTA pairs (pair_eligible) and 224 on single CTAs.
int resolve_tile_n(int tile_n, int64_t P, int64_t E, int64_t H, int64_t I);
int run_expert_pairs(const moe_expert_args *a, int phases, int *status, uint8_t *hq, uint8_t *sfb1, uint8_t *sfb2,
                     const float *w_pool, const uint8_t *xq_pool, cudaStream_t st);
int launch_combine(const uint16_t *y_pairs, const int32_t *idx, int64_t T, int k, int64_t H, uint16_t *y,
                   cudaStream_t st);

}  // namespace mxq
