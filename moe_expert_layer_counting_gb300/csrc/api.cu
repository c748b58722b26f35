// api.cu -- the fused entry point moe_forward, workspace sizing, status
// helpers and the host utilities (SM count, tensor-map encoding) used by the
// other translation units.
//
// moe_forward enqueues, on one stream: activation cast (mxq_quantize_act),
// routing (moe_route_topk), the counting-sort permute (moe_permute), the two
// grouped GEMMs (moe_expert_forward) and the combine (moe_combine) -- the
// order of the MegaMoE baseline pipeline (MegaMoE (study notes), "Baseline
// implementation"), with dispatch and combine as local gather/scatter in HBM.
// The workspace sizing mirrors the MonoMoe scratchpad discipline (MonoMoe
// kernel -- design, section 4): one caller-provided buffer whose size the
// library reports, and whatever must start at zero is reset inside the call.
#include <cstdio>
#include <mutex>

#include "host_common.h"

namespace mxq {

int num_sms() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev < 0 || dev >= 64) return 1;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
    cache[dev] = n;
  }
  return cache[dev];
}

namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}
}  // namespace

bool encode_tmap_2d(CUtensorMap *map, CUtensorMapDataType dtype, void *base, uint64_t dim0, uint64_t dim1,
                    uint64_t stride1_bytes, uint32_t box0, uint32_t box1, CUtensorMapSwizzle swz) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {dim0, dim1};
  const cuuint64_t strides[1] = {stride1_bytes};
  const cuuint32_t box[2] = {box0, box1};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, dtype, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

// moe_forward casts x straight into pool order when P * H is at most this
constexpr int64_t kPoolCastMaxValues = int64_t(16) << 20;

struct ForwardWs {
  size_t sync_end;   // status words, then the single-launch layer's arrival counters (zeroed per call)
  size_t idx, w, counts, offsets, perm, inv_perm, perm_scratch, expert, y_pairs, total;
};

ForwardWs forward_ws_layout(int64_t T, int64_t H, int64_t I, int64_t E, int64_t k) {
  const int64_t P = T * k;
  ForwardWs w;
  size_t off = kStatusBytes;
  off += round_up(fused_sync_ints(T, (int)E, (int)k) * 4, 256);
  w.sync_end = off;
  w.idx = off;          off += round_up((size_t)P * 4, 256);
  w.w = off;            off += round_up((size_t)P * 4, 256);
  w.counts = off;       off += round_up((size_t)E * 4, 256);
  w.offsets = off;      off += round_up((size_t)(E + 1) * 4, 256);
  w.perm = off;         off += round_up((size_t)P * 4, 256);
  w.inv_perm = off;     off += round_up((size_t)P * 4, 256);
  w.perm_scratch = off; off += permute_scratch_bytes(T, (int)E, (int)k);
  w.expert = off;       off += expert_ws_layout(T, H, I, E, k).total;
  w.y_pairs = off;      off += round_up((size_t)P * H * 2, 256);
  w.total = off;
  return w;
}

}  // namespace

}  // namespace mxq

using namespace mxq;

extern "C" size_t moe_workspace_size(int64_t T, int64_t H, int64_t I, int32_t E, int32_t k) {
  if (T < 0 || H <= 0 || I <= 0 || E <= 0 || k <= 0) return 0;
  return forward_ws_layout(T, H, I, E, k).total;
}

extern "C" int moe_forward(const moe_forward_args *a, cudaStream_t st) {
  if (!a || a->struct_size != sizeof(moe_forward_args)) return MOE_ERR_INVALID_ARG;
  if (a->T < 0 || a->H <= 0 || a->I <= 0 || a->E <= 0 || a->k <= 0) return MOE_ERR_INVALID_ARG;
  if (!route_mode_valid(a->route_mode)) return MOE_ERR_INVALID_ARG;
  const int phases = a->phases;
  if (phases & ~(MOE_PHASE_GEMM1 | MOE_PHASE_GEMM2 | MOE_PHASE_RESET)) return MOE_ERR_INVALID_ARG;
  if (a->schedule < MOE_SCHEDULE_DEFAULT || a->schedule > MOE_SCHEDULE_EXPERT_WAVES) return MOE_ERR_INVALID_ARG;
  if (!a->workspace) return MOE_ERR_INVALID_ARG;
  if (!aligned(a->workspace, 256)) return MOE_ERR_MISALIGNED;
  const ForwardWs lay = forward_ws_layout(a->T, a->H, a->I, a->E, a->k);
  if (a->workspace_bytes < lay.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  char *ws = reinterpret_cast<char *>(a->workspace);
  int *status = reinterpret_cast<int *>(ws);

  moe_expert_args ea{};
  ea.struct_size = sizeof(moe_expert_args);
  ea.T = a->T; ea.H = a->H; ea.I = a->I; ea.E = a->E; ea.k = a->k;
  // every front end casts x straight into the pool rows (no token-order copy)
  ea.xq = nullptr;
  ea.xs = nullptr;
  ea.phases = MOE_PHASE_GEMM1 | MOE_PHASE_GEMM2;
  ea.w1q = a->w1q; ea.w1s = a->w1s; ea.w2q = a->w2q; ea.w2s = a->w2s;
  int32_t *idx = a->topk_idx_out ? a->topk_idx_out : reinterpret_cast<int32_t *>(ws + lay.idx);
  float *wts = a->topk_w_out ? a->topk_w_out : reinterpret_cast<float *>(ws + lay.w);
  int32_t *counts = a->counts_out ? a->counts_out : reinterpret_cast<int32_t *>(ws + lay.counts);
  int32_t *offsets = a->offsets_out ? a->offsets_out : reinterpret_cast<int32_t *>(ws + lay.offsets);
  int32_t *perm = a->perm_out ? a->perm_out : reinterpret_cast<int32_t *>(ws + lay.perm);
  ea.topk_idx = idx; ea.topk_w = wts; ea.counts = counts; ea.offsets = offsets; ea.perm = perm;
  ea.y_pairs = reinterpret_cast<uint16_t *>(ws + lay.y_pairs);
  ea.tile_n = a->tile_n;
  ea.workspace = ws + lay.expert;              // not used for sizing checks below
  ea.workspace_bytes = 0;
  int rc = check_expert_args(&ea, false);
  if (rc != MOE_OK) return rc;
  if (a->T > 0) {
    if (!a->x || !a->logits || !a->y) return MOE_ERR_INVALID_ARG;
    if (!aligned(a->x, 16) || !aligned(a->logits, 16) || !aligned(a->y, 16)) return MOE_ERR_MISALIGNED;
    if ((a->topk_idx_out && !aligned(a->topk_idx_out, 16)) || (a->topk_w_out && !aligned(a->topk_w_out, 16)))
      return MOE_ERR_MISALIGNED;
  }

  // phases != 0: timing / isolation, only the layer's GEMM launch(es) on the
  // state an earlier whole-layer call left in the workspace
  const int gemms = phases & (MOE_PHASE_GEMM1 | MOE_PHASE_GEMM2);
  const int64_t P = a->T * a->k;
  ea.tile_n = resolve_tile_n(a->tile_n, P, a->E, a->H, a->I);
  const bool front = a->T > 0 && front_eligible(a->T, a->H, a->E, a->k);
  const bool fused = front && fused_eligible(a->T, a->H, a->E, a->k, ea.tile_n);
  // large problems on CTA pairs, expert-wave schedule: GEMM1 + GEMM2 +
  // combine in one launch (the default keeps three launches: measured faster)
  const bool pair_layer = a->T > 0 && !front && ea.tile_n == 208 && a->schedule == MOE_SCHEDULE_EXPERT_WAVES;
  if ((fused || pair_layer) && gemms != 0 && gemms != (MOE_PHASE_GEMM1 | MOE_PHASE_GEMM2))
    return MOE_ERR_INVALID_ARG;

  // status words and arrival counters zeroed per call: by the call's first
  // kernel (the front or the routing kernel; one graph node fewer than a
  // memset), by a memset when only GEMM launches run (phases) or T = 0
  const bool kernel_zeroes = phases == 0 && a->T > 0;
  if ((phases == 0 || (phases & MOE_PHASE_RESET)) && !kernel_zeroes &&
      cudaMemsetAsync(ws, 0, lay.sync_end, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (phases != 0) {
    if (gemms == 0 || a->T == 0) return MOE_OK;
    if (fused) return launch_fused_gemms(&ea, a->y, status + kStatusBytes / 4, status, ws + lay.expert, st);
    if (pair_layer) return launch_pair_layer(&ea, a->y, status + kStatusBytes / 4, status, ws + lay.expert, st);
    ea.phases = gemms;
    return launch_expert_forward(&ea, status, ws + lay.expert, st);
  }
  if (a->T == 0) {
    if (a->counts_out && cudaMemsetAsync(a->counts_out, 0, (size_t)a->E * 4, st) != cudaSuccess) return MOE_ERR_CUDA;
    if (a->offsets_out && cudaMemsetAsync(a->offsets_out, 0, (size_t)(a->E + 1) * 4, st) != cudaSuccess)
      return MOE_ERR_CUDA;
    return MOE_OK;
  }
  int32_t *inv_perm = reinterpret_cast<int32_t *>(ws + lay.inv_perm);
  if (front_eligible(a->T, a->H, a->E, a->k)) {
    // small problems: routing + permute + pool cast in one launch
    rc = launch_front(&ea, a->x, a->logits, a->route_mode, idx, wts, inv_perm, ws + lay.expert, status,
                      (int)(lay.sync_end / 4), st);
    if (rc != MOE_OK) return rc;
    // then, with 16-token tiles, both GEMMs and the combine in one more
    if (fused)
      return launch_fused_gemms(&ea, a->y, status + kStatusBytes / 4, status, ws + lay.expert, st);
    rc = launch_expert_forward(&ea, status, ws + lay.expert, st);
    if (rc != MOE_OK) return rc;
    return launch_combine(ea.y_pairs, idx, a->T, a->k, a->H, a->y, st);
  }
  rc = launch_route(a->logits, a->T, a->E, a->k, a->route_mode, idx, wts, st, status, (int)(lay.sync_end / 4));
  if (rc != MOE_OK) return rc;
  rc = launch_permute(idx, a->T, a->E, a->k, counts, offsets, perm, inv_perm, status, ws + lay.perm_scratch, st);
  if (rc != MOE_OK) return rc;
  if (P * a->H <= kPoolCastMaxValues) {
    // small problems: cast x straight into GEMM1's pool rows and scale chunks
    // (one launch, every load in flight at once)
    rc = launch_pool_cast(&ea, a->x, ws + lay.expert, st);
  } else {
    // large problems: cast each token once (x read once) and scatter its codes
    // to its k pool rows
    rc = launch_token_cast(&ea, a->x, inv_perm, ws + lay.expert, st);
  }
  if (rc != MOE_OK) return rc;
  if (pair_layer)   // both GEMMs and the combine in one launch
    return launch_pair_layer(&ea, a->y, status + kStatusBytes / 4, status, ws + lay.expert, st);
  rc = launch_expert_forward(&ea, status, ws + lay.expert, st);
  if (rc != MOE_OK) return rc;
  return launch_combine(ea.y_pairs, idx, a->T, a->k, a->H, a->y, st);
}

extern "C" int moe_get_device_status(const void *workspace, cudaStream_t stream, int *out) {
  if (!workspace || !out) return MOE_ERR_INVALID_ARG;
  int host = 0;
  if (cudaMemcpyAsync(&host, workspace, sizeof(int), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MOE_ERR_CUDA;
  *out = host;
  return MOE_OK;
}

extern "C" const char *moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument (null pointer, negative size or bad enum)";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape (see the shape limits in moe_mxq.h)";
    case MOE_ERR_MISALIGNED: return "misaligned pointer (16 bytes; 32 for packed FP4 weights)";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace smaller than the reported size";
    case MOE_ERR_CUDA: return "CUDA launch or driver call failed";
    case MOE_ERR_TIMEOUT: return "a device-side wait gave up (timeout)";
    case MOE_ERR_DEVICE_INDEX: return "device found an expert index out of range";
    default: return "unknown status";
  }
}

extern "C" const char *moe_version(void) { return "moe_mxq 0.1 (sm_103a, tcgen05 block-scaled)"; }
