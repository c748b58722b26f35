// gemm2sm.cu -- the expert GEMMs of large problems on CTA pairs: one
// tcgen05.mma.cta_group::2 (M = 256 weight rows, N up to 224 tokens, K = 32,
// kind::mxf8f6f4 block-scaled) drives the tensor cores of two SMs.
//
// The same GEMM1 (FP8 tokens x FP4 W1|W3, SwiGLU (.) top-k weight, FP8 + UE8M0
// requantisation) and GEMM2 (FP8 h x FP4 W2 -> BF16 per pair) as gemm.cu, on
// 224-token tiles.  Prior art: the MMA warp listing of "Warp Specialization:
// DeepEP vs Mega MoE" issues the 2-SM block-scaled MMA from the leader CTA of
// a pair, and the MegaMoE study notes ("Scheduler") run each tile on a 2-SM
// cluster.  What a pair buys on GB300:
//   * each CTA stages its own 128 weight rows but only half of the token rows
//     (the MMA reads B's halves from both CTAs), so a stage is 31.5 KB instead
//     of 45.5 KB and five stages fit per SM -- the one-CTA kernel keeps two per
//     CTA and leaves the tensor pipe waiting on loads;
//   * one thread issues for two SMs: four MMAs and three scale copies per
//     128-wide K block keep both tensor cores ~97 % busy at N = 224 (measured
//     issue rate), and token rows cross L2 -> SM once per pair, not per SM.
// Roles per CTA (320 threads): warp 0 TMA producer (both CTAs), warp 1 TMEM
// allocation (both) and the MMA issuer (rank 0 only), warps 2-9 epilogue
// (both; two halves of four warps, one TMEM lane quadrant per warp).
// Synchronisation of the pair:
//   * every load of either CTA counts on the leader's `full` barrier (TMA
//     .cta_group::2 form); the leader's producer arms it for both CTAs' bytes;
//   * the leader's commits arrive on `empty` and `tmem_full` of both CTAs
//     (multicast); each CTA's epilogue arrives on the leader's `tmem_empty`;
//   * all waits are bounded (MOE_ERR_TIMEOUT in the status words); the pair
//     meets at a cluster barrier before TMEM is freed, so no CTA exits while
//     the other still reads its shared memory or signals its barriers.
// Work order: expert-major, then weight-row pair, then token tile (as gemm.cu).
#include <cuda_bf16.h>

#include <cstdlib>
#include <utility>

#include "gemm_common.cuh"
#include "host_common.h"
#include "layer_blocks.cuh"
#include "ptx.cuh"

namespace mxq {

namespace {

struct Pair {
  static constexpr int kBN = 208;                         // token tile
  static constexpr int kHalf = kBN / 2;                   // token rows staged per CTA (TMA box height)
  static constexpr int kStreams = 2;                      // independent issue streams of a pair
  static constexpr int kStagesPerStream = 3;
  static constexpr int kStages = kStreams * kStagesPerStream;
  static constexpr int kEpiWarps = 8;
  static constexpr int kFirstEpiWarp = 2 * kStreams;      // warps 0-1 producers, 2-3 MMA issuers
  static constexpr int kThreads = 32 * (kFirstEpiWarp + kEpiWarps);
  static constexpr int kATile = kBM * kBK;                // unpacked FP4 weight tile (8-bit containers)
  static constexpr int kBTile = kHalf * kBK;
  static constexpr int kTokChunk = 1024;                  // token scales of one (tile, K block): 2 x 128 rows
  static constexpr int kSfSlot = 12;                      // TMEM columns per stage: 4 weight + 8 token scales
  static constexpr int kTmemAcc = kStreams * kBN;         // one accumulator per stream
  static constexpr int kTmemCols = kTmemAcc + kSfSlot * kStages;
  // bytes landing on the leader's full barrier per stage (both CTAs; the
  // FP4-unpacking weight load counts its packed bytes)
  static constexpr uint32_t kStageTx = 2u * (kWTileBytes + kBTile + 512 + kTokChunk);
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + kStages * kATile;
  static constexpr int kOffSfa = kOffB + kStages * kBTile;
  static constexpr int kOffSfb = kOffSfa + kStages * 512;
  static constexpr int kOffEpi = kOffSfb + kStages * kTokChunk;
  static constexpr int kOffRow = kOffEpi + 4096 * 2;      // pair id [2][BN], weight [2][BN]
  static constexpr int kOffBar = kOffRow + 16 * kBN;
  // full[kStages], empty[kStages], tmem_full[2], tmem_empty[2], mma_done[2], never
  static constexpr int kNumBars = 2 * kStages + 3 * kStreams + 1;
  static constexpr int kOffTmemPtr = (kOffBar + 8 * kNumBars + 63) & ~63;
  static constexpr int kOffScan = kOffTmemPtr + 64;
  static constexpr int kOffExp = kOffScan + 64;
  static_assert(kTmemCols <= 512, "TMEM budget");
  static_assert(kBTile % 1024 == 0 && kATile % 1024 == 0, "stage buffers stay 1024-byte aligned");
  static_assert(kHalf % 8 == 0, "token half-tiles are whole 8-row swizzle atoms");
};

size_t pair_smem_bytes(int E) { return 1024 + Pair::kOffExp + (size_t)3 * (E + 1) * 4; }

struct PairArgs {
  int E, k, T, H, I;
  int KB, MT;                       // K blocks, 128-row weight tiles per expert (even)
  int inject_wait;                  // debug: the MMA issuers first wait on a barrier nothing completes
  const uint8_t *w_codes;           // L2 prefetch ahead of the weight loads
  const int32_t *counts, *offsets, *perm;
  const float *w_pool;              // GEMM1 epilogue: top-k weight of each pool row
  uint8_t *hq, *sfb2, *hs_out;      // GEMM1 outputs
  uint16_t *y_pairs;                // GEMM2 output
  int *status;
};

template <int PHASE>
__global__ void __launch_bounds__(Pair::kThreads, 1)
    expert_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_b,
                            const __grid_constant__ CUtensorMap tmap_wsf,
                            const __grid_constant__ CUtensorMap tmap_bsf, const PairArgs args) {
  // PHASE 1: GEMM1 + SwiGLU epilogue; 2: GEMM2.
  // A cluster's j-th work item belongs to stream j % 2: producer warp s loads
  // it into stages [3s, 3s+3), MMA warp 2+s (leader) accumulates it into
  // accumulator s; the epilogue warps drain the accumulators in item order.
  using C = Pair;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                          ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
  uint64_t *full = bars;                         // leader: both CTAs' loads of a stage
  uint64_t *empty = bars + C::kStages;           // each CTA: stage consumed (leader's commit)
  uint64_t *tmem_full = bars + 2 * C::kStages;   // each CTA: accumulator s ready (leader's commit)
  uint64_t *tmem_empty = tmem_full + C::kStreams;  // leader: both CTAs' epilogues drained accumulator s
  uint64_t *mma_done = tmem_empty + C::kStreams;
  uint64_t *never = mma_done + C::kStreams;
  uint32_t *tmem_ptr = reinterpret_cast<uint32_t *>(smem + C::kOffTmemPtr);
  int *vote = reinterpret_cast<int *>(smem + C::kOffTmemPtr + 4);
  int *tile_off = reinterpret_cast<int *>(smem + C::kOffExp);
  int *cnt_sm = tile_off + (args.E + 1);
  int *off_sm = cnt_sm + (args.E + 1);
  int32_t *row_pair_buf = reinterpret_cast<int32_t *>(smem + C::kOffRow);
  float *row_w_buf = reinterpret_cast<float *>(smem + C::kOffRow + 8 * C::kBN);
  int *scan_ws = reinterpret_cast<int *>(smem + C::kOffScan);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int cluster = (int)blockIdx.x >> 1, nclusters = (int)gridDim.x >> 1;
  int *status = args.status;
#ifdef MOE_MXQ_WAIT_STATS
  // optional accounting (as in gemm.cu), 64-bit counters at byte 64 of the
  // status area: [0] producer waits on empty stages, [1] MMA waits on full
  // stages, [2] MMA waits on free accumulators, [3] epilogue waits on full
  // accumulators, [4..6] kernel cycles of warps 0..2, [7] work items,
  // [8] MMA issue cycles, [9] epilogue busy cycles (first epilogue warp)
  long long wait_acc[6] = {0, 0, 0, 0, 0, 0};
  const long long k_t0 = clock64();
  int n_items = 0;
#endif

  if (PHASE == 2) pdl_launch_dependents();
  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tmap_w);
      tma_prefetch_desc(&tmap_b);
      tma_prefetch_desc(&tmap_wsf);
      tma_prefetch_desc(&tmap_bsf);
    }
  } else if (warp == 2) {
    if (lane == 0) {
      for (int s = 0; s < C::kStages; ++s) {
        mbar_init(&full[s], 1);
        mbar_init(&empty[s], 1);
      }
      for (int a = 0; a < C::kStreams; ++a) {
        mbar_init(&tmem_full[a], 1);
        mbar_init(&tmem_empty[a], 2 * C::kEpiWarps);
        mbar_init(&mma_done[a], 1);
      }
      mbar_init(never, 1);
      fence_mbar_init();
    }
    __syncwarp();
    tmem_alloc_2sm(tmem_ptr, 512);
    tmem_relinquish_2sm();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();                  // both CTAs' barriers exist before any cross-CTA signal
  tc_fence_after();
  pdl_wait();
  if (PHASE == 1) pdl_launch_dependents();
  load_expert_table(args.counts, args.offsets, args.E, cnt_sm, off_sm);
  __syncthreads();
  block_tile_map<C::kThreads>(cnt_sm, args.E, C::kBN, tile_off, scan_ws, scan_ws + 15);
  __syncthreads();
  const uint32_t tmem_base = *tmem_ptr;
  const int MT2 = args.MT >> 1;                    // weight-row pairs per expert
  const int total_work = tile_off[args.E] * MT2;

  if (warp < C::kStreams) {
    // ------------------------------------------------------------ TMA producers (both CTAs)
    const int st = warp;
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued_mask = 0, issued_phase = 0;
    for (int w = cluster + st * nclusters; w < total_work; w += C::kStreams * nclusters) {
      const TileInfo ti = decode_work<C::kBN>(w, MT2, args.E, tile_off, cnt_sm, off_sm);
      const int n_mma = min(C::kBN, (ti.valid + 31) & ~31);
      const int mt = 2 * ti.mt + (int)rank;                       // this CTA's 128-row weight tile
      const int wtile = (ti.e * args.MT + mt) * args.KB;
      bool ok = true;
      for (int kb = 0; kb < args.KB; ++kb) {
        const int gs = st * C::kStagesPerStream + stage;
        if (!__all_sync(0xffffffffu, MXQ_TIMED_WAIT(0, mbar_wait(&empty[gs], phase ^ 1, status, kWaitLimit,
                                                                 kWaitProducerEmpty, kb)))) {
          ok = false;
          break;
        }
        if (lane == 0) {
          if (rank == 0) mbar_arrive_expect_tx(&full[gs], C::kStageTx);
          const uint32_t bar = mapa_shared(smem_u32(&full[gs]), 0);
          tma_load_2d_2sm(smem + C::kOffA + gs * C::kATile, &tmap_w, bar, 0, (wtile + kb) * kBM);
          tma_load_2d_2sm(smem + C::kOffB + gs * C::kBTile, &tmap_b, bar, kb * kBK,
                          ti.s0 + (int)rank * (n_mma >> 1));
          tma_load_2d_2sm(smem + C::kOffSfa + gs * 512, &tmap_wsf, bar, 0, (wtile + kb) * 2);
          tma_load_2d_2sm(smem + C::kOffSfb + gs * C::kTokChunk, &tmap_bsf, bar, 0, (ti.g * args.KB + kb) * 4);
          if (kb + kPrefetchAhead < args.KB)
            prefetch_l2_bulk(args.w_codes + ((size_t)wtile + kb + kPrefetchAhead) * kWTileBytes, kWTileBytes);
        }
        __syncwarp();
        issued_mask |= 1u << gs;
        issued_phase = (issued_phase & ~(1u << gs)) | (phase << gs);
        if (++stage == C::kStagesPerStream) { stage = 0; phase ^= 1; }
      }
      if (!ok) break;
    }
    // the leader never leaves with copies in flight (its full barriers count
    // both CTAs' bytes; the other CTA's copies are covered by the final
    // cluster barrier, which the leader reaches only after this drain)
    if (rank == 0)
      for (int gs = 0; gs < C::kStages; ++gs)
        if (issued_mask & (1u << gs))
          mbar_wait(&full[gs], (issued_phase >> gs) & 1u, status, kWaitLimit, kWaitProducerDrain, gs, false);
    // after a wait gave up, the other CTA may have copies in flight for a stage
    // the leader never armed (and so never drains): give them time to land
    // (~100 us; a copy takes a few) before the pair frees its shared memory
    if (lane == 0 && *reinterpret_cast<volatile int *>(status + 1) != 0) {
      const long long t0 = clock64();
      while (clock64() - t0 < 200000) __nanosleep(1000);
    }
    __syncwarp();
  } else if (warp < 2 * C::kStreams) {
    // ------------------------------------------------------------ MMA issuers (leader only)
    const int st = warp - C::kStreams;
    if (rank == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      const uint32_t d_tmem = tmem_base + (uint32_t)(st * C::kBN);
      for (int w = cluster + st * nclusters; w < total_work && ok; w += C::kStreams * nclusters) {
        const TileInfo ti = decode_work<C::kBN>(w, MT2, args.E, tile_off, cnt_sm, off_sm);
        const uint32_t n_mma = (uint32_t)min(C::kBN, (ti.valid + 31) & ~31);
        if (!__all_sync(0xffffffffu, MXQ_TIMED_WAIT(2, mbar_wait(&tmem_empty[st], acc_phase ^ 1, status, kWaitLimit,
                                                                 kWaitMmaTmemEmpty, w))))
          break;
        if (args.inject_wait == 1 && w == cluster + st * nclusters &&
            !__all_sync(0xffffffffu, mbar_wait(never, 0, status, kInjectedWaitLimit, kWaitInjected, w)))
          break;
        tc_fence_after();
        for (int kb = 0; kb < args.KB; ++kb) {
          const int gs = st * C::kStagesPerStream + stage;
          if (!__all_sync(0xffffffffu,
                          MXQ_TIMED_WAIT(1, mbar_wait(&full[gs], phase, status, kWaitLimit, kWaitMmaFull, kb)))) {
            ok = false;
            break;
          }
          tc_fence_after();
#ifdef MOE_MXQ_WAIT_STATS
          const long long t_issue = clock64();
#endif
          if (lane == 0) {
            const uint32_t sf_col = tmem_base + (uint32_t)(C::kTmemAcc + C::kSfSlot * gs);
            const uint32_t sfa = smem_u32(smem + C::kOffSfa + gs * 512);
            const uint32_t sfb = smem_u32(smem + C::kOffSfb + gs * C::kTokChunk);
            tc_cp_2sm_32x128b_warpx4(sf_col, make_smem_desc(sfa, 0, 128, kSwizzleNone));
            tc_cp_2sm_32x128b_warpx4(sf_col + 4, make_smem_desc(sfb, 0, 128, kSwizzleNone));
            if (n_mma > 128) tc_cp_2sm_32x128b_warpx4(sf_col + 8, make_smem_desc(sfb + 512, 0, 128, kSwizzleNone));
            const uint32_t a_base = smem_u32(smem + C::kOffA + gs * C::kATile);
            const uint32_t b_base = smem_u32(smem + C::kOffB + gs * C::kBTile);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t ad = make_smem_desc(a_base + kk * 32, 16, 1024, kSwizzle128B);
              const uint64_t bd = make_smem_desc(b_base + kk * 32, 16, 1024, kSwizzle128B);
              tc_mma_2sm_mxf8f6f4(d_tmem, ad, bd, make_idesc_fp4w_fp8a(n_mma, kk, 256), sf_col, sf_col + 4,
                                  (kb | kk) != 0 ? 1u : 0u);
            }
            tc_commit_2sm(&empty[gs], 3);
          }
          __syncwarp();
#ifdef MOE_MXQ_WAIT_STATS
          if (lane == 0) wait_acc[4] += clock64() - t_issue;
#endif
          if (++stage == C::kStagesPerStream) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        if (lane == 0) tc_commit_2sm(&tmem_full[st], 3);
        __syncwarp();
        acc_phase ^= 1;
      }
      // every MMA of this thread completes before the pair frees TMEM
      if (lane == 0) tc_commit_2sm(&mma_done[st], 1);
      __syncwarp();
      mbar_wait(&mma_done[st], 0, status, kWaitLimit, kWaitMmaDone, 0, false);
    }
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;
    const int ew = warp - C::kFirstEpiWarp;
    const int eh = ew >> 2;
    const int et = threadIdx.x - 32 * C::kFirstEpiWarp;
    const uint32_t bar_half = 2 + eh;
    float *ebuf_f = reinterpret_cast<float *>(smem + C::kOffEpi + 4096 * eh);
    uint16_t *ebuf_h = reinterpret_cast<uint16_t *>(smem + C::kOffEpi + 4096 * eh);
    int rb = 0;
    int j = 0;                                   // this cluster's item count
    for (int w = cluster; w < total_work; w += nclusters, ++j) {
      const int acc = j & 1;
      const uint32_t acc_phase = (uint32_t)(j >> 1) & 1u;
      TileInfo ti = decode_work<C::kBN>(w, MT2, args.E, tile_off, cnt_sm, off_sm);
      ti.mt = 2 * ti.mt + (int)rank;                              // this CTA's weight tile
      int32_t *row_pair = row_pair_buf + rb * C::kBN;
      float *row_w = row_w_buf + rb * C::kBN;
      if (et < ti.valid) {
        if (PHASE == 1) row_w[et] = __ldg(args.w_pool + ti.s0 + et);
        else row_pair[et] = __ldg(args.perm + ti.s0 + et);
      }
      const bool got = __all_sync(0xffffffffu, MXQ_TIMED_WAIT(3, mbar_wait(&tmem_full[acc], acc_phase, status,
                                                                          kWaitLimit, kWaitEpiTmemFull, w)));
#ifdef MOE_MXQ_WAIT_STATS
      const long long t_epi = clock64();
#endif
      if (lane == 0) vote[ew] = got ? 1 : 0;
      named_bar_sync(1, 32 * C::kEpiWarps);
      bool all_got = true;
      for (int i = 0; i < C::kEpiWarps; ++i) all_got = all_got && vote[i] != 0;
      if (!all_got) break;
      tc_fence_after();
      const uint32_t t_row = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(acc * C::kBN);
      for (int c0 = kChunk * eh; c0 < ti.valid; c0 += kChunk * 2) {
        uint32_t v[16];
        tmem_ld_32x32b_x16(t_row + (uint32_t)c0, v);
        tmem_ld_wait();
        if (PHASE == 1)
          epilogue_gemm1_chunk(v, c0, q, lane, ti, row_w, ebuf_f, bar_half, args.I, C::kTokChunk, args.hq,
                               args.sfb2, args.hs_out);
        else
          epilogue_gemm2_chunk(v, c0, q, lane, ti, row_pair, ebuf_h, bar_half, args.k, args.T, args.H,
                               args.y_pairs);
      }
      tc_fence_before();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&tmem_empty[acc]), 0));
#ifdef MOE_MXQ_WAIT_STATS
      if (lane == 0 && ew == 0) wait_acc[5] += clock64() - t_epi;
#endif
      rb ^= 1;
    }
  }
#ifdef MOE_MXQ_WAIT_STATS
  if (lane == 0) {
    unsigned long long *acc64 = reinterpret_cast<unsigned long long *>(reinterpret_cast<char *>(status) + 64);
    for (int i = 0; i < 4; ++i)
      if (wait_acc[i]) atomicAdd(acc64 + i, (unsigned long long)wait_acc[i]);
    if (wait_acc[4]) atomicAdd(acc64 + 8, (unsigned long long)wait_acc[4]);
    if (wait_acc[5]) atomicAdd(acc64 + 9, (unsigned long long)wait_acc[5]);
    if (warp <= 2) atomicAdd(acc64 + 4 + warp, (unsigned long long)(clock64() - k_t0));
    if (warp == 0) {
      for (int w = cluster; w < total_work; w += nclusters) ++n_items;
      atomicAdd(acc64 + 7, (unsigned long long)n_items);
    }
  }
#endif
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc_2sm(tmem_base, 512);
  }
}

template <typename Kernel>
bool set_pair_attrs(Kernel kernel, size_t smem) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) == cudaSuccess;
}

// Launch with programmatic stream serialization and 2-CTA clusters.
template <typename... KArgs, typename... Args>
int launch_pair(void (*kernel)(KArgs...), int grid, size_t smem, cudaStream_t st, Args &&...args) {
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(Pair::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace

bool pair_eligible(int64_t H, int64_t I, int E) {
  if ((2 * I / 128) % 2 != 0 || (H / 128) % 2 != 0) return false;     // weight tiles in pairs
  if (num_sms() < 2) return false;
  static int smem_optin = -1;
  if (smem_optin < 0) {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      v = 0;
    smem_optin = v;
  }
  return (int64_t)pair_smem_bytes(E) <= smem_optin;
}

int resolve_tile_n(int tile_n, int64_t P, int64_t E, int64_t H, int64_t I) {
  int bn = tile_n ? tile_n : choose_tile_n(P, E);
  if (bn == 224 || bn == Pair::kBN) bn = pair_eligible(H, I, (int)E) ? Pair::kBN : 224;
  return bn;
}

// GEMM1 (phase bit MOE_PHASE_GEMM1) and / or GEMM2 (MOE_PHASE_GEMM2) of a
// 208-token-tile problem on CTA pairs; GEMM1 reads the pool rows and token-
// scale chunks (sfb1) that the prep / cast kernels wrote and writes h (hq)
// and GEMM2's token-scale chunks (sfb2), which GEMM2 reads.
int run_expert_pairs(const moe_expert_args *a, int phases, int *status, uint8_t *hq, uint8_t *sfb1, uint8_t *sfb2,
                     const float *w_pool, const uint8_t *xq_pool, cudaStream_t st) {
  const int64_t P = a->T * a->k;
  const int E = a->E;
  const size_t sm = pair_smem_bytes(E);
  const int grid = num_sms() & ~1;
  const int64_t max_tiles = max_token_tiles(P, E, Pair::kBN);
  PairArgs g{};
  g.E = E; g.k = a->k; g.T = (int)a->T; g.H = (int)a->H; g.I = (int)a->I;
  g.counts = a->counts; g.offsets = a->offsets; g.perm = a->perm; g.w_pool = w_pool;
  g.hq = hq; g.sfb2 = sfb2; g.hs_out = a->hs; g.y_pairs = a->y_pairs; g.status = status;
  if (const char *env = getenv("MOE_MXQ_DEBUG_INJECT_WAIT")) g.inject_wait = atoi(env);
  if (phases & MOE_PHASE_GEMM1) {
    const int KB = (int)(a->H / 128), MT = (int)(2 * a->I / 128);
    const uint64_t wrows = (uint64_t)E * MT * KB * 128;
    CUtensorMap tw, tb, twsf, tbsf;
    bool ok = encode_tmap_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, (void *)a->w1q, 128, wrows, 64, 128, kBM,
                             CU_TENSOR_MAP_SWIZZLE_128B);
    ok = ok && encode_tmap_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, (void *)xq_pool, (uint64_t)a->H, (uint64_t)P,
                              (uint64_t)a->H, 128, Pair::kHalf, CU_TENSOR_MAP_SWIZZLE_128B);
    ok = ok && encode_tmap_2d(&twsf, CU_TENSOR_MAP_DATA_TYPE_UINT8, (void *)a->w1s, 256, (uint64_t)E * MT * KB * 2,
                              256, 256, 2, CU_TENSOR_MAP_SWIZZLE_NONE);
    ok = ok && encode_tmap_2d(&tbsf, CU_TENSOR_MAP_DATA_TYPE_UINT8, (void *)sfb1, 256, (uint64_t)max_tiles * KB * 4,
                              256, 256, 4, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (!ok) return MOE_ERR_CUDA;
    g.KB = KB; g.MT = MT; g.w_codes = a->w1q;
    if (!set_pair_attrs(expert_gemm_pair_kernel<1>, sm)) return MOE_ERR_CUDA;
    if (launch_pair(expert_gemm_pair_kernel<1>, grid, sm, st, tw, tb, twsf, tbsf, g) != MOE_OK) return MOE_ERR_CUDA;
  }
  if (phases & MOE_PHASE_GEMM2) {
    const int KB = (int)(a->I / 128), MT = (int)(a->H / 128);
    const uint64_t wrows = (uint64_t)E * MT * KB * 128;
    CUtensorMap tw, th, twsf, thsf;
    bool ok = encode_tmap_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, (void *)a->w2q, 128, wrows, 64, 128, kBM,
                             CU_TENSOR_MAP_SWIZZLE_128B);
    ok = ok && encode_tmap_2d(&th, CU_TENSOR_MAP_DATA_TYPE_UINT8, (void *)hq, (uint64_t)a->I, (uint64_t)P,
                              (uint64_t)a->I, 128, Pair::kHalf, CU_TENSOR_MAP_SWIZZLE_128B);
    ok = ok && encode_tmap_2d(&twsf, CU_TENSOR_MAP_DATA_TYPE_UINT8, (void *)a->w2s, 256, (uint64_t)E * MT * KB * 2,
                              256, 256, 2, CU_TENSOR_MAP_SWIZZLE_NONE);
    ok = ok && encode_tmap_2d(&thsf, CU_TENSOR_MAP_DATA_TYPE_UINT8, (void *)sfb2, 256, (uint64_t)max_tiles * KB * 4,
                              256, 256, 4, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (!ok) return MOE_ERR_CUDA;
    g.KB = KB; g.MT = MT; g.w_codes = a->w2q; g.hs_out = nullptr;
    if (!set_pair_attrs(expert_gemm_pair_kernel<2>, sm)) return MOE_ERR_CUDA;
    if (launch_pair(expert_gemm_pair_kernel<2>, grid, sm, st, tw, th, twsf, thsf, g) != MOE_OK) return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

}  // namespace mxq
