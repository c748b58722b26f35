// gemm2sm.cu -- the expert GEMMs of large problems on CTA pairs: one
// tcgen05.mma.cta_group::2 (M = 256 weight rows, N up to 208 tokens, K = 32,
// kind::mxf8f6f4 block-scaled) drives the tensor cores of two SMs.
//
// The same GEMM1 (FP8 tokens x FP4 W1|W3, SwiGLU (.) top-k weight, FP8 + UE8M0
// requantisation) and GEMM2 (FP8 h x FP4 W2 -> BF16 per pair) as gemm.cu, on
// 208-token tiles.  Prior art: the MMA warp listing of "Warp Specialization:
// DeepEP vs Mega MoE" issues the 2-SM block-scaled MMA from the leader CTA of
// a pair, and the MegaMoE study notes ("Scheduler") run each tile on a 2-SM
// cluster.  What a pair buys on GB300:
//   * each CTA stages its own 128 weight rows but only half of the token rows
//     (the MMA reads B's halves from both CTAs), so a stage is 30.5 KB instead
//     of 45.5 KB and six stages fit per SM (three per issue stream) -- the
//     one-CTA kernel keeps two per CTA and leaves the tensor pipe waiting on
//     loads;
//   * one thread issues for two SMs, and two issue streams per pair (each
//     with its own stages and accumulator) keep the tensor pipes fed while
//     one stream waits; token rows cross L2 -> SM once per pair, not per SM.
// Roles per CTA (768 threads): warps 0-1 load the weight codes of the two
// streams' stages (and arm them), warps 2-3 their token rows, warps 4-5 both
// scale parts (both CTAs; a thread's TMA copies issue one after another, so
// a stage's copies are spread over three warps), warps 6-7 the MMA issuers
// (rank 0 only), warps 8-23 the epilogue (both CTAs; four column groups of
// four warps, one TMEM lane quadrant per warp); warp 2 also initialises the
// barriers and allocates TMEM.
// Synchronisation of the pair:
//   * every load of either CTA counts on the leader's `full` barrier (TMA
//     .cta_group::2 form); the leader's weight producer arms it for both
//     CTAs' bytes;
//   * the leader's commits arrive on `empty` and `tmem_full` of both CTAs
//     (multicast); each CTA's epilogue arrives on the leader's `tmem_empty`;
//   * all waits are bounded (MOE_ERR_TIMEOUT in the status words); the pair
//     meets at a cluster barrier before TMEM is freed, so no CTA exits while
//     the other still reads its shared memory or signals its barriers.
// Work order of the separate launches: token tiles in zigzag order over the
// expert-ordered tile list, the weight-row pairs of a tile fastest.
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
  static constexpr int kEpiWarps = 16;                    // four groups of four (one TMEM lane quadrant each)
  static constexpr int kEpiGroups = kEpiWarps / 4;
  // warps 0-1 weight-code producers, 2-3 token-row producers, 4-5 scale
  // producers (one of each per stream: a thread's TMA copies issue one after
  // another, ~150 cycles each, so a stage's copies are spread over three
  // warps), 6-7 MMA issuers
  static constexpr int kFirstEpiWarp = 4 * kStreams;
  static constexpr int kThreads = 32 * (kFirstEpiWarp + kEpiWarps);
  static constexpr int kATile = kBM * kBK;                // unpacked FP4 weight tile (8-bit containers)
  static constexpr int kBTile = kHalf * kBK;
  static constexpr int kTokChunk = 1024;                  // token scales of one (tile, K block): 2 x 128 rows
  static constexpr int kSfSlot = 12;                      // TMEM columns per stage: 4 weight + 8 token scales
  static constexpr int kAccs = 2;                         // accumulators: one per stream, or two for one stream
  static constexpr int kTmemAcc = kAccs * kBN;
  static constexpr int kTmemCols = kTmemAcc + kSfSlot * kStages;
  // bytes landing on the leader's full barrier per stage (both CTAs; the
  // FP4-unpacking weight load counts its packed bytes)
  static constexpr uint32_t kStageTx = 2u * (kWTileBytes + kBTile + 512 + kTokChunk);
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + kStages * kATile;
  static constexpr int kOffSfa = kOffB + kStages * kBTile;
  static constexpr int kOffSfb = kOffSfa + kStages * 512;
  static constexpr int kOffEpi = kOffSfb + kStages * kTokChunk;
  static constexpr int kOffRow = kOffEpi + 4096 * kEpiGroups;   // y_pairs row [2][BN], weight [2][BN]
  static constexpr int kOffBar = kOffRow + 16 * kBN;
  // full[kStages], empty[kStages], tmem_full[kAccs], tmem_empty[kAccs], mma_done[kStreams], never
  static constexpr int kNumBars = 2 * kStages + 2 * kAccs + kStreams + 1;
  static constexpr int kOffTmemPtr = (kOffBar + 8 * kNumBars + 63) & ~63;
  static constexpr int kOffScan = kOffTmemPtr + 64;      // block scan: warp sums [0, 32), total [32]
  static constexpr int kOffExp = kOffScan + 256;
  static_assert(kTmemCols <= 512, "TMEM budget");
  static_assert(kBTile % 1024 == 0 && kATile % 1024 == 0, "stage buffers stay 1024-byte aligned");
  static_assert(kHalf % 8 == 0, "token half-tiles are whole 8-row swizzle atoms");
  static_assert(kThreads / 32 <= 32, "block scan: one warp sum per warp in 32 slots");
};

size_t pair_smem_bytes(int E) { return 1024 + Pair::kOffExp + (size_t)3 * (E + 1) * 4; }

// Both GEMMs' tensor maps (PHASE 1 and 2 use the set of their GEMM).
struct PairMaps {
  CUtensorMap w[2];      // weight codes (FP4, unpacked by TMA), one per GEMM
  CUtensorMap b[2];      // token rows: pool rows (GEMM1), h rows (GEMM2)
  CUtensorMap wsf[2];    // weight scale chunks, viewed as [rows][256] bytes
  CUtensorMap bsf[2];    // token scale chunks, viewed as [rows][256] bytes
};

struct PairArgs {
  int E, k, T, H, I;
  int KB[2], MT[2];                 // per GEMM: K blocks, 128-row weight tiles per expert (even)
  int inject_wait;                  // debug: the MMA issuers first wait on a barrier nothing completes
  const uint8_t *w_codes[2];        // L2 prefetch ahead of the weight loads
  const int32_t *counts, *offsets, *perm;
  const float *w_pool;              // GEMM1 epilogue: top-k weight of each pool row
  uint8_t *hq, *sfb2, *hs_out;      // GEMM1 outputs
  uint16_t *y_pairs;                // GEMM2 output
  int *status;
  // PHASE 3: arrival counters ([0] GEMM2 CTA-items done, [1 + g] GEMM1
  // CTA-items of token tile g done; zeroed before the launch) and the combine
  int *sync;
  const int32_t *topk_idx;
  uint4 *y;
};

// Expert waves of the single launch: kWaveTiles token tiles (expert-major
// order) per wave, the last wave possibly shorter.  Each wave's GEMM1 items
// (tile-major, weight-row pairs fastest) come one wave ahead of its GEMM2
// items:  [L1 w0] [L1 w1] [L2 w0] [L1 w2] [L2 w1] ... [L2 last].  A GEMM2 item
// depends only on the GEMM1 items of its own tile, which sit at least a whole
// wave of GEMM1 items (kWaveTiles * MT1/2 = 384 here, ~2.5x the items in
// flight on 152 SMs) earlier in the list, so it seldom waits, and every
// dependency points to a smaller index (the lowest unfinished item never
// waits).  h of about two waves is live in L2 at a time.
constexpr int kWaveTiles = 24;

struct PairItem {
  int gemm;                         // 0: GEMM1, 1: GEMM2
  TileInfo ti;                      // ti.mt = weight-row pair
};

// Token tile g -> expert, first pool row and valid rows (tile_off: first
// tile of each expert).
__device__ __forceinline__ void tile_rows(int g, int E, int bn, const int *tile_off, const int *cnt_sm,
                                          const int *off_sm, TileInfo &ti) {
  int lo = 0, hi = E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tile_off[mid] <= g) lo = mid; else hi = mid;
  }
  ti.e = lo;
  ti.g = g;
  const int nt = g - tile_off[lo];
  ti.s0 = off_sm[lo] + nt * bn;
  const int rem = cnt_sm[lo] - nt * bn;
  ti.valid = rem < bn ? rem : bn;
}

template <int PHASE>
__device__ __forceinline__ PairItem decode_pair_item(int w, const PairArgs &args, int NT, const int *tile_off,
                                                     const int *cnt_sm, const int *off_sm) {
  PairItem it;
  int g;
  if (PHASE != 3) {
    // separate launches: tiles in zigzag order (0, NT-1, 1, NT-2, ...), so that
    // the many-token tiles of popular experts (compute-heavy) and the
    // few-token tiles of rare experts (weight-streaming) are in flight together
    // (skewed prefill: -1.2 % per GEMM, measured; uniform routing: no change)
    const int MT2 = args.MT[PHASE - 1] >> 1;
    it.gemm = PHASE - 1;
    const int gi = w / MT2;
    it.ti.mt = w - gi * MT2;
    g = (gi & 1) ? NT - 1 - (gi >> 1) : (gi >> 1);
  } else {
    const int m1 = args.MT[0] >> 1, m2 = args.MT[1] >> 1;
    const int nw = (NT + kWaveTiles - 1) / kWaveTiles;          // waves
    const int nlast = NT - (nw - 1) * kWaveTiles;               // tiles of the last wave
    const int n0 = nw > 1 ? kWaveTiles : nlast;
    int r = w;
    // block 0: GEMM1 of wave 0
    if (r < n0 * m1) {
      it.gemm = 0; g = r / m1; it.ti.mt = r % m1;
    } else {
      r -= n0 * m1;
      // blocks 1 .. nw-2 (full size): GEMM1 of wave b, then GEMM2 of wave b-1
      const int per_block = kWaveTiles * (m1 + m2);
      const int full_blocks = nw > 2 ? nw - 2 : 0;
      if (r < full_blocks * per_block) {
        const int b = 1 + r / per_block;
        r -= (b - 1) * per_block;
        if (r < kWaveTiles * m1) {
          it.gemm = 0; g = b * kWaveTiles + r / m1; it.ti.mt = r % m1;
        } else {
          r -= kWaveTiles * m1;
          it.gemm = 1; g = (b - 1) * kWaveTiles + r / m2; it.ti.mt = r % m2;
        }
      } else {
        r -= full_blocks * per_block;
        const int b = nw - 1;                                     // the last wave
        if (nw >= 2 && r < nlast * m1) {                          // block nw-1: GEMM1 of the last wave ...
          it.gemm = 0; g = b * kWaveTiles + r / m1; it.ti.mt = r % m1;
        } else {
          if (nw >= 2) r -= nlast * m1;
          if (nw >= 2 && r < kWaveTiles * m2) {                   // ... then GEMM2 of the wave before
            it.gemm = 1; g = (b - 1) * kWaveTiles + r / m2; it.ti.mt = r % m2;
          } else {
            if (nw >= 2) r -= kWaveTiles * m2;
            it.gemm = 1; g = b * kWaveTiles + r / m2; it.ti.mt = r % m2;   // block nw: GEMM2 of the last wave
          }
        }
      }
    }
  }
  tile_rows(g, args.E, Pair::kBN, tile_off, cnt_sm, off_sm, it.ti);
  return it;
}

template <int PHASE>
__global__ void __launch_bounds__(Pair::kThreads, 1)
    expert_gemm_pair_kernel(const __grid_constant__ PairMaps maps, const PairArgs args) {
  // PHASE 1: GEMM1 + SwiGLU epilogue; 2: GEMM2; 3: expert waves of GEMM1
  // then GEMM2 items in one launch, GEMM2 items waiting on their token
  // tile's arrival counter, then the combine.
  // A cluster's j-th work item belongs to stream j % 2: producer warps s, 2+s
  // and 4+s load it into stages [3s, 3s+3), MMA warp 6+s (leader) accumulates it into
  // accumulator s; the epilogue warps drain the accumulators in item order.
  using C = Pair;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                          ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
  uint64_t *full = bars;                         // leader: both CTAs' loads of a stage
  uint64_t *empty = bars + C::kStages;           // each CTA: stage consumed (leader's commit)
  uint64_t *tmem_full = bars + 2 * C::kStages;   // each CTA: accumulator s ready (leader's commit)
  uint64_t *tmem_empty = tmem_full + C::kAccs;    // leader: both CTAs' epilogues drained accumulator a
  uint64_t *mma_done = tmem_empty + C::kAccs;     // per stream
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

  if (PHASE != 1) pdl_launch_dependents();
  if (warp == 0) {
    if (lane == 0) {
      for (int gm = 0; gm < 2; ++gm) {
        if (PHASE != 3 && gm != PHASE - 1) continue;
        tma_prefetch_desc(&maps.w[gm]);
        tma_prefetch_desc(&maps.b[gm]);
        tma_prefetch_desc(&maps.wsf[gm]);
        tma_prefetch_desc(&maps.bsf[gm]);
      }
    }
  } else if (warp == 2) {
    if (lane == 0) {
      for (int s = 0; s < C::kStages; ++s) {
        mbar_init(&full[s], 1);
        mbar_init(&empty[s], 1);
      }
      for (int a = 0; a < C::kAccs; ++a) {
        mbar_init(&tmem_full[a], 1);
        mbar_init(&tmem_empty[a], 2 * C::kEpiWarps);
      }
      for (int a = 0; a < C::kStreams; ++a) {
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
  block_tile_map<C::kThreads>(cnt_sm, args.E, C::kBN, tile_off, scan_ws, scan_ws + 32);
  __syncthreads();
  const uint32_t tmem_base = *tmem_ptr;
  const int NT = tile_off[args.E];                 // token tiles
  const int total_work = PHASE == 3 ? NT * ((args.MT[0] + args.MT[1]) >> 1) : NT * (args.MT[PHASE - 1] >> 1);
  const int n2_cta_items = 2 * NT * (args.MT[1] >> 1);   // PHASE 3: GEMM2 items x 2 CTAs

  if (warp < 3 * C::kStreams && (PHASE != 3 || warp < C::kStreams)) {
    // ------------------------------------------------------------ TMA producers (both CTAs)
    // Warp st loads the weight codes (and arms the stage), warp kStreams + st
    // the token rows and warp 2 kStreams + st both scale parts of stream st's
    // stages; all pass the same empty barriers, so a stage one of them issued
    // is issued by the others too (a wait gives up only on a barrier that has
    // not completed).  The single launch (PHASE 3) loads whole stages from the
    // weight warp, whose GEMM2 items issue their token part only after the
    // tile's counter wait.
    const int st = warp % C::kStreams;
    const int role = warp / C::kStreams;         // 0: weight codes (arms), 1: token rows, 2: both scale parts
    const bool wpart = PHASE == 3 || role == 0;
    const bool tpart = PHASE == 3 || role == 1;
    const bool spart = PHASE == 3 || role == 2;
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued_mask = 0, issued_phase = 0;
    bool ok = true;
    for (int w = cluster + st * nclusters; w < total_work && ok; w += C::kStreams * nclusters) {
      const PairItem it = decode_pair_item<PHASE>(w, args, NT, tile_off, cnt_sm, off_sm);
      const TileInfo &ti = it.ti;
      const int gm = it.gemm;
      const int KB = args.KB[gm];
      const int n_mma = min(C::kBN, (ti.valid + 31) & ~31);
      const int mt = 2 * ti.mt + (int)rank;                       // this CTA's 128-row weight tile
      const int wtile = (ti.e * args.MT[gm] + mt) * KB;
      const CUtensorMap *tw = &maps.w[gm], *tb = &maps.b[gm], *twsf = &maps.wsf[gm], *tbsf = &maps.bsf[gm];
      // one stage = the weight part (codes + scales, static data) and the
      // token part (pool rows or h + token scales); the leader's barrier
      // counts both CTAs' bytes of both parts
      auto issue_weights = [&](int gs, int kb) {
        const uint32_t bar = mapa_shared(smem_u32(&full[gs]), 0);
        if (rank == 0) mbar_arrive_expect_tx(&full[gs], C::kStageTx);
        tma_load_2d_2sm(smem + C::kOffA + gs * C::kATile, tw, bar, 0, (wtile + kb) * kBM);
        tma_load_2d_2sm(smem + C::kOffSfa + gs * 512, twsf, bar, 0, (wtile + kb) * 2);
        if (kb + kPrefetchAhead < KB)
          prefetch_l2_bulk(args.w_codes[gm] + ((size_t)wtile + kb + kPrefetchAhead) * kWTileBytes, kWTileBytes);
      };
      auto issue_tokens = [&](int gs, int kb) {
        const uint32_t bar = mapa_shared(smem_u32(&full[gs]), 0);
        tma_load_2d_2sm(smem + C::kOffB + gs * C::kBTile, tb, bar, kb * kBK, ti.s0 + (int)rank * (n_mma >> 1));
        tma_load_2d_2sm(smem + C::kOffSfb + gs * C::kTokChunk, tbsf, bar, 0, (ti.g * KB + kb) * 4);
      };
      int kb = 0;
      if (PHASE == 3 && gm == 1) {
        // GEMM2 item of the single launch: the weight part of the first
        // stages, then the wait for the tile's h (every GEMM1 CTA-item of the
        // tile published), then their token parts -- issued even after a
        // failed wait, so that every armed barrier completes
        const int npre = min(KB, C::kStagesPerStream);
        int armed = 0;
        const int st0 = stage;
        const uint32_t ph0 = phase;
        for (; armed < npre; ++armed) {
          const int gs = st * C::kStagesPerStream + stage;
          if (!__all_sync(0xffffffffu, MXQ_TIMED_WAIT(0, mbar_wait(&empty[gs], phase ^ 1, status, kWaitLimit,
                                                                   kWaitProducerEmpty, armed))))
            break;
          if (lane == 0) issue_weights(gs, armed);
          __syncwarp();
          if (++stage == C::kStagesPerStream) { stage = 0; phase ^= 1; }
        }
        bool dep_ok = true;
        if (lane == 0) {
          dep_ok = wait_counter(args.sync + 1 + ti.g, args.MT[0], status, kWaitLimit, w);
          fence_proxy_async_global();
        }
        dep_ok = __shfl_sync(0xffffffffu, dep_ok ? 1 : 0, 0) != 0;
        for (int a = 0; a < armed; ++a) {
          const int sa = (st0 + a) % C::kStagesPerStream;
          const uint32_t pa = ph0 ^ (uint32_t)((st0 + a) / C::kStagesPerStream);
          const int gs = st * C::kStagesPerStream + sa;
          if (lane == 0) issue_tokens(gs, a);
          issued_mask |= 1u << gs;
          issued_phase = (issued_phase & ~(1u << gs)) | (pa << gs);
        }
        __syncwarp();
        if (armed < npre || !dep_ok) {
          ok = false;
          break;
        }
        kb = npre;
      }
      for (; kb < KB; ++kb) {
        const int gs = st * C::kStagesPerStream + stage;
        if (!__all_sync(0xffffffffu, MXQ_TIMED_WAIT(0, mbar_wait(&empty[gs], phase ^ 1, status, kWaitLimit,
                                                                 kWaitProducerEmpty, kb)))) {
          ok = false;
          break;
        }
        if (lane == 0) {
          const uint32_t bar = mapa_shared(smem_u32(&full[gs]), 0);
          if (wpart) {
            if (rank == 0) mbar_arrive_expect_tx(&full[gs], C::kStageTx);
            tma_load_2d_2sm(smem + C::kOffA + gs * C::kATile, tw, bar, 0, (wtile + kb) * kBM);
            if (kb + kPrefetchAhead < KB)
              prefetch_l2_bulk(args.w_codes[gm] + ((size_t)wtile + kb + kPrefetchAhead) * kWTileBytes, kWTileBytes);
          }
          if (tpart)
            tma_load_2d_2sm(smem + C::kOffB + gs * C::kBTile, tb, bar, kb * kBK, ti.s0 + (int)rank * (n_mma >> 1));
          if (spart) {
            tma_load_2d_2sm(smem + C::kOffSfa + gs * 512, twsf, bar, 0, (wtile + kb) * 2);
            tma_load_2d_2sm(smem + C::kOffSfb + gs * C::kTokChunk, tbsf, bar, 0, (ti.g * KB + kb) * 4);
          }
        }
        __syncwarp();
        issued_mask |= 1u << gs;
        issued_phase = (issued_phase & ~(1u << gs)) | (phase << gs);
        if (++stage == C::kStagesPerStream) { stage = 0; phase ^= 1; }
      }
    }
    // the leader never leaves with copies in flight (its full barriers count
    // both CTAs' bytes; the other CTA's copies are covered by the final
    // cluster barrier, which the leader reaches only after this drain)
    if (rank == 0 && wpart)
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
  } else if (warp < 3 * C::kStreams) {
    // token / scale producer warps of the single launch: idle
  } else if (warp < 4 * C::kStreams) {
    // ------------------------------------------------------------ MMA issuers (leader only)
    const int st = warp - 3 * C::kStreams;
    if (rank == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int jj = 0;                                  // this stream's item count
      for (int w = cluster + st * nclusters; w < total_work && ok; w += C::kStreams * nclusters, ++jj) {
        const PairItem it = decode_pair_item<PHASE>(w, args, NT, tile_off, cnt_sm, off_sm);
        const int KB = args.KB[it.gemm];
        const uint32_t n_mma = (uint32_t)min(C::kBN, (it.ti.valid + 31) & ~31);
        // the accumulator: the stream's own (two streams), or alternating (one)
        const int acc = C::kStreams == 1 ? (jj & 1) : st;
        const uint32_t acc_use = C::kStreams == 1 ? (uint32_t)(jj >> 1) : (uint32_t)jj;   // earlier uses of it
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * C::kBN);
        if (!__all_sync(0xffffffffu, MXQ_TIMED_WAIT(2, mbar_wait(&tmem_empty[acc], (acc_use & 1u) ^ 1u, status,
                                                                 kWaitLimit, kWaitMmaTmemEmpty, w))))
          break;
        if (args.inject_wait == 1 && w == cluster + st * nclusters &&
            !__all_sync(0xffffffffu, mbar_wait(never, 0, status, kInjectedWaitLimit, kWaitInjected, w)))
          break;
        tc_fence_after();
        for (int kb = 0; kb < KB; ++kb) {
          const int gs = st * C::kStagesPerStream + stage;
          if (!__all_sync(0xffffffffu,
                          MXQ_TIMED_WAIT(1, mbar_wait(&full[gs], phase, status, kWaitLimit, kWaitMmaFull, kb)))) {
            ok = false;
            break;
          }
          // (no tcgen05 fence: the stage's bytes are published by the
          // mbarrier's transaction count, which the wait observed)
#ifdef MOE_MXQ_WAIT_STATS
          const long long t_issue = clock64();
#endif
          if (elect_one()) {
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
        if (elect_one()) tc_commit_2sm(&tmem_full[acc], 3);
        __syncwarp();
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
    const int eg = ew >> 2;                      // column group: chunks eg, eg + 4, ...
    const int et = threadIdx.x - 32 * C::kFirstEpiWarp;
    const uint32_t bar_group = 2 + eg;
    float *ebuf_f = reinterpret_cast<float *>(smem + C::kOffEpi + 4096 * eg);
    uint16_t *ebuf_h = reinterpret_cast<uint16_t *>(smem + C::kOffEpi + 4096 * eg);
    int rb = 0;
    int j = 0;                                   // this cluster's item count
    for (int w = cluster; w < total_work; w += nclusters, ++j) {
      const int acc = j & 1;
      const uint32_t acc_phase = (uint32_t)(j >> 1) & 1u;
      const PairItem it = decode_pair_item<PHASE>(w, args, NT, tile_off, cnt_sm, off_sm);
      TileInfo ti = it.ti;
      ti.mt = 2 * ti.mt + (int)rank;                              // this CTA's weight tile
      int32_t *row_pair = row_pair_buf + rb * C::kBN;
      float *row_w = row_w_buf + rb * C::kBN;
      if (et < ti.valid) {
        if (it.gemm == 0) row_w[et] = __ldg(args.w_pool + ti.s0 + et);
        else row_pair[et] = pair_row(__ldg(args.perm + ti.s0 + et), args.k, args.T);
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
      // TMEM loads one chunk ahead: the next chunk's load is in flight while
      // this one is processed
      uint32_t v[16];
      int c0 = kChunk * eg;
      if (c0 < ti.valid) tmem_ld_32x32b_x16(t_row + (uint32_t)c0, v);
      while (c0 < ti.valid) {
        tmem_ld_wait();
        uint32_t cur[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) cur[i] = v[i];
        const int cn = c0 + kChunk * C::kEpiGroups;
        if (cn < ti.valid) tmem_ld_32x32b_x16(t_row + (uint32_t)cn, v);
        if (it.gemm == 0)
          epilogue_gemm1_chunk(cur, c0, q, lane, ti, row_w, ebuf_f, bar_group, args.I, C::kTokChunk, args.hq,
                               args.sfb2, args.hs_out);
        else
          epilogue_gemm2_chunk(cur, c0, q, lane, ti, row_pair, ebuf_h, bar_group, args.H, args.y_pairs);
        c0 = cn;
      }
      tc_fence_before();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&tmem_empty[acc]), 0));
#ifdef MOE_MXQ_WAIT_STATS
      if (lane == 0 && ew == 0) wait_acc[5] += clock64() - t_epi;
#endif
      rb ^= 1;
      if (PHASE == 3) {
        // publish the CTA-item: GEMM1 -> its h rows and scale bytes (read by
        // other CTAs' TMA: proxy fence, then release), GEMM2 -> its y_pairs
        // rows (read by the combine)
        if (it.gemm == 0) fence_proxy_async_global();
        named_bar_sync(1, 32 * C::kEpiWarps);
        if (et == 0) {
          __threadfence();
          atomicAdd(it.gemm == 0 ? args.sync + 1 + ti.g : args.sync, 1);
        }
      }
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
  if (PHASE == 3) {
    // the combine, once every GEMM2 CTA-item of the launch has published its rows
    if (threadIdx.x == 0) scan_ws[0] = wait_counter(args.sync, n2_cta_items, status, kWaitLimit, total_work) ? 1 : 0;
    __syncthreads();
    if (scan_ws[0])
      combine_share(args.y_pairs, args.topk_idx, args.T, args.k, args.H, args.y,
                    (int)blockIdx.x * C::kThreads + (int)threadIdx.x, (int)gridDim.x * C::kThreads);
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

// Tensor maps of one GEMM (gm 0: GEMM1 on the pool rows, 1: GEMM2 on h).
bool encode_pair_maps(const moe_expert_args *a, int gm, const uint8_t *tokens, const uint8_t *tok_chunks,
                      PairMaps &m) {
  const int64_t P = a->T * a->k;
  const int E = a->E;
  const int KB = gm == 0 ? (int)(a->H / 128) : (int)(a->I / 128);
  const int MT = gm == 0 ? (int)(2 * a->I / 128) : (int)(a->H / 128);
  const uint64_t K = gm == 0 ? (uint64_t)a->H : (uint64_t)a->I;
  const uint64_t wrows = (uint64_t)E * MT * KB * 128;
  const int64_t max_tiles = max_token_tiles(P, E, Pair::kBN);
  const uint8_t *wq = gm == 0 ? a->w1q : a->w2q;
  const uint8_t *ws = gm == 0 ? a->w1s : a->w2s;
  bool ok = encode_tmap_2d(&m.w[gm], CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, (void *)wq, 128, wrows, 64, 128, kBM,
                           CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && encode_tmap_2d(&m.b[gm], CU_TENSOR_MAP_DATA_TYPE_UINT8, (void *)tokens, K, (uint64_t)P, K, 128,
                            Pair::kHalf, CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && encode_tmap_2d(&m.wsf[gm], CU_TENSOR_MAP_DATA_TYPE_UINT8, (void *)ws, 256, (uint64_t)E * MT * KB * 2,
                            256, 256, 2, CU_TENSOR_MAP_SWIZZLE_NONE);
  ok = ok && encode_tmap_2d(&m.bsf[gm], CU_TENSOR_MAP_DATA_TYPE_UINT8, (void *)tok_chunks, 256,
                            (uint64_t)max_tiles * KB * 4, 256, 256, 4, CU_TENSOR_MAP_SWIZZLE_NONE);
  return ok;
}

PairArgs pair_args(const moe_expert_args *a, int *status, uint8_t *hq, uint8_t *sfb2, const float *w_pool) {
  PairArgs g{};
  g.E = a->E; g.k = a->k; g.T = (int)a->T; g.H = (int)a->H; g.I = (int)a->I;
  g.KB[0] = (int)(a->H / 128); g.MT[0] = (int)(2 * a->I / 128);
  g.KB[1] = (int)(a->I / 128); g.MT[1] = (int)(a->H / 128);
  g.w_codes[0] = a->w1q; g.w_codes[1] = a->w2q;
  g.counts = a->counts; g.offsets = a->offsets; g.perm = a->perm; g.w_pool = w_pool;
  g.hq = hq; g.sfb2 = sfb2; g.hs_out = a->hs; g.y_pairs = a->y_pairs; g.status = status;
  if (const char *env = getenv("MOE_MXQ_DEBUG_INJECT_WAIT")) g.inject_wait = atoi(env);
  return g;
}

// GEMM1 (phase bit MOE_PHASE_GEMM1) and / or GEMM2 (MOE_PHASE_GEMM2) of a
// 208-token-tile problem on CTA pairs, as separate launches; GEMM1 reads the
// pool rows and token-scale chunks (sfb1) that the prep / cast kernels wrote
// and writes h (hq) and GEMM2's token-scale chunks (sfb2), which GEMM2 reads.
int run_expert_pairs(const moe_expert_args *a, int phases, int *status, uint8_t *hq, uint8_t *sfb1, uint8_t *sfb2,
                     const float *w_pool, const uint8_t *xq_pool, cudaStream_t st) {
  const size_t sm = pair_smem_bytes(a->E);
  const int grid = num_sms() & ~1;
  PairArgs g = pair_args(a, status, hq, sfb2, w_pool);
  if (phases & MOE_PHASE_GEMM1) {
    PairMaps m{};
    if (!encode_pair_maps(a, 0, xq_pool, sfb1, m)) return MOE_ERR_CUDA;
    if (!set_pair_attrs(expert_gemm_pair_kernel<1>, sm)) return MOE_ERR_CUDA;
    if (launch_pair(expert_gemm_pair_kernel<1>, grid, sm, st, m, g) != MOE_OK) return MOE_ERR_CUDA;
  }
  if (phases & MOE_PHASE_GEMM2) {
    PairMaps m{};
    if (!encode_pair_maps(a, 1, hq, sfb2, m)) return MOE_ERR_CUDA;
    g.hs_out = nullptr;
    if (!set_pair_attrs(expert_gemm_pair_kernel<2>, sm)) return MOE_ERR_CUDA;
    if (launch_pair(expert_gemm_pair_kernel<2>, grid, sm, st, m, g) != MOE_OK) return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

// GEMM1 + GEMM2 + combine of a 208-token-tile problem in one launch on CTA
// pairs (expert waves).  `sync`: 1 + max_token_tiles(P, E, 208) ints, zero on
// entry.  Every CTA of the grid must be resident at once (one per SM).
int launch_pair_fused(const moe_expert_args *a, uint16_t *y, int *sync, int *status, uint8_t *hq, uint8_t *sfb1,
                      uint8_t *sfb2, const float *w_pool, const uint8_t *xq_pool, cudaStream_t st) {
  const size_t sm = pair_smem_bytes(a->E);
  const int grid = num_sms() & ~1;
  PairMaps m{};
  if (!encode_pair_maps(a, 0, xq_pool, sfb1, m) || !encode_pair_maps(a, 1, hq, sfb2, m)) return MOE_ERR_CUDA;
  PairArgs g = pair_args(a, status, hq, sfb2, w_pool);
  g.hs_out = nullptr;
  g.sync = sync;
  g.topk_idx = a->topk_idx;
  g.y = reinterpret_cast<uint4 *>(y);
  if (!set_pair_attrs(expert_gemm_pair_kernel<3>, sm)) return MOE_ERR_CUDA;
  return launch_pair(expert_gemm_pair_kernel<3>, grid, sm, st, m, g);
}

// moe_forward's expert part for 208-token tiles: the single launch above on
// the pool rows and token-scale chunks that the prep / cast kernel left in
// the expert workspace `ews`.
int launch_pair_layer(const moe_expert_args *a, uint16_t *y, int *sync, int *status, char *ews, cudaStream_t st) {
  const ExpertWs lay = expert_ws_layout(a->T, a->H, a->I, a->E, a->k);
  uint8_t *hq = a->hq ? a->hq : reinterpret_cast<uint8_t *>(ews + lay.hq);
  return launch_pair_fused(a, y, sync, status, hq, reinterpret_cast<uint8_t *>(ews + lay.sfb1),
                           reinterpret_cast<uint8_t *>(ews + lay.sfb2), reinterpret_cast<const float *>(ews + lay.w_pool),
                           reinterpret_cast<const uint8_t *>(ews + lay.xq_pool), st);
}

}  // namespace mxq
