// gemm.cu -- grouped expert GEMMs on tcgen05 block-scaled MMA (sm_103a).
//
// GEMM1 (W1|W3, FP8 E4M3 tokens x FP4 E2M1 weights, UE8M0 per 32 along K,
// FP32 accumulate in TMEM) with the fused epilogue
//     h = silu(gate) * up * topk_w  ->  E4M3 + UE8M0 per 32 along I,
// then GEMM2 (FP8 h x FP4 W2) with a BF16 epilogue that scatters each pair's
// row to y_pairs[slot][token].
//
// Prior art: MegaMoE (study notes), "Warp roles", "Scheduler", "Wave", "L1
// epilogue", "L2 epilogue" and the gate/up interleave; Warp Specialization:
// DeepEP vs Mega MoE (MMA issue with the weights in the M slot, UTCCP copy of
// the scale factors into TMEM, epilogue listings).  What is kept on sm_103a:
//   * weights are the MMA's M operand (128 rows per tile) and tokens the N
//     operand (16..224 per tile), so decode-sized experts waste little MMA;
//   * persistent CTAs (one to three per SM, see Cfg), warp roles: warp 0 TMA
//     producer, warp 1 TMEM allocator + single-thread MMA issuer, warps 2-5
//     (2-9) epilogue (one TMEM lane quadrant each);
//   * a ring of shared-memory stages (full/empty mbarriers) and one or two
//     TMEM accumulators (tmem_full/tmem_empty) so loads, MMAs and epilogues
//     overlap;
//   * FP4 weights are unpacked into 8-bit containers by TMA
//     (16U4_ALIGN16B, 128B swizzle); token rows come from an expert-major
//     pool of FP8 rows in HBM, which replaces the pages' NVLink pull into a
//     pool buffer;
//   * scale factors travel as 512-byte chunks already in the tcgen05.cp
//     32x128b.warpx4 order and land in TMEM next to the accumulators;
//   * small problems run GEMM1, GEMM2 and the combine in one launch, GEMM2
//     items waiting on per-token-tile arrival counters (the pages' arrival
//     mask), all bounded.
// Not kept: the dispatch warps and NVLink stores (one GPU), the 2-SM
// cluster, and unbounded spins (every wait here gives up after ~1 s and
// reports MOE_ERR_TIMEOUT through the workspace status word).
//
// Work order (all roles walk the same list): expert-major, then weight tile
// mt, then token tile nt, so consecutive CTAs share a weight tile (token
// tiles of one expert) or a token tile (weight tiles of one expert) in L2.
#include <cuda_bf16.h>

#include <algorithm>
#include <cstdlib>

#include "gemm_common.cuh"
#include "host_common.h"
#include "layer_blocks.cuh"
#include "ptx.cuh"

namespace mxq {

namespace {

// Issue cost.  Every asynchronous instruction (TMA copy, tcgen05.cp,
// tcgen05.mma) takes ~80 cycles of its issuing thread, whatever its size,
// while one M=128 x N x K=32 MMA keeps the tensor core busy ~0.53 N cycles.
// So (a) a pipeline stage may cover kKBS = 2 K blocks: one TMA box of 256
// weight rows (two consecutive tiles of the tile-contiguous layout), one bulk
// copy per scale operand and one 2-D box of token rows per K block; and (b)
// small token tiles run several CTAs per SM (three for N = 16, two for
// N <= 64, with one K block per stage where shared memory is tight), giving
// the SM independent MMA issue streams without changing any accumulation
// order.
// (c) 128- and 224-token tiles run two CTAs per SM with one TMEM accumulator
// each (two accumulators would not fit twice): a CTA's epilogue is not
// overlapped with its own MMAs but with the other CTA's, and the second
// issue stream pays for that (224: GEMM1 -9 %, GEMM2 -13 % on the prefill;
// 128: -7 % / -16 %, measured).
template <int BN>
struct Cfg {
  static constexpr bool kWideTwoCta = BN >= 128;
  // tiles above 128 tokens: scales of the token operand in two 128-row
  // groups, and an 8-warp epilogue (two warps per TMEM quadrant)
  static constexpr int kKBS = (BN == 16 || BN == 64 || kWideTwoCta) ? 1 : 2;
  static constexpr int kCtasPerSm = BN == 16 ? 3 : (BN <= 64 || kWideTwoCta ? 2 : 1);
  // accumulators in TMEM (two: the epilogue of one item overlaps the MMAs of the next)
  static constexpr int kAccBufs = kWideTwoCta ? 1 : 2;
  static constexpr int kSfbGroups = (BN + 127) / 128;       // 128-row groups of token scales
  static constexpr int kTokChunk = 512 * kSfbGroups;        // bytes of one (tile, K block) token-scale chunk
  static constexpr int kSfSlot = 4 + 4 * kSfbGroups;        // TMEM columns of one K block's scales
  static constexpr int kEpiWarps = BN > 128 ? 8 : 4;
  static constexpr int kEpiHalves = kEpiWarps / 4;
  static constexpr int kThreads = 64 + 32 * kEpiWarps;
  static constexpr int kATile = kBM * kBK;                  // one unpacked FP4 tile (8-bit containers)
  static constexpr int kBTile = BN * kBK;
  static constexpr int kABytes = kKBS * kATile;
  static constexpr int kBBytes = kKBS * kBTile;
  static constexpr int kSfbBytes = BN < 32 ? BN * 16 : kTokChunk;   // used bytes of a token-scale chunk
  static constexpr int kStageBytes = kABytes + kBBytes + kKBS * (512 + kTokChunk);
  // (128-token tiles: three 33 KB stages in two CTAs' share of the SM)
  static constexpr int kSmemBudget = (kCtasPerSm == 1 ? 200 : kCtasPerSm == 2 ? (BN == 128 ? 100 : 96) : 60) * 1024;
  static constexpr int kStages = (kSmemBudget / kStageBytes) > 8 ? 8 : (kSmemBudget / kStageBytes);
  static constexpr int kTmemCols = kAccBufs * BN + kSfSlot * kKBS * kStages;
  static constexpr uint32_t kTmemAlloc = kTmemCols <= 32 ? 32 : kTmemCols <= 64 ? 64 : kTmemCols <= 128 ? 128
                                         : kTmemCols <= 256 ? 256 : 512;
  // shared memory carve-up (offsets from a 1024-aligned base)
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + kStages * kABytes;
  static constexpr int kOffSfa = kOffB + kStages * kBBytes;
  static constexpr int kOffSfb = kOffSfa + kStages * kKBS * 512;
  static constexpr int kOffEpi = kOffSfb + kStages * kKBS * kTokChunk;   // 4 KB epilogue staging per half
  // per-item row info, double-buffered by item parity: y_pairs row [2][BN], weight [2][BN]
  static constexpr int kOffRow = kOffEpi + 4096 * kEpiHalves;
  static constexpr int kOffBar = kOffRow + 16 * BN;
  static constexpr int kNumBars = 2 * kStages + 6;
  static constexpr int kOffTmemPtr = kOffBar + 8 * kNumBars;
  static constexpr int kOffScan = kOffTmemPtr + 64;         // block-scan scratch: warp sums + total
  static constexpr int kOffExp = kOffScan + 64;             // tile_off, counts, offsets: 3*(E+1) ints
  static_assert(kStages >= 2, "need at least two stages");
  static_assert(kTmemCols <= 512, "TMEM budget");
  static_assert(kTmemAlloc * kCtasPerSm <= 512, "co-resident CTAs share the SM's 512 TMEM columns");
  static_assert(kThreads / 32 <= 15, "block scan: warp sums in [0, 15), total at 15");
};

template <int BN>
size_t smem_bytes(int E) {
  return 1024 + Cfg<BN>::kOffExp + (size_t)3 * (E + 1) * 4;
}

struct GemmArgs {
  int E, k, T, H, I;
  int M, K, KB, MT;                 // weight rows / reduction / K blocks / weight tiles per expert
  int inject_wait;                  // debug: 1 = the MMA warp first waits on a barrier nothing completes
  // GEMM2 launched right after GEMM1 in the same call: the expert table and
  // the first stages' weight loads are issued before griddepcontrol.wait
  // (GEMM1 signals its dependents only after its own wait, so the routing
  // outputs are final by then; weights are never written by a kernel)
  int early_weights;
  const uint8_t *w_codes;           // this launch's weight codes (L2 prefetch ahead of the TMA)
  const int32_t *counts, *offsets, *perm;
  const int32_t *tok_pool;          // token of each pool row (GEMM1 gather)
  const float *w_pool;              // top-k weight of each pool row (GEMM1 epilogue)
  const uint8_t *w_sf;              // [E][MT][KB][512]
  const uint8_t *b_sf;              // [tiles][KB][512]
  uint8_t *hq;                      // L1 out [P][I] (pool order)
  uint8_t *sfb2;                    // L1 out [tiles][I/128][512]
  uint8_t *hs_out;                  // optional L1 out [P][I/32]
  uint16_t *y_pairs;                // L2 out [k][T][H]
  int *status;
  // GEMM1 + GEMM2 + combine in one launch (PHASE 3): GEMM2's operands, the
  // arrival counters and the combine
  int MT2, KB2;
  const uint8_t *w_sf2, *b_sf2, *w_codes2;
  int *sync;                        // [0] GEMM2 items done, [1 + g] GEMM1 items of token tile g done
  const int32_t *topk_idx;          // [T][k] (combine: dropped slots skipped)
  uint4 *y;                         // [T][H] bf16 (combine output)
};



template <int BN, int PHASE>
__global__ void __launch_bounds__(Cfg<BN>::kThreads, Cfg<BN>::kCtasPerSm)
    expert_gemm_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_b,
                       const __grid_constant__ CUtensorMap tmap_w2, const __grid_constant__ CUtensorMap tmap_b2,
                       const GemmArgs args) {
  // PHASE 1: GEMM1 + SwiGLU epilogue; 2: GEMM2; 3: both and the combine in
  // one launch (small problems): GEMM1 items, then GEMM2 items (each waiting
  // on the GEMM1 items of its token tile), then the combine
  using C = Cfg<BN>;
  constexpr bool kFused = PHASE == 3;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                          ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
  uint64_t *full = bars;
  uint64_t *empty = bars + C::kStages;
  uint64_t *tmem_full = bars + 2 * C::kStages;
  uint64_t *tmem_empty = tmem_full + 2;
  uint64_t *mma_done = tmem_full + 4;
  uint64_t *never = tmem_full + 5;          // debug wait target: initialised, never arrived on
  uint32_t *tmem_ptr = reinterpret_cast<uint32_t *>(smem + C::kOffTmemPtr);
  int *vote = reinterpret_cast<int *>(smem + C::kOffTmemPtr + 4);     // one per epilogue warp
  int *tile_off = reinterpret_cast<int *>(smem + C::kOffExp);
  int *cnt_sm = tile_off + (args.E + 1);
  int *off_sm = cnt_sm + (args.E + 1);
  int32_t *row_pair_buf = reinterpret_cast<int32_t *>(smem + C::kOffRow);
  float *row_w_buf = reinterpret_cast<float *>(smem + C::kOffRow + 8 * BN);
  int *scan_ws = reinterpret_cast<int *>(smem + C::kOffScan);            // block-scan scratch

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int *status = args.status;
#ifdef MOE_MXQ_WAIT_STATS
  long long wait_acc[4] = {0, 0, 0, 0};
  const long long k_t0 = clock64();
  int n_items = 0;
#endif

  if (PHASE != 1) pdl_launch_dependents();
  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tmap_w);
      tma_prefetch_desc(&tmap_b);
      if (kFused) {
        tma_prefetch_desc(&tmap_w2);
        tma_prefetch_desc(&tmap_b2);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      for (int s = 0; s < C::kStages; ++s) {
        mbar_init(&full[s], 1);
        mbar_init(&empty[s], 1);
      }
      for (int a = 0; a < 2; ++a) {
        mbar_init(&tmem_full[a], 1);
        mbar_init(&tmem_empty[a], C::kEpiWarps);
      }
      mbar_init(mma_done, 1);
      mbar_init(never, 1);
      fence_mbar_init();
    }
    __syncwarp();
    tmem_alloc(tmem_ptr, C::kTmemAlloc);
    tmem_relinquish();
  }
  // everything above touches no global memory; the previous kernel's outputs
  // (counts, offsets, pool rows, scales) are read only after this point --
  // except, with early_weights, the routing outputs of the kernel before the
  // previous one (L2 reads) and static weights (producer, below)
  const bool early = PHASE == 2 && args.early_weights != 0;
  if (!early) pdl_wait();
  if (PHASE == 1) pdl_launch_dependents();
  load_expert_table(args.counts, args.offsets, args.E, cnt_sm, off_sm, early);
  __syncthreads();
  block_tile_map<C::kThreads>(cnt_sm, args.E, BN, tile_off, scan_ws, scan_ws + 15);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_ptr;
  const int n1 = tile_off[args.E] * args.MT;                     // GEMM1 items (PHASE 3: then GEMM2's)
  const int n2 = kFused ? tile_off[args.E] * args.MT2 : 0;
  const int total_work = n1 + n2;
  // work item w: its tile, weight tiles per expert, K blocks, and whether it
  // is a GEMM1 item
  struct Item {
    TileInfo ti;
    int MT, KB;
    bool l1;
  };
  auto get_item = [&](int w) {
    Item it;
    it.l1 = PHASE == 1 || (kFused && w < n1);
    const bool second = kFused && !it.l1;
    it.MT = second ? args.MT2 : args.MT;
    it.KB = second ? args.KB2 : args.KB;
    it.ti = decode_work<BN>(second ? w - n1 : w, it.MT, args.E, tile_off, cnt_sm, off_sm);
    return it;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued_mask = 0, issued_phase = 0;
    bool ok = true;
    // one stage = the weight part (codes + weight scales, static data) and the
    // token part (pool rows or h, token scales, written by earlier kernels or,
    // in PHASE 3, by other CTAs); the stage's barrier expects both
    auto issue_weights = [&](int st, int kb, int nk, int wtile, const Item &it) {
      const bool second = kFused && !it.l1;
      const uint32_t sfb_bytes = (uint32_t)((nk - 1) * C::kTokChunk + C::kSfbBytes);
      // the weight box always spans kKBS tiles (rows past the tensor read as zeros);
      // the FP4-unpacking load completes the packed byte count
      mbar_arrive_expect_tx(&full[st], (uint32_t)(C::kKBS * kWTileBytes + nk * C::kBTile + nk * 512) + sfb_bytes);
      tma_load_2d(smem + C::kOffA + st * C::kABytes, second ? &tmap_w2 : &tmap_w, &full[st], 0,
                  (wtile + kb) * kBM);
      bulk_load(smem + C::kOffSfa + st * C::kKBS * 512, (second ? args.w_sf2 : args.w_sf) + ((size_t)wtile + kb) * 512,
                nk * 512, &full[st]);
    };
    auto issue_tokens = [&](int st, int kb, int nk, const Item &it) {
      const bool second = kFused && !it.l1;
      const uint32_t sfb_bytes = (uint32_t)((nk - 1) * C::kTokChunk + C::kSfbBytes);
      const uint8_t *sfb_src = (second ? args.b_sf2 : args.b_sf) + ((size_t)it.ti.g * it.KB + kb) * C::kTokChunk;
      bulk_load(smem + C::kOffSfb + st * C::kKBS * C::kTokChunk, sfb_src, sfb_bytes, &full[st]);
      unsigned char *b_dst = smem + C::kOffB + st * C::kBBytes;
      for (int i = 0; i < nk; ++i)
        tma_load_2d(b_dst + i * C::kBTile, second ? &tmap_b2 : &tmap_b, &full[st], (kb + i) * kBK, it.ti.s0);
    };
    auto advance = [&]() {
      issued_mask |= 1u << stage;
      issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
      if (++stage == C::kStages) { stage = 0; phase ^= 1; }
    };
    if (kFused) {
      // every GEMM2 item: the weight part of its first stages, then the wait
      // for the h rows of its token tile (the GEMM1 items of every weight
      // tile of that expert), then the token parts; the token parts are issued
      // even after a failed wait so that every armed barrier completes (the
      // status word says why).  GEMM1 items depend on nothing in the launch.
      for (int w = blockIdx.x; w < total_work && ok; w += gridDim.x) {
        const Item it = get_item(w);
        const int wtile = (it.ti.e * it.MT + it.ti.mt) * it.KB;
        const int nst = (it.KB + C::kKBS - 1) / C::kKBS;
        const int npre = min(nst, C::kStages);
        const int st0 = stage;
        const uint32_t ph0 = phase;
        int armed = 0;
        for (; armed < npre; ++armed) {
          if (!__all_sync(0xffffffffu, mbar_wait(&empty[stage], phase ^ 1, status, kWaitLimit, kWaitProducerEmpty,
                                                 armed * C::kKBS)))
            break;
          if (lane == 0) issue_weights(stage, armed * C::kKBS, min(C::kKBS, it.KB - armed * C::kKBS), wtile, it);
          __syncwarp();
          if (++stage == C::kStages) { stage = 0; phase ^= 1; }
        }
        bool dep_ok = true;
        if (lane == 0 && !it.l1) {
          dep_ok = wait_counter(args.sync + 1 + it.ti.g, args.MT, status, kWaitLimit, w);
          fence_proxy_async_global();
        }
        dep_ok = __shfl_sync(0xffffffffu, dep_ok ? 1 : 0, 0) != 0;
        for (int a = 0; a < armed; ++a) {
          // armed <= kStages: the ring wraps at most once inside one item
          const int st = (st0 + a) % C::kStages;
          const uint32_t ph = ph0 ^ (uint32_t)((st0 + a) / C::kStages);
          if (lane == 0) issue_tokens(st, a * C::kKBS, min(C::kKBS, it.KB - a * C::kKBS), it);
          issued_mask |= 1u << st;
          issued_phase = (issued_phase & ~(1u << st)) | (ph << st);
        }
        __syncwarp();
        if (armed < npre || !dep_ok) {
          ok = false;
          break;
        }
        for (int a = npre; a < nst; ++a) {
          const int kb = a * C::kKBS;
          if (!__all_sync(0xffffffffu, mbar_wait(&empty[stage], phase ^ 1, status, kWaitLimit, kWaitProducerEmpty, kb))) {
            ok = false;
            break;
          }
          if (lane == 0) {
            issue_weights(stage, kb, min(C::kKBS, it.KB - kb), wtile, it);
            issue_tokens(stage, kb, min(C::kKBS, it.KB - kb), it);
            if (kb + kPrefetchAhead < it.KB)
              prefetch_l2_bulk((it.l1 ? args.w_codes : args.w_codes2) + ((size_t)wtile + kb + kPrefetchAhead) * kWTileBytes,
                               kWTileBytes);
          }
          __syncwarp();
          advance();
        }
      }
    } else {
      // early_weights: the first item's first stages get their weight part now,
      // their token part after griddepcontrol.wait (all stages are free here)
      int pre = 0;
      if (early) {
        if (blockIdx.x < total_work) {
          const Item it0 = get_item(blockIdx.x);
          const int wtile0 = (it0.ti.e * it0.MT + it0.ti.mt) * it0.KB;
          for (; pre < C::kStages && pre * C::kKBS < args.KB; ++pre)
            if (lane == 0) issue_weights(pre, pre * C::kKBS, min(C::kKBS, args.KB - pre * C::kKBS), wtile0, it0);
          __syncwarp();
        }
        pdl_wait();
      }
      for (int w = blockIdx.x; w < total_work && ok; w += gridDim.x) {
        const Item it = get_item(w);
        const int wtile = (it.ti.e * it.MT + it.ti.mt) * it.KB;        // first weight tile of this item
        for (int kb = 0; kb < it.KB; kb += C::kKBS) {
          const int nk = min(C::kKBS, it.KB - kb);                     // K blocks in this stage
          const bool pre_armed = w == (int)blockIdx.x && kb < pre * C::kKBS;
          if (!pre_armed &&
              !__all_sync(0xffffffffu,
                          MXQ_TIMED_WAIT(0, mbar_wait(&empty[stage], phase ^ 1, status, kWaitLimit, kWaitProducerEmpty, kb)))) {
            ok = false;
            break;
          }
          if (lane == 0) {
            if (!pre_armed) issue_weights(stage, kb, nk, wtile, it);
            issue_tokens(stage, kb, nk, it);
            // the weight tile kPrefetchAhead K blocks on is requested into L2
            // now, so that its TMA load (issued when a stage frees) waits on
            // L2 rather than HBM (GEMM time -1 to -4 %, measured)
            if (kb + kPrefetchAhead < it.KB)
              prefetch_l2_bulk(args.w_codes + ((size_t)wtile + kb + kPrefetchAhead) * kWTileBytes, kWTileBytes);
          }
          __syncwarp();
          advance();
        }
      }
    }
    // never leave with copies in flight: wait for the last load of each stage
    for (int s = 0; s < C::kStages; ++s)
      if (issued_mask & (1u << s))
        mbar_wait(&full[s], (issued_phase >> s) & 1u, status, kWaitLimit, kWaitProducerDrain, s, false);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (early) pdl_wait();
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int w = blockIdx.x; w < total_work && ok; w += gridDim.x) {
      const Item it = get_item(w);
      // MMA N covers the valid tokens of the tile, rounded up to 16
      const uint32_t n_mma = (uint32_t)min(BN, (it.ti.valid + 15) & ~15);
      if (!__all_sync(0xffffffffu,
                      MXQ_TIMED_WAIT(2, mbar_wait(&tmem_empty[acc], acc_phase ^ 1, status, kWaitLimit, kWaitMmaTmemEmpty, w))))
        break;
      // failure-detection test hook: a wait that can only end by its timeout
      if (args.inject_wait == 1 && w == (int)blockIdx.x &&
          !__all_sync(0xffffffffu, mbar_wait(never, 0, status, kInjectedWaitLimit, kWaitInjected, w)))
        break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
      for (int kb = 0; kb < it.KB; kb += C::kKBS) {
        const int nk = min(C::kKBS, it.KB - kb);
        if (!__all_sync(0xffffffffu, MXQ_TIMED_WAIT(1, mbar_wait(&full[stage], phase, status, kWaitLimit, kWaitMmaFull, kb)))) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (elect_one()) {
          for (int i = 0; i < nk; ++i) {
            const uint32_t sf_col = tmem_base + (uint32_t)(C::kAccBufs * BN + C::kSfSlot * (stage * C::kKBS + i));
            const uint32_t sfa = smem_u32(smem + C::kOffSfa + (stage * C::kKBS + i) * 512);
            const uint32_t sfb = smem_u32(smem + C::kOffSfb + (stage * C::kKBS + i) * C::kTokChunk);
            tc_cp_32x128b_warpx4(sf_col, make_smem_desc(sfa, 0, 128, kSwizzleNone));
            // token scales: one 128-row group per 4 TMEM columns
            for (int gq = 0; gq < C::kSfbGroups && gq * 128 < (int)n_mma; ++gq)
              tc_cp_32x128b_warpx4(sf_col + 4 + 4 * gq, make_smem_desc(sfb + gq * 512, 0, 128, kSwizzleNone));
            const uint32_t a_base = smem_u32(smem + C::kOffA + stage * C::kABytes + i * C::kATile);
            const uint32_t b_base = smem_u32(smem + C::kOffB + stage * C::kBBytes + i * C::kBTile);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t ad = make_smem_desc(a_base + kk * 32, 16, 1024, kSwizzle128B);
              const uint64_t bd = make_smem_desc(b_base + kk * 32, 16, 1024, kSwizzle128B);
              tc_mma_mxf8f6f4(d_tmem, ad, bd, make_idesc_fp4w_fp8a(n_mma, kk), sf_col, sf_col + 4,
                              ((kb + i) | kk) != 0 ? 1u : 0u);
            }
          }
          tc_commit(&empty[stage]);
        }
        __syncwarp();
        if (++stage == C::kStages) { stage = 0; phase ^= 1; }
      }
      if (!ok) break;
      if (elect_one()) tc_commit(&tmem_full[acc]);
      __syncwarp();
      if (++acc == C::kAccBufs) { acc = 0; acc_phase ^= 1; }
    }
    // all MMAs issued by this thread complete before TMEM is released
    if (lane == 0) tc_commit(mma_done);
    __syncwarp();
    mbar_wait(mma_done, 0, status, kWaitLimit, kWaitMmaDone, 0, false);
  } else {
    // ------------------------------------------------------------ epilogue
    // kEpiWarps warps: quadrant q = warp % 4 of the TMEM lanes; with 8 warps the
    // two halves take alternate 16-column chunks, each with its own staging
    // buffer and named barrier.
    if (early) pdl_wait();
    const int q = warp & 3;                  // TMEM lane quadrant of this warp
    const int eh = (warp - 2) >> 2;          // epilogue half
    const int et = threadIdx.x - 64;         // 0 .. 32 * kEpiWarps - 1
    const uint32_t bar_half = 2 + eh;
    float *ebuf_f = reinterpret_cast<float *>(smem + C::kOffEpi + 4096 * eh);
    uint16_t *ebuf_h = reinterpret_cast<uint16_t *>(smem + C::kOffEpi + 4096 * eh);
    int acc = 0;
    uint32_t acc_phase = 0;
    int rb = 0;                              // row-info buffer of this item
    for (int w = blockIdx.x; w < total_work; w += gridDim.x) {
      const Item it = get_item(w);
      const TileInfo &ti = it.ti;
      // a half may start this item while the other still reads the previous
      // item's row info, so items alternate between two buffers (one is
      // reused two items later, after every warp passed this item's vote)
      int32_t *row_pair = row_pair_buf + rb * BN;
      float *row_w = row_w_buf + rb * BN;
      if (et < ti.valid) {
        if (it.l1) row_w[et] = __ldg(args.w_pool + ti.s0 + et);
        else row_pair[et] = pair_row(__ldg(args.perm + ti.s0 + et), args.k, args.T);
      }
      // the epilogue warps agree on the outcome of the bounded wait before any
      // of them enters another named barrier
      const bool got = __all_sync(0xffffffffu,
                                  MXQ_TIMED_WAIT(3, mbar_wait(&tmem_full[acc], acc_phase, status, kWaitLimit, kWaitEpiTmemFull, w)));
      if (lane == 0) vote[warp - 2] = got ? 1 : 0;
      named_bar_sync(1, 32 * C::kEpiWarps);
      bool all_got = true;
      for (int i = 0; i < C::kEpiWarps; ++i) all_got = all_got && vote[i] != 0;
      if (!all_got) break;
      tc_fence_after();
      const uint32_t t_row = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(acc * BN);
      for (int c0 = kChunk * eh; c0 < ti.valid; c0 += kChunk * C::kEpiHalves) {
        uint32_t v[16];
        tmem_ld_32x32b_x16(t_row + (uint32_t)c0, v);
        tmem_ld_wait();
        if (it.l1)
          epilogue_gemm1_chunk(v, c0, q, lane, ti, row_w, ebuf_f, bar_half, args.I, C::kTokChunk, args.hq,
                               args.sfb2, args.hs_out);
        else
          epilogue_gemm2_chunk(v, c0, q, lane, ti, row_pair, ebuf_h, bar_half, args.H, args.y_pairs);
      }
      tc_fence_before();
      if (lane == 0) mbar_arrive(&tmem_empty[acc]);
      if (++acc == C::kAccBufs) { acc = 0; acc_phase ^= 1; }
      rb ^= 1;
      if (kFused) {
        // publish the item: GEMM1 -> its h rows and scale chunk (read by other
        // CTAs' TMA: proxy fence), GEMM2 -> its y_pairs rows (the combine)
        fence_proxy_async_global();
        named_bar_sync(1, 32 * C::kEpiWarps);
        if (et == 0) {
          __threadfence();
          atomicAdd(it.l1 ? args.sync + 1 + ti.g : args.sync, 1);
        }
      }
    }
  }
#ifdef MOE_MXQ_WAIT_STATS
  if (lane == 0) {
    unsigned long long *acc64 = reinterpret_cast<unsigned long long *>(reinterpret_cast<char *>(status) + 64);
    for (int i = 0; i < 4; ++i)
      if (wait_acc[i]) atomicAdd(acc64 + i, (unsigned long long)wait_acc[i]);
    if (warp <= 2) atomicAdd(acc64 + 4 + warp, (unsigned long long)(clock64() - k_t0));
    if (warp == 0) {
      for (int w = blockIdx.x; w < total_work; w += gridDim.x) ++n_items;
      atomicAdd(acc64 + 7, (unsigned long long)n_items);
    }
  }
#endif
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemAlloc);
  }
  if (kFused) {
    // combine (MegaMoE notes, "Combine"): once every GEMM2 item of the launch
    // has published its rows, each CTA sums the k BF16 rows of its share of
    // (token, 8-value chunk) items in FP32, in slot order, and casts once
    if (threadIdx.x == 0) scan_ws[0] = wait_counter(args.sync, n2, status, kWaitLimit, total_work) ? 1 : 0;
    __syncthreads();
    if (scan_ws[0])
      combine_share(args.y_pairs, args.topk_idx, args.T, args.k, args.H, args.y,
                    (int)blockIdx.x * C::kThreads + (int)threadIdx.x, (int)gridDim.x * C::kThreads);
  }
}

// Per pool row s (expert e, tile g = tile_off[e] + rank/BN, row r = rank%BN):
//   FROM_TOKENS (before GEMM1): token t = perm[s]/k -> tok_pool[s], its top-k
//     weight -> w_pool[s], the 4 scale bytes of each K block of xs[t] into
//     chunk (g, kb) at byte (r%32)*16 + (r/32)*4, and (large token tiles) the
//     FP8 row xq[t] -> xq_pool[s];
//   otherwise (GEMM2 fed with an external h): the scale bytes of row s of
//     that h into GEMM2's chunks.
template <int BN, bool FROM_TOKENS>
__global__ void __launch_bounds__(256) prep_pool_kernel(const uint8_t *__restrict__ src_scales,
                                                        const int32_t *__restrict__ counts,
                                                        const int32_t *__restrict__ offsets,
                                                        const int32_t *__restrict__ perm,
                                                        const float *__restrict__ topk_w, int E, int k, int KB,
                                                        uint8_t *__restrict__ chunks, int32_t *__restrict__ tok_pool,
                                                        float *__restrict__ w_pool, const uint4 *__restrict__ xq,
                                                        uint4 *__restrict__ xq_pool, int row16) {
  extern __shared__ int sh[];
  int *tile_off = sh, *cnt_sm = sh + (E + 1), *off_sm = sh + 2 * (E + 1);
  pdl_launch_dependents();
  pdl_wait();
  load_expert_table(counts, offsets, E, cnt_sm, off_sm);
  __syncthreads();
  __shared__ int scan_scratch[9];
  block_tile_map<256>(cnt_sm, E, BN, tile_off, scan_scratch, scan_scratch + 8);
  __syncthreads();
  const int P = off_sm[E];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  for (int s = blockIdx.x * nwarps + warp; s < P; s += gridDim.x * nwarps) {
    int lo = 0, hi = E;                        // expert e with off[e] <= s < off[e+1]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (off_sm[mid] <= s) lo = mid; else hi = mid;
    }
    const int rank = s - off_sm[lo];
    const int g = tile_off[lo] + rank / BN, r = rank % BN;
    int row = s;
    if (FROM_TOKENS) {
      const int p = __ldg(perm + s);
      row = p / k;
      if (lane == 0) {
        tok_pool[s] = row;
        w_pool[s] = __ldg(topk_w + p);
      }
      if (xq_pool) {
        const uint4 *src = xq + (size_t)row * row16;
        uint4 *dst = xq_pool + (size_t)s * row16;
        for (int i = lane; i < row16; i += 32) dst[i] = __ldg(src + i);
      }
    }
    const uint32_t *src = reinterpret_cast<const uint32_t *>(src_scales + (size_t)row * KB * 4);
    for (int kb = lane; kb < KB; kb += 32) {
      const uint32_t wv = __ldg(src + kb);
      const int rr = r & 127;
      *reinterpret_cast<uint32_t *>(chunks + ((size_t)g * KB + kb) * Cfg<BN>::kTokChunk + (r >> 7) * 512 +
                                    (rr & 31) * 16 + (rr >> 5) * 4) = wv;
    }
  }
}

// The activation cast fused with the pool rows of GEMM1 (used by moe_forward):
// for pool row s (expert e, tile g, row r) with pair p = perm[s] and token
// t = p / k, write tok_pool[s] = t, w_pool[s] = topk_w[p], the E4M3 codes of
// x[t] to xq_pool[s] and its UE8M0 scales straight into GEMM1's scale chunks.
// One thread per 8 values of one pool row (four neighbouring lanes form a
// 32-group), so every load of the step is in flight at once; a token routed
// to k experts is cast k times, reading x[t] from L2, which saves writing and
// re-reading a token-order copy.
template <int BN>
__global__ void __launch_bounds__(256) pool_cast_kernel(const uint4 *__restrict__ x, const int32_t *__restrict__ counts,
                                                        const int32_t *__restrict__ offsets,
                                                        const int32_t *__restrict__ perm,
                                                        const float *__restrict__ topk_w, int E, int k, int H,
                                                        uint8_t *__restrict__ chunks, int32_t *__restrict__ tok_pool,
                                                        float *__restrict__ w_pool, uint2 *__restrict__ xq_pool) {
  extern __shared__ int sh[];
  int *tile_off = sh, *cnt_sm = sh + (E + 1), *off_sm = sh + 2 * (E + 1);
  pdl_launch_dependents();
  pdl_wait();
  load_expert_table(counts, offsets, E, cnt_sm, off_sm);
  __syncthreads();
  __shared__ int scan_scratch[9];
  block_tile_map<256>(cnt_sm, E, BN, tile_off, scan_scratch, scan_scratch + 8);
  __syncthreads();
  const int P = off_sm[E];
  const int H8 = H / 8, KB = H / 128;
  const int64_t items = (int64_t)P * H8;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t base = (int64_t)blockIdx.x * blockDim.x; base < items; base += stride) {
    const int64_t i = base + threadIdx.x;
    const bool valid = i < items;               // groups of 4 items are all valid or all not
    int s = 0, c = 0, t = 0, p = 0;
    if (valid) {
      s = (int)(i / H8);
      c = (int)(i - (int64_t)s * H8);
      p = __ldg(perm + s);
      t = p / k;
    }
    uint8_t sb;
    const uint2 codes = cast8_e4m3(valid ? __ldg(x + (size_t)t * H8 + c) : make_uint4(0, 0, 0, 0), valid, &sb);
    if (!valid) continue;
    xq_pool[(size_t)s * H8 + c] = codes;
    if ((c & 3) == 0) {
      int lo = 0, hi = E;                      // expert e with off[e] <= s < off[e+1]
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (off_sm[mid] <= s) lo = mid; else hi = mid;
      }
      const int rank = s - off_sm[lo];
      const int g = tile_off[lo] + rank / BN, r = rank % BN;
      const int rr = r & 127;
      chunks[((size_t)g * KB + (c >> 4)) * Cfg<BN>::kTokChunk + (r >> 7) * 512 + (rr & 31) * 16 + (rr >> 5) * 4 +
             ((c >> 2) & 3)] = sb;
      if (c == 0) {
        tok_pool[s] = t;
        w_pool[s] = __ldg(topk_w + p);
      }
    }
  }
}

// The activation cast of large problems, in token order: a warp per token
// reads its BF16 row once (a pool-order cast re-reads it k times, from DRAM
// once x outgrows L2), casts it to E4M3 with one UE8M0 scale per 32 values and
// writes the codes to the pool rows of the token's k pairs
// (s = inv_perm[t*k + j]; -1 = dropped pair).  Lanes 0..k-1 first locate
// their pair's pool row and scale-chunk position (one search per pair, not
// per value), which the column loop then takes by shuffle.  Per 256-value
// step a lane casts 8 values (four lanes form a 32-group, as pool_cast_kernel)
// and the first lane of each 16 writes the four scale bytes of its 128-value
// K block as one word; four steps' loads are issued before the first cast.
constexpr int kTokenCastUnroll = 4;

template <int BN>
__global__ void __launch_bounds__(256) token_cast_kernel(const uint4 *__restrict__ x, const int32_t *__restrict__ counts,
                                                         const int32_t *__restrict__ offsets,
                                                         const int32_t *__restrict__ inv_perm,
                                                         const float *__restrict__ topk_w, int64_t T, int E, int k,
                                                         int H, uint8_t *__restrict__ chunks,
                                                         int32_t *__restrict__ tok_pool, float *__restrict__ w_pool,
                                                         uint2 *__restrict__ xq_pool) {
  extern __shared__ int sh[];
  int *tile_off = sh, *cnt_sm = sh + (E + 1), *off_sm = sh + 2 * (E + 1);
  pdl_launch_dependents();
  pdl_wait();
  load_expert_table(counts, offsets, E, cnt_sm, off_sm);
  __syncthreads();
  __shared__ int scan_scratch[9];
  block_tile_map<256>(cnt_sm, E, BN, tile_off, scan_scratch, scan_scratch + 8);
  __syncthreads();
  const int H8 = H / 8, KB = H / 128;
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < T; t += warps) {
    // lane j < k (k <= 32): pool row of pair (t, j) and the offset of its
    // scale word in K block 0
    int s_mine = -1;
    int64_t sfo_mine = 0;
    if (lane < k) {
      const int64_t p = t * k + lane;
      s_mine = __ldg(inv_perm + p);
      if (s_mine >= 0) {
        int lo = 0, hi = E;                      // expert e with off[e] <= s < off[e+1]
        while (hi - lo > 1) {
          const int mid = (lo + hi) >> 1;
          if (off_sm[mid] <= s_mine) lo = mid; else hi = mid;
        }
        const int rank = s_mine - off_sm[lo];
        const int g = tile_off[lo] + rank / BN, r = rank % BN;
        const int rr = r & 127;
        sfo_mine = (int64_t)g * KB * Cfg<BN>::kTokChunk + (r >> 7) * 512 + (rr & 31) * 16 + (rr >> 5) * 4;
        tok_pool[s_mine] = (int32_t)t;
        w_pool[s_mine] = __ldg(topk_w + p);
      }
    }
    const uint4 *xrow = x + t * H8;
    for (int c0 = 0; c0 < H8; c0 += 32 * kTokenCastUnroll) {
      uint4 v[kTokenCastUnroll];
#pragma unroll
      for (int u = 0; u < kTokenCastUnroll; ++u) {
        const int c = c0 + 32 * u + lane;
        v[u] = c < H8 ? __ldg(xrow + c) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < kTokenCastUnroll; ++u) {
        const int cb = c0 + 32 * u;              // warp-uniform
        if (cb >= H8) break;
        const int c = cb + lane;
        const bool valid = c < H8;               // uniform over each 16 lanes (H8 % 16 == 0)
        uint8_t sb;
        const uint2 codes = cast8_e4m3(v[u], valid, &sb);
        uint32_t word = sb;                      // meaningful in lanes with c % 16 == 0
        word |= __shfl_down_sync(0xffffffffu, (uint32_t)sb, 4) << 8;
        word |= __shfl_down_sync(0xffffffffu, (uint32_t)sb, 8) << 16;
        word |= __shfl_down_sync(0xffffffffu, (uint32_t)sb, 12) << 24;
        const int64_t kb_off = (int64_t)(c >> 4) * Cfg<BN>::kTokChunk;
        for (int j = 0; j < k; ++j) {
          const int s = __shfl_sync(0xffffffffu, s_mine, j);
          const int64_t sfo = __shfl_sync(0xffffffffu, sfo_mine, j);
          if (s < 0 || !valid) continue;
          xq_pool[(size_t)s * H8 + c] = codes;
          if ((c & 15) == 0) *reinterpret_cast<uint32_t *>(chunks + sfo + kb_off) = word;
        }
      }
    }
  }
}

// Small problems in one launch.  Every CTA routes all T tokens and builds the
// whole counting-sort permutation in shared memory -- the same result in every
// CTA, so no grid-wide synchronisation is needed -- CTA 0 writes the routing
// and permute outputs, and every CTA then casts its columns (gpc 32-value
// groups) of every pool row as pool_cast_kernel does.  The x values of those
// columns for all T tokens are read into shared memory before routing starts,
// so that the cast waits on no global load.  Used for T <= 64, E <= 256 (a
// few KB of logits per CTA).
constexpr int kFrontThreads = 256;
constexpr int kFrontMaxT = 64, kFrontMaxE = 256;

template <int BN>
__global__ void __launch_bounds__(kFrontThreads) front_kernel(
    const float *__restrict__ logits, const uint4 *__restrict__ x, int T, int E, int k, int H,
    int32_t *__restrict__ idx_out, float *__restrict__ w_out, int32_t *__restrict__ counts_out,
    int32_t *__restrict__ offsets_out, int32_t *__restrict__ perm_out, int32_t *__restrict__ inv_perm_out,
    uint8_t *__restrict__ chunks, int32_t *__restrict__ tok_pool, float *__restrict__ w_pool,
    uint2 *__restrict__ xq_pool, int gpc, int mode, int *__restrict__ zero_words, int n_zero) {
  constexpr int kW = kFrontThreads / 32;
  extern __shared__ __align__(16) unsigned char fsm[];
  const int P = T * k;
  const int H8 = H / 8, KB = H / 128;
  const int cc0 = blockIdx.x * gpc * 4;                                // first 8-value column of this CTA
  const int ncols = max(0, min(gpc * 4, H8 - cc0));
  uint4 *xs = reinterpret_cast<uint4 *>(fsm);                          // [T][gpc * 4]
  int *idx_sm = reinterpret_cast<int *>(xs + (size_t)T * gpc * 4);     // [P]
  float *w_sm = reinterpret_cast<float *>(idx_sm + P);                 // [P]
  int *perm_sm = reinterpret_cast<int *>(w_sm + P);                    // [P]
  int *cnt = perm_sm + P;                                              // [E+1]
  int *off = cnt + (E + 1);                                            // [E+1]
  int *tile_off = off + (E + 1);                                       // [E+1]
  int *base = tile_off + (E + 1);                                      // [E]
  int *warp_sums = base + E;                                           // [kW]
  int *total = warp_sums + kW;                                         // [1]
  uint16_t *wc = reinterpret_cast<uint16_t *>(total + 4);              // [kW][E]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool writer = blockIdx.x == 0;
  pdl_launch_dependents();
  pdl_wait();
  // the call's status words and arrival counters (read by the launches after
  // this one, which wait for its completion)
  if (writer)
    for (int i = tid; i < n_zero; i += kFrontThreads) zero_words[i] = 0;
  // 0. this CTA's columns of x (consumed in step 3): the first 16 bytes per
  // thread are loaded into a register here and land in shared memory after
  // routing, so that their latency overlaps the logits loads
  const int nx = T * ncols;
  uint4 xv = make_uint4(0, 0, 0, 0);
  if (tid < nx) xv = __ldg(x + (size_t)(tid / ncols) * H8 + cc0 + tid % ncols);
  for (int i = tid + kFrontThreads; i < nx; i += kFrontThreads)
    xs[i] = __ldg(x + (size_t)(i / ncols) * H8 + cc0 + i % ncols);
  // 1. routing of every token, one warp per token
  for (int t = warp; t < T; t += kW) {
    int my_idx;
    float my_w;
    warp_route_token<kFrontMaxE / 32>(logits + (size_t)t * E, E, k, lane, mode, &my_idx, &my_w);
    if (lane < k) {
      idx_sm[t * k + lane] = my_idx;
      w_sm[t * k + lane] = my_w;
      if (writer) {
        idx_out[t * k + lane] = my_idx;
        w_out[t * k + lane] = my_w;
      }
    }
    __syncwarp();
  }
  if (tid < nx) xs[tid] = xv;
  for (int e = tid; e <= E; e += kFrontThreads) cnt[e] = 0;
  __syncthreads();
  // 2. count -> prefix -> stable scatter
  for (int p = tid; p < P; p += kFrontThreads) atomicAdd(&cnt[idx_sm[p]], 1);
  __syncthreads();
  const int o = block_exclusive_scan<kFrontThreads>(tid < E ? cnt[tid] : 0, warp_sums, total);
  if (tid < E) {
    off[tid] = o;
    base[tid] = o;
    if (writer) {
      counts_out[tid] = cnt[tid];
      offsets_out[tid] = o;
    }
  }
  if (tid == 0) {
    off[E] = *total;
    if (writer) offsets_out[E] = *total;
  }
  __syncthreads();
  block_tile_map<kFrontThreads>(cnt, E, BN, tile_off, warp_sums, total);
  block_stable_ranks<kFrontThreads>([&](int64_t p) { return idx_sm[p]; }, 0, P, E, base, wc,
                                    writer ? perm_out : nullptr, writer ? inv_perm_out : nullptr, perm_sm);
  // 3. this CTA's columns of every pool row (four lanes per 32-value group)
  const int items = P * ncols;
  for (int b0 = 0; b0 < items; b0 += kFrontThreads) {
    const int i = b0 + tid;
    const bool valid = i < items;
    int sr = 0, cl = 0, t = 0, pp = 0;
    if (valid) {
      sr = i / ncols;
      cl = i - sr * ncols;
      pp = perm_sm[sr];
      t = pp / k;
    }
    uint8_t sb;
    const uint2 codes = cast8_e4m3(valid ? xs[t * ncols + cl] : make_uint4(0, 0, 0, 0), valid, &sb);
    if (!valid) continue;
    const int c = cc0 + cl;
    xq_pool[(size_t)sr * H8 + c] = codes;
    if ((c & 3) == 0) {
      int lo = 0, hi = E;
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (off[mid] <= sr) lo = mid; else hi = mid;
      }
      const int rank = sr - off[lo];
      const int g = tile_off[lo] + rank / BN, r = rank % BN;
      const int rr = r & 127;
      chunks[((size_t)g * KB + (c >> 4)) * Cfg<BN>::kTokChunk + (r >> 7) * 512 + (rr & 31) * 16 + (rr >> 5) * 4 +
             ((c >> 2) & 3)] = sb;
      if (c == 0) {
        tok_pool[sr] = t;
        w_pool[sr] = w_sm[pp];
      }
    }
  }
}

size_t front_smem(int T, int E, int k, int gpc) {
  const int P = T * k;
  return (size_t)T * gpc * 64 + (size_t)3 * P * 4 +
         (size_t)3 * (E + 1) * 4 + (size_t)E * 4 + (kFrontThreads / 32) * 4 + 16 +
         (size_t)(kFrontThreads / 32) * E * 2;
}

template <int BN>
int launch_front_t(const moe_expert_args *a, const uint16_t *x, const float *logits, int mode, int32_t *idx,
                   float *wts, int32_t *inv_perm, char *ws, const ExpertWs &lay, int *zero_words, int n_zero,
                   cudaStream_t st) {
  // one CTA per 32-value column group of the pool rows, at most two per SM
  const int groups = (int)(a->H / 32);
  const int cap = num_sms() * 2;
  const int grid = groups < cap ? groups : cap;
  const int gpc = (groups + grid - 1) / grid;
  return launch_pdl(front_kernel<BN>, dim3(grid), dim3(kFrontThreads), front_smem((int)a->T, a->E, a->k, gpc), st,
                    logits, reinterpret_cast<const uint4 *>(x), (int)a->T, a->E, a->k, (int)a->H, idx, wts,
                    const_cast<int32_t *>(a->counts), const_cast<int32_t *>(a->offsets),
                    const_cast<int32_t *>(a->perm), inv_perm, reinterpret_cast<uint8_t *>(ws + lay.sfb1),
                    reinterpret_cast<int32_t *>(ws + lay.tok_pool), reinterpret_cast<float *>(ws + lay.w_pool),
                    reinterpret_cast<uint2 *>(ws + lay.xq_pool), gpc, mode, zero_words, n_zero);
}

template <int BN>
int launch_pool_cast_t(const moe_expert_args *a, const uint16_t *x, char *ws, const ExpertWs &lay, cudaStream_t st) {
  const int64_t P = a->T * a->k;
  const size_t sm = (size_t)3 * (a->E + 1) * 4;
  const int64_t blocks = ceil_div(P * (a->H / 8), 256);
  const int cap = num_sms() * 8;
  const int grid = (int)(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
  return launch_pdl(pool_cast_kernel<BN>, dim3(grid), dim3(256), sm, st, reinterpret_cast<const uint4 *>(x),
                    a->counts, a->offsets, a->perm, a->topk_w, a->E, a->k, (int)a->H,
                    reinterpret_cast<uint8_t *>(ws + lay.sfb1), reinterpret_cast<int32_t *>(ws + lay.tok_pool),
                    reinterpret_cast<float *>(ws + lay.w_pool), reinterpret_cast<uint2 *>(ws + lay.xq_pool));
}

template <int BN>
int launch_token_cast_t(const moe_expert_args *a, const uint16_t *x, const int32_t *inv_perm, char *ws,
                        const ExpertWs &lay, cudaStream_t st) {
  const size_t sm = (size_t)3 * (a->E + 1) * 4;
  const int64_t blocks = ceil_div(a->T, 8);                  // a warp per token
  const int cap = num_sms() * 8;
  const int grid = (int)(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
  return launch_pdl(token_cast_kernel<BN>, dim3(grid), dim3(256), sm, st, reinterpret_cast<const uint4 *>(x),
                    a->counts, a->offsets, inv_perm, a->topk_w, a->T, a->E, a->k, (int)a->H,
                    reinterpret_cast<uint8_t *>(ws + lay.sfb1), reinterpret_cast<int32_t *>(ws + lay.tok_pool),
                    reinterpret_cast<float *>(ws + lay.w_pool), reinterpret_cast<uint2 *>(ws + lay.xq_pool));
}

template <int BN, bool FROM_TOKENS>
int launch_prep(const uint8_t *src, const moe_expert_args *a, int KB, uint8_t *chunks, int32_t *tok_pool,
                float *w_pool, uint8_t *xq_pool, cudaStream_t st) {
  const int64_t P = a->T * a->k;
  const size_t sm = (size_t)3 * (a->E + 1) * 4;
  const int64_t blocks = ceil_div(P, 8);
  const int cap = num_sms() * 4;
  const int grid = (int)(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
  return launch_pdl(prep_pool_kernel<BN, FROM_TOKENS>, dim3(grid), dim3(256), sm, st, src, a->counts, a->offsets,
                    a->perm, a->topk_w, a->E, a->k, KB, chunks, tok_pool, w_pool,
                    reinterpret_cast<const uint4 *>(a->xq), reinterpret_cast<uint4 *>(xq_pool), (int)(a->H / 16));
}

// Shared-memory attributes of a GEMM instantiation: its dynamic size and the
// largest carveout, so that kCtasPerSm CTAs fit on one SM.  (The occupancy
// calculator reports one CTA per SM for any kernel that allocates TMEM, but
// CTAs whose allocations fit the SM's 512 columns together are co-resident.)
template <typename Kernel>
bool set_gemm_attrs(Kernel kernel, size_t smem) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) == cudaSuccess &&
         cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100) == cudaSuccess;
}

template <int BN>
int run_expert(const moe_expert_args *a, int *status, char *ws, const ExpertWs &lay, cudaStream_t st) {
  using C = Cfg<BN>;
  uint8_t *sfb1 = reinterpret_cast<uint8_t *>(ws + lay.sfb1);
  uint8_t *sfb2 = reinterpret_cast<uint8_t *>(ws + lay.sfb2);
  uint8_t *hq = a->hq ? a->hq : reinterpret_cast<uint8_t *>(ws + lay.hq);
  int32_t *tok_pool = reinterpret_cast<int32_t *>(ws + lay.tok_pool);
  float *w_pool = reinterpret_cast<float *>(ws + lay.w_pool);
  uint8_t *xq_pool = reinterpret_cast<uint8_t *>(ws + lay.xq_pool);
  const int64_t P = a->T * a->k;
  const int E = a->E;
  const int phases = a->phases ? a->phases : (MOE_PHASE_TOKEN_SCALES | MOE_PHASE_GEMM1 | MOE_PHASE_GEMM2);

  // pool rows of GEMM1: token ids, weights, token-scale chunks (+ FP8 rows for large tiles)
  if ((phases & MOE_PHASE_TOKEN_SCALES) &&
      launch_prep<BN, true>(a->xs, a, (int)(a->H / 128), sfb1, tok_pool, w_pool, xq_pool, st) != MOE_OK)
    return MOE_ERR_CUDA;
  // scale chunks of GEMM2 from a caller-provided h (instead of GEMM1's epilogue)
  if ((phases & MOE_PHASE_H_SCALES) &&
      launch_prep<BN, false>(a->hs, a, (int)(a->I / 128), sfb2, nullptr, nullptr, nullptr, st) != MOE_OK)
    return MOE_ERR_CUDA;

  if constexpr (BN == 208) {
    // the large tile on CTA pairs (gemm2sm.cu; resolve_tile_n picks 208 only
    // where the weight tiles pair up)
    const int ph = phases & (MOE_PHASE_GEMM1 | MOE_PHASE_GEMM2);
    return ph ? run_expert_pairs(a, ph, status, hq, sfb1, sfb2, w_pool, xq_pool, st) : MOE_OK;
  } else {
  GemmArgs g{};
  g.E = E; g.k = a->k; g.T = (int)a->T; g.H = (int)a->H; g.I = (int)a->I;
  g.counts = a->counts; g.offsets = a->offsets; g.perm = a->perm;
  g.tok_pool = tok_pool; g.w_pool = w_pool;
  g.hq = hq; g.sfb2 = sfb2; g.hs_out = a->hs; g.y_pairs = a->y_pairs; g.status = status;
  const size_t sm = smem_bytes<BN>(E);
  const int grid = num_sms() * C::kCtasPerSm;
  if (const char *env = getenv("MOE_MXQ_DEBUG_INJECT_WAIT")) g.inject_wait = atoi(env);
  if (phases & MOE_PHASE_GEMM1) {
    // GEMM1 + SwiGLU (.) weight + FP8 requantisation
    const uint64_t wrows = (uint64_t)E * (2 * a->I / 128) * (a->H / 128) * 128;
    CUtensorMap tw1, tb;
    bool ok = encode_tmap_2d(&tw1, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, (void *)a->w1q, 128, wrows, 64, 128,
                             C::kKBS * kBM, CU_TENSOR_MAP_SWIZZLE_128B);
    ok = ok && encode_tmap_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, (void *)xq_pool, (uint64_t)a->H, (uint64_t)P,
                              (uint64_t)a->H, 128, BN, CU_TENSOR_MAP_SWIZZLE_128B);
    if (!ok) return MOE_ERR_CUDA;
    g.M = (int)(2 * a->I); g.K = (int)a->H; g.KB = (int)(a->H / 128); g.MT = (int)(2 * a->I / 128);
    g.w_sf = a->w1s; g.b_sf = sfb1; g.w_codes = a->w1q;
    if (!set_gemm_attrs(expert_gemm_kernel<BN, 1>, sm)) return MOE_ERR_CUDA;
    if (launch_pdl(expert_gemm_kernel<BN, 1>, dim3(grid), dim3(C::kThreads), sm, st, tw1, tb, tw1, tb, g) != MOE_OK)
      return MOE_ERR_CUDA;
  }
  if (phases & MOE_PHASE_GEMM2) {
    // GEMM2 -> BF16 per pair
    const uint64_t wrows = (uint64_t)E * (a->H / 128) * (a->I / 128) * 128;
    CUtensorMap tw2, th;
    bool ok = encode_tmap_2d(&tw2, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, (void *)a->w2q, 128, wrows, 64, 128,
                             C::kKBS * kBM, CU_TENSOR_MAP_SWIZZLE_128B);
    ok = ok && encode_tmap_2d(&th, CU_TENSOR_MAP_DATA_TYPE_UINT8, (void *)hq, (uint64_t)a->I, (uint64_t)P,
                              (uint64_t)a->I, 128, BN, CU_TENSOR_MAP_SWIZZLE_128B);
    if (!ok) return MOE_ERR_CUDA;
    g.M = (int)a->H; g.K = (int)a->I; g.KB = (int)(a->I / 128); g.MT = (int)(a->H / 128);
    g.w_sf = a->w2s; g.b_sf = sfb2; g.w_codes = a->w2q;
    g.early_weights = (phases & MOE_PHASE_GEMM1) ? 1 : 0;
    g.hs_out = nullptr;
    if (!set_gemm_attrs(expert_gemm_kernel<BN, 2>, sm)) return MOE_ERR_CUDA;
    if (launch_pdl(expert_gemm_kernel<BN, 2>, dim3(grid), dim3(C::kThreads), sm, st, tw2, th, tw2, th, g) != MOE_OK)
      return MOE_ERR_CUDA;
  }
  return MOE_OK;
  }
}

}  // namespace

int launch_pool_cast(const moe_expert_args *a, const uint16_t *x, void *scratch, cudaStream_t st) {
  const ExpertWs lay = expert_ws_layout(a->T, a->H, a->I, a->E, a->k);
  if (a->T == 0) return MOE_OK;
  char *ws = reinterpret_cast<char *>(scratch);
  const int bn = resolve_tile_n(a->tile_n, a->T * a->k, a->E, a->H, a->I);
  switch (bn) {
    case 16: return launch_pool_cast_t<16>(a, x, ws, lay, st);
    case 32: return launch_pool_cast_t<32>(a, x, ws, lay, st);
    case 64: return launch_pool_cast_t<64>(a, x, ws, lay, st);
    case 128: return launch_pool_cast_t<128>(a, x, ws, lay, st);
    case 208: return launch_pool_cast_t<208>(a, x, ws, lay, st);
    case 224: return launch_pool_cast_t<224>(a, x, ws, lay, st);
    default: return MOE_ERR_INVALID_ARG;
  }
}

int launch_token_cast(const moe_expert_args *a, const uint16_t *x, const int32_t *inv_perm, void *scratch,
                      cudaStream_t st) {
  const ExpertWs lay = expert_ws_layout(a->T, a->H, a->I, a->E, a->k);
  if (a->T == 0) return MOE_OK;
  char *ws = reinterpret_cast<char *>(scratch);
  const int bn = resolve_tile_n(a->tile_n, a->T * a->k, a->E, a->H, a->I);
  switch (bn) {
    case 16: return launch_token_cast_t<16>(a, x, inv_perm, ws, lay, st);
    case 32: return launch_token_cast_t<32>(a, x, inv_perm, ws, lay, st);
    case 64: return launch_token_cast_t<64>(a, x, inv_perm, ws, lay, st);
    case 128: return launch_token_cast_t<128>(a, x, inv_perm, ws, lay, st);
    case 208: return launch_token_cast_t<208>(a, x, inv_perm, ws, lay, st);
    case 224: return launch_token_cast_t<224>(a, x, inv_perm, ws, lay, st);
    default: return MOE_ERR_INVALID_ARG;
  }
}

bool front_eligible(int64_t T, int64_t H, int E, int k) {
  return T >= 1 && T <= kFrontMaxT && E <= kFrontMaxE && T * k * H <= (int64_t(4) << 20);
}

int launch_front(const moe_expert_args *a, const uint16_t *x, const float *logits, int mode, int32_t *idx,
                 float *wts, int32_t *inv_perm, void *scratch, int *zero_words, int n_zero, cudaStream_t st) {
  const ExpertWs lay = expert_ws_layout(a->T, a->H, a->I, a->E, a->k);
  char *ws = reinterpret_cast<char *>(scratch);
  const int bn = resolve_tile_n(a->tile_n, a->T * a->k, a->E, a->H, a->I);
  switch (bn) {
    case 16: return launch_front_t<16>(a, x, logits, mode, idx, wts, inv_perm, ws, lay, zero_words, n_zero, st);
    case 32: return launch_front_t<32>(a, x, logits, mode, idx, wts, inv_perm, ws, lay, zero_words, n_zero, st);
    case 64: return launch_front_t<64>(a, x, logits, mode, idx, wts, inv_perm, ws, lay, zero_words, n_zero, st);
    case 128: return launch_front_t<128>(a, x, logits, mode, idx, wts, inv_perm, ws, lay, zero_words, n_zero, st);
    case 208: return launch_front_t<208>(a, x, logits, mode, idx, wts, inv_perm, ws, lay, zero_words, n_zero, st);
    case 224: return launch_front_t<224>(a, x, logits, mode, idx, wts, inv_perm, ws, lay, zero_words, n_zero, st);
    default: return MOE_ERR_INVALID_ARG;
  }
}

// GEMM1 + GEMM2 + combine in one launch (16-token tiles, after the
// small-problem front kernel).  Its CTAs wait on one another's arrival
// counters, so all of them must be resident at once: kCtasPerSm CTAs of this
// shared-memory size have to fit on an SM.
bool fused_eligible(int64_t T, int64_t H, int E, int k, int tile_n) {
  if (!front_eligible(T, H, E, k)) return false;
  if (tile_n != 0 && tile_n != 16) return false;
  if (choose_tile_n(T * k, E) != 16) return false;
  static int smem_per_sm = -1;
  if (smem_per_sm < 0) {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess)
      v = 0;
    smem_per_sm = v;
  }
  return (int64_t)Cfg<16>::kCtasPerSm * ((int64_t)smem_bytes<16>(E) + 1024) <= smem_per_sm;
}

size_t fused_sync_ints(int64_t T, int E, int k) { return 1 + (size_t)max_token_tiles(T * k, E, 16); }

int launch_fused_gemms(const moe_expert_args *a, uint16_t *y, int *sync, int *status, char *ews, cudaStream_t st) {
  using C = Cfg<16>;
  constexpr int BN = 16;
  const ExpertWs lay = expert_ws_layout(a->T, a->H, a->I, a->E, a->k);
  const int64_t P = a->T * a->k;
  const int E = a->E;
  uint8_t *sfb1 = reinterpret_cast<uint8_t *>(ews + lay.sfb1);
  uint8_t *sfb2 = reinterpret_cast<uint8_t *>(ews + lay.sfb2);
  uint8_t *hq = reinterpret_cast<uint8_t *>(ews + lay.hq);
  uint8_t *xq_pool = reinterpret_cast<uint8_t *>(ews + lay.xq_pool);
  CUtensorMap tw1, tb, tw2, th;
  const uint64_t wrows1 = (uint64_t)E * (2 * a->I / 128) * (a->H / 128) * 128;
  const uint64_t wrows2 = (uint64_t)E * (a->H / 128) * (a->I / 128) * 128;
  bool ok = encode_tmap_2d(&tw1, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, (void *)a->w1q, 128, wrows1, 64, 128,
                           C::kKBS * kBM, CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && encode_tmap_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, (void *)xq_pool, (uint64_t)a->H, (uint64_t)P,
                            (uint64_t)a->H, 128, BN, CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && encode_tmap_2d(&tw2, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, (void *)a->w2q, 128, wrows2, 64, 128,
                            C::kKBS * kBM, CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && encode_tmap_2d(&th, CU_TENSOR_MAP_DATA_TYPE_UINT8, (void *)hq, (uint64_t)a->I, (uint64_t)P,
                            (uint64_t)a->I, 128, BN, CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) return MOE_ERR_CUDA;
  GemmArgs g{};
  g.E = E; g.k = a->k; g.T = (int)a->T; g.H = (int)a->H; g.I = (int)a->I;
  g.M = (int)(2 * a->I); g.K = (int)a->H; g.KB = (int)(a->H / 128); g.MT = (int)(2 * a->I / 128);
  g.MT2 = (int)(a->H / 128); g.KB2 = (int)(a->I / 128);
  g.counts = a->counts; g.offsets = a->offsets; g.perm = a->perm;
  g.tok_pool = reinterpret_cast<int32_t *>(ews + lay.tok_pool);
  g.w_pool = reinterpret_cast<float *>(ews + lay.w_pool);
  g.w_sf = a->w1s; g.b_sf = sfb1; g.w_sf2 = a->w2s; g.b_sf2 = sfb2; g.w_codes = a->w1q;
  g.w_codes2 = a->w2q;
  g.hq = hq; g.sfb2 = sfb2; g.hs_out = nullptr; g.y_pairs = a->y_pairs; g.status = status;
  g.sync = sync; g.topk_idx = a->topk_idx; g.y = reinterpret_cast<uint4 *>(y);
  if (const char *env = getenv("MOE_MXQ_DEBUG_INJECT_WAIT")) g.inject_wait = atoi(env);
  const size_t sm = smem_bytes<BN>(E);
  if (!set_gemm_attrs(expert_gemm_kernel<BN, 3>, sm)) return MOE_ERR_CUDA;
  return launch_pdl(expert_gemm_kernel<BN, 3>, dim3(num_sms() * C::kCtasPerSm), dim3(C::kThreads), sm, st, tw1, tb,
                    tw2, th, g);
}

int launch_expert_forward(const moe_expert_args *a, int *status, void *scratch, cudaStream_t st) {
  const ExpertWs lay = expert_ws_layout(a->T, a->H, a->I, a->E, a->k);
  if (a->T == 0) return MOE_OK;
  char *ws = reinterpret_cast<char *>(scratch);
  const int bn = resolve_tile_n(a->tile_n, a->T * a->k, a->E, a->H, a->I);
  switch (bn) {
    case 16: return run_expert<16>(a, status, ws, lay, st);
    case 32: return run_expert<32>(a, status, ws, lay, st);
    case 64: return run_expert<64>(a, status, ws, lay, st);
    case 128: return run_expert<128>(a, status, ws, lay, st);
    case 208: return run_expert<208>(a, status, ws, lay, st);
    case 224: return run_expert<224>(a, status, ws, lay, st);
    default: return MOE_ERR_INVALID_ARG;
  }
}

int check_expert_args(const moe_expert_args *a, bool need_ws) {
  if (!a) return MOE_ERR_INVALID_ARG;
  if (a->struct_size != sizeof(moe_expert_args)) return MOE_ERR_INVALID_ARG;
  if (a->T < 0 || a->H <= 0 || a->I <= 0 || a->E <= 0 || a->k <= 0) return MOE_ERR_INVALID_ARG;
  if (a->H % 128 || a->I % 128 || a->E > kMaxE || a->k > a->E || a->k > 32) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (a->T * (int64_t)a->k >= ((int64_t)1 << 31) || a->H * a->E >= ((int64_t)1 << 31) ||
      2 * a->I * a->E >= ((int64_t)1 << 31))
    return MOE_ERR_UNSUPPORTED_SHAPE;
  if (a->tile_n != 0 && a->tile_n != 16 && a->tile_n != 32 && a->tile_n != 64 && a->tile_n != 128 &&
      a->tile_n != 208 && a->tile_n != 224)
    return MOE_ERR_INVALID_ARG;
  if (a->phases & ~15) return MOE_ERR_INVALID_ARG;
  if ((a->phases & MOE_PHASE_H_SCALES) && (!a->hq || !a->hs)) return MOE_ERR_INVALID_ARG;
  if (need_ws) {
    if (!a->workspace) return MOE_ERR_INVALID_ARG;
    if (!aligned(a->workspace, 256)) return MOE_ERR_MISALIGNED;
    if (a->workspace_bytes < kStatusBytes + expert_ws_layout(a->T, a->H, a->I, a->E, a->k).total)
      return MOE_ERR_WORKSPACE_TOO_SMALL;
  }
  if (a->T == 0) return MOE_OK;
  // the token step (phases 0 includes it) reads xq / xs
  const bool token_step = a->phases == 0 || (a->phases & MOE_PHASE_TOKEN_SCALES);
  if ((token_step && (!a->xq || !a->xs)) || !a->w1q || !a->w1s || !a->w2q || !a->w2s || !a->topk_idx ||
      !a->topk_w || !a->counts || !a->offsets || !a->perm || !a->y_pairs)
    return MOE_ERR_INVALID_ARG;
  if (!aligned(a->w1q, 32) || !aligned(a->w2q, 32)) return MOE_ERR_MISALIGNED;
  if ((token_step && (!aligned(a->xq, 16) || !aligned(a->xs, 16))) || !aligned(a->w1s, 16) ||
      !aligned(a->w2s, 16) || !aligned(a->y_pairs, 16) || (a->hq && !aligned(a->hq, 16)))
    return MOE_ERR_MISALIGNED;
  return MOE_OK;
}

}  // namespace mxq

using namespace mxq;

extern "C" size_t moe_expert_workspace_size(int64_t T, int64_t H, int64_t I, int32_t E, int32_t k) {
  if (T < 0 || H <= 0 || I <= 0 || E <= 0 || k <= 0) return 0;
  return kStatusBytes + expert_ws_layout(T, H, I, E, k).total;
}

extern "C" int moe_expert_forward(const moe_expert_args *args, cudaStream_t stream) {
  const int rc = check_expert_args(args, true);
  if (rc != MOE_OK) return rc;
  if (cudaMemsetAsync(args->workspace, 0, 32, stream) != cudaSuccess) return MOE_ERR_CUDA;
  return launch_expert_forward(args, reinterpret_cast<int *>(args->workspace),
                               reinterpret_cast<char *>(args->workspace) + kStatusBytes, stream);
}
