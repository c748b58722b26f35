// ptx.cuh -- hand-written inline-PTX wrappers for sm_103a: mbarrier, TMA
// (tiled, gather4, bulk), tcgen05 (alloc, cp, mma block_scale, commit, ld),
// FP8/FP4 conversions and the UE8M0 exponent rule.
#pragma once
#include <cstdint>
#include <cuda.h>

namespace mxq {

// ---------------------------------------------------------------- status words
// Every workspace starts with int32 status words: [0] first error (0 = ok),
// [1] abort flag raised by a device-side wait that gave up, [2] the site of
// the first wait that gave up (see the kWait* codes), [3] its block index,
// [4] its loop position.
enum : int { kStatusOk = 0, kStatusTimeout = 6, kStatusBadIndex = 7 };

__device__ __forceinline__ void report_status(int *status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// ---------------------------------------------------------------- misc
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Orders this thread's generic-proxy global accesses with later async-proxy
// (TMA) accesses: a writer runs it after stores that another CTA's TMA will
// read, a reader after it acquired the flag that publishes them.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ int ld_acquire_gpu(const int *p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// ---------------------------------------------------------------- programmatic dependent launch
// A kernel launched with programmatic stream serialization may start while the
// previous kernel of the stream is still running.  pdl_wait() blocks until
// that kernel has completed and its memory is visible; every kernel here
// calls it before its first global-memory access, so only setup that touches
// no global memory (barrier init, TMEM allocation, tensor-map prefetch)
// overlaps the previous kernel.  pdl_launch_dependents() lets the next kernel
// of the stream be scheduled early.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" :::); }

// One lane of the (converged) warp, the same for every lane to agree on:
// elect.sync.  Issuing tcgen05 instructions under it rather than under
// `lane == 0` keeps the issue path warp-uniform (measured: the MMA issue block
// of the CTA-pair GEMM took ~2.5x fewer cycles).
__device__ __forceinline__ bool elect_one() {
  uint32_t e;
  asm volatile("{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}" : "=r"(e));
  return e != 0;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Sites of bounded waits, recorded in status word [2] on a timeout.
enum : int {
  kWaitProducerEmpty = 1,
  kWaitMmaTmemEmpty = 2,
  kWaitMmaFull = 3,
  kWaitEpiTmemFull = 4,
  kWaitProducerDrain = 5,
  kWaitMmaDone = 6,
  kWaitInjected = 7,      // debug: a wait on a barrier that nothing completes
  kWaitArrival = 8        // single-launch layer: a CTA waiting on other CTAs' arrival counter
};

// Waits for phase `parity` of `bar` to complete.  Gives up after `limit`
// clock cycles, or (honor_abort) as soon as the abort flag is raised, and
// returns false.  On a timeout it raises the abort flag and records the
// status, the wait site and the loop position `pos` itself.  Waits for the
// CTA's own asynchronous copies and MMAs before it exits pass
// honor_abort = false: those always complete, and the CTA must not release
// shared memory or TMEM they still write.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, int *ws_status,
                                          long long limit, int site = 0, int pos = 0, bool honor_abort = true) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  volatile int *abort_flag = ws_status + 1;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (honor_abort && *abort_flag) return false;
    if (clock64() - t0 > limit) {
      if (atomicCAS(ws_status + 2, 0, site) == 0) {
        ws_status[3] = (int)blockIdx.x;
        ws_status[4] = pos;
      }
      report_status(ws_status, kStatusTimeout);
      atomicExch(ws_status + 1, 1);
      return false;
    }
  }
}

// Waits (bounded) until *counter >= target, the counter being raised by
// other CTAs of the same launch (release: fence + atomic add).  Acquire load,
// so their earlier writes are visible to this thread afterwards.  Same
// timeout and abort protocol as mbar_wait.  One thread calls it.
__device__ __forceinline__ bool wait_counter(const int *counter, int target, int *ws_status, long long limit,
                                             int pos = 0) {
  if (ld_acquire_gpu(counter) >= target) return true;
  const long long t0 = clock64();
  volatile int *abort_flag = ws_status + 1;
  while (true) {
    if (ld_acquire_gpu(counter) >= target) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > limit) {
      if (atomicCAS(ws_status + 2, 0, kWaitArrival) == 0) {
        ws_status[3] = (int)blockIdx.x;
        ws_status[4] = pos;
      }
      report_status(ws_status, kStatusTimeout);
      atomicExch(ws_status + 1, 1);
      return false;
    }
    __nanosleep(128);
  }
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, uint64_t *bar, int32_t x,
                                            int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}

// Plain bulk copy global -> shared (both 16-byte aligned, bytes % 16 == 0).
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Hint: bring `bytes` (multiple of 16, 16-byte aligned) of global memory into L2.
__device__ __forceinline__ void prefetch_l2_bulk(const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(src)), "r"(bytes)
               : "memory");
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Arrives once on `bar` when every tcgen05 operation issued so far by this
// thread has completed.
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}
// 32 rows x 128 bits from shared memory into TMEM, replicated into all four
// 32-lane quadrants.
__device__ __forceinline__ void tc_cp_32x128b_warpx4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
// D[tmem] (+)= A[smem] x B[smem]^T with per-32-K UE8M0 scales from TMEM.
__device__ __forceinline__ void tc_mma_mxf8f6f4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                                uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                                uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p;\n\t"
      "}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Each thread of the warp reads its own TMEM lane (warp's quadrant base +
// lane id), 16 consecutive 32-bit columns starting at the address's column.
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32"
      " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// Shared-memory matrix descriptor (tcgen05 format): start address, leading
// and stride byte offsets (all >> 4), version 1, swizzle mode in bits 61..63.
enum : uint32_t { kSwizzleNone = 0, kSwizzle128B = 2 };
__device__ __forceinline__ uint64_t make_smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t swz) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFF);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)(swz & 7) << 61;
  return d;
}

// Instruction descriptor of kind::mxf8f6f4 with block scaling:
// A = E2M1 (code 5), B = E4M3 (code 0), both K-major, UE8M0 scales,
// M = m (128, or 256 for the 2-SM form), N = n; sf_id picks the byte of the
// 32-bit scale cell.
__device__ __forceinline__ uint32_t make_idesc_fp4w_fp8a(uint32_t n, uint32_t sf_id, uint32_t m = 128) {
  uint32_t d = 0;
  d |= (sf_id & 3u) << 4;      // B scale-factor byte
  d |= 5u << 7;                // A format: E2M1
  d |= 0u << 10;               // B format: E4M3
  d |= ((n >> 3) & 0x3Fu) << 17;
  d |= 1u << 23;               // scale format UE8M0
  d |= ((m >> 4) & 0x1Fu) << 24;
  d |= (sf_id & 3u) << 29;     // A scale-factor byte
  return d;
}

// ---------------------------------------------------------------- 2-SM (cta_group::2) forms
// A CTA pair of a 2-CTA cluster shares one MMA: the even CTA (rank 0) issues
// tcgen05.mma.cta_group::2 with M = 256, each CTA holding 128 rows of A and
// of D (its own TMEM) and N/2 rows of B (CTA r supplies columns
// [r*N/2, (r+1)*N/2)); the A scales are each CTA's own rows, the B scales all
// N columns in each CTA's TMEM; tcgen05.cp.cta_group::2 copies each CTA's
// shared memory into its own TMEM.  A kernel uses one cta_group throughout.
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Barrier over both CTAs of the cluster (release / acquire at cluster scope).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address in the shared memory of cluster CTA `rank` of the variable at
// shared::cta address `addr` of this CTA.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// Arrive (release, cluster scope) on an mbarrier given by its shared::cluster address.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// Both CTAs' warps allocate / free the same TMEM columns together.
__device__ __forceinline__ void tmem_alloc_2sm(uint32_t *dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_2sm() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_2sm(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// Arrives once on the mbarrier at `bar`'s offset in every CTA of `cta_mask`
// when all tcgen05 operations issued so far by this thread have completed.
__device__ __forceinline__ void tc_commit_2sm(uint64_t *bar, uint16_t cta_mask) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
               ::"r"(smem_u32(bar)), "h"(cta_mask)
               : "memory");
}
__device__ __forceinline__ void tc_cp_2sm_32x128b_warpx4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
__device__ __forceinline__ void tc_mma_2sm_mxf8f6f4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                    uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p;\n\t"
      "}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}
// TMA tile load into this CTA's shared memory whose completion is counted on
// an mbarrier of either CTA of the pair (`bar_cluster`: shared::cluster address).
__device__ __forceinline__ void tma_load_2d_2sm(void *dst, const CUtensorMap *map, uint32_t bar_cluster, int32_t x,
                                                int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y)
      : "memory");
}

// ---------------------------------------------------------------- formats
// UE8M0 exponent of a non-negative finite float amax: the smallest integer e
// with Q * 2^e >= amax (Q = 448 for E4M3, 6 for E2M1), from the bits of amax,
// clamped to [-127, 127].  amax = 0 (and float subnormals, whose exponent is
// far below the clamp) give -127.
template <bool kE4M3>
__device__ __forceinline__ int ue8m0_exponent(float amax) {
  const uint32_t b = __float_as_uint(amax);
  const int exp_field = (int)((b >> 23) & 0xFF);
  if (exp_field == 0) return -127;
  const uint32_t man = b & 0x7FFFFFu;
  // amax = 1.m * 2^(E-127); with Q = 1.75 * 2^8 (E4M3) or 1.5 * 2^2 (E2M1).
  const int e = kE4M3 ? (exp_field - 127 - 8 + (man > 0x600000u ? 1 : 0))
                      : (exp_field - 127 - 2 + (man > 0x400000u ? 1 : 0));
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// 2^-e as a float for e in [-127, 127] (2^-127 is a float subnormal).
__device__ __forceinline__ float pow2_neg(int e) {
  const int be = 127 - e;
  return be >= 1 ? __uint_as_float((uint32_t)be << 23) : __uint_as_float(0x00400000u);
}

// Two floats -> two E4M3 codes (round to nearest even, saturating); `lo` ends
// up in the low byte.
__device__ __forceinline__ uint16_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two floats -> two E2M1 codes in one byte; `lo` in the low nibble.
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
      "cvt.u32.u8 %0, t;\n\t}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

// One lane's share of the activation cast: 8 consecutive BF16 values (one
// 16-byte load), four neighbouring lanes forming one 32-group.  All 32 lanes
// of the warp must call it together (`valid` false for lanes without data).
// Returns the 8 E4M3 codes; *scale_byte gets the group's UE8M0 byte.
__device__ __forceinline__ uint2 cast8_e4m3(const uint4 &v, bool valid, uint8_t *scale_byte) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  float f[8];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = bf16_bits_to_float(w[i] & 0xFFFFu);
    f[2 * i + 1] = bf16_bits_to_float(w[i] >> 16);
  }
  if (valid) {
#pragma unroll
    for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
  }
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  const int e = ue8m0_exponent<true>(amax);
  const float inv = pow2_neg(e);
  uint32_t c[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) c[j] = cvt_e4m3x2(f[2 * j] * inv, f[2 * j + 1] * inv);
  *scale_byte = (uint8_t)(e + 127);
  return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

}  // namespace mxq
