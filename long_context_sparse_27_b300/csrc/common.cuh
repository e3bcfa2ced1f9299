// common.cuh -- device helpers shared by the CSA2 kernels (sm_103a).
//
// Number formats (E2M1 / UE8M0 / E4M3), bounded mbarrier waits, TMA and
// tcgen05 wrappers written as inline PTX.  Nothing here allocates.
#pragma once

#include <cuda.h>  // CUtensorMap (type only; the driver entry point is fetched at run time)
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/csa2.h"

namespace csa2 {

// ---------------------------------------------------------------------------
// scalar formats
// ---------------------------------------------------------------------------

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) {
  return __uint_as_float(b << 16);
}

// floor(log2(a)) for finite a > 0, exact (normal and subnormal floats).
__device__ __forceinline__ int floor_log2_pos(float a) {
  uint32_t u = __float_as_uint(a);
  int ef = (int)((u >> 23) & 0xFF);
  if (ef != 0) return ef - 127;
  return (31 - __clz(u & 0x7FFFFF)) - 149;  // a = m * 2^-149
}

// 2^e as a float for e in [-149, 127].
__device__ __forceinline__ float exp2_int(int e) {
  if (e >= -126) return __uint_as_float((uint32_t)(e + 127) << 23);
  return __uint_as_float(1u << (e + 149));
}

// E2M1 code of y: nearest of {0, .5, 1, 1.5, 2, 3, 4, 6}, ties to the even
// code, |y| > 6 -> 6, sign bit 3 copied from y (so -0 and negative values
// that round to zero give 8).  Each comparison decides one step of the
// grid; ">" at a midpoint whose lower neighbour has the even code, ">="
// where the upper neighbour has it.
__device__ __forceinline__ uint32_t e2m1_encode(float y) {
  float a = fabsf(y);
  uint32_t c = (uint32_t)(a > 0.25f) + (uint32_t)(a >= 0.75f) + (uint32_t)(a > 1.25f) +
               (uint32_t)(a >= 1.75f) + (uint32_t)(a > 2.5f) + (uint32_t)(a >= 3.5f) +
               (uint32_t)(a > 5.0f);
  return c | ((__float_as_uint(y) >> 31) << 3);
}

// E2M1 value of a 4-bit code: exponent field ef = bits 2..1 (bias 1),
// mantissa bit 0; ef = 0 is subnormal (0 or 0.5).  Built as float bits.
__device__ __forceinline__ float e2m1_value(uint32_t c) {
  uint32_t ef = (c >> 1) & 3u, m = c & 1u;
  uint32_t bits = ef ? (((ef + 126u) << 23) | (m << 22)) : (m ? 0x3F000000u : 0u);
  return __uint_as_float(bits | ((c & 8u) << 28));
}

// UE8M0 scale byte -> 2^(s - 127) as a float (s = 0 gives the subnormal 2^-127).
__device__ __forceinline__ float ue8m0_value(uint32_t s) { return exp2_int((int)s - 127); }

// Exponent e of the indexer-Q scale 2^e for a head whose largest magnitude
// is amax > 0: the smallest e (>= -126) with amax / 2^e <= 448 = 1.75 * 2^8.
// With amax = m 2^E (m in [1, 2)), e = E - 8 when m <= 1.75, else E - 7.
__device__ __forceinline__ int index_q_exponent(float amax) {
  const int E = floor_log2_pos(amax);
  // fraction bits of m, normalising a subnormal amax first
  const uint32_t u = __float_as_uint(amax);
  uint32_t frac = u & 0x7FFFFFu;
  if (((u >> 23) & 0xFFu) == 0) frac = (frac << (__clz(frac) - 8)) & 0x7FFFFFu;
  const int e = (frac <= 0x600000u) ? E - 8 : E - 7;  // 0x600000: fraction of 1.75
  return e < -126 ? -126 : e;
}

// E4M3 with round-to-nearest-even and saturation to +-448.
__device__ __forceinline__ uint32_t e4m3_encode(float x) {
  return (uint32_t)__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
}

// Eight bf16 values (a 16-byte load) as floats, element i of the load in v[i].
__device__ __forceinline__ void bf16x8_to_float(uint4 raw, float v[8]) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = bf16_bits_to_float(w[i] & 0xFFFFu);
    v[2 * i + 1] = bf16_bits_to_float(w[i] >> 16);
  }
}

// a1: eight consecutive elements of a 32-element block whose largest
// magnitude is amax -> eight E2M1 codes (element i in nibble i) and the
// block's UE8M0 scale byte: X = 2^(floor(log2 amax) - 2), exponent clamped
// to [-127, 127]; an all-zero block has scale byte 0 and zero codes.
__device__ __forceinline__ uint32_t fp4_encode8(const float v[8], float amax, uint32_t& sbyte) {
  uint32_t packed = 0;
  sbyte = 0;
  if (amax > 0.f) {
    int e = floor_log2_pos(amax) - 2;
    e = max(-127, min(127, e));
    sbyte = (uint32_t)(e + 127);
    const float inv = exp2_int(-e);  // -e in [-127, 127]: exact power of two
#pragma unroll
    for (int i = 0; i < 8; ++i) packed |= e2m1_encode(v[i] * inv) << (4 * i);
  }
  return packed;
}

// a1, indexer keys: eight bf16 values (a 16-byte load) -> eight E4M3 bytes,
// element i in byte i.
__device__ __forceinline__ uint2 e4m3_encode8(uint4 raw) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
  uint32_t lo = 0, hi = 0;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    lo |= e4m3_encode(bf16_bits_to_float(w[i] & 0xFFFFu)) << (16 * i);
    lo |= e4m3_encode(bf16_bits_to_float(w[i] >> 16)) << (16 * i + 8);
    hi |= e4m3_encode(bf16_bits_to_float(w[i + 2] & 0xFFFFu)) << (16 * i);
    hi |= e4m3_encode(bf16_bits_to_float(w[i + 2] >> 16)) << (16 * i + 8);
  }
  return make_uint2(lo, hi);
}

// ---------------------------------------------------------------------------
// top-k keys and histograms
// ---------------------------------------------------------------------------

// Order-preserving 32-bit key of a score: a larger float gives a larger key;
// -0 maps like +0 (the two compare equal).
__device__ __forceinline__ uint32_t score_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

constexpr int kTopkBins = 4096;  // first-level digit: the key's top 12 bits
// A row's level-1 histogram in global memory: the 4096 fine bins, then 64
// coarse bins (the key's top 6 bits; coarse bin c = fine bins 64c .. 64c+63),
// so that a reader can find the threshold bin from 128 counts.
constexpr int kTopkCoarse = 64;
constexpr int kTopkHistStride = kTopkBins + kTopkCoarse;

// ---------------------------------------------------------------------------
// programmatic dependent launch
// ---------------------------------------------------------------------------

// Every kernel of this library is launched with programmatic stream
// serialisation.  Each kernel waits for the previous kernel on the stream to
// finish and its writes to be visible (pdl_wait) before its first global-
// memory access, and lets the next kernel launch once its own CTAs are
// finishing (pdl_trigger near its end; a CTA that exits counts as having
// triggered).  The next kernel's launch and prologue (shared-memory setup,
// barrier init, tensor-memory allocation) thereby overlap this kernel's
// drain; the data order is the stream order.  Triggering at kernel entry
// was measured slower: the early CTAs of the next kernel took SM resources
// from the running one.  Both are no-ops for a launch without the attribute.
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------------------
// device status
// ---------------------------------------------------------------------------

__device__ __forceinline__ void raise_flag(int32_t* dev_status, int32_t flag) {
  if (dev_status) atomicOr(dev_status, flag);
}

// Pool row of entry j of sequence b in a paged cache (csa2_pages), or -1
// with CSA2_DEVFLAG_BOUNDS raised when the block table names a page outside
// [0, num_pages).
__device__ __forceinline__ int64_t paged_row(const csa2_pages& pg, int64_t b, int64_t j,
                                             int32_t* dev_status) {
  // entries fit 32 bits (indices are int32): 32-bit division
  const uint32_t jj = (uint32_t)j, pr = (uint32_t)pg.page_rows;
  const uint32_t pi = jj / pr;
  const int32_t page = pg.block_table[b * pg.bt_ld + pi];
  if (page < 0 || page >= pg.num_pages) {
    raise_flag(dev_status, CSA2_DEVFLAG_BOUNDS);
    return -1;
  }
  return (int64_t)page * pg.page_rows + (jj - pi * pr);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------------------
// shared memory / mbarrier
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of an mbarrier to complete, giving up after
// `limit_ns` of wall time or as soon as *abort is set by another warp.
// On a time-out it sets *abort and the TIMEOUT bit of dev_status.
// Returns true if the phase completed.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          int32_t* dev_status, uint64_t limit_ns) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(a, parity)) return true;
    if ((it & 63) == 0) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > limit_ns) {
        *abort = 1;
        raise_flag(dev_status, CSA2_DEVFLAG_TIMEOUT);
        return false;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// TMA (bulk tensor copies into shared memory, completion on an mbarrier)
// ---------------------------------------------------------------------------

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void tma_load_2d(const CUtensorMap* map, uint64_t* bar, void* dst,
                                            int32_t x, int32_t y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(const CUtensorMap* map, uint64_t* bar, void* dst,
                                            int32_t x, int32_t y, int32_t z, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z),
      "l"(policy)
      : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05 (5th-generation tensor cores, accumulators in tensor memory)
// ---------------------------------------------------------------------------

// Allocate `ncols` (power of two >= 32) TMEM columns; the base address is
// written to shared memory at `slot`.  Whole warp.
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor for a K-major operand stored in the
// 128-byte swizzle layout written by TMA (CU_TENSOR_MAP_SWIZZLE_128B):
// rows of 128 bytes, 8-row groups 1024 bytes apart.  Fields: start
// address >> 4 (bits 0-13), leading-byte offset >> 4 (16-29, unused for
// this layout, 1), stride-byte offset >> 4 (32-45), fixed 0b001 (46-48),
// base offset 0 (49-51, tiles are 1024-byte aligned), swizzle mode 2 =
// 128-byte (61-63).
__device__ __forceinline__ uint64_t sdesc_k_sw128(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor, kind::f8f6f4 with E4M3 A and B, f32 accumulate,
// both operands K-major: D format (bits 4-5) = 1, A / B format (7-9 /
// 10-12) = 0, transpose bits 15 / 16 = 0, N >> 3 at 17-22, M >> 4 at 24-28.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Instruction descriptor, kind::f16 with BF16 A and B (format 1), f32
// accumulate, both operands K-major: D format (bits 4-5) = 1, A / B format
// (7-9 / 10-12) = 1, N >> 3 at 17-22, M >> 4 at 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tc_mma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every tcgen05 operation issued so far by this
// thread has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// 32 consecutive 32-bit TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
      "[%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// (d0, d1) += (a0, a1) * (b0, b1): two fp32 fused multiply-adds, each
// rounded once, in one packed instruction.
__device__ __forceinline__ void ffma2(float& d0, float& d1, float a0, float a1, float b0,
                                      float b1) {
  uint64_t d, a, b;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(d0), "f"(d1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(a0), "f"(a1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(b) : "f"(b0), "f"(b1));
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(d) : "l"(a), "l"(b));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(d0), "=f"(d1) : "l"(d));
}

// 16 lanes x 64 consecutive 32-bit columns from lane (taddr >> 16): thread
// t holds lanes t / 4 and t / 4 + 8, columns 8 k + 2 (t % 4) and the one
// after it, as v[4 k + 2 i + b] = (lane t / 4 + 8 i, column 8 k + 2 (t % 4) + b).
__device__ __forceinline__ void tmem_ld16x256b_x8(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x8.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
      "[%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Generic-proxy writes to shared memory (st.shared, cp.async) made visible
// to the async proxy (tcgen05.mma operand reads); each writing thread
// executes it before the barrier that precedes the MMA issue.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Thread-block-cluster barrier in two halves: arrive (release: this
// thread's earlier writes, global ones included, are ordered before) and
// wait (acquire).  Every thread of every CTA of the cluster executes both.
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------------------
// cp.async (16-byte global -> shared copies, completion per thread)
// ---------------------------------------------------------------------------

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)),
               "l"(gmem_src)
               : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// ---------------------------------------------------------------------------
// warp-level bf16 MMA (m16n8k16) used by the attention kernel
// ---------------------------------------------------------------------------

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                            uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                                  uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma_bf16_16816(float* c, uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Eight E2M1 codes (4 bytes; element 2i in the low nibble of byte i), each
// times the power of two held in both halves of sc2, as eight bf16 in four
// 32-bit words (element 2i in the low half).  Byte-permute table lookups:
// the unscaled magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6} have bf16 high bytes
// {00,3F,3F,3F,40,40,40,40} and low bytes {00,00,80,C0,00,40,80,C0}; the
// code's sign bit becomes bit 15.  The scale multiply is exact when every
// product is a normal bf16 (the caller checks the scale's range).
__device__ __forceinline__ void e2m1x8_to_bf16(uint32_t code4, __nv_bfloat162 sc2,
                                               uint32_t out[4]) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t c16 = (code4 >> (16 * h)) & 0xFFFFu;  // four codes
    const uint32_t mag = c16 & 0x7777u;
    const uint32_t lo = prmt(0xC0800000u, 0xC0804000u, mag);
    uint32_t hi = prmt(0x3F3F3F00u, 0x40404040u, mag);
    // selector bit 3 (the code's sign) makes prmt replicate the selected
    // byte's top bit: 0x7F -> 0x00 for negative codes, 0x7F for positive
    const uint32_t t = prmt(0x7F7F7F7Fu, 0x7F7F7F7Fu, c16);
    hi |= ((t + 0x01010101u) & 0x80808080u) ^ 0x80808080u;
    const uint32_t w0 = prmt(lo, hi, 0x5140u);  // elements 4h, 4h+1
    const uint32_t w1 = prmt(lo, hi, 0x7362u);  // elements 4h+2, 4h+3
    const __nv_bfloat162 p0 = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&w0), sc2);
    const __nv_bfloat162 p1 = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&w1), sc2);
    out[2 * h] = *reinterpret_cast<const uint32_t*>(&p0);
    out[2 * h + 1] = *reinterpret_cast<const uint32_t*>(&p1);
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // .x = lo (low half), .y = hi
  return *reinterpret_cast<uint32_t*>(&v);
}

}  // namespace csa2
