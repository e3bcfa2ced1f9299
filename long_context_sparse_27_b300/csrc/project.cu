// project.cu -- the decoder's global KV: the final encoder hidden state times
// a layer's projection, quantised straight into the FP4 main-KV cache.
//
// "Unlocking Extreme Context Scaling with DeepSeek-V4.1-Flash", Causal
// Encoder-Decoder (CED) Efficiency: the decoder derives its global KV cache
// from the final encoder hidden state using per-layer projections; the main
// KV is FP4 E2M1 ("Deployment and Infrastructure") with the per-32-element
// power-of-two block scale of the library's quantiser.
//
// The hidden dimension is split over the 8 CTAs of a thread-block cluster,
// so that a few rows (a decode step's new entries) still spread the weight
// stream over many SMs.  A CTA owns (64 rows, 64 output columns, 1/8 of the
// hidden features), 4 warps of 16 rows: its share is walked in steps of 32
// through a cp.async ring of h and w tiles, m16n8k16 bf16 MMAs accumulate in
// fp32, and the partial tile goes to shared memory.  After one cluster
// barrier CTA r sums rows 8r .. 8r + 7 of the 8 partials in rank order over
// distributed shared memory (a fixed order: the projection is
// deterministic), and quantises them: each 32-column block of a row lives in
// 8 threads (4 values each), whose amax is three shuffles away.  The codes
// are decided on the fp32 projection, which can also be written out.
#include "common.cuh"
#include "internal.h"

namespace csa2 {

namespace {

constexpr int kPjRows = 64;        // rows per CTA
constexpr int kPjCols = 64;        // output columns per CTA (two FP4 blocks)
constexpr int kPjK = 32;           // hidden features per step
constexpr int kPjThreads = 128;    // 4 warps x 16 rows
constexpr int kPjSplit = 8;        // CTAs of a cluster: shares of the hidden dimension
constexpr int kPjStride = kPjK + 8;  // padded smem row (bf16): conflict-free ldmatrix
constexpr int kPjTile = kPjRows * kPjStride;  // elements of one h (or w) tile
constexpr int kPjStages = 6;       // copies in flight: steps ks + 1 .. ks + 5 load during step ks
constexpr int kPjPartLd = kPjCols + 4;  // padded fp32 row of the partial tile
constexpr int kPjSmem = 2 * kPjStages * kPjTile * 2;  // the h and w rings (bytes)
static_assert(kPjRows * kPjPartLd * 4 <= kPjSmem, "the partial tile reuses the rings");
static_assert(kPjRows / kPjSplit * kPjCols / 4 == kPjThreads,
              "the reduction gives each thread 4 columns of one row");

__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
// wait until at most N of this thread's committed copy groups are pending
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// the address of the same shared-memory location in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t cluster_addr(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
__device__ __forceinline__ float4 ld_cluster_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

__global__ void __launch_bounds__(kPjThreads)
    project_fp4_kernel(const uint16_t* __restrict__ h, int64_t h_ld,
                       const uint16_t* __restrict__ w, int64_t w_ld, int64_t rows,
                       int32_t hidden, uint8_t* __restrict__ codes, int64_t codes_ld,
                       uint8_t* __restrict__ scales, int64_t scales_ld, float* __restrict__ out,
                       int64_t out_ld) {
  extern __shared__ __align__(16) uint16_t pj_smem[];
  uint16_t* sh = pj_smem;                          // [kPjStages][kPjTile]
  uint16_t* sw = pj_smem + kPjStages * kPjTile;    // [kPjStages][kPjTile]
  float* part = reinterpret_cast<float*>(pj_smem);  // [kPjRows][kPjPartLd], after the loop
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rank = (int)(blockIdx.x % kPjSplit);
  const int64_t r0 = (int64_t)(blockIdx.x / kPjSplit) * kPjRows;
  const int64_t c0 = (int64_t)blockIdx.y * kPjCols;
  // this CTA's steps of the hidden dimension
  const int steps_all = hidden / kPjK;
  const int per = (steps_all + kPjSplit - 1) / kPjSplit;
  const int ks0 = min(steps_all, rank * per);
  const int steps = min(steps_all, ks0 + per) - ks0;
  pdl_wait();

  // stage s of step ks: 64 rows x 32 features of h and of w (4 16-byte
  // pieces per row); rows past the end are zeros
  auto load = [&](int s, int ks) {
    const int64_t f0 = (int64_t)(ks0 + ks) * kPjK;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int i = tid + u * kPjThreads;  // 0 .. 255
      const int r = i >> 2, p = i & 3;
      uint16_t* dh = sh + s * kPjTile + r * kPjStride + p * 8;
      if (r0 + r < rows)
        cp_async16(dh, h + (r0 + r) * h_ld + f0 + p * 8);
      else
        *reinterpret_cast<uint4*>(dh) = make_uint4(0, 0, 0, 0);
      cp_async16(sw + s * kPjTile + r * kPjStride + p * 8, w + (c0 + r) * w_ld + f0 + p * 8);
    }
  };

  float acc[kPjCols / 8][4];
#pragma unroll
  for (int nt = 0; nt < kPjCols / 8; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
  // a ring of kPjStages stages, one copy group per step (empty groups past
  // the end keep the count uniform)
#pragma unroll
  for (int i = 0; i < kPjStages - 1; ++i) {
    if (i < steps) load(i, i);
    cp_async_commit();
  }
  for (int ks = 0; ks < steps; ++ks) {
    const int s = ks % kPjStages;
    cp_async_wait_group<kPjStages - 2>();  // step ks's group has landed
    __syncthreads();  // ... for every thread; every warp is done with step ks - 1's stage
    if (ks + kPjStages - 1 < steps) load((ks + kPjStages - 1) % kPjStages, ks + kPjStages - 1);
    cp_async_commit();
    const uint16_t* th = sh + s * kPjTile;
    const uint16_t* tw = sw + s * kPjTile;
#pragma unroll
    for (int kk = 0; kk < kPjK / 16; ++kk) {
      uint32_t a0, a1, a2, a3;
      ldmatrix_x4(smem_u32(th + (16 * warp + (lane & 15)) * kPjStride + kk * 16 + (lane >> 4) * 8),
                  a0, a1, a2, a3);
#pragma unroll
      for (int np = 0; np < kPjCols / 16; ++np) {
        // columns 16 np .. 16 np + 15 as two n8 tiles, k halves of 8
        const int n = 16 * np + (lane & 7) + ((lane >> 4) << 3);
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4(smem_u32(tw + n * kPjStride + kk * 16 + ((lane >> 3) & 1) * 8), b0, b1, b2,
                    b3);
        mma_bf16_16816(acc[2 * np], a0, a1, a2, a3, b0, b1);
        mma_bf16_16816(acc[2 * np + 1], a0, a1, a2, a3, b2, b3);
      }
    }
  }
  pdl_trigger();
  cp_async_wait_group<0>();
  __syncthreads();  // the rings are free: the partial tile takes their place

  // thread (g = lane / 4, t = lane % 4) holds rows g and g + 8 of the
  // warp's 16 at columns 8 nt + 2 t, + 1
  {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      float* prow = part + (16 * warp + g + 8 * half) * kPjPartLd + 2 * t;
#pragma unroll
      for (int nt = 0; nt < kPjCols / 8; ++nt)
        *reinterpret_cast<float2*>(prow + 8 * nt) =
            make_float2(acc[nt][2 * half], acc[nt][2 * half + 1]);
    }
  }
  cluster_arrive_release();
  cluster_wait_acquire();

  // rows 8 rank .. 8 rank + 7: thread tid takes row 8 rank + tid / 16,
  // columns 4 (tid % 16) .. + 3, summed over the cluster's partials in
  // rank order; lanes 8b .. 8b + 7 of a row hold its 32-column block b
  const int lr = kPjRows / kPjSplit * rank + tid / 16;
  const int col = 4 * (tid % 16);
  const int64_t row = r0 + lr;
  if (row < rows) {
    const uint32_t local = smem_u32(part + lr * kPjPartLd + col);
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int q = 0; q < kPjSplit; ++q) {
      const float4 x = ld_cluster_f4(cluster_addr(local, (uint32_t)q));
      v.x += x.x;
      v.y += x.y;
      v.z += x.z;
      v.w += x.w;
    }
    float amax = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
    // the 8 lanes of the block (whole rows per warp: every lane is here or
    // none of its 16-lane row group is, and the two groups are whole rows)
    const uint32_t grp = 0xFFu << (lane & 24);
    amax = fmaxf(amax, __shfl_xor_sync(grp, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(grp, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(grp, amax, 4));
    uint32_t sbyte = 0, b0 = 0, b1 = 0;
    if (amax > 0.f) {
      int e = floor_log2_pos(amax) - 2;
      e = max(-127, min(127, e));
      sbyte = (uint32_t)(e + 127);
      const float inv = exp2_int(-e);
      b0 = e2m1_encode(v.x * inv) | (e2m1_encode(v.y * inv) << 4);
      b1 = e2m1_encode(v.z * inv) | (e2m1_encode(v.w * inv) << 4);
    }
    uint8_t* crow = codes + row * codes_ld + (c0 + col) / 2;
    crow[0] = (uint8_t)b0;
    crow[1] = (uint8_t)b1;
    if ((tid & 7) == 0) scales[row * scales_ld + (c0 + col) / 32] = (uint8_t)sbyte;
    if (out) {
      float* orow = out + row * out_ld + c0 + col;
      *reinterpret_cast<float2*>(orow) = make_float2(v.x, v.y);
      *reinterpret_cast<float2*>(orow + 2) = make_float2(v.z, v.w);
    }
  }
  // no CTA leaves while another may still read its partial
  cluster_arrive_release();
  cluster_wait_acquire();
}

std::atomic<uint64_t> g_project_attr{0};  // devices on which the kernel's attributes are set

// ---------------------------------------------------------------------------
// few rows (at most 16, a decode step's new entries): the weight stream is
// the whole cost, so every CTA issues all of its loads at once
// ---------------------------------------------------------------------------
//
// A CTA owns (16 rows, one 32-column FP4 block, 1/8 of the hidden features);
// the 8 CTAs of a cluster split the hidden dimension, so d / 32 x 8 CTAs
// (128 for d = 512) stream the weights.  The CTA's h and w slices arrive in
// one round of cp.async copies; its 4 warps take a quarter of the features
// each (m16n8k16 bf16 MMAs, fp32 accumulators), their partials are summed in
// shared memory, and after a cluster barrier CTA r sums rows 2r, 2r + 1 of
// the 8 CTA partials in rank order over distributed shared memory (a fixed
// order) and quantises them like the other projection kernels.

constexpr int kPsRows = 16;
constexpr int kPsCols = 32;         // one FP4 block
constexpr int kPsThreads = 128;     // 4 warps
constexpr int kPsSplit = 8;         // CTAs of a cluster
constexpr int kPsWorkers = kPsSplit * kPsThreads / 32;  // warps over the hidden dimension
constexpr int kPsPartLd = kPsCols + 4;
constexpr int kPsMaxFeatures = 2048;  // per CTA: the slices fit in shared memory
constexpr int kPsMaxHidden = kPsSplit * kPsMaxFeatures;

// features of the CTA share / of one warp (multiples of 16)
__host__ __device__ constexpr int ps_warp_steps(int hidden) {
  return (hidden / 16 + kPsWorkers - 1) / kPsWorkers;
}
__host__ __device__ constexpr int ps_stride(int hidden) {  // padded smem row (bf16)
  return 4 * 16 * ps_warp_steps(hidden) + 8;
}
__host__ __device__ constexpr int ps_smem(int hidden) {
  return (kPsRows + kPsCols) * ps_stride(hidden) * 2 +
         (kPsThreads / 32 + 1) * kPsRows * kPsPartLd * 4;
}

__global__ void __launch_bounds__(kPsThreads)
    project_few_kernel(const uint16_t* __restrict__ h, int64_t h_ld,
                       const uint16_t* __restrict__ w, int64_t w_ld, int32_t rows,
                       int32_t hidden, uint8_t* __restrict__ codes, int64_t codes_ld,
                       uint8_t* __restrict__ scales, int64_t scales_ld, float* __restrict__ out,
                       int64_t out_ld) {
  extern __shared__ __align__(16) uint16_t ps_smem_raw[];
  const int stride = ps_stride(hidden);
  uint16_t* sh = ps_smem_raw;                    // [16][stride]
  uint16_t* sw = ps_smem_raw + kPsRows * stride;  // [32][stride]
  // [4 warps + the CTA sum][16][kPsPartLd]
  float* part = reinterpret_cast<float*>(ps_smem_raw + (kPsRows + kPsCols) * stride);
  float* cpart = part + (kPsThreads / 32) * kPsRows * kPsPartLd;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rank = (int)(blockIdx.x % kPsSplit);
  const int64_t c0 = (int64_t)blockIdx.y * kPsCols;
  const int wsteps = ps_warp_steps(hidden);
  const int ksteps = hidden / 16;
  // the CTA's features [f0, f1): warps rank * 4 .. rank * 4 + 3 of the split
  const int s0 = min(ksteps, rank * 4 * wsteps), s1 = min(ksteps, (rank + 1) * 4 * wsteps);
  const int f0 = 16 * s0, nf = 16 * (s1 - s0);
  pdl_wait();

  // every copy of the CTA in flight at once: 8-element pieces of the 16 h
  // rows (zeros past the last row) and of the 32 w rows
  const int pieces = nf / 8;
  for (int i = tid; i < (kPsRows + kPsCols) * pieces; i += kPsThreads) {
    const int r = i / pieces, p = i % pieces;
    if (r < kPsRows) {
      uint16_t* d = sh + r * stride + p * 8;
      if (r < rows)
        cp_async16(d, h + (int64_t)r * h_ld + f0 + p * 8);
      else
        *reinterpret_cast<uint4*>(d) = make_uint4(0, 0, 0, 0);
    } else {
      cp_async16(sw + (r - kPsRows) * stride + p * 8, w + (c0 + r - kPsRows) * w_ld + f0 + p * 8);
    }
  }
  cp_async_wait_all();
  __syncthreads();

  // warp: k-steps [ws0, ws1) of the CTA's share
  float acc[kPsCols / 8][4];
#pragma unroll
  for (int nt = 0; nt < kPsCols / 8; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
  const int ws0 = min(s1 - s0, warp * wsteps), ws1 = min(s1 - s0, (warp + 1) * wsteps);
  for (int kk = ws0; kk < ws1; ++kk) {
    uint32_t a0, a1, a2, a3;
    ldmatrix_x4(smem_u32(sh + (lane & 15) * stride + kk * 16 + (lane >> 4) * 8), a0, a1, a2, a3);
#pragma unroll
    for (int np = 0; np < kPsCols / 16; ++np) {
      const int n = 16 * np + (lane & 7) + ((lane >> 4) << 3);
      uint32_t b0, b1, b2, b3;
      ldmatrix_x4(smem_u32(sw + n * stride + kk * 16 + ((lane >> 3) & 1) * 8), b0, b1, b2, b3);
      mma_bf16_16816(acc[2 * np], a0, a1, a2, a3, b0, b1);
      mma_bf16_16816(acc[2 * np + 1], a0, a1, a2, a3, b2, b3);
    }
  }
  pdl_trigger();
  {  // thread (g = lane / 4, t = lane % 4): rows g, g + 8, columns 8 nt + 2 t, + 1
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      float* prow = part + (warp * kPsRows + g + 8 * half) * kPsPartLd + 2 * t;
#pragma unroll
      for (int nt = 0; nt < kPsCols / 8; ++nt)
        *reinterpret_cast<float2*>(prow + 8 * nt) =
            make_float2(acc[nt][2 * half], acc[nt][2 * half + 1]);
    }
  }
  __syncthreads();
  // the CTA's partial: the 4 warps' in warp order
  for (int i = tid; i < kPsRows * kPsCols; i += kPsThreads) {
    const int r = i / kPsCols, c = i % kPsCols;
    float v = 0.f;
#pragma unroll
    for (int q = 0; q < kPsThreads / 32; ++q) v += part[(q * kPsRows + r) * kPsPartLd + c];
    cpart[r * kPsPartLd + c] = v;
  }
  cluster_arrive_release();
  cluster_wait_acquire();

  // rows 2 rank, 2 rank + 1: thread tid < 16 takes row 2 rank + tid / 8,
  // columns 4 (tid % 8) .. + 3 (the 8 lanes of a row hold its block)
  if (tid < 2 * 8) {
    const int lr = 2 * rank + tid / 8, col = 4 * (tid % 8);
    if (lr < rows) {
      const uint32_t local = smem_u32(cpart + lr * kPsPartLd + col);
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int q = 0; q < kPsSplit; ++q) {
        const float4 x = ld_cluster_f4(cluster_addr(local, (uint32_t)q));
        v.x += x.x;
        v.y += x.y;
        v.z += x.z;
        v.w += x.w;
      }
      float amax = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
      const uint32_t grp = 0xFFu << (lane & 8);  // the 8 lanes of the row (both rows or none)
      amax = fmaxf(amax, __shfl_xor_sync(grp, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(grp, amax, 2));
      amax = fmaxf(amax, __shfl_xor_sync(grp, amax, 4));
      uint32_t sbyte = 0, b0 = 0, b1 = 0;
      if (amax > 0.f) {
        int e = floor_log2_pos(amax) - 2;
        e = max(-127, min(127, e));
        sbyte = (uint32_t)(e + 127);
        const float inv = exp2_int(-e);
        b0 = e2m1_encode(v.x * inv) | (e2m1_encode(v.y * inv) << 4);
        b1 = e2m1_encode(v.z * inv) | (e2m1_encode(v.w * inv) << 4);
      }
      uint8_t* crow = codes + (int64_t)lr * codes_ld + (c0 + col) / 2;
      crow[0] = (uint8_t)b0;
      crow[1] = (uint8_t)b1;
      if ((tid & 7) == 0) scales[(int64_t)lr * scales_ld + c0 / 32] = (uint8_t)sbyte;
      if (out) {
        float* orow = out + (int64_t)lr * out_ld + c0 + col;
        *reinterpret_cast<float2*>(orow) = make_float2(v.x, v.y);
        *reinterpret_cast<float2*>(orow + 2) = make_float2(v.z, v.w);
      }
    }
  }
  // no CTA leaves while another may still read its partial
  cluster_arrive_release();
  cluster_wait_acquire();
}

std::atomic<uint64_t> g_project_few_attr{0};

// ---------------------------------------------------------------------------
// tensor-core path (from 64 rows): tcgen05 bf16 MMAs, accumulators in TMEM
// ---------------------------------------------------------------------------
//
// A CTA owns (128 rows, N = 128 output columns (64 where d is not a multiple
// of 128), 1/4 of the hidden features); the 4 CTAs of a cluster split the
// hidden dimension.  Warp 0 streams 128 x 64 tiles of h and N x 64 tiles of
// w by TMA (128-byte swizzle) through a 4-stage mbarrier ring, warp 1 issues
// tcgen05.mma.kind::f16 (M = 128, N, K = 16; four per stage) into one TMEM
// accumulator, and warps 2 .. 5
// (one TMEM lane quarter each) move the accumulator to a shared-memory
// partial tile.  After one cluster barrier CTA r sums rows 32 r .. 32 r + 31
// of the 4 partials in rank order over distributed shared memory and
// quantises them, one thread per (row, 32-column block).  Every wait is
// bounded; a wait that gives up sets CSA2_DEVFLAG_TIMEOUT and the CTA's
// abort flag, and the CTA still takes part in both cluster barriers.
constexpr int kTcM = 128;                  // rows per CTA (MMA M, TMEM lanes)
constexpr int kTcK = 64;                   // features per stage: 128-byte rows
constexpr int kTcStages = 4;
constexpr int kTcSplit = 4;                // CTAs of a cluster: shares of the hidden dimension
constexpr int kTcThreads = 192;            // producer, MMA issuer, 4 epilogue warps
constexpr int kTcATile = kTcM * kTcK * 2;  // 16 KB

// N output columns per CTA (MMA N): 128 where d allows (each h tile then
// serves twice the columns), else 64 (two CTAs per SM)
template <int N>
struct TcPj {
  static constexpr int BTile = N * kTcK * 2;           // 8 or 16 KB
  static constexpr int PartLd = N + 4;                 // padded fp32 row of the partial tile
  static constexpr int OffB = kTcStages * kTcATile;
  static constexpr int OffBar = OffB + kTcStages * BTile;
  static constexpr int Smem = OffBar + 256;            // barriers, TMEM slot, abort flag
  static constexpr int SmemAlloc = Smem + 1024;        // 1024-byte alignment of the tiles
  static constexpr int CtasPerSm = N == 64 ? 2 : 1;
  static_assert(kTcM * PartLd * 4 <= OffBar, "the partial tile reuses the rings");
  static_assert((kTcM / kTcSplit) * (N / 32) <= kTcThreads, "one thread per (row, block)");
  static_assert(CtasPerSm * (SmemAlloc + 1024) <= 228 * 1024, "CTAs per SM");
};

template <int N>
__global__ void __launch_bounds__(kTcThreads, TcPj<N>::CtasPerSm)
    project_tc_kernel(const __grid_constant__ CUtensorMap hmap,
                      const __grid_constant__ CUtensorMap wmap, int64_t rows, int32_t hidden,
                      uint8_t* __restrict__ codes, int64_t codes_ld,
                      uint8_t* __restrict__ scales, int64_t scales_ld, float* __restrict__ out,
                      int64_t out_ld, int32_t* dev_status, uint64_t wait_ns) {
  using C = TcPj<N>;
  extern __shared__ uint8_t tc_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(tc_raw) + 1023) & ~(uintptr_t)1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OffBar);
  uint64_t* empty = full + kTcStages;
  uint64_t* accb = empty + kTcStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accb + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* part = reinterpret_cast<float*>(smem);  // [kTcM][C::PartLd], after the main loop

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rank = (int)(blockIdx.x % kTcSplit);
  const int64_t r0 = (int64_t)(blockIdx.x / kTcSplit) * kTcM;
  const int c0 = (int)blockIdx.y * N;
  const int nkb_all = hidden / kTcK;
  const int per = (nkb_all + kTcSplit - 1) / kTcSplit;
  const int kb0 = min(nkb_all, rank * per);
  const int nkb = min(nkb_all, kb0 + per) - kb0;

  if (tid == 0) {
    for (int i = 0; i < kTcStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(accb, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&hmap);
    tma_prefetch_desc(&wmap);
  }
  if (warp == 1) tmem_alloc(tmem_slot, N);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0 && nkb > 0) {
      const uint64_t pol = l2_policy_evict_normal();  // h and w tiles are read by several CTAs
      int issued = 0;
      for (int i = 0; i < nkb; ++i) {
        const int s = i % kTcStages;
        if (!mbar_wait(&empty[s], (uint32_t)(((i / kTcStages) & 1) ^ 1), abort_flag, dev_status,
                       wait_ns))
          break;
        mbar_arrive_expect_tx(&full[s], kTcATile + C::BTile);
        const int32_t x = (kb0 + i) * kTcK;
        tma_load_2d(&hmap, &full[s], smem + s * kTcATile, x, (int32_t)r0, pol);
        tma_load_2d(&wmap, &full[s], smem + C::OffB + s * C::BTile, x, c0, pol);
        ++issued;
      }
      // on an abort, let the copies in flight land before shared memory is reused
      int dummy = 0;
      for (int u = issued > kTcStages ? issued - kTcStages : 0; u < issued; ++u)
        mbar_wait(&full[u % kTcStages], (uint32_t)((u / kTcStages) & 1), &dummy, nullptr,
                  wait_ns);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0 && nkb > 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(kTcM, N);
      for (int i = 0; i < nkb; ++i) {
        const int s = i % kTcStages;
        if (!mbar_wait(&full[s], (uint32_t)((i / kTcStages) & 1), abort_flag, dev_status, wait_ns))
          break;
        tc_fence_after();
        const uint64_t a = sdesc_k_sw128(smem_u32(smem + s * kTcATile));
        const uint64_t b = sdesc_k_sw128(smem_u32(smem + C::OffB + s * C::BTile));
#pragma unroll
        for (int kk = 0; kk < kTcK / 16; ++kk)  // K = 16 bf16 = 32 bytes = 2 descriptor units
          tc_mma_bf16(tmem_base, a + 2 * kk, b + 2 * kk, idesc, (i > 0 || kk > 0) ? 1u : 0u);
        tc_commit(&empty[s]);
      }
      tc_commit(accb);  // every MMA issued has completed
    }
  } else {
    // ---------------- accumulator -> shared-memory partial ----------------
    const int quarter = warp & 3;  // TMEM lanes 32 quarter .. (warp % 4 rule)
    const int row = 32 * quarter + lane;
    bool got = false;
    if (nkb > 0) got = __all_sync(0xffffffffu, mbar_wait(accb, 0, abort_flag, dev_status, wait_ns));
    if (got) tc_fence_after();
    // the rings are free once the accumulator is complete (every stage's
    // loads landed and its MMAs read it)
    asm volatile("bar.sync 1, %0;" ::"n"(4 * 32) : "memory");
    float* prow = part + row * C::PartLd;
#pragma unroll 1
    for (int c = 0; c < N; c += 32) {  // 32 columns at a time
      float v[32];
      if (got) {
        tmem_ld32(tmem_base + ((uint32_t)(32 * quarter) << 16) + c, v);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0.f;
      }
#pragma unroll
      for (int i = 0; i < 32; i += 4)
        *reinterpret_cast<float4*>(prow + c + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
    }
  }
  // the producer's copies have landed (or were never issued) before the
  // partial tile overwrites the rings: the epilogue wrote only after the
  // accumulator barrier, which follows every stage's full barrier
  tc_fence_before();
  __syncthreads();
  pdl_trigger();
  cluster_arrive_release();
  cluster_wait_acquire();

  // ---- rows 32 rank .. 32 rank + 31: one thread per (row, 32-column block)
  if (tid < (kTcM / kTcSplit) * (N / 32)) {
    const int lr = (kTcM / kTcSplit) * rank + tid / (N / 32);
    const int blk = tid % (N / 32);
    const int64_t grow = r0 + lr;
    if (grow < rows) {
      float x[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) x[i] = 0.f;
      const uint32_t local = smem_u32(part + lr * C::PartLd + 32 * blk);
#pragma unroll
      for (int q = 0; q < kTcSplit; ++q) {
        const uint32_t ra = cluster_addr(local, (uint32_t)q);
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          const float4 t = ld_cluster_f4(ra + 4 * i);
          x[i] += t.x;
          x[i + 1] += t.y;
          x[i + 2] += t.z;
          x[i + 3] += t.w;
        }
      }
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(x[i]));
      uint32_t sbyte = 0, pk[4];
#pragma unroll
      for (int g = 0; g < 4; ++g) pk[g] = fp4_encode8(x + 8 * g, amax, sbyte);
      const int64_t col = c0 + 32 * blk;
      *reinterpret_cast<uint4*>(codes + grow * codes_ld + col / 2) =
          make_uint4(pk[0], pk[1], pk[2], pk[3]);
      scales[grow * scales_ld + col / 32] = (uint8_t)sbyte;
      if (out) {
        float* orow = out + grow * out_ld + col;
#pragma unroll
        for (int i = 0; i < 32; i += 2)
          *reinterpret_cast<float2*>(orow + i) = make_float2(x[i], x[i + 1]);
      }
    }
  }
  // no CTA leaves (or frees its tensor memory) while another may still read its partial
  cluster_arrive_release();
  cluster_wait_acquire();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, N);
  }
}

std::atomic<uint64_t> g_project_tc_attr[2] = {{0}, {0}};  // N = 64, 128


template <int N>
csa2_status launch_project_tc(const csa2_project_args& a, cudaStream_t s) {
  using C = TcPj<N>;
  EncodeTiledFn enc = tensor_map_encoder();
  if (!enc) return cuda_fail(cudaErrorNotSupported);
  CUtensorMap hmap, wmap;
  {
    cuuint64_t dims[2] = {(cuuint64_t)a.hidden, (cuuint64_t)a.rows};
    cuuint64_t strides[1] = {(cuuint64_t)a.h_ld * 2};
    cuuint32_t box[2] = {kTcK, kTcM};
    cuuint32_t es[2] = {1, 1};
    if (enc(&hmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.h), dims, strides,
            box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return CSA2_ERR_INVALID_ARG;
  }
  {
    cuuint64_t dims[2] = {(cuuint64_t)a.hidden, (cuuint64_t)a.d};
    cuuint64_t strides[1] = {(cuuint64_t)a.w_ld * 2};
    cuuint32_t box[2] = {kTcK, N};
    cuuint32_t es[2] = {1, 1};
    if (enc(&wmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.w), dims, strides,
            box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return CSA2_ERR_INVALID_ARG;
  }
  cudaError_t e = once_per_device(g_project_tc_attr[N == 128 ? 1 : 0], [] {
    return cudaFuncSetAttribute(project_tc_kernel<N>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                C::SmemAlloc);
  });
  if (e != cudaSuccess) return cuda_fail(e);
  const int64_t row_tiles = (a.rows + kTcM - 1) / kTcM;
  if (row_tiles * kTcSplit > 0x7FFFFFFF) return CSA2_ERR_UNSUPPORTED;
  const dim3 grid((unsigned)(row_tiles * kTcSplit), (unsigned)(a.d / N));
  return launch_kernel(project_tc_kernel<N>, grid, dim3(kTcThreads), (size_t)C::SmemAlloc, s,
                       kTcSplit, hmap, wmap, a.rows, a.hidden, a.codes, a.codes_ld, a.scales,
                       a.scales_ld, a.out, a.out_ld, a.dev_status, wait_limit_ns());
}

}  // namespace

csa2_status launch_project_fp4(const csa2_project_args& a, cudaStream_t s) {
  if (a.rows == 0) return CSA2_OK;
  const bool tc = a.rows >= 64 && a.hidden % (kTcK * kTcSplit) == 0 &&
                  (reinterpret_cast<uintptr_t>(a.codes) & 15) == 0 && a.codes_ld % 16 == 0;
  if (tc) return a.d % 128 == 0 ? launch_project_tc<128>(a, s) : launch_project_tc<64>(a, s);
  if (a.rows <= kPsRows && a.hidden <= kPsMaxHidden) {
    cudaError_t e = once_per_device(g_project_few_attr, [] {
      return cudaFuncSetAttribute(project_few_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  ps_smem(kPsMaxHidden));
    });
    if (e != cudaSuccess) return cuda_fail(e);
    const dim3 grid((unsigned)kPsSplit, (unsigned)(a.d / kPsCols));
    return launch_kernel(project_few_kernel, grid, dim3(kPsThreads), (size_t)ps_smem(a.hidden), s,
                         kPsSplit, static_cast<const uint16_t*>(a.h), a.h_ld,
                         static_cast<const uint16_t*>(a.w), a.w_ld, (int32_t)a.rows, a.hidden,
                         a.codes, a.codes_ld, a.scales, a.scales_ld, a.out, a.out_ld);
  }
  cudaError_t e = once_per_device(g_project_attr, [] {
    return cudaFuncSetAttribute(project_fp4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kPjSmem);
  });
  if (e != cudaSuccess) return cuda_fail(e);
  const int64_t row_tiles = (a.rows + kPjRows - 1) / kPjRows;
  if (row_tiles * kPjSplit > 0x7FFFFFFF) return CSA2_ERR_UNSUPPORTED;
  const dim3 grid((unsigned)(row_tiles * kPjSplit), (unsigned)(a.d / kPjCols));
  return launch_kernel(project_fp4_kernel, grid, dim3(kPjThreads), (size_t)kPjSmem, s, kPjSplit,
                       static_cast<const uint16_t*>(a.h), a.h_ld,
                       static_cast<const uint16_t*>(a.w), a.w_ld, a.rows, a.hidden, a.codes,
                       a.codes_ld, a.scales, a.scales_ld, a.out, a.out_ld);
}

}  // namespace csa2
