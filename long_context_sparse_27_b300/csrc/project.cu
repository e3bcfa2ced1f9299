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

}  // namespace

csa2_status launch_project_fp4(const csa2_project_args& a, cudaStream_t s) {
  if (a.rows == 0) return CSA2_OK;
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
