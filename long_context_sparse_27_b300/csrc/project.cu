// project.cu -- the decoder's global KV: the final encoder hidden state times
// a layer's projection, quantised straight into the FP4 main-KV cache.
//
// "Unlocking Extreme Context Scaling with DeepSeek-V4.1-Flash", Causal
// Encoder-Decoder (CED) Efficiency: the decoder derives its global KV cache
// from the final encoder hidden state using per-layer projections; the main
// KV is FP4 E2M1 ("Deployment and Infrastructure") with the per-32-element
// power-of-two block scale of the library's quantiser.
//
// One CTA per (64 rows, 64 output columns), 4 warps of 16 rows: the hidden
// dimension is walked in steps of 32 through a 4-stage cp.async ring of h
// and w tiles (three steps in flight), m16n8k16 bf16 MMAs accumulate in
// fp32, and the epilogue quantises the accumulators in registers: each 32-column block of a row
// lives in the four threads of a quad (8 values each), whose amax is two
// shuffles away.  The codes are decided on the fp32 projection, which can
// also be written out.
#include "common.cuh"
#include "internal.h"

namespace csa2 {

namespace {

constexpr int kPjRows = 64;        // rows per CTA
constexpr int kPjCols = 64;        // output columns per CTA (two FP4 blocks)
constexpr int kPjK = 32;           // hidden features per step
constexpr int kPjThreads = 128;    // 4 warps x 16 rows
constexpr int kPjStride = kPjK + 8;  // padded smem row (bf16): conflict-free ldmatrix
constexpr int kPjTile = kPjRows * kPjStride;  // elements of one h (or w) tile
constexpr int kPjStages = 4;       // copies in flight: steps ks + 1 .. ks + 3 load during step ks

__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
// wait until at most N of this thread's committed copy groups are pending
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__global__ void __launch_bounds__(kPjThreads)
    project_fp4_kernel(const uint16_t* __restrict__ h, int64_t h_ld,
                       const uint16_t* __restrict__ w, int64_t w_ld, int64_t rows,
                       int32_t hidden, uint8_t* __restrict__ codes, int64_t codes_ld,
                       uint8_t* __restrict__ scales, int64_t scales_ld, float* __restrict__ out,
                       int64_t out_ld) {
  __shared__ __align__(16) uint16_t sh[kPjStages][kPjTile];
  __shared__ __align__(16) uint16_t sw[kPjStages][kPjTile];
  pdl_wait();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t r0 = (int64_t)blockIdx.x * kPjRows;
  const int64_t c0 = (int64_t)blockIdx.y * kPjCols;

  // stage s of step ks: 64 rows x 32 features of h and of w (4 16-byte
  // pieces per row); rows past the end are zeros
  auto load = [&](int s, int ks) {
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int i = tid + u * kPjThreads;  // 0 .. 255
      const int r = i >> 2, p = i & 3;
      uint16_t* dh = &sh[s][r * kPjStride + p * 8];
      if (r0 + r < rows)
        cp_async16(dh, h + (r0 + r) * h_ld + (int64_t)ks * kPjK + p * 8);
      else
        *reinterpret_cast<uint4*>(dh) = make_uint4(0, 0, 0, 0);
      cp_async16(&sw[s][r * kPjStride + p * 8], w + (c0 + r) * w_ld + (int64_t)ks * kPjK + p * 8);
    }
  };

  float acc[kPjCols / 8][4];
#pragma unroll
  for (int nt = 0; nt < kPjCols / 8; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
  const int steps = hidden / kPjK;
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
#pragma unroll
    for (int kk = 0; kk < kPjK / 16; ++kk) {
      uint32_t a0, a1, a2, a3;
      ldmatrix_x4(smem_u32(&sh[s][(16 * warp + (lane & 15)) * kPjStride + kk * 16 +
                                  (lane >> 4) * 8]),
                  a0, a1, a2, a3);
#pragma unroll
      for (int np = 0; np < kPjCols / 16; ++np) {
        // columns 16 np .. 16 np + 15 as two n8 tiles, k halves of 8
        const int n = 16 * np + (lane & 7) + ((lane >> 4) << 3);
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4(smem_u32(&sw[s][n * kPjStride + kk * 16 + ((lane >> 3) & 1) * 8]), b0, b1,
                    b2, b3);
        mma_bf16_16816(acc[2 * np], a0, a1, a2, a3, b0, b1);
        mma_bf16_16816(acc[2 * np + 1], a0, a1, a2, a3, b2, b3);
      }
    }
  }
  pdl_trigger();

  // epilogue: thread (g = lane / 4, t = lane % 4) holds rows g and g + 8 of
  // the warp's 16 at columns 8 nt + 2t, + 1; block b = n-tiles 4b .. 4b + 3
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int64_t row = r0 + 16 * warp + g + 8 * half;
#pragma unroll
    for (int b = 0; b < kPjCols / 32; ++b) {
      float v[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        v[2 * i] = acc[4 * b + i][2 * half];
        v[2 * i + 1] = acc[4 * b + i][2 * half + 1];
      }
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      if (row >= rows) continue;
      uint32_t sbyte = 0;
      uint32_t byte[4] = {0u, 0u, 0u, 0u};
      if (amax > 0.f) {
        int e = floor_log2_pos(amax) - 2;
        e = max(-127, min(127, e));
        sbyte = (uint32_t)(e + 127);
        const float inv = exp2_int(-e);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          byte[i] = e2m1_encode(v[2 * i] * inv) | (e2m1_encode(v[2 * i + 1] * inv) << 4);
      }
      // columns 8 (4b + i) + 2t, + 1 are byte (c0 + 32 b + 8 i + 2 t) / 2 of the row
      uint8_t* crow = codes + row * codes_ld + (c0 + 32 * b) / 2;
#pragma unroll
      for (int i = 0; i < 4; ++i) crow[4 * i + t] = (uint8_t)byte[i];
      if (t == 0) scales[row * scales_ld + (c0 + 32 * b) / 32] = (uint8_t)sbyte;
      if (out) {
        float* orow = out + row * out_ld + c0 + 32 * b;
#pragma unroll
        for (int i = 0; i < 4; ++i)
          *reinterpret_cast<float2*>(orow + 8 * i + 2 * t) = make_float2(v[2 * i], v[2 * i + 1]);
      }
    }
  }
}

}  // namespace

csa2_status launch_project_fp4(const csa2_project_args& a, cudaStream_t s) {
  if (a.rows == 0) return CSA2_OK;
  const dim3 grid((unsigned)((a.rows + kPjRows - 1) / kPjRows), (unsigned)(a.d / kPjCols));
  return launch_kernel(project_fp4_kernel, grid, dim3(kPjThreads), 0, s, 1,
                       static_cast<const uint16_t*>(a.h), a.h_ld,
                       static_cast<const uint16_t*>(a.w), a.w_ld, a.rows, a.hidden, a.codes,
                       a.codes_ld, a.scales, a.scales_ld, a.out, a.out_ld);
}

}  // namespace csa2
