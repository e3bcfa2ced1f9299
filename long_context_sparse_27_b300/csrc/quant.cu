// quant.cu -- a1 (FP4 E2M1 main-KV quantiser + E4M3 indexer-K cast) and
// a2 (indexer-Q E4M3 quantiser).
//
// a1 follows the FP4 main-KV cache of "Unlocking Extreme Context Scaling
// with DeepSeek-V4.1-Flash" ("Deployment and Infrastructure") in the E2M1
// format named on the aiany.app DeepSeek-V4.1-Flash page ("What Sets It
// Apart"), with the OCP MX v1.0 per-32 power-of-two scale:
// X = 2^(floor(log2 amax) - 2).  Memory-bound and tiny (one new row per
// sequence per decode step): each thread converts 8 elements (one 16-byte
// load), four threads share a 32-element block and reduce its amax with
// two shuffles.
#include "common.cuh"
#include "internal.h"

namespace csa2 {

namespace {

constexpr int kQuantThreads = 256;

// Threads [0, kv_threads) quantise main-KV rows; threads from the next
// multiple of 32 on cast indexer-K rows.  Every thread of a warp takes part
// in the shuffles; threads past the end work on zeros and store nothing.
__global__ void __launch_bounds__(kQuantThreads)
    quant_fp4_kernel(const uint16_t* __restrict__ x, int64_t rows, int32_t d, int64_t x_ld,
                     uint8_t* __restrict__ codes, int64_t codes_ld, uint8_t* __restrict__ scales,
                     int64_t scales_ld, const uint16_t* __restrict__ kx, int32_t di,
                     int64_t k_ld, uint8_t* __restrict__ k8, int64_t k8_ld, int64_t kv_threads,
                     int64_t k_begin, const csa2_pages pages, int64_t rows_per_seq,
                     int64_t entry0, int32_t* dev_status) {
  pdl_wait();
  // destination row of source row r: r itself, or its entry's row in the
  // page pool (-1: a page outside the pool, nothing written)
  auto dst_row = [&](int64_t r) -> int64_t {
    if (!pages.block_table) return r;
    return paged_row(pages, r / rows_per_seq, entry0 + r % rows_per_seq, dev_status);
  };
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (gid < k_begin) {
    const int64_t per_row = d / 8;
    const bool live = gid < kv_threads;
    const int64_t row = live ? gid / per_row : 0;
    const int64_t part = live ? gid % per_row : 0;
    uint4 raw = make_uint4(0, 0, 0, 0);
    if (live) raw = *reinterpret_cast<const uint4*>(x + row * x_ld + part * 8);
    float v[8];
    bf16x8_to_float(raw, v);
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    if (!live) return;
    const int64_t drow = dst_row(row);
    if (drow < 0) return;
    uint32_t sbyte;
    const uint32_t packed = fp4_encode8(v, amax, sbyte);
    *reinterpret_cast<uint32_t*>(codes + drow * codes_ld + part * 4) = packed;
    if ((part & 3) == 0) scales[drow * scales_ld + part / 4] = (uint8_t)sbyte;
  } else {
    const int64_t t = gid - k_begin;
    const int64_t per_row = di / 8;
    if (t >= rows * per_row) return;
    const int64_t row = t / per_row, part = t % per_row;
    const int64_t drow = dst_row(row);
    if (drow < 0) return;
    const uint4 raw = *reinterpret_cast<const uint4*>(kx + row * k_ld + part * 8);
    *reinterpret_cast<uint2*>(k8 + drow * k8_ld + part * 8) = e4m3_encode8(raw);
  }
}

// a2: one warp per (row, head); each lane holds di/32 consecutive values.
template <int DI>
__global__ void __launch_bounds__(256)
    quant_index_q_kernel(const uint16_t* __restrict__ q, const float* __restrict__ w,
                         int64_t n_heads_total, uint8_t* __restrict__ q8, float* __restrict__ c) {
  constexpr int PER = DI / 32;
  pdl_wait();
  const int64_t head = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (head >= n_heads_total) return;  // whole warp leaves together
  const uint16_t* src = q + head * DI + lane * PER;
  float v[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) v[i] = bf16_bits_to_float(src[i]);
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < PER; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const int e = amax > 0.f ? index_q_exponent(amax) : 0;
  const float inv = exp2_int(-e);
  uint8_t out[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) out[i] = amax > 0.f ? (uint8_t)e4m3_encode(v[i] * inv) : 0;
#pragma unroll
  for (int i = 0; i < PER; ++i) q8[head * DI + lane * PER + i] = out[i];
  if (lane == 0) c[head] = w[head] * exp2_int(e);
}

}  // namespace

csa2_status launch_quantize_fp4(const csa2_quant_args& a, cudaStream_t s, int32_t* dev_status) {
  if (a.rows == 0) return CSA2_OK;
  const int64_t kv_threads = a.rows * (a.d / 8);
  const int64_t k_begin = (kv_threads + 31) / 32 * 32;
  const int64_t k_threads = a.idxk ? a.rows * (a.di / 8) : 0;
  const int64_t total = k_begin + k_threads;
  const int64_t blocks = (total + kQuantThreads - 1) / kQuantThreads;
  return launch_kernel(quant_fp4_kernel, dim3((unsigned)blocks), dim3(kQuantThreads), 0, s, 1,
                       static_cast<const uint16_t*>(a.x), a.rows, a.d, a.x_ld, a.codes,
                       a.codes_ld, a.scales, a.scales_ld, static_cast<const uint16_t*>(a.idxk),
                       a.di, a.idxk_ld, a.idxk_e4m3, a.idxk_e4m3_ld, kv_threads, k_begin,
                       a.pages, a.rows_per_seq, a.entry0, dev_status);
}

csa2_status launch_quantize_index_q(const void* q, const float* w, int64_t nq, int32_t hi,
                                    int32_t di, uint8_t* q8, float* c, cudaStream_t s) {
  const int64_t heads = nq * hi;
  if (heads == 0) return CSA2_OK;
  const unsigned blocks = (unsigned)((heads + 7) / 8);
  const uint16_t* qp = static_cast<const uint16_t*>(q);
  switch (di) {
    case 32: return launch_kernel(quant_index_q_kernel<32>, dim3(blocks), dim3(256), 0, s, 1, qp, w, heads, q8, c);
    case 64: return launch_kernel(quant_index_q_kernel<64>, dim3(blocks), dim3(256), 0, s, 1, qp, w, heads, q8, c);
    case 128: return launch_kernel(quant_index_q_kernel<128>, dim3(blocks), dim3(256), 0, s, 1, qp, w, heads, q8, c);
    case 256: return launch_kernel(quant_index_q_kernel<256>, dim3(blocks), dim3(256), 0, s, 1, qp, w, heads, q8, c);
    default: return CSA2_ERR_UNSUPPORTED;
  }
}

}  // namespace csa2
