// block_keys.cu -- block-level representations of the indexer keys, the
// first level of the Hierarchical Sparse Indexer ("DeepSeek-V4.1-Flash:
// Pushing the Limits of KV Cache Compression", Method: indexers restricted
// to a candidate pool chosen by an earlier indexer; Related Work: scoring
// token-level entries and pruning them on block-level representations).
//
// This library's definition: the entries of a sequence form blocks of G
// consecutive entries; a block's key is E4M3((sum of its entries' decoded
// E4M3 keys) / G), entries past the end of the sequence counting as zero.
// Every E4M3 value is a multiple of 2^-9 of magnitude <= 448, so the fp32
// sum of at most 2^16 of them is exact in any order (it needs at most 24
// significant bits) and the division by a power-of-two G is exact: the cast
// is the only rounding.
#include "common.cuh"
#include "internal.h"

namespace csa2 {

namespace {

// E4M3 value of a code (bias 7, 3 mantissa bits; exponent field 0 is
// subnormal, 2^-6 * m / 8).  The casts of this library never write the NaN
// codes 0x7F / 0xFF.
__device__ __forceinline__ float e4m3_value(uint32_t c) {
  const uint32_t e = (c >> 3) & 15u, m = c & 7u;
  const float mag = e ? exp2_int((int)e - 7) * (1.f + (float)m * 0.125f)
                      : (float)m * 0.001953125f;  // m * 2^-9
  return (c & 0x80u) ? -mag : mag;
}

// One CTA per (block, sequence), one thread per key byte.
__global__ void __launch_bounds__(128)
    block_keys_kernel(const uint8_t* __restrict__ k8, int64_t n, int64_t k_ld,
                      int64_t k_seq_stride, const csa2_pages pages, int32_t G, int64_t blk0,
                      uint8_t* __restrict__ out, int64_t out_ld, int64_t out_seq_stride,
                      int32_t* dev_status) {
  pdl_wait();
  const int64_t blk = blk0 + blockIdx.x, b = blockIdx.y;
  const int t = threadIdx.x;
  const int64_t j0 = blk * G, j1 = min(n, j0 + G);
  float sum = 0.f;
  for (int64_t j = j0; j < j1; ++j) {
    const uint8_t* row;
    if (pages.block_table) {
      const int64_t r = paged_row(pages, b, j, dev_status);
      if (r < 0) continue;  // a page outside the pool reads as zeros
      row = k8 + r * k_ld;
    } else {
      row = k8 + b * k_seq_stride + j * k_ld;
    }
    sum += e4m3_value(row[t]);
  }
  pdl_trigger();
  out[b * out_seq_stride + blk * out_ld + t] = (uint8_t)e4m3_encode(sum / (float)G);
}

}  // namespace

csa2_status launch_block_keys(const uint8_t* k8, int64_t B, int64_t n, int64_t k_ld,
                              int64_t k_seq_stride, const csa2_pages& pages, int32_t G,
                              int64_t blk0, int64_t nblk, uint8_t* out, int64_t out_ld,
                              int64_t out_seq_stride, int32_t* dev_status, cudaStream_t s) {
  if (B == 0 || nblk == 0) return CSA2_OK;
  return launch_kernel(block_keys_kernel, dim3((unsigned)nblk, (unsigned)B), dim3(128), 0, s, 1,
                       k8, n, k_ld, k_seq_stride, pages, G, blk0, out, out_ld, out_seq_stride,
                       dev_status);
}

}  // namespace csa2
