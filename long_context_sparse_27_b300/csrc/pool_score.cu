// pool_score.cu -- the restricted scoring step of the Hierarchical Sparse
// Indexer: an indexer that scores only a shared candidate pool chosen by an
// earlier indexer ("DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache
// Compression", Method; "Unlocking Extreme Context Scaling with DeepSeek-
// V4.1-Flash", "Compressed Sparse Attention 2 (CSA2)").  The score is the
// FP8 indexer's: s = sum_h c[q,h] * max(0, <q8[q,h], k_j>) with E4M3 q8 / k.
//
// One CTA per (query, 128 pool slots), pools of up to 2048 slots: the
// slots' indexer-K rows (128 B each, scattered over the sequence) are
// gathered into shared memory with cp.async, next to the query's 64 x 128
// E4M3 heads; each of the 8 warps scores 16 slots against the 64 heads with
// m16n8k32 E4M3 MMAs (fp32 accumulate) and reduces ReLU x c over the heads
// in registers.  The work
// is small (a pool of P entries per query instead of the whole sequence),
// so the kernel is bound by the gather latency, not by MMA throughput.
#include "common.cuh"
#include "internal.h"

namespace csa2 {

namespace {

constexpr int kPSlots = 128;          // pool slots per CTA
constexpr int kPThreads = 256;        // 8 warps x 16 slots
constexpr int kPHeads = 64;           // indexer heads
constexpr int kPDim = 128;            // indexer dim (E4M3 bytes per row)
constexpr int kPRow = kPDim + 16;     // padded row: conflict-free 32-bit fragment loads

// D[16 x 8] += A[16 x 32] . B[32 x 8], E4M3 inputs, fp32 accumulate.
// A: a0 / a1 rows g / g + 8 bytes 4t .. 4t+3, a2 / a3 the same + 16;
// B: b0 bytes (k) 4t .. 4t+3 of column g, b1 the same + 16;
// D: d0 / d1 row g columns 2t, 2t + 1, d2 / d3 row g + 8 (g = lane / 4,
// t = lane % 4).
__device__ __forceinline__ void mma_e4m3_16832(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__global__ void __launch_bounds__(kPThreads)
    pool_score_kernel(const uint8_t* __restrict__ q8, const float* __restrict__ c,
                      const uint8_t* __restrict__ k, int64_t k_ld, int64_t k_seq_stride,
                      int64_t q_per_seq, int64_t n, const int32_t* __restrict__ pool,
                      int64_t pool_ld, int32_t pool_n, float* __restrict__ scores,
                      int64_t scores_ld, int32_t* dev_status, const csa2_pages pages) {
  __shared__ __align__(16) uint8_t sk[kPSlots * kPRow];
  __shared__ __align__(16) uint8_t sq[kPHeads * kPRow];
  __shared__ float sc[kPHeads];
  __shared__ int64_t sj[kPSlots];  // byte offset of the slot's key row from k, -1: empty
  pdl_wait();
  const int64_t qi = blockIdx.x;
  const int s0 = blockIdx.y * kPSlots;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t b = (uint32_t)qi / (uint32_t)q_per_seq;  // queries fit 32 bits

  if (tid < kPSlots) {
    const int slot = s0 + tid;
    int32_t j = slot < pool_n ? pool[qi * pool_ld + slot] : -1;
    if (j < -1 || j >= n) {
      raise_flag(dev_status, CSA2_DEVFLAG_BOUNDS);
      j = -1;
    }
    int64_t off = -1;
    if (j >= 0) {
      if (pages.block_table) {  // paged keys: the entry's row in the pool
        const int64_t row = paged_row(pages, b, j, dev_status);
        off = row < 0 ? -1 : row * k_ld;
      } else {
        off = b * k_seq_stride + (int64_t)j * k_ld;
      }
    }
    sj[tid] = off;
  }
  if (tid < kPHeads) sc[tid] = c[qi * kPHeads + tid];
  for (int i = tid; i < kPHeads * (kPDim / 16); i += kPThreads) {
    const int h = i / (kPDim / 16), p = i % (kPDim / 16);
    cp_async16(sq + h * kPRow + p * 16, q8 + (qi * kPHeads + h) * kPDim + p * 16);
  }
  __syncthreads();
  for (int i = tid; i < kPSlots * (kPDim / 16); i += kPThreads) {
    const int r = i / (kPDim / 16), p = i % (kPDim / 16);
    const int64_t off = sj[r];
    uint8_t* dst = sk + r * kPRow + p * 16;
    if (off >= 0)
      cp_async16(dst, k + off + p * 16);
    else
      *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
  }
  cp_async_wait_all();
  __syncthreads();

  // warp w: slots 16w .. 16w + 15 (MMA rows) against heads 8 nt .. (MMA columns)
  const int g = lane >> 2, t = lane & 3;
  float acc[kPHeads / 8][4];
#pragma unroll
  for (int nt = 0; nt < kPHeads / 8; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
  const uint8_t* arow = sk + (16 * warp + g) * kPRow + 4 * t;
#pragma unroll
  for (int ks = 0; ks < kPDim / 32; ++ks) {
    const uint32_t a0 = *reinterpret_cast<const uint32_t*>(arow + ks * 32);
    const uint32_t a1 = *reinterpret_cast<const uint32_t*>(arow + 8 * kPRow + ks * 32);
    const uint32_t a2 = *reinterpret_cast<const uint32_t*>(arow + ks * 32 + 16);
    const uint32_t a3 = *reinterpret_cast<const uint32_t*>(arow + 8 * kPRow + ks * 32 + 16);
#pragma unroll
    for (int nt = 0; nt < kPHeads / 8; ++nt) {
      const uint8_t* brow = sq + (8 * nt + g) * kPRow + 4 * t + ks * 32;
      const uint32_t b0 = *reinterpret_cast<const uint32_t*>(brow);
      const uint32_t b1 = *reinterpret_cast<const uint32_t*>(brow + 16);
      mma_e4m3_16832(acc[nt], a0, a1, a2, a3, b0, b1);
    }
  }
  // ReLU x c summed over this thread's heads (8 nt + 2t, + 1), then over the
  // four threads of a row group
  float s_lo = 0.f, s_hi = 0.f;
#pragma unroll
  for (int nt = 0; nt < kPHeads / 8; ++nt) {
    const float c0 = sc[8 * nt + 2 * t], c1 = sc[8 * nt + 2 * t + 1];
    s_lo = fmaf(c0, fmaxf(acc[nt][0], 0.f), s_lo);
    s_lo = fmaf(c1, fmaxf(acc[nt][1], 0.f), s_lo);
    s_hi = fmaf(c0, fmaxf(acc[nt][2], 0.f), s_hi);
    s_hi = fmaf(c1, fmaxf(acc[nt][3], 0.f), s_hi);
  }
#pragma unroll
  for (int o = 1; o < 4; o <<= 1) {
    s_lo += __shfl_xor_sync(0xffffffffu, s_lo, o);
    s_hi += __shfl_xor_sync(0xffffffffu, s_hi, o);
  }
  if (t == 0) {
    const int r_lo = 16 * warp + g, r_hi = r_lo + 8;
    if (s0 + r_lo < pool_n)
      scores[qi * scores_ld + s0 + r_lo] = sj[r_lo] >= 0 ? s_lo : -INFINITY;
    if (s0 + r_hi < pool_n)
      scores[qi * scores_ld + s0 + r_hi] = sj[r_hi] >= 0 ? s_hi : -INFINITY;
  }
  pdl_trigger();
}

}  // namespace

csa2_status launch_index_score_pool(const csa2_index_args& a, const uint8_t* q8, const float* c,
                                    const int32_t* pool, int64_t pool_ld, int32_t pool_n,
                                    float* scores, int64_t scores_ld, cudaStream_t s) {
  if (a.hi != kPHeads || a.di != kPDim) return CSA2_ERR_UNSUPPORTED;
  const int64_t nq = a.B * a.q_per_seq;
  if (nq == 0 || pool_n == 0) return CSA2_OK;
  if (pool_n > 2048) return CSA2_ERR_UNSUPPORTED;
  const dim3 grid((unsigned)nq, (unsigned)((pool_n + kPSlots - 1) / kPSlots));
  return launch_kernel(pool_score_kernel, grid, dim3(kPThreads), 0, s, 1, q8, c,
                       static_cast<const uint8_t*>(a.k), a.k_ld, a.k_seq_stride, a.q_per_seq,
                       a.n, pool, pool_ld, pool_n, scores, scores_ld, a.dev_status, a.pages);
}

}  // namespace csa2
