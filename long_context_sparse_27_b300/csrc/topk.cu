// topk.cu -- a4, per-row top-k with the lowest index winning ties.
//
// Full mode selects new Top-512 entries for each query ("Unlocking Extreme
// Context Scaling with DeepSeek-V4.1-Flash", "Compressed Sparse Attention 2
// (CSA2)").  Order is (score descending, index ascending); the output row
// holds the chosen indices ascending, padded with -1.
//
// Radix select on an order-preserving 32-bit key (+0 and -0 share a key):
//   1. topk_hist_kernel     (chunks x rows CTAs) 4096-bin histogram of the
//                           key's top 12 bits into the workspace.
//   2. topk_compact_kernel  (chunks x rows) every CTA finds the threshold bin
//                           T1 from the histogram; entries above it are
//                           written out as selected, entries in it are
//                           appended as 64-bit (key, ~index) candidates and
//                           histogrammed on the next 12 key bits.
//   3. topk_final_kernel    (one CTA per row) finds the second-level bin T2,
//                           takes the candidates above it, sorts the few in
//                           it exactly, and writes the k indices ascending.
// A row whose threshold bins overflow the candidate buffers (huge runs of
// equal scores) is finished by an exact 8-pass radix select over its
// 64-bit (key, ~index) values inside topk_final_kernel.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace csa2 {

namespace {

constexpr int kBins = 4096;       // 12-bit digits
constexpr int kCandCap = 4096;    // first-level candidates kept per row
constexpr int kTinyCap = 2048;    // second-level ties sorted in shared memory
constexpr int kMaxK = 2048;
constexpr int kThreads = 512;

struct RowWS {
  uint32_t hist1[kBins];
  uint32_t hist2[kBins];
  uint32_t n_sel;   // entries above T1 written to sel
  uint32_t n_cand;  // entries in T1 (may exceed kCandCap: then only counted)
  int32_t t1;       // threshold bin (-1: every visible entry is selected)
  uint32_t above1;  // visible entries in bins above t1
  uint32_t pad[60];
};

size_t row_stride_bytes(int32_t k) {
  return align256(sizeof(RowWS)) + align256((size_t)k * 4) + align256((size_t)kCandCap * 8);
}

struct RowPtrs {
  RowWS* ws;
  int32_t* sel;
  uint64_t* cand;
};

__device__ __forceinline__ RowPtrs row_ptrs(void* base, int64_t row, int32_t k) {
  const size_t h = (sizeof(RowWS) + 255) & ~(size_t)255;
  const size_t s = ((size_t)k * 4 + 255) & ~(size_t)255;
  const size_t c = ((size_t)kCandCap * 8 + 255) & ~(size_t)255;
  uint8_t* p = static_cast<uint8_t*>(base) + (size_t)row * (h + s + c);
  return {reinterpret_cast<RowWS*>(p), reinterpret_cast<int32_t*>(p + h),
          reinterpret_cast<uint64_t*>(p + h + s)};
}

// order-preserving key: larger float -> larger key; -0 maps like +0
__device__ __forceinline__ uint32_t score_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ uint64_t composite(uint32_t key, int64_t j) {
  return ((uint64_t)key << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)j);
}

__device__ __forceinline__ int64_t row_nvalid(const int32_t* n_valid, int64_t row, int64_t n) {
  int64_t nv = n_valid ? (int64_t)n_valid[row] : n;
  return nv < 0 ? 0 : (nv > n ? n : nv);
}

// Block-wide: the largest bin t with (sum of hist[b], b >= t) >= target, and
// the count strictly above it.  t = -1 if the whole histogram holds fewer
// than `target`.  nbins = kBins, blockDim = kThreads (8 bins per thread,
// thread 0 owning the top bins).  Results in *t_out / *above_out (shared).
__device__ void find_threshold(const uint32_t* hist, uint32_t target, int* t_out,
                               uint32_t* above_out, uint32_t* scratch /* [kThreads/32] */) {
  constexpr int PER = kBins / kThreads;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid / 32;
  const int hi_bin = kBins - 1 - tid * PER;  // bins hi_bin .. hi_bin-PER+1
  uint32_t local = 0;
#pragma unroll
  for (int i = 0; i < PER; ++i) local += hist[hi_bin - i];
  // exclusive prefix over threads in order tid = 0, 1, ... (top bins first)
  uint32_t incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) scratch[warp] = incl;
  if (tid == 0) *t_out = -1;
  __syncthreads();
  uint32_t warp_off = 0;
  for (int w = 0; w < warp; ++w) warp_off += scratch[w];
  const uint32_t before = warp_off + incl - local;
  if (before < target && before + local >= target) {
    uint32_t cum = before;
    for (int i = 0; i < PER; ++i) {
      const uint32_t h = hist[hi_bin - i];
      if (cum + h >= target) {
        *t_out = hi_bin - i;
        *above_out = cum;
        break;
      }
      cum += h;
    }
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kThreads)
    topk_hist_kernel(const float* __restrict__ scores, int64_t n, int64_t ld,
                     const int32_t* __restrict__ n_valid, int32_t k, void* ws, int64_t chunk) {
  __shared__ uint32_t h[kBins];
  const int64_t row = blockIdx.y;
  for (int i = threadIdx.x; i < kBins; i += kThreads) h[i] = 0;
  __syncthreads();
  const int64_t nv = row_nvalid(n_valid, row, n);
  const int64_t j0 = (int64_t)blockIdx.x * chunk;
  const int64_t j1 = min(nv, j0 + chunk);
  const float* s = scores + row * ld;
  for (int64_t j = j0 + threadIdx.x; j < j1; j += kThreads)
    atomicAdd(&h[score_key(s[j]) >> 20], 1u);
  __syncthreads();
  RowPtrs rp = row_ptrs(ws, row, k);
  for (int i = threadIdx.x; i < kBins; i += kThreads)
    if (h[i]) atomicAdd(&rp.ws->hist1[i], h[i]);
}

__global__ void __launch_bounds__(kThreads)
    topk_compact_kernel(const float* __restrict__ scores, int64_t n, int64_t ld,
                        const int32_t* __restrict__ n_valid, int32_t k, void* ws,
                        int64_t chunk) {
  __shared__ uint32_t h[kBins];
  __shared__ uint32_t scratch[kThreads / 32];
  __shared__ int t1;
  __shared__ uint32_t above1;
  const int64_t row = blockIdx.y;
  RowPtrs rp = row_ptrs(ws, row, k);
  const int64_t nv = row_nvalid(n_valid, row, n);
  if (nv <= k) return;  // every visible entry is selected; the final kernel writes them
  for (int i = threadIdx.x; i < kBins; i += kThreads) h[i] = rp.ws->hist1[i];
  __syncthreads();
  find_threshold(h, (uint32_t)k, &t1, &above1, scratch);
  const int T1 = t1;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    rp.ws->t1 = T1;
    rp.ws->above1 = above1;
  }
  const int64_t j0 = (int64_t)blockIdx.x * chunk;
  const int64_t j1 = min(nv, j0 + chunk);
  const float* s = scores + row * ld;
  for (int64_t j = j0 + threadIdx.x; j < j1; j += kThreads) {
    const uint32_t key = score_key(s[j]);
    const int b1 = (int)(key >> 20);
    if (b1 > T1) {
      const uint32_t pos = atomicAdd(&rp.ws->n_sel, 1u);
      if (pos < (uint32_t)k) rp.sel[pos] = (int32_t)j;
    } else if (b1 == T1) {
      const uint32_t pos = atomicAdd(&rp.ws->n_cand, 1u);
      if (pos < (uint32_t)kCandCap) {
        rp.cand[pos] = composite(key, j);
        atomicAdd(&rp.ws->hist2[(key >> 8) & (kBins - 1)], 1u);
      }
    }
  }
}

// Rank sort of `cnt` distinct indices held in shared memory, written
// ascending to out[0 .. cnt).
__device__ void write_ascending(const int32_t* list, int cnt, int32_t* out) {
  for (int i = threadIdx.x; i < cnt; i += kThreads) {
    const int32_t x = list[i];
    int rank = 0;
    for (int t = 0; t < cnt; ++t) rank += (list[t] < x);
    out[rank] = x;
  }
}

// Bitonic sort (descending) of m <= kTinyCap 64-bit values in shared memory,
// padded with zeros to a power of two.
__device__ void bitonic_desc(uint64_t* v, int m) {
  int p = 1;
  while (p < m) p <<= 1;
  for (int i = m + threadIdx.x; i < p; i += kThreads) v[i] = 0;
  __syncthreads();
  for (int size = 2; size <= p; size <<= 1) {
    for (int stride = size / 2; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < p / 2; i += kThreads) {
        const int lo = 2 * i - (i & (stride - 1));
        const int hi = lo + stride;
        const bool desc = ((lo & size) == 0);
        const uint64_t a = v[lo], b = v[hi];
        if ((a < b) == desc) {
          v[lo] = b;
          v[hi] = a;
        }
      }
      __syncthreads();
    }
  }
}

__global__ void __launch_bounds__(kThreads)
    topk_final_kernel(const float* __restrict__ scores, int64_t n, int64_t ld,
                      const int32_t* __restrict__ n_valid, int32_t k, void* ws,
                      int32_t* __restrict__ idx_out, int64_t idx_ld) {
  __shared__ int32_t outl[kMaxK];
  __shared__ uint64_t tiny[kTinyCap];
  __shared__ uint32_t h2[kBins];
  __shared__ uint32_t scratch[kThreads / 32];
  __shared__ uint32_t n_out, n_tiny;
  __shared__ int t2;
  __shared__ uint32_t above2;
  __shared__ int slow;
  const int64_t row = blockIdx.x;
  RowPtrs rp = row_ptrs(ws, row, k);
  int32_t* out = idx_out + row * idx_ld;
  const int64_t nv = row_nvalid(n_valid, row, n);
  if (nv <= k) {
    for (int64_t i = threadIdx.x; i < k; i += kThreads) out[i] = i < nv ? (int32_t)i : -1;
    return;
  }
  const uint32_t above1 = rp.ws->above1;
  const uint32_t m1 = rp.ws->n_cand;
  const uint32_t r1 = (uint32_t)k - above1;  // needed from bin T1 (>= 1)
  if (threadIdx.x == 0) {
    n_out = 0;
    n_tiny = 0;
    slow = m1 > (uint32_t)kCandCap;
  }
  for (int i = threadIdx.x; i < (int)above1; i += kThreads) outl[i] = rp.sel[i];
  __syncthreads();
  if (!slow) {
    for (int i = threadIdx.x; i < kBins; i += kThreads) h2[i] = rp.ws->hist2[i];
    __syncthreads();
    find_threshold(h2, r1, &t2, &above2, scratch);
    const int T2 = t2;
    const uint32_t m2 = h2[T2];
    if (threadIdx.x == 0) {
      n_out = above1;
      if (m2 > (uint32_t)kTinyCap) slow = 1;
    }
    __syncthreads();
    if (!slow) {
      for (uint32_t i = threadIdx.x; i < m1; i += kThreads) {
        const uint64_t c = rp.cand[i];
        const int b2 = (int)((c >> 40) & (kBins - 1));
        const int32_t j = (int32_t)(0xFFFFFFFFu - (uint32_t)c);
        if (b2 > T2)
          outl[atomicAdd(&n_out, 1u)] = j;
        else if (b2 == T2)
          tiny[atomicAdd(&n_tiny, 1u)] = c;
      }
      __syncthreads();
      const int mt = (int)n_tiny;
      bitonic_desc(tiny, mt);
      const uint32_t r2 = r1 - above2;
      const uint32_t base = n_out;
      for (uint32_t i = threadIdx.x; i < r2; i += kThreads)
        outl[base + i] = (int32_t)(0xFFFFFFFFu - (uint32_t)tiny[i]);
      __syncthreads();
    }
  }
  if (slow) {
    // exact radix select over every visible entry's (key, ~index), 8 bits
    // at a time from the top; the values are distinct, so the k-th largest
    // V leaves exactly k entries >= V
    uint32_t* hh = h2;  // first 256 bins reused
    __shared__ uint64_t prefix;
    __shared__ uint32_t need;
    if (threadIdx.x == 0) {
      prefix = 0;
      need = (uint32_t)k;
    }
    __syncthreads();
    const float* s = scores + row * ld;
    for (int shift = 56; shift >= 0; shift -= 8) {
      for (int i = threadIdx.x; i < 256; i += kThreads) hh[i] = 0;
      __syncthreads();
      const uint64_t pre = prefix;
      const uint64_t mask_hi = (shift == 56) ? 0 : (~0ull << (shift + 8));
      for (int64_t j = threadIdx.x; j < nv; j += kThreads) {
        const uint64_t c = composite(score_key(s[j]), j);
        if ((c & mask_hi) == pre) atomicAdd(&hh[(c >> shift) & 255], 1u);
      }
      __syncthreads();
      if (threadIdx.x == 0) {
        uint32_t cum = 0;
        int d = 255;
        for (; d > 0; --d) {
          if (cum + hh[d] >= need) break;
          cum += hh[d];
        }
        need -= cum;
        prefix = pre | ((uint64_t)d << shift);
      }
      __syncthreads();
    }
    const uint64_t V = prefix;
    if (threadIdx.x == 0) n_out = 0;
    __syncthreads();
    for (int64_t j = threadIdx.x; j < nv; j += kThreads)
      if (composite(score_key(s[j]), j) >= V) outl[atomicAdd(&n_out, 1u)] = (int32_t)j;
    __syncthreads();
  }
  write_ascending(outl, k, out);
}

}  // namespace

size_t topk_workspace_bytes(int64_t rows, int64_t n, int32_t k) {
  (void)n;
  return (size_t)rows * row_stride_bytes(k);
}

csa2_status launch_topk(const float* scores, int64_t rows, int64_t n, int64_t ld,
                        const int32_t* n_valid, int32_t k, int32_t* idx_out, int64_t idx_ld,
                        void* ws, int32_t* dev_status, cudaStream_t s) {
  (void)dev_status;
  if (rows == 0) return CSA2_OK;
  const size_t stride = row_stride_bytes(k);
  // zero the histograms and counters of every row (the selected / candidate
  // lists need no clearing: only their counted prefix is read)
  const size_t head = align256(sizeof(RowWS));
  cudaError_t e = cudaMemset2DAsync(ws, stride, 0, head, (size_t)rows, s);
  if (e != cudaSuccess) return cuda_fail(e);
  // chunks per row: enough CTAs to cover the GPU about twice
  const int64_t want = (2 * (int64_t)sm_count() + rows - 1) / rows;
  const int64_t max_chunks = (n + 4095) / 4096;
  const int64_t chunks = std::max<int64_t>(1, std::min<int64_t>(want, max_chunks));
  const int64_t chunk = (n + chunks - 1) / chunks;
  if (n > 0) {
    dim3 grid((unsigned)chunks, (unsigned)rows);
    topk_hist_kernel<<<grid, kThreads, 0, s>>>(scores, n, ld, n_valid, k, ws, chunk);
    csa2_status st = check_launch();
    if (st != CSA2_OK) return st;
    topk_compact_kernel<<<grid, kThreads, 0, s>>>(scores, n, ld, n_valid, k, ws, chunk);
    st = check_launch();
    if (st != CSA2_OK) return st;
  }
  topk_final_kernel<<<(unsigned)rows, kThreads, 0, s>>>(scores, n, ld, n_valid, k, ws, idx_out,
                                                        idx_ld);
  return check_launch();
}

}  // namespace csa2

// ===========================================================================
// Variant without allocation: the scratch lives in the library itself, for
// callers that cannot allocate device memory.  All calls share this array.
// ===========================================================================

namespace csa2 {
namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)4 << 20;  // 4 MiB per device
static __device__ __align__(256) uint8_t g_topk_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the array, looked up once per device (host code cannot
// use the array's name as a device pointer).
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64] = {nullptr};

}  // namespace
}  // namespace csa2

extern "C" csa2_status csa2_topk_noalloc(const float* scores, int64_t rows, int64_t n,
                                         int64_t ld, const int32_t* n_valid, int32_t k,
                                         int32_t* idx_out, int64_t idx_ld, int32_t* dev_status,
                                         csa2_stream_t stream) {
  using namespace csa2;
  if (rows < 0 || n < 0 || k < 1 || idx_ld < k || ld < n) return CSA2_ERR_INVALID_ARG;
  if (k > kMaxK || n >= ((int64_t)1 << 31)) return CSA2_ERR_UNSUPPORTED;
  if (rows == 0) return CSA2_OK;
  if (!idx_out || (n > 0 && !scores)) return CSA2_ERR_INVALID_ARG;
  if (topk_workspace_bytes(rows, n, k) > kNoAllocScratchBytes) return CSA2_ERR_WORKSPACE;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= 64) return CSA2_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
      e = cudaGetSymbolAddress(&scratch, g_topk_noalloc_scratch);
      if (e != cudaSuccess) return cuda_fail(e);
      g_noalloc_ptr[dev] = scratch;
    }
    scratch = g_noalloc_ptr[dev];
  }
  // launch_topk clears the histograms and counters of every row it uses
  return launch_topk(scores, rows, n, ld, n_valid, k, idx_out, idx_ld, scratch, dev_status,
                     reinterpret_cast<cudaStream_t>(stream));
}
