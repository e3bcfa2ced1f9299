// topk.cu -- a4, per-row top-k with the lowest index winning ties.
//
// Full mode selects new Top-512 entries for each query ("Unlocking Extreme
// Context Scaling with DeepSeek-V4.1-Flash", "Compressed Sparse Attention 2
// (CSA2)").  Order is (score descending, index ascending); the output row
// holds the chosen indices ascending, padded with -1.
//
// Radix select on an order-preserving 32-bit key (+0 and -0 share a key),
// one row per thread-block cluster of kTkCluster CTAs, each CTA owning a
// contiguous chunk of the row:
//   level 1   the row's 4096-bin histogram of the key's top 12 bits comes
//             from global memory (topk_hist_kernel, or the indexer epilogue
//             that produced the scores); every CTA finds the threshold bin
//             T1 itself and keeps its entries in bins >= T1, in index order;
//   level 2/3 if bin T1 holds more entries than are still needed, the CTAs
//             histogram the next 12 (then 8) key bits of those entries and
//             combine the histograms through distributed shared memory;
//   ties      entries whose whole key equals the threshold key are taken in
//             index order, CTA by CTA;
//   output    each CTA learns how many entries the CTAs before it keep and
//             writes its own ascending, so the row needs no final sort.
// Every CTA of a cluster takes the same branches (they derive the same
// thresholds from the same histograms), so the cluster barriers match.
#include <cooperative_groups.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace csa2 {

namespace {

namespace cg = cooperative_groups;

constexpr int kBins = kTopkBins;    // 12-bit digits (levels 1 and 2)
constexpr int kBins3 = 256;         // 8-bit digit (level 3)
constexpr int kMaxK = 2048;
constexpr int kTkThreads = 512;
constexpr int kTkWarps = kTkThreads / 32;
constexpr int kTkCluster = 8;       // CTAs per row (portable cluster size)
constexpr int kLCap = 512;          // per-warp ordered list of entries in bins >= T1
constexpr int kTkDynSmem = 2 * kTkWarps * kLCap * 4;  // keys + indices
constexpr int kHistThreads = 512;

__device__ __forceinline__ int64_t row_nvalid(const int32_t* n_valid, int64_t row, int64_t n) {
  int64_t nv = n_valid ? (int64_t)n_valid[row] : n;
  return nv < 0 ? 0 : (nv > n ? n : nv);
}

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// ---------------------------------------------------------------------------
// level-1 histogram of a row's visible keys (when the scores come from
// elsewhere than the fused indexer epilogue)
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(kHistThreads)
    topk_hist_kernel(const float* __restrict__ scores, int64_t n, int64_t ld,
                     const int32_t* __restrict__ n_valid, uint32_t* __restrict__ hist1,
                     int64_t chunk) {
  __shared__ uint32_t h[kBins];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < kBins; i += kHistThreads) h[i] = 0;
  pdl_wait();
  __syncthreads();
  const int64_t row = blockIdx.y;
  const int64_t nv = row_nvalid(n_valid, row, n);
  const int64_t j0 = (int64_t)blockIdx.x * chunk;
  const int64_t j1 = min(nv, j0 + chunk);
  const float* s = scores + row * ld;
  constexpr int U = 4;
  for (int64_t base = j0 + warp * 32; base < j1; base += (int64_t)kHistThreads * U) {
    float x[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t j = base + u * kHistThreads + lane;
      x[u] = j < j1 ? s[j] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t j = base + u * kHistThreads + lane;
      if (j < j1) atomicAdd(&h[score_key(x[u]) >> 20], 1u);
    }
  }
  __syncthreads();
  pdl_trigger();
  for (int i = tid; i < kBins; i += kHistThreads)
    if (h[i]) atomicAdd(&hist1[row * kBins + i], h[i]);
}

// ---------------------------------------------------------------------------
// selection
// ---------------------------------------------------------------------------

struct TkTmp {
  uint32_t wsum[kTkWarps];
  uint32_t tot[kTkCluster];
  int t;            // find_top: bin
  uint32_t above;   // find_top: entries in higher bins
  int R;            // cluster_top: slice holding the threshold
  uint32_t cum;     // cluster_top: entries in higher slices
  uint32_t T, A, cnt;  // cluster_top results: bin, entries above it, entries in it
};

// Largest bin t with sum(h[t .. nb)) >= target, and above = sum(h[t+1 ..
// nb)).  Needs 1 <= target <= sum(h).  Block-wide; results in tmp->t /
// tmp->above.  Thread i owns bins nb-1-i*per down to nb-(i+1)*per.
__device__ void find_top(const uint32_t* h, int nb, uint32_t target, TkTmp* tmp) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (nb + kTkThreads - 1) / kTkThreads;
  const int hi = nb - 1 - tid * per;
  uint32_t local = 0;
  for (int i = 0; i < per; ++i)
    if (hi - i >= 0) local += h[hi - i];
  uint32_t incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) tmp->wsum[warp] = incl;
  __syncthreads();
  uint32_t woff = 0;
  for (int w = 0; w < warp; ++w) woff += tmp->wsum[w];
  const uint32_t before = woff + incl - local;
  if (local > 0 && before < target && before + local >= target) {
    uint32_t cum = before;
    for (int i = 0; i < per; ++i) {
      const uint32_t x = h[hi - i];
      if (cum + x >= target) {
        tmp->t = hi - i;
        tmp->above = cum;
        break;
      }
      cum += x;
    }
  }
  __syncthreads();
}

// The cluster-wide histogram is the sum of every CTA's `hist` (nb bins).
// CTA r reduces bins [r*sl, (r+1)*sl) (sl = nb / C) into `slice`; then every
// CTA finds the slice that holds the target-th largest entry and the bin in
// it.  All CTAs end with the same tmp->T / A / cnt.  `hist` is overwritten.
template <int C>
__device__ void cluster_top(cg::cluster_group& cluster, uint32_t* hist, uint32_t* slice,
                            uint32_t* s_tot, int nb, uint32_t target, TkTmp* tmp) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int r = (int)cluster.block_rank();
  const int sl = nb / C;
  cluster.sync();  // every CTA's histogram is complete
  uint32_t part = 0;
  for (int i = tid; i < sl; i += kTkThreads) {
    uint32_t v = 0;
#pragma unroll
    for (int c = 0; c < C; ++c) v += *cluster.map_shared_rank(hist + r * sl + i, c);
    slice[i] = v;
    part += v;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
  if (lane == 0) tmp->wsum[warp] = part;
  __syncthreads();
  if (tid == 0) {
    uint32_t t = 0;
    for (int w = 0; w < kTkWarps; ++w) t += tmp->wsum[w];
    *s_tot = t;
  }
  cluster.sync();  // every slice and slice total is complete
  if (tid < C) tmp->tot[tid] = *cluster.map_shared_rank(s_tot, tid);
  __syncthreads();
  if (tid == 0) {
    uint32_t cum = 0;
    int R = C - 1;
    for (; R > 0; --R) {
      if (cum + tmp->tot[R] >= target) break;
      cum += tmp->tot[R];
    }
    tmp->R = R;
    tmp->cum = cum;
  }
  __syncthreads();
  const int R = tmp->R;
  // the other CTAs no longer read this CTA's `hist`: reuse it for slice R
  for (int i = tid; i < sl; i += kTkThreads) hist[i] = *cluster.map_shared_rank(slice + i, R);
  __syncthreads();
  find_top(hist, sl, target - tmp->cum, tmp);
  if (tid == 0) {
    tmp->T = (uint32_t)(R * sl + tmp->t);
    tmp->A = tmp->cum + tmp->above;
    tmp->cnt = hist[tmp->t];
  }
  __syncthreads();
}

template <int C>
__global__ void __launch_bounds__(kTkThreads, 1)
    topk_select_kernel(const float* __restrict__ scores, int64_t n, int64_t ld,
                       const int32_t* __restrict__ n_valid, int32_t k,
                       uint32_t* __restrict__ hist1, int32_t* __restrict__ idx_out,
                       int64_t idx_ld, int vec, const int32_t* __restrict__ remap,
                       int64_t remap_ld, int clear) {
  cg::cluster_group cluster = cg::this_cluster();
  extern __shared__ __align__(16) uint8_t dyn[];
  uint32_t* lkey = reinterpret_cast<uint32_t*>(dyn);
  int32_t* lj = reinterpret_cast<int32_t*>(dyn + kTkWarps * kLCap * 4);
  __shared__ uint32_t hist[kBins];
  __shared__ uint32_t slice[kBins / C];
  __shared__ TkTmp tmp;
  __shared__ uint32_t s_tot, s_gt, s_tie, s_off, s_quota;
  __shared__ uint32_t wgt[kTkWarps], wtie[kTkWarps];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_wait();
  const int r = (int)cluster.block_rank();
  const int64_t row = blockIdx.x / C;
  const int64_t nv = row_nvalid(n_valid, row, n);
  int32_t* out = idx_out + row * idx_ld;
  // The row's histogram goes back to zero once read (unless the caller
  // selects from it again), ready for the next selection that uses the same
  // workspace: CTA r clears bins r*512 .. (after every CTA has read them).
  // With `remap`, entry j of the row stands for remap[row * remap_ld + j]
  // (its position in a candidate pool) and that is what is written.
  uint32_t* hrow = hist1 + row * kBins;
  const int32_t* rmap = remap ? remap + row * remap_ld : nullptr;
  if (nv <= k) {  // every visible entry is selected (the whole cluster returns here)
    for (int64_t i = (int64_t)r * kTkThreads + tid; i < k; i += (int64_t)C * kTkThreads)
      out[i] = i < nv ? (rmap ? rmap[i] : (int32_t)i) : -1;
    if (clear)
      for (int i = tid; i < kBins / C; i += kTkThreads) hrow[r * (kBins / C) + i] = 0;
    return;
  }
  const float* s = scores + row * ld;

  // ---- level 1: threshold bin from the row's histogram (all loads in flight)
  {
    uint32_t hv[kBins / kTkThreads];
#pragma unroll
    for (int u = 0; u < kBins / kTkThreads; ++u) hv[u] = hrow[tid + u * kTkThreads];
#pragma unroll
    for (int u = 0; u < kBins / kTkThreads; ++u) hist[tid + u * kTkThreads] = hv[u];
  }
  __syncthreads();
  find_top(hist, kBins, (uint32_t)k, &tmp);
  const uint32_t T1 = (uint32_t)tmp.t;
  uint32_t need = (uint32_t)k - tmp.above;
  const uint32_t cnt1 = hist[T1];

  // ---- this CTA's chunk; warp w scans its contiguous segment in order and
  // keeps (key, index) of every entry in a bin >= T1
  const int64_t chunk = (((nv + C - 1) / C) + 31) & ~(int64_t)31;
  const int64_t j0 = min(nv, (int64_t)r * chunk), j1 = min(nv, j0 + chunk);
  const int64_t seg = (((chunk + kTkWarps - 1) / kTkWarps) + 31) & ~(int64_t)31;
  const int64_t wj0 = min(j1, j0 + warp * seg), wj1 = min(j1, wj0 + seg);
  uint32_t* mykey = lkey + warp * kLCap;
  int32_t* myj = lj + warp * kLCap;
  uint32_t cnt = 0;
  {
    constexpr int U = 8;  // 8 x 4 scores per lane in flight
    for (int64_t base = wj0; base < wj1; base += 128 * U) {
      float4 x[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t j = base + u * 128 + lane * 4;
        if (vec && j + 3 < wj1) {
          x[u] = __ldcs(reinterpret_cast<const float4*>(s + j));
        } else {
          x[u].x = j < wj1 ? s[j] : 0.f;
          x[u].y = j + 1 < wj1 ? s[j + 1] : 0.f;
          x[u].z = j + 2 < wj1 ? s[j + 2] : 0.f;
          x[u].w = j + 3 < wj1 ? s[j + 3] : 0.f;
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t j = base + u * 128 + lane * 4;
        const float xv[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
        uint32_t key[4];
        bool p[4];
        uint32_t c = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          key[e] = score_key(xv[e]);
          p[e] = (j + e < wj1) && (key[e] >> 20) >= T1;
          c += p[e];
        }
        // most steps hold no entry in the top bins: skip the lane scan
        if (__ballot_sync(0xffffffffu, c != 0) == 0) continue;
        uint32_t incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += v;
        }
        uint32_t pos = cnt + incl - c;
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (p[e]) {
            if (pos < (uint32_t)kLCap) {
              mykey[pos] = key[e];
              myj[pos] = (int32_t)(j + e);
            }
            ++pos;
          }
        cnt += __shfl_sync(0xffffffffu, incl, 31);
      }
    }
  }
  // A warp whose list overflowed re-reads its segment instead (rare: it needs
  // more than kLCap entries in the top bins of one segment).
  const bool ovf = cnt > (uint32_t)kLCap;
  // f(key, index, valid) over the warp's kept entries in index order; all
  // lanes take the same number of steps.
  auto walk = [&](auto&& f) {
    if (!ovf) {
      for (uint32_t base = 0; base < cnt; base += 32) {
        const uint32_t i = base + lane;
        const bool v = i < cnt;
        f(v ? mykey[i] : 0u, v ? myj[i] : 0, v);
      }
    } else {
      for (int64_t base = wj0; base < wj1; base += 32) {
        const int64_t j = base + lane;
        bool v = j < wj1;
        const uint32_t key = v ? score_key(s[j]) : 0u;
        v = v && (key >> 20) >= T1;
        f(key, (int32_t)j, v);
      }
    }
  };
  __syncwarp();

  // ---- levels 2 and 3 (only while the threshold bin holds surplus entries)
  int depth = 1;        // key digits resolved: 1 -> 12 bits, 2 -> 24, 3/4 -> 32
  uint32_t thr = T1;    // threshold key prefix
  if (cnt1 != need) {
    __syncthreads();
    for (int i = tid; i < kBins; i += kTkThreads) hist[i] = 0;
    __syncthreads();
    walk([&](uint32_t key, int32_t, bool v) {
      if (v && (key >> 20) == T1) atomicAdd(&hist[(key >> 8) & (kBins - 1)], 1u);
    });
    __syncthreads();
    cluster_top<C>(cluster, hist, slice, &s_tot, kBins, need, &tmp);
    need -= tmp.A;
    depth = 2;
    thr = (T1 << 12) | tmp.T;
    if (tmp.cnt != need) {
      for (int i = tid; i < kBins3; i += kTkThreads) hist[i] = 0;
      __syncthreads();
      const uint32_t t12 = thr;
      walk([&](uint32_t key, int32_t, bool v) {
        if (v && (key >> 8) == t12) atomicAdd(&hist[key & (kBins3 - 1)], 1u);
      });
      __syncthreads();
      cluster_top<C>(cluster, hist, slice, &s_tot, kBins3, need, &tmp);
      need -= tmp.A;
      thr = (thr << 8) | tmp.T;
      depth = tmp.cnt != need ? 4 : 3;
    }
  }
  const int shift = depth == 1 ? 20 : (depth == 2 ? 8 : 0);
  // g: kept for sure; t: a tie on the full key, kept in index order up to `need`
  auto is_g = [&](uint32_t key) {
    return (key >> shift) > thr || (depth <= 3 && (key >> shift) == thr);
  };
  auto is_t = [&](uint32_t key) { return depth == 4 && key == thr; };

  // ---- counts, offsets, output
  uint32_t ng = 0, nt = 0;
  walk([&](uint32_t key, int32_t, bool v) {
    ng += __popc(__ballot_sync(0xffffffffu, v && is_g(key)));
    nt += __popc(__ballot_sync(0xffffffffu, v && is_t(key)));
  });
  if (lane == 0) {
    wgt[warp] = ng;
    wtie[warp] = nt;
  }
  __syncthreads();
  if (tid == 0) {
    uint32_t g = 0, t = 0;
    for (int w = 0; w < kTkWarps; ++w) {
      g += wgt[w];
      t += wtie[w];
    }
    s_gt = g;
    s_tie = t;
  }
  cluster.sync();  // every CTA's counts are visible
  if (tid < C) {  // every CTA's counts, one remote load per thread
    tmp.tot[tid] = *cluster.map_shared_rank(&s_gt, tid);
    tmp.wsum[tid] = *cluster.map_shared_rank(&s_tie, tid);
  }
  cluster.sync();  // no CTA reads another's shared memory after this point
  // every CTA read the row's histogram at its start: clear this CTA's share
  if (clear)
    for (int i = tid; i < kBins / C; i += kTkThreads) hrow[r * (kBins / C) + i] = 0;
  if (tid == 0) {
    uint32_t pre_sel = 0, pre_tie = 0;
    for (int c = 0; c < r; ++c) {
      const uint32_t qc = min(tmp.wsum[c], need > pre_tie ? need - pre_tie : 0u);
      pre_tie += tmp.wsum[c];
      pre_sel += tmp.tot[c] + qc;
    }
    s_quota = min(s_tie, need > pre_tie ? need - pre_tie : 0u);
    s_off = pre_sel;
  }
  __syncthreads();
  uint32_t woff = s_off, tq = s_quota;
  for (int w = 0; w < warp; ++w) {
    const uint32_t qw = min(wtie[w], tq);
    tq -= qw;
    woff += wgt[w] + qw;
  }
  const uint32_t myq = min(wtie[warp], tq);
  pdl_trigger();
  uint32_t run_sel = 0, run_tie = 0;
  const uint32_t lt = lanemask_lt();
  walk([&](uint32_t key, int32_t j, bool v) {
    const bool g = v && is_g(key);
    const bool t = v && is_t(key);
    const uint32_t tm = __ballot_sync(0xffffffffu, t);
    const bool sel = g || (t && run_tie + __popc(tm & lt) < myq);
    const uint32_t sm = __ballot_sync(0xffffffffu, sel);
    const uint32_t pos = woff + run_sel + __popc(sm & lt);
    if (sel && pos < (uint32_t)k) out[pos] = rmap ? rmap[j] : j;
    run_sel += __popc(sm);
    run_tie += __popc(tm);
  });
}

// ---------------------------------------------------------------------------
// short rows (a candidate pool): one CTA per row, every key in shared memory

constexpr int kSmallN = 4096;  // longest row

// Row r of n <= kSmallN values (the first n_valid[r] of them when n_valid
// is given): value i is scores[r * ld + i], or with `gather` scores[r * ld +
// gather[r * gather_ld + i]] (an index < 0 is an empty slot, below every
// value).  The k largest (value descending, position
// ascending) are written ascending by position to out[r * out_ld ..] as
// remap[r * remap_ld + i] (remap may be null: i), padded with -1.  The
// same radix select as topk_select_kernel, on one CTA: 12 / 12 / 8-bit
// digits, then ties on the whole key in position order.
__global__ void __launch_bounds__(kTkThreads)
    topk_small_kernel(const float* __restrict__ scores, int64_t ld,
                      const int32_t* __restrict__ gather, int64_t gather_ld, int32_t n_row,
                      const int32_t* __restrict__ n_valid, int32_t k,
                      const int32_t* __restrict__ remap, int64_t remap_ld,
                      int32_t* __restrict__ out, int64_t out_ld) {
  __shared__ uint32_t key[kSmallN];
  __shared__ uint32_t hist[kBins];
  __shared__ TkTmp tmp;
  __shared__ uint32_t wg[kTkWarps], wt[kTkWarps];
  pdl_wait();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t row = blockIdx.x;
  const int n = (int)row_nvalid(n_valid, row, n_row);  // positions >= n_valid[row] do not exist
  const float* s = scores + row * ld;
  const int32_t* gi = gather ? gather + row * gather_ld : nullptr;
  const int32_t* rm = remap ? remap + row * remap_ld : nullptr;
  int32_t* o = out + row * out_ld;
  for (int i = tid; i < kBins; i += kTkThreads) hist[i] = 0;
  __syncthreads();
  for (int i = tid; i < n; i += kTkThreads) {
    uint32_t kk = 0;  // an empty slot
    if (!gi) {
      kk = score_key(s[i]);
    } else {
      const int32_t j = gi[i];
      if (j >= 0) kk = score_key(s[j]);
    }
    key[i] = kk;
    atomicAdd(&hist[kk >> 20], 1u);
  }
  __syncthreads();
  const int m = min(k, n);
  if (m == 0) {  // an empty row (the whole CTA returns here)
    for (int i = tid; i < k; i += kTkThreads) o[i] = -1;
    return;
  }
  // threshold: depth 1 (12 bits), 2 (24), 3 (32) or 4 (32 bits, ties)
  find_top(hist, kBins, (uint32_t)m, &tmp);
  uint32_t thr = (uint32_t)tmp.t;
  uint32_t need = (uint32_t)m - tmp.above;
  uint32_t cnt = hist[thr];
  int depth = 1;
  if (cnt != need) {
    __syncthreads();
    for (int i = tid; i < kBins; i += kTkThreads) hist[i] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += kTkThreads)
      if ((key[i] >> 20) == thr) atomicAdd(&hist[(key[i] >> 8) & (kBins - 1)], 1u);
    __syncthreads();
    find_top(hist, kBins, need, &tmp);
    need -= tmp.above;
    thr = (thr << 12) | (uint32_t)tmp.t;
    cnt = hist[tmp.t];
    depth = 2;
    if (cnt != need) {
      __syncthreads();
      for (int i = tid; i < kBins3; i += kTkThreads) hist[i] = 0;
      __syncthreads();
      for (int i = tid; i < n; i += kTkThreads)
        if ((key[i] >> 8) == thr) atomicAdd(&hist[key[i] & (kBins3 - 1)], 1u);
      __syncthreads();
      find_top(hist, kBins3, need, &tmp);
      need -= tmp.above;
      thr = (thr << 8) | (uint32_t)tmp.t;
      cnt = hist[tmp.t];
      depth = cnt != need ? 4 : 3;
    }
  }
  const int shift = depth == 1 ? 20 : (depth == 2 ? 8 : 0);
  // thread t owns positions [t * per, (t + 1) * per): counts, then offsets
  const int per = (n + kTkThreads - 1) / kTkThreads;
  const int i0 = min(n, tid * per), i1 = min(n, i0 + per);
  uint32_t g = 0, t = 0;
  for (int i = i0; i < i1; ++i) {
    const uint32_t x = key[i] >> shift;
    g += x > thr || (depth <= 3 && x == thr);
    t += depth == 4 && key[i] == thr;
  }
  // block-wide exclusive scans of g and t
  uint32_t ig = g, it = t;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t vg = __shfl_up_sync(0xffffffffu, ig, d);
    const uint32_t vt = __shfl_up_sync(0xffffffffu, it, d);
    if (lane >= d) {
      ig += vg;
      it += vt;
    }
  }
  if (lane == 31) {
    wg[warp] = ig;
    wt[warp] = it;
  }
  __syncthreads();
  uint32_t bg = 0, bt = 0;
  for (int w = 0; w < warp; ++w) {
    bg += wg[w];
    bt += wt[w];
  }
  uint32_t gpre = bg + ig - g, tpre = bt + it - t;  // before this thread's range
  // ties before this range taken (at most need), so positions before it
  uint32_t pos = gpre + min(tpre, need);
  for (int i = i0; i < i1; ++i) {
    const uint32_t x = key[i] >> shift;
    bool sel = x > thr || (depth <= 3 && x == thr);
    if (!sel && depth == 4 && key[i] == thr) sel = tpre++ < need;
    if (sel) {
      if (pos < (uint32_t)m) o[pos] = rm ? rm[i] : i;
      ++pos;
    }
  }
  pdl_trigger();
  for (int i = m + tid; i < k; i += kTkThreads) o[i] = -1;
}

std::atomic<uint64_t> g_select_attr{0};  // devices on which the selector's attributes are set

}  // namespace

size_t topk_workspace_bytes(int64_t rows, int64_t n, int32_t k) {
  (void)n;
  (void)k;
  return (size_t)rows * kBins * sizeof(uint32_t);
}

csa2_status clear_topk_hist(uint32_t* hist1, int64_t rows, cudaStream_t s) {
  if (rows == 0) return CSA2_OK;
  cudaError_t e = cudaMemsetAsync(hist1, 0, (size_t)rows * kBins * sizeof(uint32_t), s);
  return e == cudaSuccess ? CSA2_OK : cuda_fail(e);
}

csa2_status launch_topk_select(const float* scores, int64_t rows, int64_t n, int64_t ld,
                               const int32_t* n_valid, int32_t k, uint32_t* hist1,
                               int32_t* idx_out, int64_t idx_ld, cudaStream_t s,
                               const int32_t* remap, int64_t remap_ld, bool clear_hist) {
  if (rows == 0) return CSA2_OK;
  cudaError_t e = once_per_device(g_select_attr, [] {
    return cudaFuncSetAttribute(topk_select_kernel<kTkCluster>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, kTkDynSmem);
  });
  if (e != cudaSuccess) return cuda_fail(e);
  const int vec = (ld % 4 == 0 && (reinterpret_cast<uintptr_t>(scores) % 16) == 0) ? 1 : 0;
  return launch_kernel(topk_select_kernel<kTkCluster>, dim3((unsigned)(rows * kTkCluster)),
                       dim3(kTkThreads), (size_t)kTkDynSmem, s, kTkCluster, scores, n, ld, n_valid,
                       k, hist1, idx_out, idx_ld, vec, remap, remap_ld, clear_hist ? 1 : 0);
}

csa2_status launch_topk_small(const float* scores, int64_t ld, const int32_t* gather,
                              int64_t gather_ld, int64_t rows, int32_t n, const int32_t* n_valid,
                              int32_t k, const int32_t* remap, int64_t remap_ld, int32_t* idx_out,
                              int64_t idx_ld, cudaStream_t s) {
  if (rows == 0) return CSA2_OK;
  if (n < 0 || n > kSmallN || k < 1 || k > kMaxK) return CSA2_ERR_UNSUPPORTED;
  return launch_kernel(topk_small_kernel, dim3((unsigned)rows), dim3(kTkThreads), 0, s, 1, scores,
                       ld, gather, gather_ld, n, n_valid, k, remap, remap_ld, idx_out, idx_ld);
}

csa2_status launch_topk_hist(const float* scores, int64_t rows, int64_t n, int64_t ld,
                             const int32_t* n_valid, uint32_t* hist1, cudaStream_t s) {
  if (rows == 0 || n == 0) return CSA2_OK;
  // enough CTAs to cover the GPU about twice
  const int64_t want = (2 * (int64_t)sm_count() + rows - 1) / rows;
  const int64_t max_chunks = (n + 4095) / 4096;
  const int64_t chunks = std::max<int64_t>(1, std::min<int64_t>(want, max_chunks));
  const int64_t chunk = (n + chunks - 1) / chunks;
  return launch_kernel(topk_hist_kernel, dim3((unsigned)chunks, (unsigned)rows),
                       dim3(kHistThreads), 0, s, 1, scores, n, ld, n_valid, hist1, chunk);
}

csa2_status launch_topk(const float* scores, int64_t rows, int64_t n, int64_t ld,
                        const int32_t* n_valid, int32_t k, int32_t* idx_out, int64_t idx_ld,
                        void* ws, int32_t* dev_status, cudaStream_t s) {
  (void)dev_status;
  if (rows == 0) return CSA2_OK;
  // short rows: one CTA per row with every key in shared memory
  if (n <= kSmallN)
    return launch_topk_small(scores, ld, nullptr, 0, rows, (int32_t)n, n_valid, k, nullptr, 0,
                             idx_out, idx_ld, s);
  uint32_t* hist1 = static_cast<uint32_t*>(ws);
  csa2_status st = clear_topk_hist(hist1, rows, s);
  if (st != CSA2_OK) return st;
  if ((st = launch_topk_hist(scores, rows, n, ld, n_valid, hist1, s)) != CSA2_OK) return st;
  return launch_topk_select(scores, rows, n, ld, n_valid, k, hist1, idx_out, idx_ld, s);
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

// Device address of the array.  Host code cannot use the array's name as a
// device pointer, so the address is looked up with cudaGetSymbolAddress,
// with the device current, and kept per device together with the unique ID
// of the CUDA context it was looked up in.  A call made in another context
// (after cudaDeviceReset, or from a context other than the primary one)
// looks it up again: the library's module, and with it the array, may then
// sit at another address.  Context IDs are never reused within a process.
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64] = {nullptr};
unsigned long long g_noalloc_ctx[64] = {0};

// Unique ID of the calling thread's current context (0 if there is none or
// the driver cannot say).
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static bool looked = false;
  if (!looked) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
    looked = true;
  }
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

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
  csa2_status st = injected("topk_noalloc");
  if (st != CSA2_OK) return st;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= 64) return CSA2_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    unsigned long long ctx = current_context_id();
    if (!g_noalloc_ptr[dev] || ctx == 0 || ctx != g_noalloc_ctx[dev]) {
      e = cudaGetSymbolAddress(&scratch, g_topk_noalloc_scratch);
      if (e != cudaSuccess) return cuda_fail(e);
      g_noalloc_ptr[dev] = scratch;
      // the lookup made the context current if there was none
      g_noalloc_ctx[dev] = ctx != 0 ? ctx : current_context_id();
    }
    scratch = g_noalloc_ptr[dev];
  }
  // launch_topk clears the parts of the scratch that must start at zero
  return launch_topk(scores, rows, n, ld, n_valid, k, idx_out, idx_ld, scratch, dev_status,
                     reinterpret_cast<cudaStream_t>(stream));
}
