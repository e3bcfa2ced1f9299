// topk.cu -- a4, per-row top-k with the lowest index winning ties.
//
// Full mode selects new Top-512 entries for each query ("Unlocking Extreme
// Context Scaling with DeepSeek-V4.1-Flash", "Compressed Sparse Attention 2
// (CSA2)").  Order is (score descending, index ascending); the output row
// holds the chosen indices ascending, padded with -1.
//
// Radix select on an order-preserving 32-bit key (+0 and -0 share a key).
// Level 1 is the row's 4096-bin histogram of the key's top 12 bits; it comes
// from global memory (topk_hist_kernel, or the indexer epilogue that
// produced the scores).  Its threshold bin T1 splits the row into entries
// surely selected (bins above T1), candidates (bin T1) and the rest.
//
// Long rows (topk_scan_kernel): a row is cut into S slices, one CTA each.
// Every CTA finds T1 from the histogram, scans its slice once and keeps the
// entries in bins >= T1, in index order, in shared memory; with S > 1 it
// publishes them to its slot in the workspace and the last CTA of the row to
// finish (an atomic counter) gathers every slot.  That CTA then resolves the
// threshold bin among the gathered entries (next 12, then 8 key bits, then
// ties on the whole key in index order) and writes the selection ascending.
// A slice with more kept entries than its slot holds (massive ties, sorted
// rows) makes the last CTA run the same levels as passes over the whole row
// in global memory instead: slower, same result.
//
// Short rows (topk_small_kernel, n <= 4096): one CTA per row with every key
// in shared memory, the same levels.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace csa2 {

namespace {

constexpr int kBins = kTopkBins;    // 12-bit digits (levels 1 and 2)
constexpr int kBins3 = 256;         // 8-bit digit (level 3)
constexpr int kMaxK = 2048;
constexpr int kTkThreads = 512;
constexpr int kTkWarps = kTkThreads / 32;
constexpr int kHistThreads = 512;
constexpr int kRound = kTkThreads * 4;        // scores per round: one float4 per thread
constexpr int kRounds = 4;                    // rounds whose loads are in flight together
constexpr int kBatch = kRound * kRounds;      // 8192 scores per batch
constexpr int kCandCap = 8192;                // kept entries a CTA holds in shared memory
constexpr int kSlotCap = 1024;                // kept entries a slice may publish
constexpr int kMaxSlices = 64;
constexpr int kSliceTarget = 296;             // CTAs of one launch to aim for (2 per SM)
constexpr int kSmallN = (int)kTopkShortRow;   // longest row of topk_small_kernel
// dynamic shared memory of topk_scan_kernel: histogram (fine and coarse
// bins) | keys | indices
constexpr int kScanSmem = (kTopkHistStride + 2 * kCandCap) * 4;

__device__ __forceinline__ int64_t row_nvalid(const int32_t* n_valid, int64_t row, int64_t n) {
  int64_t nv = n_valid ? (int64_t)n_valid[row] : n;
  return nv < 0 ? 0 : (nv > n ? n : nv);
}

// ---------------------------------------------------------------------------
// level-1 histogram of a row's visible keys (when the scores come from
// elsewhere than the fused indexer epilogue)
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(kHistThreads)
    topk_hist_kernel(const float* __restrict__ scores, int64_t n, int64_t ld,
                     const int32_t* __restrict__ n_valid, uint32_t* __restrict__ hist1,
                     int64_t chunk, const uint32_t* __restrict__ within, int vec, int exclusive) {
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
  // level 1: every key by its top 12 bits; within a bin: that bin's keys by
  // their next 12 bits
  const bool sub = within != nullptr;
  const uint32_t t1 = sub ? within[row] >> 20 : 0u;
  auto count = [&](float x) {
    const uint32_t key = score_key(x);
    if (!sub || (key >> 20) == t1) atomicAdd(&h[sub ? (key >> 8) & (kBins - 1) : key >> 20], 1u);
  };
  constexpr int U = 4;
  if (vec) {
    // 16 scores per thread in flight: float4 u of thread t at b + 2048 u + 4 t
    // (chunks start on multiples of 4 scores)
    for (int64_t b = j0; b < j1; b += (int64_t)kHistThreads * 4 * U) {
      float4 x[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t j = b + (int64_t)u * kHistThreads * 4 + 4 * tid;
        if (j + 3 < j1) {
          x[u] = __ldcs(reinterpret_cast<const float4*>(s + j));
        } else {
          x[u].x = j < j1 ? s[j] : 0.f;
          x[u].y = j + 1 < j1 ? s[j + 1] : 0.f;
          x[u].z = j + 2 < j1 ? s[j + 2] : 0.f;
          x[u].w = j + 3 < j1 ? s[j + 3] : 0.f;
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t j = b + (int64_t)u * kHistThreads * 4 + 4 * tid;
        if (j < j1) count(x[u].x);
        if (j + 1 < j1) count(x[u].y);
        if (j + 2 < j1) count(x[u].z);
        if (j + 3 < j1) count(x[u].w);
      }
    }
  } else {
    for (int64_t base = j0 + warp * 32; base < j1; base += (int64_t)kHistThreads * U) {
      float x[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t j = base + u * kHistThreads + lane;
        x[u] = j < j1 ? s[j] : 0.f;
      }
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (base + u * kHistThreads + lane < j1) count(x[u]);
    }
  }
  __syncthreads();
  pdl_trigger();
  uint32_t* hrow = hist1 + row * kTopkHistStride;
  if (exclusive) {  // the row's only CTA: its counts are the row's (stores, no atomics)
    for (int i = tid; i < kBins; i += kHistThreads) hrow[i] = h[i];
    if (tid < kTopkCoarse) {
      uint32_t v = 0;
      for (int i = 0; i < kBins / kTopkCoarse; ++i) v += h[tid * (kBins / kTopkCoarse) + i];
      hrow[kBins + tid] = v;
    }
    return;
  }
  for (int i = tid; i < kBins; i += kHistThreads)
    if (h[i]) atomicAdd(&hrow[i], h[i]);
  if (tid < kTopkCoarse) {  // coarse bin t: fine bins 64t .. 64t + 63
    uint32_t v = 0;
    for (int i = 0; i < kBins / kTopkCoarse; ++i) v += h[tid * (kBins / kTopkCoarse) + i];
    if (v) atomicAdd(&hrow[kBins + tid], v);
  }
}

// ---------------------------------------------------------------------------
// block-wide pieces of the selection (kTkThreads threads)
// ---------------------------------------------------------------------------

struct TkTmp {
  uint32_t wsum[kTkWarps * kRounds];
  int t;            // find_top: bin
  uint32_t above;   // find_top: entries in higher bins
  uint32_t total;   // scans: running count
  uint32_t flag;
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
  // exclusive prefix of the warp totals: lane w < kTkWarps of every warp
  // scans them (kTkWarps <= 32)
  uint32_t wv = lane < kTkWarps ? tmp->wsum[lane] : 0u;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, wv, o);
    if (lane >= o) wv += y;
  }
  const uint32_t woff = __shfl_sync(0xffffffffu, wv, (warp + 31) & 31) * (warp > 0);
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

// The threshold below level 1: among the entries whose top 12 key bits equal
// T1 (cnt1 of them), `need` more are selected.  Resolves the next 12 and 8
// key bits through histograms built by `each` (each(f) calls f(key) for
// every entry) and returns depth / thr: depth 1, 2, 3 -> an entry is selected
// iff (key >> shift) > thr or == thr (shift 20, 8, 0); depth 4 -> (key > thr)
// or (key == thr and it is among the first `need` such entries in index
// order).  `hist` is overwritten.
struct Threshold {
  int depth;
  uint32_t thr, need;
  __device__ int shift() const { return depth == 1 ? 20 : (depth == 2 ? 8 : 0); }
  __device__ bool sure(uint32_t key) const {
    const uint32_t x = key >> shift();
    return x > thr || (depth <= 3 && x == thr);
  }
  __device__ bool tie(uint32_t key) const { return depth == 4 && key == thr; }
};

template <class Each>
__device__ Threshold resolve_threshold(uint32_t T1, uint32_t need, uint32_t cnt1, uint32_t* hist,
                                       TkTmp* tmp, Each&& each) {
  const int tid = threadIdx.x;
  Threshold th{1, T1, need};
  if (cnt1 == need) return th;
  __syncthreads();
  for (int i = tid; i < kBins; i += kTkThreads) hist[i] = 0;
  __syncthreads();
  each([&](uint32_t key) {
    if ((key >> 20) == T1) atomicAdd(&hist[(key >> 8) & (kBins - 1)], 1u);
  });
  __syncthreads();
  find_top(hist, kBins, th.need, tmp);
  th.need -= tmp->above;
  th.thr = (T1 << 12) | (uint32_t)tmp->t;
  th.depth = 2;
  if (hist[tmp->t] == th.need) return th;
  __syncthreads();
  for (int i = tid; i < kBins3; i += kTkThreads) hist[i] = 0;
  __syncthreads();
  const uint32_t t12 = th.thr;
  each([&](uint32_t key) {
    if ((key >> 8) == t12) atomicAdd(&hist[key & (kBins3 - 1)], 1u);
  });
  __syncthreads();
  find_top(hist, kBins3, th.need, tmp);
  th.need -= tmp->above;
  th.thr = (th.thr << 8) | (uint32_t)tmp->t;
  th.depth = hist[tmp->t] != th.need ? 4 : 3;
  __syncthreads();
  return th;
}

// Scores [j0, j1) of row s in index order, kBatch at a time (each thread a
// float4 per round, the rounds' loads in flight together).  cls(key, j)
// returns 0 (skip), 1 (take) or 2 (a tie: taken while fewer than `quota`
// ties precede it in index order).  emit(pos, key, j) receives every taken
// entry with its rank among taken entries.  Returns the number taken.
// Block-wide (every thread calls it with the same arguments).
// This thread's float4s of the batch starting at b0 (scores [b0, j1)).
__device__ __forceinline__ void load_batch(const float* __restrict__ s, int64_t b0, int64_t j1,
                                           int vec, float4* x) {
  const int tid = threadIdx.x;
#pragma unroll
  for (int u = 0; u < kRounds; ++u) {
    const int64_t j = b0 + (int64_t)u * kRound + tid * 4;
    if (vec && j + 3 < j1) {
      x[u] = __ldcs(reinterpret_cast<const float4*>(s + j));
    } else {
      x[u].x = j < j1 ? s[j] : 0.f;
      x[u].y = j + 1 < j1 ? s[j + 1] : 0.f;
      x[u].z = j + 2 < j1 ? s[j + 2] : 0.f;
      x[u].w = j + 3 < j1 ? s[j + 3] : 0.f;
    }
  }
}

template <class Cls, class Emit>
__device__ uint32_t ordered_take(const float* __restrict__ s, int64_t j0, int64_t j1, int vec,
                                 uint32_t quota, TkTmp* tmp, Cls&& cls, Emit&& emit) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t taken1 = 0, ties = 0;  // block-uniform: class-1 entries and ties of earlier batches
  for (int64_t b0 = j0; b0 < j1; b0 += kBatch) {
    float4 x[kRounds];
    load_batch(s, b0, j1, vec, x);
    uint32_t c[kRounds], incl[kRounds];
    uint32_t cl[kRounds];  // 2 bits per element: its class
#pragma unroll
    for (int u = 0; u < kRounds; ++u) {
      const int64_t j = b0 + (int64_t)u * kRound + tid * 4;
      const float xv[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
      uint32_t packed = 0, cnt = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t k2 = (j + e < j1) ? cls(score_key(xv[e]), j + e) : 0u;
        packed |= k2 << (2 * e);
        cnt += (k2 == 1u) + ((k2 == 2u) << 16);  // low half: takes, high half: ties
      }
      cl[u] = packed;
      c[u] = cnt;
      uint32_t v = cnt;
      if (__ballot_sync(0xffffffffu, cnt != 0)) {  // most rounds of a warp keep nothing
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(0xffffffffu, v, o);
          if (lane >= o) v += y;
        }
      }
      incl[u] = v;
      if (lane == 31) tmp->wsum[u * kTkWarps + warp] = v;
    }
    __syncthreads();
    if (warp == 0) {
      // exclusive prefix over (round, warp) in index order; ties are capped
      // by the quota only when positions are assigned below
      uint32_t v[kRounds * kTkWarps / 32];
      uint32_t run = 0;
#pragma unroll
      for (int i = 0; i < kRounds * kTkWarps / 32; ++i) {
        const uint32_t w = tmp->wsum[i * 32 + lane];
        uint32_t sc = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(0xffffffffu, sc, o);
          if (lane >= o) sc += y;
        }
        v[i] = run + sc - w;
        run += __shfl_sync(0xffffffffu, sc, 31);
      }
      __syncwarp();
#pragma unroll
      for (int i = 0; i < kRounds * kTkWarps / 32; ++i) tmp->wsum[i * 32 + lane] = v[i];
      if (lane == 0) tmp->total = run;
    }
    __syncthreads();
    const uint32_t batch_total = tmp->total;
#pragma unroll
    for (int u = 0; u < kRounds; ++u) {
      if (__ballot_sync(0xffffffffu, c[u] != 0) == 0) continue;
      // rank among taken entries: class-1 entries before it plus the ties
      // before it, capped by the quota
      const uint32_t before = tmp->wsum[u * kTkWarps + warp] + incl[u] - c[u];
      uint32_t t_before = ties + (before >> 16);
      uint32_t c1 = taken1 + (before & 0xFFFFu);
      const int64_t j = b0 + (int64_t)u * kRound + tid * 4;
      const float xv[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t k2 = (cl[u] >> (2 * e)) & 3u;
        if (k2 == 1u || (k2 == 2u && t_before < quota))
          emit(c1 + min(t_before, quota), score_key(xv[e]), j + e);
        c1 += k2 == 1u;
        t_before += k2 == 2u;
      }
    }
    taken1 += batch_total & 0xFFFFu;
    ties += batch_total >> 16;
    __syncthreads();  // tmp->wsum is rewritten by the next batch
  }
  return taken1 + min(ties, quota);
}

// Every key of the row, in any order (histogram passes of the fallback).
template <class F>
__device__ __forceinline__ void for_each_key(const float* __restrict__ s, int64_t nv, int vec,
                                             const F& f) {
  const int tid = threadIdx.x;
  for (int64_t b0 = 0; b0 < nv; b0 += kBatch) {
    float4 x[kRounds];
#pragma unroll
    for (int u = 0; u < kRounds; ++u) {
      const int64_t j = b0 + (int64_t)u * kRound + tid * 4;
      if (vec && j + 3 < nv) {
        x[u] = __ldcs(reinterpret_cast<const float4*>(s + j));
      } else {
        x[u].x = j < nv ? s[j] : 0.f;
        x[u].y = j + 1 < nv ? s[j + 1] : 0.f;
        x[u].z = j + 2 < nv ? s[j + 2] : 0.f;
        x[u].w = j + 3 < nv ? s[j + 3] : 0.f;
      }
    }
#pragma unroll
    for (int u = 0; u < kRounds; ++u) {
      const int64_t j = b0 + (int64_t)u * kRound + tid * 4;
      if (j < nv) f(score_key(x[u].x));
      if (j + 1 < nv) f(score_key(x[u].y));
      if (j + 2 < nv) f(score_key(x[u].z));
      if (j + 3 < nv) f(score_key(x[u].w));
    }
  }
}

// Writes the entries of key[0..nc) (positions in index order) that `th`
// selects, ascending by position, as map(position) to o[0..m), and -1 to
// o[m..k).  Thread t owns positions [t * per, (t + 1) * per).
// expand = G > 0: each selected position p goes out as the G entries p * G
// + t (t < G; -1 from expand_n on) in slots pos * G + t; o holds k * G slots.
template <class Map>
__device__ void write_selected(const uint32_t* key, int nc, const Threshold& th, uint32_t m,
                               int32_t k, int32_t* o, TkTmp* tmp, Map&& map, int32_t expand = 0,
                               int64_t expand_n = 0) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (nc + kTkThreads - 1) / kTkThreads;
  const int i0 = min(nc, tid * per), i1 = min(nc, i0 + per);
  uint32_t g = 0, t = 0;
  for (int i = i0; i < i1; ++i) {
    g += th.sure(key[i]);
    t += th.tie(key[i]);
  }
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
  __syncthreads();
  if (lane == 31) {
    tmp->wsum[warp] = ig;
    tmp->wsum[kTkWarps + warp] = it;
  }
  __syncthreads();
  uint32_t bg = 0, bt = 0;
  for (int w = 0; w < warp; ++w) {
    bg += tmp->wsum[w];
    bt += tmp->wsum[kTkWarps + w];
  }
  uint32_t tpre = bt + it - t;
  uint32_t pos = bg + ig - g + min(tpre, th.need);
  for (int i = i0; i < i1; ++i) {
    bool sel = th.sure(key[i]);
    if (!sel && th.tie(key[i])) sel = tpre++ < th.need;
    if (sel) {
      if (pos < m) {
        if (expand > 0) {
          const int64_t e0 = (int64_t)map(i) * expand;
          for (int t = 0; t < expand; ++t)
            o[(int64_t)pos * expand + t] = e0 + t < expand_n ? (int32_t)(e0 + t) : -1;
        } else {
          o[pos] = map(i);
        }
      }
      ++pos;
    }
  }
  const int64_t per_slot = expand > 0 ? expand : 1;
  for (int64_t i = (int64_t)m * per_slot + tid; i < (int64_t)k * per_slot; i += kTkThreads)
    o[i] = -1;
}

// ---------------------------------------------------------------------------
// long rows
// ---------------------------------------------------------------------------

// Lane l of the calling warp holds bins 63 - 2l and 62 - 2l of a 64-bin
// row: the largest bin b whose count from the top reaches target, the
// count above it (above) and its own count (returned).  bin = 0 / above = 0
// when the bins hold fewer than target entries.
// SH: the bins are in shared memory (else global memory, read through L2).
template <bool SH = false>
__device__ uint32_t pick64(const uint32_t* bins, uint32_t target, uint32_t& bin,
                          uint32_t& above) {
  const int lane = threadIdx.x & 31;
  const uint32_t hi = SH ? bins[63 - 2 * lane] : __ldcg(bins + 63 - 2 * lane);
  const uint32_t lo = SH ? bins[62 - 2 * lane] : __ldcg(bins + 62 - 2 * lane);
  uint32_t incl = hi + lo;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  const uint32_t before = incl - hi - lo;
  const uint32_t who = __ballot_sync(0xffffffffu, before < target && incl >= target);
  const int src = who ? __ffs(who) - 1 : 31;
  const bool in_hi = before + hi >= target;
  const uint32_t b = in_hi ? 63 - 2 * lane : 62 - 2 * lane;
  const uint32_t ab = in_hi ? before : before + hi;
  bin = who ? __shfl_sync(0xffffffffu, b, src) : 0u;
  above = who ? __shfl_sync(0xffffffffu, ab, src) : 0u;
  return __shfl_sync(0xffffffffu, in_hi ? hi : lo, src);
}

// Workspace of a long-row selection: per row its level-1 histogram, a
// counter (the slices done) and S slots of (count, kSlotCap keys, kSlotCap
// indices).
struct ScanLayout {
  int64_t rows;
  int S;
  __host__ __device__ size_t hist_bytes() const { return (size_t)rows * kTopkHistStride * 4; }
  __host__ __device__ size_t counter_off() const { return hist_bytes(); }
  __host__ __device__ size_t slot_off() const {
    return align256_hd(counter_off() + (size_t)rows * 16);
  }
  static constexpr size_t kSlotBytes = 16 + (size_t)kSlotCap * 8;
  __host__ __device__ size_t total() const {
    return S > 0 ? slot_off() + (size_t)rows * S * kSlotBytes : hist_bytes();
  }
  __host__ __device__ static size_t align256_hd(size_t x) { return (x + 255) & ~(size_t)255; }
};

// Slices per row: about kSliceTarget CTAs per launch (every CTA resident),
// each slice at least 4096 scores, at most kMaxSlices.  0 for short rows.
int scan_slices(int64_t rows, int64_t n) {
  if (n <= kSmallN || rows <= 0) return 0;
  const int64_t want = (kSliceTarget + rows - 1) / rows;
  const int64_t most = std::min<int64_t>(kMaxSlices, (n + 4095) / 4096);
  return (int)std::max<int64_t>(1, std::min(want, most));
}

__global__ void __launch_bounds__(kTkThreads, 2)
    topk_scan_kernel(const float* __restrict__ scores, int64_t n, int64_t ld,
                     const int32_t* __restrict__ n_valid, int32_t k,
                     uint32_t* __restrict__ hist1, uint32_t* __restrict__ counters,
                     uint8_t* __restrict__ slots, int S, int64_t slice,
                     int32_t* __restrict__ idx_out, int64_t idx_ld, int vec,
                     const int32_t* __restrict__ remap, int64_t remap_ld, int clear) {
  extern __shared__ __align__(16) uint32_t dyn[];
  uint32_t* hist = dyn;                                     // [kTopkHistStride]
  uint32_t* ckey = dyn + kTopkHistStride;                   // [kCandCap] kept keys
  int32_t* cidx = reinterpret_cast<int32_t*>(ckey + kCandCap);  // their indices
  __shared__ TkTmp tmp;
  __shared__ uint32_t s_last, s_base[kMaxSlices + 1], s_cnt[kMaxSlices];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_wait();
  const int64_t row = blockIdx.x / S;
  const int sl = (int)(blockIdx.x % S);
  const int64_t nv = row_nvalid(n_valid, row, n);
  const uint32_t m = (uint32_t)(nv < (int64_t)k ? nv : (int64_t)k);
  int32_t* out = idx_out + row * idx_ld;
  uint32_t* hrow = hist1 + row * kTopkHistStride;
  const int32_t* rmap = remap ? remap + row * remap_ld : nullptr;
  const float* s = scores + row * ld;
  if (nv <= k) {  // every visible entry is selected; slice 0 writes the row
    if (sl == 0) {
      for (int64_t i = tid; i < k; i += kTkThreads)
        out[i] = i < nv ? (rmap ? rmap[i] : (int32_t)i) : -1;
      if (clear)
        for (int i = tid; i < kTopkHistStride; i += kTkThreads) hrow[i] = 0;
    }
    return;
  }

  const int64_t j0 = min(nv, (int64_t)sl * slice), j1 = min(nv, j0 + slice);
  uint8_t* slot = slots + ((size_t)row * S + sl) * ScanLayout::kSlotBytes;
  uint32_t T1, need, cnt1, kept;
  if (S > 1) {
    // ---- a slice: in each batch of kBatch scores warp w takes the
    // contiguous 512 from b0 + 512 w (lane l the float4 at 128 u + 4 l, u <
    // kRounds).  The row's histogram and the first batch's scores are loaded
    // together; warp 0 then finds the threshold bin in shared memory
    // (coarse, then fine bins); the entries in bins >= T1 go straight to the
    // slot in index order, the only block-wide step per batch being the
    // prefix over the 16 warps' counts (double-buffered: one barrier per
    // batch).
    uint32_t* sk = reinterpret_cast<uint32_t*>(slot + 16);
    int32_t* sj = reinterpret_cast<int32_t*>(slot + 16 + (size_t)kSlotCap * 4);
    uint32_t* wtot = tmp.wsum;  // [2][kTkWarps] per-warp counts of a batch
    // the row's level-1 histogram (fine and coarse bins) into shared memory
    // in one round of cp.async, so the threshold bin costs one round trip
    for (int i = tid; i < kTopkHistStride / 4; i += kTkThreads)
      cp_async16(hist + 4 * i, hrow + 4 * i);
    float4 x[kRounds];
    auto load = [&](int64_t b0) {
      const int64_t wb = b0 + (int64_t)warp * (kBatch / kTkWarps);
#pragma unroll
      for (int u = 0; u < kRounds; ++u) {
        const int64_t j = wb + 128 * u + 4 * lane;
        if (vec && j + 3 < j1) {
          x[u] = __ldcs(reinterpret_cast<const float4*>(s + j));
        } else {
          x[u].x = j < j1 ? s[j] : 0.f;
          x[u].y = j + 1 < j1 ? s[j + 1] : 0.f;
          x[u].z = j + 2 < j1 ? s[j + 2] : 0.f;
          x[u].w = j + 3 < j1 ? s[j + 3] : 0.f;
        }
      }
    };
    if (j0 < j1) load(j0);  // the first batch's scores are in flight during the pick
    cp_async_wait_all();
    __syncthreads();
    if (warp == 0) {  // coarse, then fine bins
      uint32_t cbin, cabove, fbin, fabove;
      pick64<true>(hist + kBins, m, cbin, cabove);
      const uint32_t c1 =
          pick64<true>(hist + cbin * (kBins / kTopkCoarse), m - cabove, fbin, fabove);
      if (lane == 0) {
        tmp.t = (int)(cbin * (kBins / kTopkCoarse) + fbin);
        tmp.above = cabove + fabove;
        tmp.total = c1;
      }
    }
    __syncthreads();
    T1 = (uint32_t)tmp.t;
    need = m - tmp.above;
    cnt1 = tmp.total;
    uint32_t base = 0;  // entries kept by earlier batches (block-uniform)
    int par = 0;
    for (int64_t b0 = j0; b0 < j1; b0 += kBatch) {
      if (b0 != j0) load(b0);
      const int64_t wb = b0 + (int64_t)warp * (kBatch / kTkWarps);
      // 4 bits per float4: which of its scores are kept
      uint32_t bits[kRounds], cnt = 0;
#pragma unroll
      for (int u = 0; u < kRounds; ++u) {
        const int64_t j = wb + 128 * u + 4 * lane;
        const float xv[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
        uint32_t b = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e)
          b |= (uint32_t)(j + e < j1 && (score_key(xv[e]) >> 20) >= T1) << e;
        bits[u] = b;
        cnt += __popc(b);
      }
      uint32_t wsum = cnt;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
      if (lane == 0) wtot[par * kTkWarps + warp] = wsum;
      __syncthreads();
      uint32_t pos = base, batch = 0;
#pragma unroll
      for (int w = 0; w < kTkWarps; ++w) {
        const uint32_t c = wtot[par * kTkWarps + w];
        pos += w < warp ? c : 0u;
        batch += c;
      }
      if (wsum) {
#pragma unroll
        for (int u = 0; u < kRounds; ++u) {
          const uint32_t c = __popc(bits[u]);
          if (!__ballot_sync(0xffffffffu, c != 0)) continue;
          uint32_t incl = c;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
          }
          uint32_t p = pos + incl - c;
          const int64_t j = wb + 128 * u + 4 * lane;
          const float xv[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            if ((bits[u] >> e) & 1u) {
              if (p < (uint32_t)kSlotCap) {
                sk[p] = score_key(xv[e]);
                sj[p] = (int32_t)(j + e);
              }
              ++p;
            }
          }
          pos += __shfl_sync(0xffffffffu, incl, 31);
        }
      }
      base += batch;
      par ^= 1;
    }
    kept = base;
  } else {
    // ---- one CTA per row: the row's first scores move into L1 (a prefetch
    // holds no registers) while warp 0 finds the threshold bin; the entries
    // in bins >= T1 are kept in shared memory in index order
#pragma unroll
    for (int u = 0; u < kRounds; ++u) {
      const int64_t j = j0 + (int64_t)u * kRound + tid * 4;
      if (j < j1) asm volatile("prefetch.global.L1 [%0];" ::"l"(s + j));
    }
    if (warp == 0) {
      uint32_t cbin, cabove, fbin, fabove;
      pick64(hrow + kBins, m, cbin, cabove);
      const uint32_t cnt = pick64(hrow + cbin * (kBins / kTopkCoarse), m - cabove, fbin, fabove);
      if (lane == 0) {
        tmp.t = (int)(cbin * (kBins / kTopkCoarse) + fbin);
        tmp.above = cabove + fabove;
        tmp.total = cnt;
      }
    }
    __syncthreads();
    T1 = (uint32_t)tmp.t;
    need = m - tmp.above;
    cnt1 = tmp.total;
    __syncthreads();  // tmp is rewritten by the scan
    kept = ordered_take(
        s, j0, j1, vec, 0u, &tmp,
        [&](uint32_t key, int64_t) { return (key >> 20) >= T1 ? 1u : 0u; },
        [&](uint32_t pos, uint32_t key, int64_t j) {
          if (pos < (uint32_t)kCandCap) {
            ckey[pos] = key;
            cidx[pos] = (int32_t)j;
          }
        });
  }
  __syncthreads();

  bool overflow;
  int nc;
  if (S == 1) {
    overflow = kept > (uint32_t)kCandCap;
    nc = (int)min(kept, (uint32_t)kCandCap);
  } else {
    // the slice's entries are in its slot: count the slice as done; the last
    // slice of the row to finish gathers every slot
    if (tid == 0) *reinterpret_cast<uint32_t*>(slot) = kept;
    __syncthreads();  // the CTA's slot writes happen before thread 0's fence
    if (tid == 0) {
      __threadfence();
      s_last = atomicAdd(&counters[row * 4], 1u) == (uint32_t)(S - 1);
      if (s_last) __threadfence();  // every other slice's writes are visible from here
    }
    __syncthreads();
    if (!s_last) {
      pdl_trigger();
      return;
    }
    // every slot's count and its first 32 (key, index) pairs in one round
    // of cp.async copies into shared memory (the histogram's space is free
    // until the threshold is resolved): slot c's pairs land at hist[64 c ..]
    static_assert(kMaxSlices * 64 <= kBins, "staging fits in the histogram");
    for (int c = warp; c < S; c += kTkWarps) {
      const uint8_t* sc = slots + ((size_t)row * S + c) * ScanLayout::kSlotBytes;
      asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(hist + 64 * c + lane)),
                   "l"(sc + 16 + lane * 4) : "memory");
      asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(
                       smem_u32(hist + 64 * c + 32 + lane)),
                   "l"(sc + 16 + (size_t)kSlotCap * 4 + lane * 4) : "memory");
      if (lane == 0)
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(&s_base[c])),
                     "l"(sc) : "memory");
    }
    cp_async_wait_all();
    __syncthreads();
    // counts -> offsets (slice order = index order)
    if (warp == 0) {
      uint32_t cc[2], ovf = 0;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int c = lane + 32 * h;
        cc[h] = c < S ? s_base[c] : 0u;
        ovf |= cc[h] > (uint32_t)kSlotCap;
      }
      __syncwarp();
      uint32_t run = 0;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t incl = cc[h];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const int c = lane + 32 * h;
        if (c < S) s_cnt[c] = cc[h];
        if (c < S) s_base[c] = run + incl - cc[h];
        run += __shfl_sync(0xffffffffu, incl, 31);
      }
      ovf = __any_sync(0xffffffffu, ovf != 0);
      if (lane == 0) {
        s_base[S] = run;
        tmp.flag = ovf || run > (uint32_t)kCandCap;
        counters[row * 4] = 0;  // ready for the next selection on this workspace
      }
    }
    __syncthreads();
    overflow = tmp.flag != 0;
    nc = (int)s_base[S];
    if (!overflow) {
      for (int c = warp; c < S; c += kTkWarps) {
        const uint32_t b = s_base[c], cnt = s_cnt[c];
        if ((uint32_t)lane < cnt) {
          ckey[b + lane] = hist[64 * c + lane];
          cidx[b + lane] = (int32_t)hist[64 * c + 32 + lane];
        }
        if (cnt > 32) {  // the rest of a long slot
          const uint8_t* sc = slots + ((size_t)row * S + c) * ScanLayout::kSlotBytes;
          const uint32_t* sk2 = reinterpret_cast<const uint32_t*>(sc + 16);
          const int32_t* sj2 = reinterpret_cast<const int32_t*>(sc + 16 + (size_t)kSlotCap * 4);
          for (uint32_t i = 32 + lane; i < cnt; i += 32) {
            ckey[b + i] = __ldcg(sk2 + i);
            cidx[b + i] = __ldcg(sj2 + i);
          }
        }
      }
    }
    __syncthreads();
  }
  pdl_trigger();

  if (!overflow) {
    // every entry of bins >= T1 is in shared memory, in index order
    const Threshold th = resolve_threshold(T1, need, cnt1, hist, &tmp, [&](const auto& f) {
      for (int i = tid; i < nc; i += kTkThreads) f(ckey[i]);
    });
    write_selected(ckey, nc, th, m, k, out, &tmp,
                   [&](int i) { return rmap ? rmap[cidx[i]] : cidx[i]; });
  } else {
    // some slice kept more than its slot: the same levels over the whole row
    const Threshold th = resolve_threshold(T1, need, cnt1, hist, &tmp, [&](const auto& f) {
      for_each_key(s, nv, vec, f);
    });
    const uint32_t taken = ordered_take(
        s, 0, nv, vec, th.need, &tmp,
        [&](uint32_t key, int64_t) { return th.sure(key) ? 1u : (th.tie(key) ? 2u : 0u); },
        [&](uint32_t pos, uint32_t, int64_t j) {
          if (pos < m) out[pos] = rmap ? rmap[j] : (int32_t)j;
        });
    (void)taken;
    for (int i = (int)m + tid; i < k; i += kTkThreads) out[i] = -1;
  }
  if (clear)  // every slice read the histogram before counting itself done
    for (int i = tid; i < kTopkHistStride; i += kTkThreads) hrow[i] = 0;
}

// ---------------------------------------------------------------------------
// short rows (a candidate pool): one CTA per row, every key in shared memory

// Row r of n <= kSmallN values (the first n_valid[r] of them when n_valid
// is given): value i is scores[r * ld + i], or with `gather` scores[r * ld +
// gather[r * gather_ld + i]] (an index < 0 is an empty slot, below every
// value).  The k largest (value descending, position ascending) are written
// ascending by position to out[r * out_ld ..] as remap[r * remap_ld + i]
// (remap may be null: i), padded with -1.  The same levels as the long
// rows: 12 / 12 / 8-bit digits, then ties on the whole key in position order.
__global__ void __launch_bounds__(kTkThreads)
    topk_small_kernel(const float* __restrict__ scores, int64_t ld,
                      const int32_t* __restrict__ gather, int64_t gather_ld, int32_t n_row,
                      const int32_t* __restrict__ n_valid, int32_t k,
                      const int32_t* __restrict__ remap, int64_t remap_ld,
                      int32_t* __restrict__ out, int64_t out_ld, int32_t expand,
                      int64_t expand_n) {
  __shared__ uint32_t key[kSmallN];
  __shared__ uint32_t hist[kBins];
  __shared__ TkTmp tmp;
  pdl_wait();
  const int tid = threadIdx.x;
  const int64_t row = blockIdx.x;
  const int n = (int)row_nvalid(n_valid, row, n_row);  // positions >= n_valid[row] do not exist
  const float* s = scores + row * ld;
  const int32_t* gi = gather ? gather + row * gather_ld : nullptr;
  const int32_t* rm = remap ? remap + row * remap_ld : nullptr;
  int32_t* o = out + row * out_ld;
  for (int i = tid; i < kBins; i += kTkThreads) hist[i] = 0;
  // every position's source, then every score: the loads of each round are
  // in flight together (a gathered score is two dependent loads)
  constexpr int kPer = kSmallN / kTkThreads;
  int32_t src[kPer];
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int i = tid + u * kTkThreads;
    src[u] = i < n ? (gi ? gi[i] : i) : -1;
  }
  float v[kPer];
#pragma unroll
  for (int u = 0; u < kPer; ++u) v[u] = src[u] >= 0 ? s[src[u]] : 0.f;
  __syncthreads();  // the histogram is cleared
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int i = tid + u * kTkThreads;
    if (i < n) {
      const uint32_t kk = src[u] >= 0 ? score_key(v[u]) : 0u;  // 0: an empty slot
      key[i] = kk;
      atomicAdd(&hist[kk >> 20], 1u);
    }
  }
  __syncthreads();
  const uint32_t m = (uint32_t)min(k, n);
  if (m == 0) {  // an empty row (the whole CTA returns here)
    const int64_t slots = (int64_t)k * (expand > 0 ? expand : 1);
    for (int64_t i = tid; i < slots; i += kTkThreads) o[i] = -1;
    return;
  }
  find_top(hist, kBins, m, &tmp);
  const uint32_t T1 = (uint32_t)tmp.t;
  const uint32_t need = m - tmp.above;
  const uint32_t cnt1 = hist[T1];
  const Threshold th = resolve_threshold(T1, need, cnt1, hist, &tmp, [&](const auto& f) {
    for (int i = tid; i < n; i += kTkThreads) f(key[i]);
  });
  pdl_trigger();
  write_selected(key, n, th, m, k, o, &tmp, [&](int i) { return rm ? rm[i] : i; }, expand,
                 expand_n);
}

// ---------------------------------------------------------------------------
// selection from candidates (a prefill chunk without its score matrix)
// ---------------------------------------------------------------------------


// The k-th largest key of a sample of row r (its histogram in hist1), one
// warp per row, in two levels of 12 bits.  Level 0: T1 = the level-1 bin
// holding it; theta[r] = T1 << 20, cand_cnt[r] = its rank among the keys of
// bin T1.  Level 1 (the histogram now holds bin T1's keys by their next 12
// bits): T2 = the sub-bin holding that rank; theta[r] |= T2 << 8, the lowest
// key of the 24-bit prefix, and cand_cnt[r] = 0 for the emitting pass.
// theta[r] is at most the sample's k-th largest key, so no entry of the
// row's top k lies below it.  A sample of fewer than k keys (in either
// level) gives bin 0: every visible entry becomes a candidate.  Each level
// clears the row's histogram.
__global__ void __launch_bounds__(128)
    topk_theta_kernel(uint32_t* __restrict__ hist1, int64_t rows, int32_t k,
                      uint32_t* __restrict__ theta, uint32_t* __restrict__ cand_cnt, int level) {
  pdl_wait();
  const int64_t row = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
  if (row >= rows) return;  // whole warps leave together
  const int lane = threadIdx.x & 31;
  uint32_t* hrow = hist1 + row * kTopkHistStride;
  const uint32_t target = level == 0 ? (uint32_t)k : cand_cnt[row];
  uint32_t cbin, cabove, fbin, fabove;
  pick64(hrow + kTopkBins, target, cbin, cabove);
  pick64(hrow + cbin * (kTopkBins / kTopkCoarse), target - cabove, fbin, fabove);
  const uint32_t bin = cbin * (kTopkBins / kTopkCoarse) + fbin;
  __syncwarp();
  if (lane == 0) {
    if (level == 0) {
      theta[row] = bin << 20;
      cand_cnt[row] = target - cabove - fabove;  // >= 1 when the bin holds the k-th
    } else {
      theta[row] |= bin << 8;
      cand_cnt[row] = 0;
    }
  }
  for (int i = lane; i < kTopkHistStride; i += 32) hrow[i] = 0;
  pdl_trigger();
}

// Row r's candidates cand[r * cap .. + min(cand_cnt[r], cap)) as (key,
// entry), in any order (entry 0xFFFFFFFF: an empty slot): the m = min(k, n_valid[r], candidates) largest by
// (key descending, entry ascending), written ascending to out[r * out_ld ..],
// padded with -1.  The same radix levels as the other selectors resolve the
// threshold; the output is read off a bitmap of the row's n entries in
// entry order (ties at the threshold key through a second bitmap, the
// lowest entries first).  More candidates than cap raise
// CSA2_DEVFLAG_CAPACITY (the selection is then among the first cap).
__global__ void __launch_bounds__(kTkThreads)
    topk_cand_kernel(const uint2* __restrict__ cand, const uint32_t* __restrict__ cand_cnt,
                     int64_t cap, int64_t n, const int32_t* __restrict__ n_valid, int32_t k,
                     int32_t* __restrict__ out, int64_t out_ld, int32_t* dev_status) {
  extern __shared__ __align__(16) uint32_t dyn[];
  uint32_t* hist = dyn;                                 // [kBins]
  uint32_t* ckey = dyn + kBins;                         // [cap]
  uint32_t* cidx = ckey + cap;                          // [cap]
  const int64_t words = (n + 31) / 32;
  uint32_t* selb = cidx + cap;                          // [words] selected entries
  uint32_t* tieb = selb + words;                        // [words] ties at the threshold key
  __shared__ TkTmp tmp;
  pdl_wait();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t row = blockIdx.x;
  int32_t* o = out + row * out_ld;
  const uint32_t total = cand_cnt[row];
  if (total > (uint64_t)cap && tid == 0) raise_flag(dev_status, CSA2_DEVFLAG_CAPACITY);
  const int slots = (int)min((uint64_t)total, (uint64_t)cap);
  const int64_t nv = row_nvalid(n_valid, row, n);
  __shared__ uint32_t s_nc;
  for (int i = tid; i < kBins; i += kTkThreads) hist[i] = 0;
  for (int64_t i = tid; i < 2 * words; i += kTkThreads) selb[i] = 0;
  if (tid == 0) s_nc = 0;
  __syncthreads();
  // the filled slots (an unused reserved slot holds entry 0xFFFFFFFF),
  // compacted in any order
  const uint2* cr = cand + row * cap;
  const uint32_t lt = (1u << lane) - 1u;
  for (int i0 = 0; i0 < slots; i0 += kTkThreads) {
    const int i = i0 + tid;
    uint2 c = make_uint2(0u, 0xFFFFFFFFu);
    if (i < slots) c = __ldcg(cr + i);
    const bool ok = c.y != 0xFFFFFFFFu;
    const uint32_t mask = __ballot_sync(0xffffffffu, ok);
    if (mask) {
      uint32_t b = 0;
      if (lane == 0) b = atomicAdd(&s_nc, (uint32_t)__popc(mask));
      b = __shfl_sync(0xffffffffu, b, 0);
      if (ok) {
        const uint32_t pos = b + __popc(mask & lt);
        ckey[pos] = c.x;
        cidx[pos] = c.y;
        atomicAdd(&hist[c.x >> 20], 1u);
      }
    }
  }
  __syncthreads();
  const int nc = (int)s_nc;
  const uint32_t m = (uint32_t)min((int64_t)min(k, nc), nv);
  if (m > 0) {
    find_top(hist, kBins, m, &tmp);
    const uint32_t T1 = (uint32_t)tmp.t;
    const uint32_t need = m - tmp.above;
    const uint32_t cnt1 = hist[T1];
    const Threshold th = resolve_threshold(T1, need, cnt1, hist, &tmp, [&](const auto& f) {
      for (int i = tid; i < nc; i += kTkThreads) f(ckey[i]);
    });
    for (int i = tid; i < nc; i += kTkThreads) {
      const uint32_t key = ckey[i], j = cidx[i];
      if (th.sure(key))
        atomicOr(&selb[j >> 5], 1u << (j & 31));
      else if (th.tie(key))
        atomicOr(&tieb[j >> 5], 1u << (j & 31));
    }
    __syncthreads();
    // thread t owns words [t * per, (t + 1) * per) of both bitmaps
    const int64_t per = (words + kTkThreads - 1) / kTkThreads;
    const int64_t w0 = min(words, (int64_t)tid * per), w1 = min(words, w0 + per);
    auto block_excl = [&](uint32_t v) {  // block-wide exclusive prefix in thread order
      uint32_t incl = v;
#pragma unroll
      for (int o2 = 1; o2 < 32; o2 <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o2);
        if (lane >= o2) incl += y;
      }
      __syncthreads();
      if (lane == 31) tmp.wsum[warp] = incl;
      __syncthreads();
      uint32_t wv = lane < kTkWarps ? tmp.wsum[lane] : 0u;
#pragma unroll
      for (int o2 = 1; o2 < 32; o2 <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, wv, o2);
        if (lane >= o2) wv += y;
      }
      const uint32_t woff = __shfl_sync(0xffffffffu, wv, (warp + 31) & 31) * (warp > 0);
      return woff + incl - v;
    };
    if (th.depth == 4) {
      // ties: the first `need` tie entries in entry order join the selection
      uint32_t t = 0;
      for (int64_t w = w0; w < w1; ++w) t += __popc(tieb[w]);
      uint32_t rank = block_excl(t);
      for (int64_t w = w0; w < w1; ++w) {
        uint32_t bits = tieb[w];
        while (bits) {
          const int b = __ffs(bits) - 1;
          bits &= bits - 1;
          if (rank++ < th.need) selb[w] |= 1u << b;
        }
      }
      __syncthreads();
    }
    uint32_t c = 0;
    for (int64_t w = w0; w < w1; ++w) c += __popc(selb[w]);
    uint32_t pos = block_excl(c);
    for (int64_t w = w0; w < w1; ++w) {
      uint32_t bits = selb[w];
      while (bits) {
        const int b = __ffs(bits) - 1;
        bits &= bits - 1;
        if (pos < m) o[pos] = (int32_t)(w * 32 + b);
        ++pos;
      }
    }
  }
  pdl_trigger();
  for (int i = (int)m + tid; i < k; i += kTkThreads) o[i] = -1;
}

std::atomic<uint64_t> g_scan_attr{0};  // devices on which the scan kernel's attributes are set
std::atomic<uint64_t> g_cand_attr{0};  // the same for the candidate selector

}  // namespace

size_t topk_workspace_bytes(int64_t rows, int64_t n, int32_t k) {
  (void)k;
  ScanLayout L{rows, scan_slices(rows, n)};
  return L.total();
}

csa2_status clear_topk_hist(uint32_t* hist1, int64_t rows, int64_t n, cudaStream_t s) {
  if (rows == 0) return CSA2_OK;
  ScanLayout L{rows, scan_slices(rows, n)};
  // the histograms and (long rows) the per-row counters start at zero
  const size_t bytes = L.S > 0 ? L.slot_off() : L.hist_bytes();
  cudaError_t e = cudaMemsetAsync(hist1, 0, bytes, s);
  return e == cudaSuccess ? CSA2_OK : cuda_fail(e);
}

csa2_status launch_topk_select(const float* scores, int64_t rows, int64_t n, int64_t ld,
                               const int32_t* n_valid, int32_t k, uint32_t* hist1,
                               int32_t* idx_out, int64_t idx_ld, cudaStream_t s,
                               const int32_t* remap, int64_t remap_ld, bool clear_hist) {
  if (rows == 0) return CSA2_OK;
  ScanLayout L{rows, scan_slices(rows, n)};
  if (L.S == 0) return CSA2_ERR_UNSUPPORTED;  // short rows take topk_small_kernel
  cudaError_t e = once_per_device(g_scan_attr, [] {
    return cudaFuncSetAttribute(topk_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kScanSmem);
  });
  if (e != cudaSuccess) return cuda_fail(e);
  const int vec = (ld % 4 == 0 && (reinterpret_cast<uintptr_t>(scores) % 16) == 0) ? 1 : 0;
  // slices are multiples of 4 scores long, so every float4 of a slice is
  // aligned (a slice's last batch is partly past its end: those loads are
  // bounded by the slice)
  const int64_t per = (n + L.S - 1) / L.S;
  const int64_t slice = (per + 3) / 4 * 4;
  uint8_t* base = reinterpret_cast<uint8_t*>(hist1);
  return launch_kernel(topk_scan_kernel, dim3((unsigned)(rows * L.S)), dim3(kTkThreads),
                       (size_t)kScanSmem, s, 1, scores, n, ld, n_valid, k, hist1,
                       reinterpret_cast<uint32_t*>(base + L.counter_off()), base + L.slot_off(),
                       L.S, slice, idx_out, idx_ld, vec, remap, remap_ld, clear_hist ? 1 : 0);
}

csa2_status launch_topk_small(const float* scores, int64_t ld, const int32_t* gather,
                              int64_t gather_ld, int64_t rows, int32_t n, const int32_t* n_valid,
                              int32_t k, const int32_t* remap, int64_t remap_ld, int32_t* idx_out,
                              int64_t idx_ld, cudaStream_t s, int32_t expand, int64_t expand_n) {
  if (rows == 0) return CSA2_OK;
  if (n < 0 || n > kSmallN || k < 1 || k > kMaxK || expand < 0) return CSA2_ERR_UNSUPPORTED;
  return launch_kernel(topk_small_kernel, dim3((unsigned)rows), dim3(kTkThreads), 0, s, 1, scores,
                       ld, gather, gather_ld, n, n_valid, k, remap, remap_ld, idx_out, idx_ld,
                       expand, expand_n);
}

csa2_status launch_topk_theta(uint32_t* hist1, int64_t rows, int32_t k, uint32_t* theta,
                              uint32_t* cand_cnt, int level, cudaStream_t s) {
  if (rows == 0) return CSA2_OK;
  return launch_kernel(topk_theta_kernel, dim3((unsigned)((rows + 3) / 4)), dim3(128), 0, s, 1,
                       hist1, rows, k, theta, cand_cnt, level);
}

size_t topk_cand_smem(int64_t cap, int64_t n) {
  return (size_t)(kBins + 2 * cap + 2 * ((n + 31) / 32)) * 4;
}

// Dynamic shared memory the candidate selector may take: a CTA holds at most
// 227 KB of static and dynamic shared memory together, and the kernel's
// static part (its TkTmp) is well under the 1 KB kept back here.
constexpr size_t kCandDynMax = 227 * 1024 - 1024;
static_assert(sizeof(TkTmp) <= 1024, "static shared memory of the candidate selector");

bool topk_cand_fits(int64_t cap, int64_t n) { return topk_cand_smem(cap, n) <= kCandDynMax; }

csa2_status launch_topk_cand(const uint2* cand, const uint32_t* cand_cnt, int64_t cap,
                             int64_t rows, int64_t n, const int32_t* n_valid, int32_t k,
                             int32_t* out, int64_t out_ld, int32_t* dev_status, cudaStream_t s) {
  if (rows == 0) return CSA2_OK;
  const size_t smem = topk_cand_smem(cap, n);
  if (smem > kCandDynMax || k < 1 || k > kMaxK) return CSA2_ERR_UNSUPPORTED;
  cudaError_t e = once_per_device(g_cand_attr, [] {
    return cudaFuncSetAttribute(topk_cand_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kCandDynMax);
  });
  if (e != cudaSuccess) return cuda_fail(e);
  return launch_kernel(topk_cand_kernel, dim3((unsigned)rows), dim3(kTkThreads), smem, s, 1, cand,
                       cand_cnt, cap, n, n_valid, k, out, out_ld, dev_status);
}

csa2_status launch_topk_hist(const float* scores, int64_t rows, int64_t n, int64_t ld,
                             const int32_t* n_valid, uint32_t* hist1, cudaStream_t s,
                             const uint32_t* within) {
  if (rows == 0 || n == 0) return CSA2_OK;
  // enough CTAs to cover the GPU about twice
  const int64_t want = (2 * (int64_t)sm_count() + rows - 1) / rows;
  const int64_t max_chunks = (n + 4095) / 4096;
  int64_t chunks = std::max<int64_t>(1, std::min<int64_t>(want, max_chunks));
  const int64_t chunk = ((n + chunks - 1) / chunks + 3) / 4 * 4;  // multiples of 4 scores
  chunks = (n + chunk - 1) / chunk;
  const int vec = (ld % 4 == 0 && (reinterpret_cast<uintptr_t>(scores) % 16) == 0) ? 1 : 0;
  // with one CTA per row the row's histogram is that CTA's counts, written
  // outright (every caller hands over rows at zero, which several CTAs add to)
  return launch_kernel(topk_hist_kernel, dim3((unsigned)chunks, (unsigned)rows),
                       dim3(kHistThreads), 0, s, 1, scores, n, ld, n_valid, hist1, chunk,
                       within, vec, chunks == 1 ? 1 : 0);
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
  csa2_status st = clear_topk_hist(hist1, rows, n, s);
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
