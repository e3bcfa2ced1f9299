// index_score.cu -- a3, the indexer score
//   s[q, j] = sum_h w'[q, h] * max(0, <q_h, k_j>)   (j < n_valid[q], else -inf)
// over every compressed entry of the query's sequence.  The pages name an
// indexer Q scored against indexer K per layer ("Unlocking Extreme Context
// Scaling with DeepSeek-V4.1-Flash", "Compressed Sparse Attention 2
// (CSA2)"); the weighted-ReLU head sum is this library's definition.
//
// Two kernels:
//  * idx_score_f32_kernel  fp32 q / k on CUDA cores (small indexers).
//  * idx_score_tc_kernel   E4M3 q8 / k on tcgen05 tensor cores.  Per tile of
//    128 entries: D[128 x 64*QG] = K_tile[128 x 128] . Q8[64*QG x 128]^T in
//    tensor memory, then an epilogue applies ReLU, the head weights c and the
//    head sum.  Warp 0 streams K tiles with TMA into a ring of 16 KB stages,
//    warp 1 issues the MMAs into a ring of two tensor-memory accumulators,
//    and the epilogue warpgroups drain alternate tiles (two in decode,
//    warps 2-5 and 6-9; in a prefill chunk two per tile, each taking two of
//    its four queries), so several warps per SM sub-partition hide each
//    other's tcgen05.ld and FMA latency.  In decode (QG = 1) the kernel is a stream over the indexer
//    keys (128 B per entry): one CTA's load -> MMA -> epilogue -> accumulator
//    hand-back chain is latency-bound well short of HBM speed, so two CTAs
//    with 3-stage rings share each SM and overlap their chains.  In a prefill
//    chunk (QG = 4, 4 queries x 64 heads per MMA) it is a dense contraction,
//    one CTA per SM with a 6-stage ring.
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include "common.cuh"
#include "internal.h"

namespace csa2 {

// ===========================================================================
// fp32 path
// ===========================================================================

namespace {

constexpr int kF32Warps = 8;

// block = (entry chunk, query); warp w handles entries j = chunk*8*R + w, +8, ...
__global__ void __launch_bounds__(kF32Warps * 32)
    idx_score_f32_kernel(const float* __restrict__ q, const float* __restrict__ w,
                         const float* __restrict__ k, int64_t q_per_seq, int32_t hi, int32_t di,
                         int64_t n, int64_t k_ld, int64_t k_seq_stride,
                         const int32_t* __restrict__ n_valid, float* __restrict__ scores,
                         int64_t scores_ld, int64_t per_block, const csa2_pages pages,
                         int32_t* dev_status) {
  extern __shared__ float sq[];  // [hi * di] query, then [hi] weights
  pdl_wait();
  const int64_t qi = blockIdx.y;
  const float* qsrc = q + qi * (int64_t)hi * di;
  for (int i = threadIdx.x; i < hi * di; i += blockDim.x) sq[i] = qsrc[i];
  for (int i = threadIdx.x; i < hi; i += blockDim.x) sq[hi * di + i] = w[qi * hi + i];
  __syncthreads();
  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  const int64_t nv = n_valid ? (int64_t)n_valid[qi] : n;
  const int64_t b = qi / q_per_seq;
  const float* kseq = k + b * k_seq_stride;
  const int64_t j0 = (int64_t)blockIdx.x * per_block;
  const int64_t j1 = min(n, j0 + per_block);
  for (int64_t j = j0 + warp; j < j1; j += kF32Warps) {
    if (j >= nv) {
      if (lane == 0) scores[qi * scores_ld + j] = -INFINITY;
      continue;
    }
    const float* kj = kseq + j * k_ld;
    if (pages.block_table) {  // paged keys: the entry's row in the pool
      const int64_t row = paged_row(pages, b, j, dev_status);
      kj = row < 0 ? nullptr : k + row * k_ld;
    }
    float kv[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) kv[t] = (kj && lane + 32 * t < di) ? kj[lane + 32 * t] : 0.f;
    float s = 0.f;
    for (int h = 0; h < hi; ++h) {
      float dot = 0.f;
#pragma unroll
      for (int t = 0; t < 8; ++t)
        if (lane + 32 * t < di) dot = fmaf(sq[h * di + lane + 32 * t], kv[t], dot);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
      s = fmaf(sq[hi * di + h], fmaxf(dot, 0.f), s);
    }
    if (lane == 0) scores[qi * scores_ld + j] = s;
  }
  pdl_trigger();
}

}  // namespace

csa2_status launch_index_score_f32(const csa2_index_args& a, cudaStream_t s) {
  const int64_t nq = a.B * a.q_per_seq;
  if (nq == 0 || a.n == 0) return CSA2_OK;
  const int64_t per_block = 256;
  dim3 grid((unsigned)((a.n + per_block - 1) / per_block), (unsigned)nq);
  const size_t smem = sizeof(float) * ((size_t)a.hi * a.di + a.hi);
  return launch_kernel(idx_score_f32_kernel, grid, dim3(kF32Warps * 32), smem, s, 1,
                       static_cast<const float*>(a.q), a.w, static_cast<const float*>(a.k),
                       a.q_per_seq, a.hi, a.di, a.n, a.k_ld, a.k_seq_stride, a.n_valid, a.scores,
                       a.scores_ld, per_block, a.pages, a.dev_status);
}

// ===========================================================================
// FP8 tcgen05 path
// ===========================================================================

namespace {

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far beyond any legal wait

// Limit of the pipeline waits of one launch: 2 s, or CSA2_WAIT_LIMIT_NS
// when set (read at every launch; a test hook that makes the waits run out
// and the kernel return CSA2_DEVFLAG_TIMEOUT).  Waits for copies or MMAs
// already in flight keep fixed limits, so a CTA never leaves with either
// outstanding.
uint64_t pipeline_wait_ns() {
  const char* e = std::getenv("CSA2_WAIT_LIMIT_NS");
  if (!e || !*e) return kWaitLimitNs;
  const unsigned long long v = std::strtoull(e, nullptr, 10);
  return v > 0 ? (uint64_t)v : kWaitLimitNs;
}

// CSA2_TEST_STALL_LOADS=1 (read at every launch; a test hook): the TMA
// producer issues no key loads, so the MMA and epilogue waits wait for data
// that never comes and run out after pipeline_wait_ns(); no copy or MMA is
// ever in flight, and the launch ends with CSA2_DEVFLAG_TIMEOUT.
bool stall_loads() {
  const char* e = std::getenv("CSA2_TEST_STALL_LOADS");
  return e && e[0] == '1';
}


template <int QG>
struct TcCfg {
  static constexpr int BM = 128;        // entries per tile (MMA M)
  static constexpr int BN = 64 * QG;    // 64 heads x QG queries (MMA N)
  static constexpr int BK = 128;        // indexer dim: 128 E4M3 bytes per row
  static constexpr int CTAS_PER_SM = QG == 1 ? 2 : 1;
  static constexpr int STAGES = QG == 1 ? 3 : 8;
  // epilogue: STREAMS tiles drained at once, each by SPLIT warpgroups that
  // share its queries.  A prefill tile holds 4 queries x 64 heads, two
  // queries per warpgroup.  Its threads read the accumulator in 16x256b
  // shape (4 threads per entry, 16 heads each), so each thread keeps its
  // 2 x 16 head weights in registers: read from shared memory for every
  // entry, the weights cost 512 B of load traffic per thread and tile,
  // more than the MMAs' time
  static constexpr int SPLIT = QG == 1 ? 1 : 2;
  static constexpr int STREAMS = 2;
  static constexpr bool REG_W = QG > 1;
  static constexpr int EPI_WGS = STREAMS * SPLIT;  // epilogue warpgroups
  static constexpr int QPW = QG / SPLIT;           // queries per epilogue warpgroup
  static constexpr int NACC = 2;        // accumulators in tensor memory
  static constexpr int KTILE = BM * BK;  // 16 KB
  static constexpr int QTILE = BN * BK;  // 8 KB or 32 KB
  static constexpr int TMEM_USED = NACC * BN;
  static constexpr int TMEM_COLS = TMEM_USED <= 32 ? 32 : TMEM_USED <= 64 ? 64 : TMEM_USED <= 128 ? 128
                                 : TMEM_USED <= 256 ? 256 : 512;  // power of two
  static constexpr int EPI_WARPS = 4 * EPI_WGS;
  static constexpr int THREADS = 64 + 32 * EPI_WARPS;
  // shared memory carve-up (offsets from a 1024-byte aligned base)
  static constexpr int OFF_K = 0;
  static constexpr int OFF_Q = OFF_K + STAGES * KTILE;
  // float [EPI_WARPS][2][BN]: each epilogue warp's copy of its group's head
  // weights (none when they live in registers)
  static constexpr int OFF_C = OFF_Q + 2 * QTILE;
  static constexpr int OFF_CQ = OFF_C + (REG_W ? 0 : EPI_WARPS * 2 * BN * 4);  // float [2][BN], fused Q
  // fused first-level top-k histogram (decode): two group slots of 4096 bins
  static constexpr int OFF_H = OFF_CQ + (QG == 1 ? 2 * BN * 4 : 0);
  // decode: the first HSLOTS groups of a CTA's range keep their histograms
  // in shared memory (later ones add to the global histogram directly)
  static constexpr int HSLOTS = QG == 1 ? 2 : 0;
  static constexpr int HIST_BYTES = HSLOTS * kTopkBins * 4;
  static constexpr int OFF_BAR = OFF_H + HIST_BYTES;
  // barriers: full[S], empty[S], qfull[2], qempty[2], tfull[NACC], tempty[NACC], fin, nrdy
  static constexpr int NBAR = 2 * STAGES + 4 + 2 * NACC + 2;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;         // tmem slot, abort flag
  static constexpr int SMEM = OFF_MISC + 16;
  static constexpr int SMEM_ALLOC = SMEM + 1024;
  static_assert(NACC % STREAMS == 0 && QG % SPLIT == 0,
                "accumulator a is drained by the warpgroups of stream a % STREAMS");
  static_assert(TMEM_USED <= 512, "tensor memory holds 512 columns");
  static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory per CTA");
  static_assert(CTAS_PER_SM * (SMEM_ALLOC + 1024) <= 228 * 1024, "CTAs resident per SM");
  static_assert(CTAS_PER_SM * TMEM_COLS <= 512, "tensor memory shared by the SM's CTAs");
};

struct TcParams {
  const float* c;          // [nq, 64] head weights (w * sigma); unused when qbf is set
  // decode with the indexer-Q quantiser fused in: bf16 Q [nq, 64, 128] and
  // raw weights w [nq, 64]; the kernel quantises the (at most two) query
  // groups of each CTA itself instead of loading q8 by TMA
  const uint16_t* qbf;
  const float* w;
  const int32_t* n_valid;  // [nq] or null
  float* scores;
  int64_t scores_ld;
  int64_t n;               // entries per sequence
  int64_t q_per_seq;
  int64_t groups;          // nq / QG
  int64_t ktiles;          // ceil(n / 128)
  int32_t* dev_status;
  uint32_t* hist1;         // QG = 1: [nq][4096] first-level top-k histograms to add to, or null
  int reverse;             // walk each CTA's tile range from its end
  int keep_in_l2;          // load keys with the normal L2 policy instead of evict-first
  // paged keys (pages.block_table set): kmap is a 2-D map over the pool
  // with boxes of pg_box rows (128 when pages hold a multiple of 128
  // entries, so a tile lies in one page; else 64); a tile is 128 / pg_box
  // boxes, each inside one page
  csa2_pages pages;
  int pg_box;
  int pg_shift;            // log2(page_rows) when a power of two, else -1
  uint64_t wait_ns;        // limit of each pipeline wait (drain waits keep their own)
  int stall_loads;         // test hook: the producer issues no loads (waits run out)
  // sampled launches: the cursor's tile kt is key tile kt * tile_stride, and
  // its scores go to columns kt * 128 .. of the (compact) score rows
  int tile_stride;
  // emitting launches (cand set): no scores are stored; every visible entry
  // whose order-preserving key is >= theta[q] is appended to query q's
  // candidates cand[q * cand_cap ..] as (key, entry), in slots reserved 32 at
  // a time through the counter cand_cnt[q]; reserved slots left unused hold
  // (0, 0xFFFFFFFF).  The counter may end above cand_cap: the overflow is
  // the reader's to detect
  const uint32_t* theta;
  uint32_t* cand_cnt;
  uint2* cand;
  int64_t cand_cap;
  // slots a (warp, query) stream reserves at a time: 32 (one atomic per 32
  // candidates), or 0: exactly the slots a tile's takes need.  A stream's
  // unused reserved slots count against cand_cap, so the host takes 0 when a
  // query's tiles are spread over so many CTAs that they could add up
  uint32_t cand_chunk;
  // decode Full layers (one query per sequence): the step's new rows, which
  // the epilogue warps quantise first; the producer waits for them (nrdy)
  // before loading a tile that holds one (nr.kv null: none)
  NewRows nr;
};


// (group, tile within the group) of the CTA's tiles, moved without 64-bit
// divisions: tile t is group t / ktiles, tile t % ktiles.
struct TileCursor {
  int64_t g, kt, ktiles;
  __device__ TileCursor(int64_t t, int64_t ktiles_) : g(t / ktiles_), kt(t % ktiles_), ktiles(ktiles_) {}
  __device__ void advance(int64_t by) {
    kt += by;
    while (kt >= ktiles) {
      kt -= ktiles;
      ++g;
    }
    while (kt < 0) {
      kt += ktiles;
      --g;
    }
  }
};

// ReLU on the FMA pipe: an accumulator value x = <q_h, k_j> of E4M3 codes
// has |x| <= 128 * 448^2 < 2^25, so the saturating product x * 2^-25 is
// max(x, 0) * 2^-25 exactly (a power-of-two scaling, far from the fp32
// subnormals: the smallest nonzero |x| is 2^-18).  Each fused product-add
// (w * 2^25) * that + s rounds the same real value as w max(x, 0) + s, so
// the head sum is bit-identical to the one taken with a max.  Where
// w * 2^25 could overflow (a weight of the warp's queries >= 2^100) the
// kernel sums w * (x * 2^-25) and multiplies the sum by 2^25 instead: the
// same sum, scaled, wherever its terms and partial sums stay above the fp32
// subnormals (2^-101 before the scaling).  The epilogue's FMNMX
// instructions would otherwise keep the ALU pipe the busiest.
constexpr float kReluScale = 33554432.f;  // 2^25
__device__ __forceinline__ float relu_scaled(float x) {
  float y;
  asm("mul.rn.sat.f32 %0, %1, 0f33000000;" : "=f"(y) : "f"(x));  // x * 2^-25 clamped to [0, 1]
  return y;
}

// The smallest score x with score_key(x) >= t: keys order the scores as
// floats do (-0 counts as +0), so score_key(x) >= t exactly when x >= the
// returned value.  Keys below every negative float's (t = 0 among them) give
// -inf: every score; keys above every positive float's give a NaN, which no
// score reaches.
__device__ __forceinline__ float key_floor(uint32_t t) {
  if (t & 0x80000000u) return __uint_as_float(t ^ 0x80000000u);  // +0 .. +inf, or NaN above
  const float x = __uint_as_float(~t);                             // -0 .. -inf, or NaN below
  return x != x ? -INFINITY : x;
}

template <int QG>
__global__ void __launch_bounds__(TcCfg<QG>::THREADS, TcCfg<QG>::CTAS_PER_SM)
    idx_score_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap qmap, const TcParams p) {
  using C = TcCfg<QG>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t* kbuf = smem + C::OFF_K;
  uint8_t* qbuf = smem + C::OFF_Q;
  float* cbuf = reinterpret_cast<float*>(smem + C::OFF_C);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* full = bars;
  uint64_t* empty = bars + C::STAGES;
  uint64_t* qfull = bars + 2 * C::STAGES;
  uint64_t* qempty = qfull + 2;
  uint64_t* tfull = qempty + 2;
  uint64_t* tempty = tfull + C::NACC;
  uint64_t* fin = tempty + C::NACC;
  uint64_t* nrdy = fin + 1;  // the CTA's new rows are in the caches
  uint32_t* hslot = reinterpret_cast<uint32_t*>(smem + C::OFF_H);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  const int64_t total = p.groups * p.ktiles;
  const int64_t t_begin = (int64_t)blockIdx.x * total / gridDim.x;
  const int64_t t_end = (int64_t)(blockIdx.x + 1) * total / gridDim.x;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::STAGES; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      // fused Q: every epilogue warp arrives once its share of the slot is written
      mbar_init(&qfull[i], p.qbf ? C::EPI_WARPS : 1);
      mbar_init(&qempty[i], 1);
    }
    for (int i = 0; i < C::NACC; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 4 * C::SPLIT);  // the warps of the warpgroups that share a tile
    }
    mbar_init(fin, 1);
    mbar_init(nrdy, C::EPI_WARPS);  // every epilogue warp, once its new-row share is written
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&kmap);
    if (!p.qbf) tma_prefetch_desc(&qmap);
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
  if constexpr (QG == 1) {
    for (int i = threadIdx.x; i < C::HSLOTS * kTopkBins; i += C::THREADS) hslot[i] = 0;
  }
  const int64_t g_first = total > 0 ? t_begin / p.ktiles : 0;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();  // the setup above overlapped the previous kernel; global data from here on

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    // Lane 0 issues the barrier operations and the copies.  Paged keys: the
    // whole warp runs the loop and looks up the pool rows of the next 32
    // tiles (lane l those of tile i0 + 32 + l, loads in flight while lane 0
    // works through tiles i0 .. i0 + 31), and lane 0 takes tile i's rows from
    // lane i % 32 by a shuffle: no lookup latency and no 64-bit division in
    // the loop.
    const bool paged_keys = p.pages.block_table != nullptr;
    if (t_begin < t_end && !p.stall_loads && (paged_keys || lane == 0)) {
      const uint64_t pol_k = p.keep_in_l2 ? l2_policy_evict_normal() : l2_policy_evict_first();
      const uint64_t pol_q = l2_policy_evict_last();
      int stage = 0;
      uint32_t ph = 0;
      int64_t g_prev = -1, qcount = 0, issued = 0;
      bool ok = true, nr_seen = false;
      const int64_t dir = p.reverse ? -1 : 1;
      TileCursor cur(p.reverse ? t_end - 1 : t_begin, p.ktiles);
      const bool paged = paged_keys;  // the whole warp runs the loop; else lane 0 alone
      const int64_t ntiles = t_end - t_begin;
      const uint32_t qps = (uint32_t)p.q_per_seq;
      const uint32_t pr = paged ? (uint32_t)p.pages.page_rows : 1u;
      const int boxes = C::BM / (paged ? p.pg_box : C::BM);
      // pool rows of the two 64-row halves of the CTA's tile i (-1: none)
      auto rows_of = [&](int64_t i, int32_t* y) {
        y[0] = y[1] = -1;
        if (i >= ntiles) return;
        const TileCursor c(p.reverse ? t_end - 1 - i : t_begin + i, p.ktiles);
        const int64_t kt = c.kt * p.tile_stride;
        const int32_t* bt = p.pages.block_table + (int64_t)((uint32_t)(c.g * QG) / qps) * p.pages.bt_ld;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t j = (uint32_t)(kt * C::BM + 64 * h);
          if (h >= boxes || (int64_t)j >= p.n) continue;  // past the rows: masked
          const uint32_t pi = p.pg_shift >= 0 ? j >> p.pg_shift : j / pr;
          const int32_t page = __ldg(bt + pi);
          if (page < 0 || page >= p.pages.num_pages) {
            raise_flag(p.dev_status, CSA2_DEVFLAG_BOUNDS);
            continue;
          }
          y[h] = (int32_t)((int64_t)page * pr + (j - pi * pr));
        }
      };
      int64_t b_of = -1, b = 0;  // the sequence of group b_of
      // lane 0: the barrier waits and copies of tile (g, kt); paged keys at
      // pool rows y0 / y1 (-1: that half is not loaded).  False: a wait gave up.
      auto issue_tile = [&](int64_t g, int64_t kt, int32_t y0, int32_t y1) -> bool {
        if (g != b_of) {
          b_of = g;
          b = (uint32_t)(g * QG) / qps;
        }
        if (g != g_prev && !p.qbf) {
          const int qs = (int)(qcount & 1);
          const uint32_t qph = (uint32_t)((qcount >> 1) & 1);
          if (!mbar_wait(&qempty[qs], qph ^ 1, abort_flag, p.dev_status, p.wait_ns)) return false;
          mbar_arrive_expect_tx(&qfull[qs], C::QTILE);
          tma_load_2d(&qmap, &qfull[qs], qbuf + qs * C::QTILE, 0, (int32_t)(g * C::BN), pol_q);
          ++qcount;
          g_prev = g;
        }
        if (!mbar_wait(&empty[stage], ph ^ 1, abort_flag, p.dev_status, p.wait_ns)) return false;
        if (p.nr.kv && !nr_seen && kt * C::BM < p.nr.row0 + p.nr.rows &&
            (kt + 1) * C::BM > p.nr.row0) {
          // this tile holds new rows: the epilogue warps have written them
          // (their proxy fence orders the stores before this TMA load)
          if (!mbar_wait(nrdy, 0, abort_flag, p.dev_status, p.wait_ns)) return false;
          nr_seen = true;
        }
        if (!paged) {
          mbar_arrive_expect_tx(&full[stage], C::KTILE);
          tma_load_3d(&kmap, &full[stage], kbuf + stage * C::KTILE, 0, (int32_t)(kt * C::BM),
                      (int32_t)b, pol_k);
        } else {
          const uint32_t box_bytes = (uint32_t)p.pg_box * C::BK;
          mbar_arrive_expect_tx(&full[stage],
                                (y0 >= 0 ? box_bytes : 0u) + (y1 >= 0 ? box_bytes : 0u));
          if (y0 >= 0) tma_load_2d(&kmap, &full[stage], kbuf + stage * C::KTILE, 0, y0, pol_k);
          if (y1 >= 0)
            tma_load_2d(&kmap, &full[stage], kbuf + stage * C::KTILE + C::KTILE / 2, 0, y1,
                        pol_k);
        }
        ++issued;
        if (++stage == C::STAGES) {
          stage = 0;
          ph ^= 1;
        }
        return true;
      };
      if (paged) {
        // the whole warp: the rows of tiles i0 .. i0 + 31 in ycur (lane l:
        // tile i0 + l), those of the next 32 in flight in ynext
        int32_t ycur[2], ynext[2];
        rows_of(lane, ycur);
        rows_of(32 + lane, ynext);
        for (int64_t i = 0; i < ntiles; ++i, cur.advance(dir)) {
          if (i > 0 && (i & 31) == 0) {
            ycur[0] = ynext[0];
            ycur[1] = ynext[1];
            rows_of(i + 32 + lane, ynext);
          }
          const int32_t y0 = __shfl_sync(0xffffffffu, ycur[0], (int)(i & 31));
          const int32_t y1 = __shfl_sync(0xffffffffu, ycur[1], (int)(i & 31));
          if (lane == 0) ok = issue_tile(cur.g, cur.kt * p.tile_stride, y0, y1);
          if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
        }
      } else {
        for (int64_t i = 0; i < ntiles && ok; ++i, cur.advance(dir))
          ok = issue_tile(cur.g, cur.kt * p.tile_stride, -1, -1);
      }
      if (lane == 0 && !ok) {
        // let the copies already in flight land before the CTA's shared
        // memory goes away: wait (bounded, ignoring the abort flag) for the
        // full barrier of every stage filled but possibly not consumed
        int dummy = 0;
        const int64_t first = issued > C::STAGES ? issued - C::STAGES : 0;
        for (int64_t u = first; u < issued; ++u)
          mbar_wait(&full[u % C::STAGES], (uint32_t)((u / C::STAGES) & 1), &dummy, nullptr,
                    kWaitLimitNs / 20);
        if (qcount > 0)
          mbar_wait(&qfull[(qcount - 1) & 1], (uint32_t)(((qcount - 1) >> 1) & 1), &dummy,
                    nullptr, kWaitLimitNs / 20);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0 && t_begin < t_end) {
      constexpr uint32_t idesc = idesc_e4m3_f32(C::BM, C::BN);
      int stage = 0, acc = 0;
      uint32_t ph = 0, aph = 0;
      int64_t g_prev = -1, qcount = 0;
      int qs = 0;
      bool any = false;
      const int64_t dir = p.reverse ? -1 : 1;
      TileCursor cur(p.reverse ? t_end - 1 : t_begin, p.ktiles);
      for (int64_t i = 0; i < t_end - t_begin; ++i, cur.advance(dir)) {
        const int64_t g = cur.g;
        if (g != g_prev) {
          if (g_prev >= 0) tc_commit(&qempty[qs]);  // old Q free once its MMAs finish
          qs = (int)(qcount & 1);
          if (!mbar_wait(&qfull[qs], (uint32_t)((qcount >> 1) & 1), abort_flag, p.dev_status,
                         p.wait_ns))
            break;
          ++qcount;
          g_prev = g;
        }
        if (!mbar_wait(&tempty[acc], aph ^ 1, abort_flag, p.dev_status, p.wait_ns)) break;
        tc_fence_after();
        if (!mbar_wait(&full[stage], ph, abort_flag, p.dev_status, p.wait_ns)) break;
        tc_fence_after();
        const uint64_t adesc = sdesc_k_sw128(smem_u32(kbuf + stage * C::KTILE));
        const uint64_t bdesc = sdesc_k_sw128(smem_u32(qbuf + qs * C::QTILE));
        const uint32_t dtm = tmem_base + (uint32_t)(acc * C::BN);
#pragma unroll
        for (int kk = 0; kk < C::BK / 32; ++kk)  // K = 32 E4M3 per MMA: +32 B = +2 in the address field
          tc_mma_f8(dtm, adesc + 2 * kk, bdesc + 2 * kk, idesc, kk > 0 ? 1u : 0u);
        tc_commit(&empty[stage]);
        tc_commit(&tfull[acc]);
        any = true;
        if (++stage == C::STAGES) {
          stage = 0;
          ph ^= 1;
        }
        if (++acc == C::NACC) {
          acc = 0;
          aph ^= 1;
        }
      }
      if (any) {
        // every MMA issued has completed before tensor memory is released
        int dummy = 0;
        tc_commit(fin);
        mbar_wait(fin, 0, &dummy, p.dev_status, kWaitLimitNs);
      }
    }
  } else {
    // ---------------- epilogue ----------------
    // warpgroup wg belongs to stream wg / SPLIT, which drains the tiles with
    // local number li = stream, stream + STREAMS, ...; tile li sits in
    // accumulator li % NACC; the warpgroup takes queries q0 .. q0 + QPW - 1.
    const int ew = warp - 2;          // 0 .. EPI_WARPS-1
    const int wg = ew >> 2;
    const int stream = wg / C::SPLIT;
    const int q0 = (wg % C::SPLIT) * C::QPW;
    const int lq = warp & 3;          // TMEM lane quarter this warp may access
    // entry within the tile (REG_W: the entry this thread keeps after the
    // quad's sum, see below)
    const int row = C::REG_W ? lq * 32 + (lane >> 2) + 8 * (lane & 3) : lq * 32 + lane;
    int64_t g_prev = -1;
    // each warp keeps its own double-buffered copy of the group's head weights
    float* my_c = cbuf + ew * 2 * C::BN;
    int cb = 1;
    // fused Q (decode): slot 0 holds the first group in processing order,
    // slot 1 the other end of the CTA's range (the host launches this form
    // only when no range spans more than two groups)
    const int64_t gq0 = (p.reverse ? t_end - 1 : t_begin) / p.ktiles;
    // [2][BN] folded weights c = w * sigma of the two slots
    float* cq = reinterpret_cast<float*>(smem + C::OFF_CQ);
    if constexpr (QG == 1) {  // (the prefill form has no room for cq and never fuses)
      if (p.qbf && t_begin < t_end) {
        const int64_t gq1 = (p.reverse ? t_begin : t_end - 1) / p.ktiles;
        // warp ew quantises heads 8 ew .. 8 ew + 7; lanes 4h'.. 4h'+3 hold
        // the four 32-element quarters of head 8 ew + h'
        const int h = (C::BN / C::EPI_WARPS) * ew + (lane >> 2), part = lane & 3;
        for (int slot = 0; slot < 2; ++slot) {
          const int64_t g = slot == 0 ? gq0 : gq1;
          if (slot == 1 && gq1 == gq0) break;
          const uint4* src =
              reinterpret_cast<const uint4*>(p.qbf + (g * C::BN + h) * C::BK + part * 32);
          uint4 raw[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) raw[i] = __ldg(src + i);
          float v[32];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t wv[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              v[8 * i + 2 * j] = bf16_bits_to_float(wv[j] & 0xFFFFu);
              v[8 * i + 2 * j + 1] = bf16_bits_to_float(wv[j] >> 16);
            }
          }
          float amax = 0.f;
#pragma unroll
          for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
          const int e = amax > 0.f ? index_q_exponent(amax) : 0;
          const float inv = exp2_int(-e);
          uint32_t pk[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            uint32_t wd = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j)
              wd |= (amax > 0.f ? e4m3_encode(v[4 * i + j] * inv) : 0u) << (8 * j);
            pk[i] = wd;
          }
          // bytes 32 part .. of row h: 16-byte pieces 2 part, 2 part + 1 of
          // the 128-byte swizzle row (piece index XOR h % 8), as TMA writes
          uint8_t* qrow = qbuf + slot * C::QTILE + h * C::BK;
          *reinterpret_cast<uint4*>(qrow + (((2 * part) ^ (h & 7)) << 4)) =
              make_uint4(pk[0], pk[1], pk[2], pk[3]);
          *reinterpret_cast<uint4*>(qrow + (((2 * part + 1) ^ (h & 7)) << 4)) =
              make_uint4(pk[4], pk[5], pk[6], pk[7]);
          if (part == 0) cq[slot * C::BN + h] = p.w[g * C::BN + h] * exp2_int(e);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&qfull[slot]);
        }
        // every epilogue warp's share of cq is written
        asm volatile("bar.sync 1, %0;" ::"n"(C::EPI_WARPS * 32) : "memory");
      }
      if (p.nr.kv && t_begin < t_end) {
        // a1 for the new rows inside this CTA's tiles: work items (sequence,
        // row, piece), piece < d / 256 a 256-element part of the main-KV row
        // (lane l: elements 8 l .. 8 l + 7; a 32-element block in 4 lanes),
        // the last piece the 128-element indexer key (lanes 0 .. 15); item
        // u goes to epilogue warp u % EPI_WARPS
        const int kvp = p.nr.d / 256;
        const int64_t g_lo = t_begin / p.ktiles, g_hi = (t_end - 1) / p.ktiles;
        int u = 0;
        for (int64_t b = g_lo; b <= g_hi; ++b) {
          for (int r = 0; r < p.nr.rows; ++r) {
            const int64_t j = p.nr.row0 + r;
            const int64_t t = b * p.ktiles + j / C::BM;
            if (t < t_begin || t >= t_end || j >= p.n) continue;
            for (int piece = 0; piece <= kvp; ++piece, ++u) {
              if (u % C::EPI_WARPS != ew) continue;
              const int64_t crow =
                  p.pages.block_table ? paged_row(p.pages, b, j, p.dev_status) : b * p.n + j;
              const int64_t src = b * p.nr.rows + r;
              if (piece < kvp) {
                const int e0 = 256 * piece + 8 * lane;
                float v[8];
                bf16x8_to_float(
                    __ldg(reinterpret_cast<const uint4*>(p.nr.kv + src * p.nr.d + e0)), v);
                float amax = 0.f;
#pragma unroll
                for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
                uint32_t sbyte;
                const uint32_t packed = fp4_encode8(v, amax, sbyte);
                if (crow >= 0) {
                  *reinterpret_cast<uint32_t*>(p.nr.codes + crow * (p.nr.d / 2) + e0 / 2) = packed;
                  if ((lane & 3) == 0) p.nr.scales[crow * (p.nr.d / 32) + e0 / 32] = (uint8_t)sbyte;
                }
              } else if (lane < C::BK / 8 && crow >= 0) {
                const uint4 raw =
                    __ldg(reinterpret_cast<const uint4*>(p.nr.idxk + src * C::BK + 8 * lane));
                *reinterpret_cast<uint2*>(p.nr.k8 + crow * C::BK + 8 * lane) = e4m3_encode8(raw);
              }
            }
          }
        }
        // the key stores are ordered before the producer's TMA loads (async
        // proxy) of their tiles, which wait for every warp's arrival
        asm volatile("fence.proxy.async.global;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(nrdy);
      }
    }
    // per query of the current group: entries visible (below n and
    // n_valid), the candidate threshold and the score row
    int32_t vis[C::QPW];
    uint32_t th[C::QPW];
    float thf[C::QPW];  // the smallest score whose key reaches th (see key_floor)
    float* srow[C::QPW];
    // REG_W: this thread's 16 head weights per query, times kReluScale
    // unless the head sums are scaled instead (relu_post = kReluScale)
    float wr[C::REG_W ? 16 * C::QPW : 1];
    float relu_post = 1.f;
    // emitting launches: each (warp, query) stream reserves its candidate
    // slots 32 at a time (one atomic per 32 candidates); slots [cpos, cend)
    // of the current chunk are still free, and are filled with the empty
    // candidate (entry 0xFFFFFFFF) when the stream leaves the query
    uint32_t cpos[C::QPW], cend[C::QPW];
#pragma unroll
    for (int i = 0; i < C::QPW; ++i) cpos[i] = cend[i] = 0;
    auto flush_chunks = [&](int64_t gq) {
#pragma unroll
      for (int qq = 0; qq < C::QPW; ++qq) {
        const uint32_t pos = cpos[qq] + lane;
        if (pos < cend[qq] && pos < (uint64_t)p.cand_cap)
          p.cand[(gq * QG + q0 + qq) * p.cand_cap + pos] = make_uint2(0u, 0xFFFFFFFFu);
        cpos[qq] = cend[qq] = 0;
      }
    };
    // li counts tiles in processing order (from the range's end when
    // reversed); the cursor is (group g, tile kt).  The host keeps a
    // launch's tiles and entries below 2^31, so the per-tile arithmetic is
    // 32-bit.
    const int32_t dir = p.reverse ? -1 : 1;
    const int32_t ntiles = (int32_t)(t_end - t_begin), ktiles = (int32_t)p.ktiles;
    const int32_t kstep = p.tile_stride * C::BM;  // entries from one cursor tile to the next
    const int32_t n32 = (int32_t)p.n;
    const int64_t tc0 = p.reverse ? t_end - 1 - stream : t_begin + stream;
    int64_t g = tc0 / p.ktiles;
    int32_t kt = (int32_t)(tc0 % p.ktiles);
    auto advance = [&]() {
      kt += dir * C::STREAMS;
      while (kt >= ktiles) {
        kt -= ktiles;
        ++g;
      }
      while (kt < 0) {
        kt += ktiles;
        --g;
      }
    };
    for (uint32_t li = stream; li < (uint32_t)ntiles; li += C::STREAMS, advance()) {
      const int acc = li % C::NACC;
      const uint32_t aph = (uint32_t)((li / C::NACC) & 1);
      if (g != g_prev) {
        if (p.cand && g_prev >= 0) flush_chunks(g_prev);
        cb ^= 1;
        __syncwarp();
        if constexpr (C::REG_W) {
          // heads 8 k + 2 (lane % 4) + b of the warpgroup's queries
#pragma unroll
          for (int qq = 0; qq < C::QPW; ++qq)
#pragma unroll
            for (int k = 0; k < 8; ++k)
#pragma unroll
              for (int b = 0; b < 2; ++b)
                wr[16 * qq + 2 * k + b] =
                    __ldg(p.c + g * C::BN + (q0 + qq) * 64 + 8 * k + 2 * (lane & 3) + b);
          // the ReLU's 2^-25 is undone on the weights, or, where a weight
          // of the warp's queries reaches 2^100 (times 2^25 it could
          // overflow), on the head sums
          bool big = false;
#pragma unroll
          for (int i = 0; i < 16 * C::QPW; ++i) big = big || !(fabsf(wr[i]) < 0x1p100f);
          big = __any_sync(0xffffffffu, big);
          relu_post = big ? kReluScale : 1.f;
#pragma unroll
          for (int i = 0; i < 16 * C::QPW; ++i) wr[i] *= big ? 1.f : kReluScale;
        } else if (p.qbf) {
          for (int i = lane; i < C::BN; i += 32)
            my_c[cb * C::BN + i] = cq[(g == gq0 ? 0 : 1) * C::BN + i];
        } else {
          for (int i = lane; i < C::BN; i += 32) my_c[cb * C::BN + i] = p.c[g * C::BN + i];
        }
        __syncwarp();
#pragma unroll
        for (int i = 0; i < C::QPW; ++i) {
          const int64_t qi = g * QG + q0 + i;
          vis[i] = p.n_valid ? min(n32, p.n_valid[qi]) : n32;
          th[i] = p.cand ? p.theta[qi] : 0u;
          thf[i] = key_floor(th[i]);
          srow[i] = p.scores ? p.scores + qi * p.scores_ld : nullptr;
        }
        g_prev = g;
      }
      // every lane waits; the warp goes on only if all of them saw the phase
      // complete, so the warp-collective loads below never run diverged
      const bool got = mbar_wait(&tfull[acc], aph, abort_flag, p.dev_status, p.wait_ns);
      if (!__all_sync(0xffffffffu, got)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(lq * 32) << 16) + (uint32_t)(acc * C::BN);
      float sc[C::QPW];
      if constexpr (C::REG_W) {
#pragma unroll
        for (int qq = 0; qq < C::QPW; ++qq) {
          // part[m]: this thread's 16 heads of entry lq * 32 + lane / 4 + 8 m
          float part[4];
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            float v[32];
            tmem_ld16x256b_x8(taddr + ((uint32_t)(16 * half) << 16) + (q0 + qq) * 64, v);
            tmem_ld_wait();
            if (qq == C::QPW - 1 && half == 1) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&tempty[acc]);
            }
            const float* w = wr + 16 * qq;
            float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
#pragma unroll
            for (int k = 0; k < 8; ++k) {  // heads 8 k + 2 (lane % 4) + {0, 1} of two entries
              ffma2(a0, a1, w[2 * k], w[2 * k + 1], relu_scaled(v[4 * k]), relu_scaled(v[4 * k + 1]));
              ffma2(b0, b1, w[2 * k], w[2 * k + 1], relu_scaled(v[4 * k + 2]),
                    relu_scaled(v[4 * k + 3]));
            }
            part[2 * half] = a0 + a1;
            part[2 * half + 1] = b0 + b1;
          }
          // sum over the 4 threads of the entry's quad, thread j of the quad
          // keeping entry m = j: two exchange steps (lane ^ 1, then lane ^ 2)
          const int jq = lane & 3;
          const bool odd = jq & 1;
          float k0 = odd ? part[1] : part[0], k1 = odd ? part[3] : part[2];
          k0 += __shfl_xor_sync(0xffffffffu, odd ? part[0] : part[1], 1);
          k1 += __shfl_xor_sync(0xffffffffu, odd ? part[2] : part[3], 1);
          const bool hi = jq & 2;
          float kk = hi ? k1 : k0;
          kk += __shfl_xor_sync(0xffffffffu, hi ? k0 : k1, 2);
          sc[qq] = kk * relu_post;
        }
      } else {
#pragma unroll
        for (int qq = 0; qq < C::QPW; ++qq) {
          float s8[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) s8[i] = 0.f;
          // two halves of 32 heads: 32 accumulator values live at a time
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            float v[32];
            tmem_ld32(taddr + (q0 + qq) * 64 + half * 32, v);
            tmem_ld_wait();
            if (qq == C::QPW - 1 && half == 1) {
              // the accumulator is in registers: hand it back to the MMA warp
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&tempty[acc]);
            }
            const float4* cw =
                reinterpret_cast<const float4*>(my_c + cb * C::BN + (q0 + qq) * 64 + half * 32);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float4 f = cw[i];
              s8[(4 * i) & 7] = fmaf(f.x, fmaxf(v[4 * i], 0.f), s8[(4 * i) & 7]);
              s8[(4 * i + 1) & 7] = fmaf(f.y, fmaxf(v[4 * i + 1], 0.f), s8[(4 * i + 1) & 7]);
              s8[(4 * i + 2) & 7] = fmaf(f.z, fmaxf(v[4 * i + 2], 0.f), s8[(4 * i + 2) & 7]);
              s8[(4 * i + 3) & 7] = fmaf(f.w, fmaxf(v[4 * i + 3], 0.f), s8[(4 * i + 3) & 7]);
            }
          }
          sc[qq] = ((s8[0] + s8[1]) + (s8[2] + s8[3])) + ((s8[4] + s8[5]) + (s8[6] + s8[7]));
        }
      }
      const int32_t jc = kt * C::BM + row;  // score column (compact when sampled)
      const int32_t j = kt * kstep + row;   // the entry
      if (p.cand) {
        // candidates of the exact selection: the warp's takes fill its
        // current chunk, then (one atomic) a new chunk of 32
        const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
        for (int qq = 0; qq < C::QPW; ++qq) {
          const bool take = j < vis[qq] && sc[qq] >= thf[qq];
          const uint32_t mask = __ballot_sync(0xffffffffu, take);
          if (mask) {
            const uint32_t cnt = __popc(mask), r = __popc(mask & lt);
            const uint32_t avail = cend[qq] - cpos[qq];
            uint32_t pos = cpos[qq] + r;
            if (cnt <= avail) {
              cpos[qq] += cnt;
            } else {
              const uint32_t rsv = max(cnt - avail, p.cand_chunk);
              uint32_t nb = 0;
              if (lane == 0) nb = atomicAdd(&p.cand_cnt[g * QG + q0 + qq], rsv);
              nb = __shfl_sync(0xffffffffu, nb, 0);
              if (r >= avail) pos = nb + (r - avail);
              cpos[qq] = nb + (cnt - avail);
              cend[qq] = nb + rsv;
            }
            if (take && pos < (uint64_t)p.cand_cap)
              p.cand[(g * QG + q0 + qq) * p.cand_cap + pos] =
                  make_uint2(score_key(sc[qq]), (uint32_t)j);
          }
        }
      } else if (j < n32 || p.tile_stride > 1) {
        // (a sampled row is compact: its columns past the entries read -inf)
#pragma unroll
        for (int qq = 0; qq < C::QPW; ++qq) srow[qq][jc] = j < vis[qq] ? sc[qq] : -INFINITY;
      }
      if constexpr (QG == 1) {
        // first-level histogram of the visible keys (the top-k's level 1):
        // the CTA's first two groups in shared memory, any later one (short
        // rows) straight to global memory
        if (p.hist1 && j < vis[0]) {
          const uint32_t bin = score_key(sc[0]) >> 20;
          const int64_t slot = g - g_first;
          if (slot < C::HSLOTS)
            atomicAdd(hslot + slot * kTopkBins + bin, 1u);
          else
          {
            atomicAdd(p.hist1 + g * kTopkHistStride + bin, 1u);
            atomicAdd(p.hist1 + g * kTopkHistStride + kTopkBins + (bin >> 6), 1u);
          }
        }
      }
    }
    if (p.cand && g_prev >= 0) flush_chunks(g_prev);
  }

  tc_fence_before();
  __syncthreads();
  pdl_trigger();  // the next kernel may start launching while this one drains
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
  if constexpr (QG == 1) {
    if (p.hist1 && t_end > t_begin) {
      const int64_t g_last = (t_end - 1) / p.ktiles;
      for (int sl = 0; sl < C::HSLOTS && g_first + sl <= g_last; ++sl)
        {
          uint32_t* hrow = p.hist1 + (g_first + sl) * kTopkHistStride;
          for (int i = threadIdx.x; i < kTopkBins; i += C::THREADS) {
            const uint32_t v = hslot[sl * kTopkBins + i];
            if (v) atomicAdd(&hrow[i], v);
          }
          if (threadIdx.x < kTopkCoarse) {  // coarse bin t: fine bins 64t .. 64t + 63
            uint32_t v = 0;
            for (int i = 0; i < kTopkBins / kTopkCoarse; ++i)
              v += hslot[sl * kTopkBins + threadIdx.x * (kTopkBins / kTopkCoarse) + i];
            if (v) atomicAdd(&hrow[kTopkBins + threadIdx.x], v);
          }
        }
    }
  }
}

// ---- host side: tensor maps ----

EncodeTiledFn encode_fn() { return tensor_map_encoder(); }

// CTAs of a launch over `total` tiles (at most CTAS_PER_SM per SM).
template <int QG>
int64_t tc_grid(int64_t total) {
  return std::min<int64_t>(total, (int64_t)TcCfg<QG>::CTAS_PER_SM * sm_count());
}

// q8 / c: the quantised queries; or, both null, bf16 queries a.q and raw
// weights a.w quantised inside the kernel (decode only, see TcParams::qbf).
template <int QG>
csa2_status launch_tc(const csa2_index_args& a, const uint8_t* q8, const float* c,
                      uint32_t* hist1, IndexTuning tune, cudaStream_t s,
                      const IndexSelect* sel = nullptr, const NewRows* nr = nullptr) {
  using C = TcCfg<QG>;
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cuda_fail(cudaErrorNotSupported);
  const int64_t nq = a.B * a.q_per_seq;
  const bool fuse_q = q8 == nullptr;
  CUtensorMap kmap, qmap;
  std::memset(&qmap, 0, sizeof(qmap));
  if (a.pages.block_table) {
    // the page pool as rows of 128 bytes, loaded in 64-row boxes
    cuuint64_t dims[2] = {(cuuint64_t)a.di,
                          (cuuint64_t)a.pages.num_pages * (cuuint64_t)a.pages.page_rows};
    cuuint64_t strides[1] = {(cuuint64_t)a.k_ld};
    cuuint32_t box[2] = {128, (cuuint32_t)(a.pages.page_rows % 128 == 0 ? 128 : 64)};
    cuuint32_t es[2] = {1, 1};
    if (enc(&kmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(a.k), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return CSA2_ERR_INVALID_ARG;
  } else {
    cuuint64_t dims[3] = {(cuuint64_t)a.di, (cuuint64_t)a.n, (cuuint64_t)a.B};
    cuuint64_t strides[2] = {(cuuint64_t)a.k_ld, (cuuint64_t)a.k_seq_stride};
    cuuint32_t box[3] = {128, 128, 1};
    cuuint32_t es[3] = {1, 1, 1};
    if (enc(&kmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(a.k), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return CSA2_ERR_INVALID_ARG;
  }
  if (!fuse_q) {
    cuuint64_t dims[2] = {(cuuint64_t)a.di, (cuuint64_t)(nq * a.hi)};
    cuuint64_t strides[1] = {(cuuint64_t)a.di};
    cuuint32_t box[2] = {128, (cuuint32_t)C::BN};
    cuuint32_t es[2] = {1, 1};
    if (enc(&qmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(q8), dims, strides,
            box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return CSA2_ERR_INVALID_ARG;
  }
  // the kernel's per-tile arithmetic is 32-bit: entries and tiles of a
  // launch stay below 2^31
  if (a.n > ((int64_t)1 << 30) || (nq / QG) * ((a.n + C::BM - 1) / C::BM) >= ((int64_t)1 << 31) ||
      (sel && sel->tile_stride > 1024))
    return CSA2_ERR_UNSUPPORTED;
  TcParams p;
  p.c = c;
  p.qbf = fuse_q ? static_cast<const uint16_t*>(a.q) : nullptr;
  p.w = fuse_q ? a.w : nullptr;
  p.n_valid = a.n_valid;
  p.scores = a.scores;
  p.scores_ld = a.scores_ld;
  p.n = a.n;
  p.q_per_seq = a.q_per_seq;
  p.groups = nq / QG;
  p.ktiles = (a.n + C::BM - 1) / C::BM;
  if (sel && sel->tile_stride > 1)  // sampled: every tile_stride-th tile
    p.ktiles = (p.ktiles + sel->tile_stride - 1) / sel->tile_stride;
  p.dev_status = a.dev_status;
  p.hist1 = QG == 1 ? hist1 : nullptr;
  p.reverse = tune.reverse ? 1 : 0;
  p.keep_in_l2 = tune.keep_in_l2 ? 1 : 0;
  p.pages = a.pages;
  p.pg_box = a.pages.page_rows % 128 == 0 ? 128 : 64;
  p.pg_shift = -1;
  if (a.pages.page_rows > 0 && (a.pages.page_rows & (a.pages.page_rows - 1)) == 0)
    for (p.pg_shift = 0; (1 << p.pg_shift) < a.pages.page_rows; ++p.pg_shift) {
    }
  p.wait_ns = pipeline_wait_ns();
  p.stall_loads = stall_loads() ? 1 : 0;
  p.tile_stride = sel && sel->tile_stride > 1 ? sel->tile_stride : 1;
  p.theta = sel ? sel->theta : nullptr;
  p.cand_cnt = sel ? sel->cand_cnt : nullptr;
  p.cand = sel ? sel->cand : nullptr;
  p.cand_cap = sel ? sel->cand_cap : 0;
  if (nr) p.nr = *nr;
  const int64_t total = p.groups * p.ktiles;
  if (total == 0) return CSA2_OK;
  const int grid = (int)tc_grid<QG>(total);
  {
    // a query's (warp, query) streams: STREAMS tile streams x 4 warps in each CTA
    // whose range meets the query's group; each may leave up to 31 reserved
    // slots unused.  Chunks of 32 while that waste stays within a quarter of
    // the buffer, else exact reservations.
    const int64_t per_cta = (total + grid - 1) / grid;
    const int64_t ctas_per_group = (p.ktiles + per_cta - 1) / per_cta + 1;
    const int64_t waste = (int64_t)C::STREAMS * 4 * ctas_per_group * 31;
    p.cand_chunk = waste * 4 <= p.cand_cap ? 32u : 0u;
  }
  static std::atomic<uint64_t> attr_done{0};
  cudaError_t e = once_per_device(attr_done, [] {
    return cudaFuncSetAttribute(idx_score_tc_kernel<QG>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
  });
  if (e != cudaSuccess) return cuda_fail(e);
  return launch_kernel(idx_score_tc_kernel<QG>, dim3(grid), dim3(C::THREADS),
                       (size_t)C::SMEM_ALLOC, s, 1, kmap, qmap, p);
}

}  // namespace

csa2_status launch_index_score_fp8(const csa2_index_args& a, const uint8_t* q8, const float* c,
                                   uint32_t* hist1, IndexTuning tune, cudaStream_t s) {
  if (a.hi != 64 || a.di != 128) return CSA2_ERR_UNSUPPORTED;
  if (a.B * a.q_per_seq == 0 || a.n == 0) return CSA2_OK;
  if (a.q_per_seq % 4 == 0) return launch_tc<4>(a, q8, c, nullptr, tune, s);
  return launch_tc<1>(a, q8, c, hist1, tune, s);
}

bool index_bf16q_supported(const csa2_index_args& a, const NewRows* nr) {
  if (a.hi != 64 || a.di != 128 || a.q_dtype != CSA2_BF16 || a.k_dtype != CSA2_E4M3 ||
      a.q_per_seq % 4 == 0)
    return false;
  const int64_t nq = a.B * a.q_per_seq;
  if (nq > 0 && a.n > 0) {
    // every CTA's tile range must span at most two query groups
    const int64_t ktiles = (a.n + TcCfg<1>::BM - 1) / TcCfg<1>::BM;
    const int64_t total = nq * ktiles;
    const int64_t grid = tc_grid<1>(total);
    if ((total + grid - 1) / grid > ktiles + 1) return false;
  }
  if ((reinterpret_cast<uintptr_t>(a.q) & 15) != 0) return false;
  if (nr) {
    // one query per sequence (each key tile read by one CTA), a few new rows
    // of whole 256-element parts, 16-byte rows, inside the caches
    if (a.q_per_seq != 1 || nr->rows < 1 || nr->rows > 128 || nr->d < 256 || nr->d % 256 != 0)
      return false;
    if (nr->row0 < 0 || nr->row0 + nr->rows > a.n) return false;
    if (!nr->kv || !nr->idxk || !nr->codes || !nr->scales || !nr->k8) return false;
    if (((reinterpret_cast<uintptr_t>(nr->kv) | reinterpret_cast<uintptr_t>(nr->idxk) |
          reinterpret_cast<uintptr_t>(nr->k8)) & 15) != 0 ||
        (reinterpret_cast<uintptr_t>(nr->codes) & 3) != 0)
      return false;
    if (nr->k8 != a.k || a.k_ld != 128 || (!a.pages.block_table && a.k_seq_stride != a.n * 128))
      return false;  // the keys the launch reads are the cache the new rows go to
  }
  return true;
}

csa2_status launch_index_score_bf16q(const csa2_index_args& a, uint32_t* hist1, IndexTuning tune,
                                     cudaStream_t s, const NewRows* nr) {
  if (!index_bf16q_supported(a, nr)) return CSA2_ERR_UNSUPPORTED;
  const int64_t nq = a.B * a.q_per_seq;
  if (nq == 0 || a.n == 0) return CSA2_OK;
  return launch_tc<1>(a, nullptr, nullptr, hist1, tune, s, nullptr, nr);
}

csa2_status launch_index_select_prefill(const csa2_index_args& a, const uint8_t* q8,
                                        const float* c, const IndexSelect& sel, cudaStream_t s) {
  if (a.hi != 64 || a.di != 128 || a.q_per_seq % 4 != 0) return CSA2_ERR_UNSUPPORTED;
  if (a.B * a.q_per_seq == 0 || a.n == 0) return CSA2_OK;
  return launch_tc<4>(a, q8, c, nullptr, IndexTuning{}, s, &sel);
}

EncodeTiledFn tensor_map_encoder() {
  static std::atomic<EncodeTiledFn> fn{nullptr};
  EncodeTiledFn f = fn.load(std::memory_order_acquire);
  if (!f) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      f = reinterpret_cast<EncodeTiledFn>(p);
      fn.store(f, std::memory_order_release);
    }
  }
  return f;
}

uint64_t wait_limit_ns() { return pipeline_wait_ns(); }

bool index_fuses_topk_hist(const csa2_index_args& a) {
  return (a.q_dtype == CSA2_BF16 || a.q_dtype == CSA2_E4M3) && a.k_dtype == CSA2_E4M3 &&
         a.q_per_seq % 4 != 0;
}

}  // namespace csa2
