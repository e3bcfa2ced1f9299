// sparse_attn.cu -- a5, attention over the selected FP4 entries joined with
// the bf16 sliding window under one softmax.
//
// The selected compressed entries are gathered from the FP4 E2M1 main KV
// cache (aiany.app DeepSeek-V4.1-Flash page, "What Sets It Apart") and
// attended together with the layer-local sliding window ("DeepSeek-V4.1-
// Flash: Pushing the Limits of KV Cache Compression", Introduction: a
// global branch beside local sliding-window attention).  One latent row is
// both key and value.
//
// attn_f32_kernel    fp32 queries, one CTA per (query, head), CUDA cores.
// attn_bf16_kernel   bf16 queries, d = 512: one CTA per (80-key chunk, 16
//                    heads, query).  The chunk's rows are gathered and
//                    dequantised into shared memory as bf16 (exact: every
//                    E2M1 value times a UE8M0 scale is a bf16 value), then
//                    S = Q K^T and O = P V run as m16n8k16 bf16 MMAs with
//                    fp32 accumulation (at 16 heads the operands are too
//                    thin for the tcgen05 path: every tcgen05 MMA would
//                    re-read a 4 KB key tile from shared memory); P is split
//                    into two bf16 terms (p = hi + lo) so the probabilities
//                    keep ~16 bits.  Each chunk writes its (max, sum,
//                    unnormalised O) to the workspace; the chunks of one
//                    (query, head group) form a thread-block cluster and,
//                    after one cluster barrier, each merges a slice of the
//                    output.  With more than 8 chunks attn_combine_kernel
//                    merges instead.
#include <cooperative_groups.h>

#include "common.cuh"
#include "internal.h"

namespace csa2 {

namespace {

// Where key t of query q comes from: an FP4 row, a window row, or nothing.
struct KeySrc {
  const uint8_t* codes;  // FP4 row (null if not FP4)
  const uint8_t* scales;
  const uint16_t* win;   // bf16 window row (null if not window)
};

__device__ __forceinline__ KeySrc key_source(const csa2_attn_args& a, int64_t qi, int64_t t,
                                             int32_t ws, int32_t wl) {
  KeySrc r{nullptr, nullptr, nullptr};
  const int64_t b = (uint32_t)qi / (uint32_t)a.q_per_seq;  // queries fit 32 bits
  if (t < a.k) {
    const int32_t j = a.idx[qi * a.idx_ld + t];
    if (j < -1 || j >= a.n) {
      raise_flag(a.dev_status, CSA2_DEVFLAG_BOUNDS);
      return r;
    }
    if (j < 0) return r;
    if (a.pages.block_table) {  // paged: the entry's row in the pool
      const int64_t row = paged_row(a.pages, b, j, a.dev_status);
      if (row < 0) return r;
      r.codes = a.codes + row * a.codes_ld;
      r.scales = a.scales + row * a.scales_ld;
      return r;
    }
    r.codes = a.codes + b * a.codes_seq_stride + (int64_t)j * a.codes_ld;
    r.scales = a.scales + b * a.scales_seq_stride + (int64_t)j * a.scales_ld;
    return r;
  }
  const int64_t u = t - a.k;
  if (u < wl) {
    const int64_t row = (int64_t)ws + u;
    if (row < 0 || row >= a.w_rows) {
      raise_flag(a.dev_status, CSA2_DEVFLAG_BOUNDS);
      return r;
    }
    r.win = static_cast<const uint16_t*>(a.window) + b * a.win_seq_stride + row * a.win_ld;
  }
  return r;
}

// The query's window rows [ws, ws + wl).  A length above the launch's bound
// win_max is clipped to it and raises CSA2_DEVFLAG_BOUNDS, like a row outside
// [0, w_rows) (the launch only has room for win_max window keys).
__device__ __forceinline__ void window_of(const csa2_attn_args& a, int64_t qi, int32_t& ws,
                                          int32_t& wl) {
  ws = a.win_start ? a.win_start[qi] : 0;
  wl = a.win_len ? a.win_len[qi] : a.w_rows;
  if (wl < 0) wl = 0;
  if (wl > a.win_max) {
    raise_flag(a.dev_status, CSA2_DEVFLAG_BOUNDS);
    wl = a.win_max;
  }
}

// ---------------------------------------------------------------------------
// fp32 path
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(128) attn_f32_kernel(const csa2_attn_args a) {
  extern __shared__ float sm[];  // q [d], logits [k + win_max]
  pdl_wait();
  const int64_t qi = blockIdx.y;
  const int h = blockIdx.x;
  const int d = a.d;
  float* sq = sm;
  float* lg = sm + d;
  __shared__ float red[4];
  const float* qsrc = static_cast<const float*>(a.q) + (qi * a.hq + h) * (int64_t)d;
  for (int i = threadIdx.x; i < d; i += blockDim.x) sq[i] = qsrc[i];
  int32_t ws, wl;
  window_of(a, qi, ws, wl);
  const int64_t nkeys = a.k + wl;
  __syncthreads();
  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  // logits: one warp per key
  for (int64_t t = warp; t < nkeys; t += 4) {
    const KeySrc src = key_source(a, qi, t, ws, wl);
    float dot = 0.f;
    const bool valid = src.codes || src.win;
    if (valid) {
      for (int i = lane; i < d; i += 32) {
        float kv;
        if (src.codes) {
          const uint32_t byte = src.codes[i >> 1];
          kv = e2m1_value((byte >> ((i & 1) * 4)) & 15u) * ue8m0_value(src.scales[i >> 5]);
        } else {
          kv = bf16_bits_to_float(src.win[i]);
        }
        dot = fmaf(sq[i], kv, dot);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
    }
    if (lane == 0) lg[t] = valid ? dot * a.softmax_scale : -INFINITY;
  }
  __syncthreads();
  // softmax statistics
  float mx = -INFINITY;
  for (int64_t t = threadIdx.x; t < nkeys; t += blockDim.x) mx = fmaxf(mx, lg[t]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (lane == 0) red[warp] = mx;
  __syncthreads();
  mx = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
  __syncthreads();
  float sum = 0.f;
  for (int64_t t = threadIdx.x; t < nkeys; t += blockDim.x) {
    const float p = (mx == -INFINITY) ? 0.f : expf(lg[t] - mx);
    lg[t] = p;
    sum += p;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (lane == 0) red[warp] = sum;
  __syncthreads();
  sum = red[0] + red[1] + red[2] + red[3];
  const float inv = sum > 0.f ? 1.f / sum : 0.f;
  float* out = a.out + (qi * a.hq + h) * (int64_t)d;
  for (int i = threadIdx.x; i < d; i += blockDim.x) {
    float acc = 0.f;
    for (int64_t t = 0; t < nkeys; ++t) {
      const float p = lg[t];
      if (p == 0.f) continue;
      const KeySrc src = key_source(a, qi, t, ws, wl);
      float kv;
      if (src.codes) {
        const uint32_t byte = src.codes[i >> 1];
        kv = e2m1_value((byte >> ((i & 1) * 4)) & 15u) * ue8m0_value(src.scales[i >> 5]);
      } else {
        kv = bf16_bits_to_float(src.win[i]);
      }
      acc = fmaf(p, kv, acc);
    }
    out[i] = acc * inv;
  }
}

// ---------------------------------------------------------------------------
// bf16 tensor-core path (d = 512, 16 heads per CTA, 80 keys per chunk)
// ---------------------------------------------------------------------------

constexpr int kD = 512;
// 16 heads per CTA keep two CTAs on an SM (about 104 KB of shared memory
// each), so the 8-CTA clusters of a 1M-context decode step all run at once.
constexpr int kHG = 16;                  // heads per CTA
constexpr int kKC = 80;                  // keys per chunk
constexpr int kPairs = kKC / 16;         // key pairs of 16 (two n8 tiles)
constexpr int kAttnWarps = 8;
constexpr int kAttnThreads = 32 * kAttnWarps;
constexpr int kSWarps = kPairs;          // S = Q K^T: warp w < kSWarps owns keys 16w .. 16w + 15
constexpr int kPVSlice = kD / kAttnWarps;  // O = P V: warp w owns 64 dims
constexpr int kMaxClusterChunks = 8;     // portable cluster size
constexpr int kRowBytes = kD * 2 + 16;   // padded bf16 row (conflict-free ldmatrix)
constexpr int kPRow = kKC * 2 + 16;      // padded P row
constexpr int kSmemQ = kHG * kRowBytes;
constexpr int kSmemK = kKC * kRowBytes;
constexpr int kSmemP = 2 * kHG * kPRow;  // P split into bf16 hi and lo
constexpr int kAttnSmem = kSmemQ + kSmemK + kSmemP;
constexpr int kPieces = kD / 8;          // 16-byte pieces of a bf16 row (8 elements)
constexpr int kBlocks = kD / 32;         // 32-element blocks of a row (16 code bytes each)
constexpr int kBItems = kKC * kBlocks / kAttnThreads;  // K-tile blocks per thread
constexpr int kQItems = kHG * kPieces / kAttnThreads;  // Q-tile pieces per thread
static_assert(kKC * kBlocks % kAttnThreads == 0 && kAttnThreads % kBlocks == 0 &&
                  kHG * kPieces % kAttnThreads == 0,
              "tiles split evenly over the threads, one block column per thread");
static_assert(kSWarps <= kAttnWarps && kKC % 16 == 0, "S tiling");
static_assert(kPVSlice == 64, "PV tiling");

struct PartialLayout {
  // per (query, head group, chunk): O [kHG][512] f32 (unnormalised), then m [kHG], l [kHG]
  static constexpr int64_t kFloats = (int64_t)kHG * kD + 2 * kHG;
};

// Rows of one chunk: a FP4 row (codes + scales), a bf16 window row, or none.
struct ChunkRows {
  const uint8_t* codes[kKC];
  const uint8_t* scales[kKC];
  const uint16_t* win[kKC];
};

// Dequantises 32 E2M1 codes (16 bytes, element 2i in the low nibble of byte
// i) with scale byte sb into four 16-byte bf16 pieces at d0 .. d3 (piece v =
// elements 8v .. 8v + 7).  Exact: every E2M1 value times a UE8M0 scale in
// [2^-127, 2^125] is a bf16 value.  Out of line: the instruction cache holds
// one copy of this code, whatever the number of call sites.
__device__ __noinline__ void dequant_block(uint4 cw, uint32_t sb, uint8_t* d0, uint8_t* d1,
                                           uint8_t* d2, uint8_t* d3) {
  // scale 2^(sb - 127) in [2^-119, 2^123]: every product is a normal bf16,
  // so the bf16x2 multiply is exact; other scales take fp32
  if (sb >= 8 && sb <= 250) {
    const __nv_bfloat16 sc1 = __float2bfloat16_rn(ue8m0_value(sb));
    const __nv_bfloat162 sc2 = __halves2bfloat162(sc1, sc1);
    uint32_t p[4];
    e2m1x8_to_bf16(cw.x, sc2, p);
    *reinterpret_cast<uint4*>(d0) = make_uint4(p[0], p[1], p[2], p[3]);
    e2m1x8_to_bf16(cw.y, sc2, p);
    *reinterpret_cast<uint4*>(d1) = make_uint4(p[0], p[1], p[2], p[3]);
    e2m1x8_to_bf16(cw.z, sc2, p);
    *reinterpret_cast<uint4*>(d2) = make_uint4(p[0], p[1], p[2], p[3]);
    e2m1x8_to_bf16(cw.w, sc2, p);
    *reinterpret_cast<uint4*>(d3) = make_uint4(p[0], p[1], p[2], p[3]);
    return;
  }
  const float scf = ue8m0_value(sb);
  auto slow = [&](uint32_t word, uint8_t* dst) {
    uint32_t p[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const uint32_t byte = (word >> (8 * b)) & 0xFFu;
      p[b] = pack_bf16x2(e2m1_value(byte & 15u) * scf, e2m1_value(byte >> 4) * scf);
    }
    *reinterpret_cast<uint4*>(dst) = make_uint4(p[0], p[1], p[2], p[3]);
  };
  slow(cw.x, d0);
  slow(cw.y, d1);
  slow(cw.z, d2);
  slow(cw.w, d3);
}

// One CTA = (key chunk, 16 heads, query), 8 warps, two CTAs per SM.  Phases:
//  1. key sources of the chunk (idx reads); Q rows copying by cp.async;
//  2. K tile: window rows by cp.async; FP4 rows load their code and scale
//     bytes into registers (every load in flight), then dequantise exactly
//     to bf16; keys without a row are zero rows;
//  3. S = Q K^T (warps 0..4, m16n8k16 bf16 MMA, fp32 accumulate), the
//     chunk's softmax statistics per head, P = e^(S - m) split into bf16 hi +
//     lo (~16 significant bits);
//  4. O = P V (8 warps, 64 dims each);
//  5. the unnormalised O, m and l go to this chunk's partial in the
//     workspace.  CLUSTER: the chunks of one (query, head group) are a
//     thread-block cluster; after one cluster barrier each CTA merges
//     1/nchunks of the output from every chunk's partial.  Otherwise
//     attn_combine_kernel merges.
// pre: Q, the window rows and the window ranges may be read before the
// programmatic-launch wait (the caller knows the kernels still running on the
// stream do not write them): Q and the first chunk's window rows are copied
// into shared memory while the previous kernel drains.
// MODE: kModeCombine (chunk partials, merged by attn_combine_kernel),
// kModeCluster (the chunks of a query and head group are a cluster and merge
// their partials through L2) or kModeSeq (one CTA per query and head group
// walks its chunks in order with a running softmax: no partials).
constexpr int kModeCombine = 0, kModeCluster = 1, kModeSeq = 2;

template <int MODE>
__global__ void __launch_bounds__(kAttnThreads, 2)
    attn_bf16_kernel(const csa2_attn_args a, int nchunks, int fk, float* __restrict__ partial,
                     int pre) {
  extern __shared__ __align__(16) uint8_t sm_raw[];
  uint8_t* sQ = sm_raw;
  uint8_t* sK = sm_raw + kSmemQ;
  uint8_t* sPh = sK + kSmemK;
  uint8_t* sPl = sPh + kHG * kPRow;
  __shared__ ChunkRows rows;
  __shared__ float red_m[kPairs][kHG], red_l[kPairs][kHG];
  // kModeSeq: the running softmax state of each head and this chunk's rescale
  __shared__ float run_m[kHG], run_l[kHG], run_f[kHG];

  const int hg = blockIdx.y;
  const int64_t qi = blockIdx.z;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid & 31;
  const int ngroups = (a.hq + kHG - 1) / kHG;
  // heads of this group that exist (hq may be an odd multiple of 16)
  const int hvalid = min(kHG, a.hq - hg * kHG);
  auto load_q = [&] {
    const uint8_t* qsrc = static_cast<const uint8_t*>(a.q) +
                          ((qi * a.hq + (int64_t)hg * kHG) * kD) * 2;
#pragma unroll
    for (int u = 0; u < kQItems; ++u) {
      const int i = tid + u * kAttnThreads;
      const int r = i / kPieces, c = i % kPieces;
      if (r < hvalid)
        cp_async16(sQ + r * kRowBytes + c * 16, qsrc + r * kD * 2 + c * 16);
      else
        *reinterpret_cast<uint4*>(sQ + r * kRowBytes + c * 16) = make_uint4(0, 0, 0, 0);
    }
  };
  int32_t ws = 0, wl = 0;
  int64_t nkeys = 0;
  if (pre) {
    load_q();
    window_of(a, qi, ws, wl);
    nkeys = a.k + wl;
  }

  // the key list index of row r of chunk c (-1: no key)
  auto key_of = [&](int c, int r) -> int64_t {
    if (fk > 0) {
      if (r < fk) {
        const int64_t i = (int64_t)c * fk + r;
        return i < a.k ? i : -1;
      }
      const int64_t u = (int64_t)c * (kKC - fk) + (r - fk);
      return u < wl ? a.k + u : -1;
    }
    const int64_t t = (int64_t)c * kKC + r;
    return t < nkeys ? t : -1;
  };
  // the first chunk's window rows (inputs no earlier kernel writes, like Q)
  // are copied before the programmatic-launch wait
  const int c_first = MODE == kModeSeq ? 0 : (int)blockIdx.x;
  if (pre) {
    const int c = tid % kBlocks;
    const int rot = (tid >> 1) & 3;
#pragma unroll
    for (int u = 0; u < kBItems; ++u) {
      const int r = tid / kBlocks + u * (kAttnThreads / kBlocks);
      const int64_t t = key_of(c_first, r);
      if (t >= a.k) {
        const KeySrc src = key_source(a, qi, t, ws, wl);
        if (src.win) {
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const int vv = (v + rot) & 3;
            cp_async16(sK + r * kRowBytes + c * 64 + vv * 16, src.win + c * 32 + vv * 8);
          }
        }
      }
    }
  }
  pdl_wait();
  if (!pre) {
    load_q();
    window_of(a, qi, ws, wl);
    nkeys = a.k + wl;
  }
  const int d0 = warp * kPVSlice;
  const int r0 = lane >> 2;  // rows (heads) r0 and r0 + 8 of this thread's MMA fragments
  float o[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  if constexpr (MODE == kModeSeq) {
    if (tid < kHG) {
      run_m[tid] = -INFINITY;
      run_l[tid] = 0.f;
    }
  }
  for (int chunk = MODE == kModeSeq ? 0 : (int)blockIdx.x;
       chunk < (MODE == kModeSeq ? nchunks : (int)blockIdx.x + 1); ++chunk) {
    if constexpr (MODE == kModeSeq) __syncthreads();  // the previous chunk's tiles are read
  // ---- 1. key sources.  fk > 0: chunk c holds selected keys fk c .. fk c +
  // fk - 1 and window rows (kKC - fk) c .., so every chunk gathers the same
  // mix (the softmax is over the set of keys, in any order); fk = 0: keys
  // t = kKC c .. of the list (selected keys, then the window)
  if (tid < kKC) {
    const int64_t t = key_of(chunk, tid);
    KeySrc src{nullptr, nullptr, nullptr};
    if (t >= 0) src = key_source(a, qi, t, ws, wl);
    rows.codes[tid] = src.codes;
    rows.scales[tid] = src.scales;
    rows.win[tid] = src.win;
  }
  __syncthreads();

  // ---- 2. K tile: item = (row r, 32-element block c) = 16 code bytes -> 64
  // bf16 bytes; thread t always takes block c = t % 16 of rows t / 16 + 16u.
  // FP4 items load their 16 code bytes and scale byte into registers first
  // (every load in flight at once); window items copy 64 bytes with
  // cp.async.  An item's four 16-byte output pieces go out in the order
  // (v + t / 2) % 4, so each group of 8 lanes covers all 8 bank quads of its
  // 128-byte wavefront.
  {
    const int c = tid % kBlocks;
    const int rot = (tid >> 1) & 3;
    uint4 cw[kBItems];
    uint32_t sb[kBItems];
#pragma unroll
    for (int u = 0; u < kBItems; ++u) {
      const int r = tid / kBlocks + u * (kAttnThreads / kBlocks);
      const uint8_t* cp = rows.codes[r];
      cw[u] = cp ? __ldg(reinterpret_cast<const uint4*>(cp) + c) : make_uint4(0, 0, 0, 0);
      sb[u] = cp ? (uint32_t)__ldg(rows.scales[r] + c) : 0u;
      if (const uint16_t* wrow = rows.win[r]; wrow && !(pre && chunk == c_first)) {
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const int vv = (v + rot) & 3;
          cp_async16(sK + r * kRowBytes + c * 64 + vv * 16, wrow + c * 32 + vv * 8);
        }
      }
    }
#pragma unroll  // small: the dequantiser is one out-of-line copy
    for (int u = 0; u < kBItems; ++u) {
      const int r = tid / kBlocks + u * (kAttnThreads / kBlocks);
      if (rows.win[r]) continue;  // copied by cp.async
      uint8_t* row = sK + r * kRowBytes + c * 64;
      if (rows.codes[r]) {
        // piece v (code word v) always lands at row + 16 v; the words are
        // handed over starting at piece rot, so the stores go out in the
        // rotated order
        const uint4 w = cw[u];
        auto word = [&](int v) {
          v &= 3;
          return v == 0 ? w.x : (v == 1 ? w.y : (v == 2 ? w.z : w.w));
        };
        dequant_block(make_uint4(word(rot), word(rot + 1), word(rot + 2), word(rot + 3)), sb[u],
                      row + ((0 + rot) & 3) * 16, row + ((1 + rot) & 3) * 16,
                      row + ((2 + rot) & 3) * 16, row + ((3 + rot) & 3) * 16);
      } else {  // no key: a zero row (finite values where P is 0)
#pragma unroll
        for (int v = 0; v < 4; ++v)
          *reinterpret_cast<uint4*>(row + v * 16) = make_uint4(0, 0, 0, 0);
      }
    }
  }
  cp_async_wait_all();
  __syncthreads();
  if constexpr (MODE == kModeSeq) {
    // the next chunk's rows move into L2 while this chunk is computed
    if (tid < kKC && chunk + 1 < nchunks) {
      const int64_t t = key_of(chunk + 1, tid);
      if (t >= 0) {
        const KeySrc src = key_source(a, qi, t, ws, wl);
        if (src.codes) {
          asm volatile("prefetch.global.L2 [%0];" ::"l"(src.codes));
          asm volatile("prefetch.global.L2 [%0];" ::"l"(src.codes + 128));
          asm volatile("prefetch.global.L2 [%0];" ::"l"(src.scales));
        } else if (src.win) {
#pragma unroll
          for (int b = 0; b < kD * 2; b += 128)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const uint8_t*>(src.win) + b));
        }
      }
    }
  }

  // ---- 3. S = Q K^T and the chunk softmax (warps 0 .. kSWarps-1)
  if (warp < kSWarps) {
    const int pr = warp;
    // two independent accumulator chains per n-tile: dims 0..255 and 256..511
    float s1[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    float s2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    const uint32_t qbase = smem_u32(sQ) + (lane & 15) * kRowBytes + (lane >> 4) * 16;
    const int krow = pr * 16 + (lane & 7) + ((lane >> 4) << 3);
    const uint32_t kbase = smem_u32(sK) + krow * kRowBytes + ((lane >> 3) & 1) * 16;
#pragma unroll 4
    for (int ks = 0; ks < kD / 32; ++ks) {
      uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
      uint32_t c0, c1, c2, c3, d0, d1, d2, d3;
      ldmatrix_x4(qbase + ks * 32, a0, a1, a2, a3);
      ldmatrix_x4(kbase + ks * 32, b0, b1, b2, b3);
      ldmatrix_x4(qbase + (ks + kD / 32) * 32, c0, c1, c2, c3);
      ldmatrix_x4(kbase + (ks + kD / 32) * 32, d0, d1, d2, d3);
      mma_bf16_16816(s1[0], a0, a1, a2, a3, b0, b1);
      mma_bf16_16816(s1[1], a0, a1, a2, a3, b2, b3);
      mma_bf16_16816(s2[0], c0, c1, c2, c3, d0, d1);
      mma_bf16_16816(s2[1], c0, c1, c2, c3, d2, d3);
    }
    // rows (heads) r0 (e = 0, 1) and r0 + 8 (e = 2, 3); keys 16pr + 8nt + 2(lane%4) + (e&1)
    float sc[2][4];
    float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = pr * 16 + nt * 8 + 2 * (lane & 3) + (e & 1);
        const bool valid = rows.codes[key] || rows.win[key];
        sc[nt][e] = valid ? (s1[nt][e] + s2[nt][e]) * a.softmax_scale : -INFINITY;
        if (e < 2)
          m0 = fmaxf(m0, sc[nt][e]);
        else
          m1 = fmaxf(m1, sc[nt][e]);
      }
#pragma unroll
    for (int o = 1; o < 4; o <<= 1) {
      m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, o));
      m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, o));
    }
    if ((lane & 3) == 0) {
      red_m[pr][r0] = m0;
      red_m[pr][r0 + 8] = m1;
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kSWarps * 32) : "memory");  // S warps only
    m0 = m1 = -INFINITY;
#pragma unroll
    for (int w = 0; w < kPairs; ++w) {
      m0 = fmaxf(m0, red_m[w][r0]);
      m1 = fmaxf(m1, red_m[w][r0 + 8]);
    }
    if constexpr (MODE == kModeSeq) {  // P against the running maximum
      m0 = fmaxf(m0, run_m[r0]);
      m1 = fmaxf(m1, run_m[r0 + 8]);
    }
    float l0 = 0.f, l1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      float p[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float m = e < 2 ? m0 : m1;
        p[e] = (sc[nt][e] == -INFINITY) ? 0.f : __expf(sc[nt][e] - m);
      }
      l0 += p[0] + p[1];
      l1 += p[2] + p[3];
      const int col = pr * 16 + nt * 8 + 2 * (lane & 3);
      // p = hi + lo with hi = bf16(p), lo = bf16(p - hi): ~16 significant bits
      const __nv_bfloat162 h01 = __floats2bfloat162_rn(p[0], p[1]);
      const __nv_bfloat162 h23 = __floats2bfloat162_rn(p[2], p[3]);
      const float2 f01 = __bfloat1622float2(h01), f23 = __bfloat1622float2(h23);
      *reinterpret_cast<__nv_bfloat162*>(sPh + r0 * kPRow + col * 2) = h01;
      *reinterpret_cast<__nv_bfloat162*>(sPh + (r0 + 8) * kPRow + col * 2) = h23;
      *reinterpret_cast<uint32_t*>(sPl + r0 * kPRow + col * 2) =
          pack_bf16x2(p[0] - f01.x, p[1] - f01.y);
      *reinterpret_cast<uint32_t*>(sPl + (r0 + 8) * kPRow + col * 2) =
          pack_bf16x2(p[2] - f23.x, p[3] - f23.y);
    }
#pragma unroll
    for (int o = 1; o < 4; o <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, o);
      l1 += __shfl_xor_sync(0xffffffffu, l1, o);
    }
    if ((lane & 3) == 0) {
      red_l[pr][r0] = l0;
      red_l[pr][r0 + 8] = l1;
    }
  }
  __syncthreads();
  if constexpr (MODE == kModeSeq) {
    if (tid < kHG) {  // head tid: m_new = max(m_old, chunk max), l = l f + chunk sum
      float mc = run_m[tid], l = 0.f;
#pragma unroll
      for (int w = 0; w < kPairs; ++w) {
        mc = fmaxf(mc, red_m[w][tid]);
        l += red_l[w][tid];
      }
      const float f = run_m[tid] == -INFINITY ? 0.f : __expf(run_m[tid] - mc);
      run_f[tid] = f;
      run_l[tid] = run_l[tid] * f + l;
      run_m[tid] = mc;
    }
    __syncthreads();
  }

  // ---- 4. O = P V: dims d0 .. d0+63 (8 n-tiles), keys as the K dimension
  if constexpr (MODE == kModeSeq) {
    // the running state moves on: O and l scale by e^(m_old - m_new)
    const float f0 = run_f[r0], f1 = run_f[r0 + 8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      o[i][0] *= f0;
      o[i][1] *= f0;
      o[i][2] *= f1;
      o[i][3] *= f1;
    }
  }
  {
    const uint32_t pbase_h = smem_u32(sPh) + (lane & 15) * kPRow + (lane >> 4) * 16;
    const uint32_t pbase_l = smem_u32(sPl) + (lane & 15) * kPRow + (lane >> 4) * 16;
    const int vrow = (lane & 7) + ((lane >> 3) & 1) * 8;
    const uint32_t vbase = smem_u32(sK) + vrow * kRowBytes + (d0 + (lane >> 4) * 8) * 2;
#pragma unroll
    for (int ks = 0; ks < kKC / 16; ++ks) {
      uint32_t h0r, h1r, h2r, h3r, l0r, l1r, l2r, l3r;
      ldmatrix_x4(pbase_h + ks * 32, h0r, h1r, h2r, h3r);
      ldmatrix_x4(pbase_l + ks * 32, l0r, l1r, l2r, l3r);
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4_trans(vbase + ks * 16 * kRowBytes + np * 32, b0, b1, b2, b3);
        mma_bf16_16816(o[2 * np], h0r, h1r, h2r, h3r, b0, b1);
        mma_bf16_16816(o[2 * np], l0r, l1r, l2r, l3r, b0, b1);
        mma_bf16_16816(o[2 * np + 1], h0r, h1r, h2r, h3r, b2, b3);
        mma_bf16_16816(o[2 * np + 1], l0r, l1r, l2r, l3r, b2, b3);
      }
    }
  }

  }  // chunks

  if constexpr (MODE == kModeSeq) {
    // ---- 5. the output: O / l (no key: 0)
    pdl_trigger();
    const float i0 = run_l[r0] > 0.f ? 1.f / run_l[r0] : 0.f;
    const float i1 = run_l[r0 + 8] > 0.f ? 1.f / run_l[r0 + 8] : 0.f;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const int col = d0 + nt * 8 + 2 * (lane & 3);
      if (r0 < hvalid)
        *reinterpret_cast<float2*>(a.out + (qi * a.hq + (int64_t)hg * kHG + r0) * kD + col) =
            make_float2(o[nt][0] * i0, o[nt][1] * i0);
      if (r0 + 8 < hvalid)
        *reinterpret_cast<float2*>(a.out + (qi * a.hq + (int64_t)hg * kHG + r0 + 8) * kD + col) =
            make_float2(o[nt][2] * i1, o[nt][3] * i1);
    }
    return;
  }
  const int chunk = blockIdx.x;
  // ---- 5. this chunk's partial: O (unnormalised), then m and l per head
  float* part = partial + ((qi * ngroups + hg) * (int64_t)nchunks + chunk) *
                              PartialLayout::kFloats;
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) {
    const int col = d0 + nt * 8 + 2 * (lane & 3);
    *reinterpret_cast<float2*>(part + r0 * kD + col) = make_float2(o[nt][0], o[nt][1]);
    *reinterpret_cast<float2*>(part + (r0 + 8) * kD + col) = make_float2(o[nt][2], o[nt][3]);
  }
  if (tid < kHG) {
    float m = -INFINITY, l = 0.f;
#pragma unroll
    for (int w = 0; w < kPairs; ++w) {
      m = fmaxf(m, red_m[w][tid]);
      l += red_l[w][tid];
    }
    part[kHG * kD + tid] = m;
    part[kHG * kD + kHG + tid] = l;
  }

  if constexpr (MODE == kModeCluster) {
    // every chunk's partial is written (release) and visible (acquire)
    cluster_arrive_release();
    cluster_wait_acquire();
    pdl_trigger();
    const int rank = chunk;  // the cluster spans the chunks along x
    const float* base =
        partial + ((qi * ngroups + hg) * (int64_t)nchunks) * PartialLayout::kFloats;
    constexpr int kVec = kHG * kD / 4;  // float4s of the [kHG][512] output
    const int v0 = rank * kVec / nchunks, v1 = (rank + 1) * kVec / nchunks;
    for (int v = v0 + tid; v < v1; v += kAttnThreads) {
      const int h = (v * 4) / kD, d = (v * 4) % kD;
      if (h >= hvalid) break;  // v grows with h
      float2 ml[kMaxClusterChunks];
      float4 x[kMaxClusterChunks];
#pragma unroll
      for (int c = 0; c < kMaxClusterChunks; ++c) {
        if (c < nchunks) {
          const float* pc = base + c * PartialLayout::kFloats;
          ml[c] = make_float2(__ldcg(pc + kHG * kD + h), __ldcg(pc + kHG * kD + kHG + h));
          x[c] = __ldcg(reinterpret_cast<const float4*>(pc + h * kD + d));
        } else {
          ml[c] = make_float2(-INFINITY, 0.f);
          x[c] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      float M = -INFINITY;
#pragma unroll
      for (int c = 0; c < kMaxClusterChunks; ++c) M = fmaxf(M, ml[c].x);
      float L = 0.f, f[kMaxClusterChunks];
#pragma unroll
      for (int c = 0; c < kMaxClusterChunks; ++c) {
        f[c] = (ml[c].x == -INFINITY) ? 0.f : __expf(ml[c].x - M);
        L += f[c] * ml[c].y;
      }
      const float inv = L > 0.f ? 1.f / L : 0.f;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int c = 0; c < kMaxClusterChunks; ++c) {
        const float w = f[c] * inv;
        acc.x += w * x[c].x;
        acc.y += w * x[c].y;
        acc.z += w * x[c].z;
        acc.w += w * x[c].w;
      }
      *reinterpret_cast<float4*>(a.out + (qi * a.hq + (int64_t)hg * kHG + h) * kD + d) = acc;
    }
  } else {
    pdl_trigger();
  }
}

// out[q, h, :] = sum_c e^(m_c - M) O_c / sum_c e^(m_c - M) l_c
__global__ void __launch_bounds__(128)
    attn_combine_kernel(const float* __restrict__ partial, int nchunks, int hq,
                        float* __restrict__ out) {
  const int h = blockIdx.x;
  const int64_t qi = blockIdx.y;
  const int hg = h / kHG, hr = h % kHG;
  pdl_wait();
  const int ngroups = (hq + kHG - 1) / kHG;
  const float* base =
      partial + ((qi * ngroups + hg) * (int64_t)nchunks) * PartialLayout::kFloats;
  float M = -INFINITY;
  for (int c = 0; c < nchunks; ++c)
    M = fmaxf(M, base[c * PartialLayout::kFloats + kHG * kD + hr]);
  float L = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (M != -INFINITY) {
    for (int c = 0; c < nchunks; ++c) {
      const float* pc = base + c * PartialLayout::kFloats;
      const float m = pc[kHG * kD + hr];
      if (m == -INFINITY) continue;
      const float f = expf(m - M);
      L += f * pc[kHG * kD + kHG + hr];
      const float4 v = *reinterpret_cast<const float4*>(pc + hr * kD + threadIdx.x * 4);
      acc.x += f * v.x;
      acc.y += f * v.y;
      acc.z += f * v.z;
      acc.w += f * v.w;
    }
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  *reinterpret_cast<float4*>(out + (qi * hq + h) * (int64_t)kD + threadIdx.x * 4) =
      make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
}

int win_bound(const csa2_attn_args& a) { return a.win_max > 0 ? a.win_max : a.w_rows; }

int attn_chunks(const csa2_attn_args& a) {
  return (int)((a.k + win_bound(a) + kKC - 1) / kKC);
}

}  // namespace

// Many queries (a prefill chunk): one CTA per (query, head group) walking its
// chunks fills the GPU at least twice over, and no partial goes through
// memory; few queries (decode): one CTA per chunk, merged in a cluster.
bool attn_sequential(const csa2_attn_args& a) {
  const int64_t ctas = a.nq * ((a.hq + kHG - 1) / kHG);
  return ctas >= 4 * (int64_t)sm_count();
}

size_t attn_workspace_bytes(const csa2_attn_args& a) {
  if (a.q_dtype != CSA2_BF16 || attn_sequential(a)) return 0;
  // every chunk's partial (O, m, l) goes through the workspace
  const int64_t nchunks = attn_chunks(a);
  return (size_t)a.nq * ((a.hq + kHG - 1) / kHG) * nchunks * PartialLayout::kFloats *
         sizeof(float);
}

csa2_status launch_sparse_attn(const csa2_attn_args& in, cudaStream_t s, bool q_ready) {
  if (in.nq == 0) return CSA2_OK;
  csa2_attn_args a = in;
  a.win_max = win_bound(in);
  if (a.q_dtype == CSA2_F32) {
    const size_t smem = sizeof(float) * ((size_t)a.d + a.k + a.win_max);
    if (smem > 48 * 1024) return CSA2_ERR_UNSUPPORTED;
    return launch_kernel(attn_f32_kernel, dim3((unsigned)a.hq, (unsigned)a.nq), dim3(128), smem, s,
                         1, a);
  }
  const int nchunks = attn_chunks(a);
  if (nchunks == 0) {
    cudaError_t e = cudaMemsetAsync(a.out, 0, (size_t)a.nq * a.hq * kD * sizeof(float), s);
    return e == cudaSuccess ? CSA2_OK : cuda_fail(e);
  }
  static std::atomic<uint64_t> attr_done{0};
  cudaError_t e = once_per_device(attr_done, [] {
    cudaError_t r = cudaFuncSetAttribute(attn_bf16_kernel<kModeCluster>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kAttnSmem);
    if (r == cudaSuccess)
      r = cudaFuncSetAttribute(attn_bf16_kernel<kModeCombine>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, kAttnSmem);
    if (r == cudaSuccess)
      r = cudaFuncSetAttribute(attn_bf16_kernel<kModeSeq>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, kAttnSmem);
    return r;
  });
  if (e != cudaSuccess) return cuda_fail(e);
  float* partial = static_cast<float*>(a.workspace);
  const int pre = q_ready ? 1 : 0;
  // spread the selected keys and the window rows evenly over the chunks when
  // the split holds every key (the window rows' bf16 loads are four times
  // an FP4 row's bytes: a chunk of window rows alone would finish last)
  int fk = (int)((a.k + nchunks - 1) / nchunks);
  if (fk > kKC || (int64_t)(kKC - fk) * nchunks < a.win_max) fk = 0;
  const unsigned ngroups = (unsigned)((a.hq + kHG - 1) / kHG);
  if (attn_sequential(a))
    return launch_kernel(attn_bf16_kernel<kModeSeq>, dim3(1, ngroups, (unsigned)a.nq),
                         dim3(kAttnThreads), (size_t)kAttnSmem, s, 1, a, nchunks, fk, partial,
                         pre);
  const dim3 grid((unsigned)nchunks, ngroups, (unsigned)a.nq);
  if (nchunks <= kMaxClusterChunks)
    return launch_kernel(attn_bf16_kernel<kModeCluster>, grid, dim3(kAttnThreads),
                         (size_t)kAttnSmem, s, (unsigned)nchunks, a, nchunks, fk, partial, pre);
  csa2_status st = launch_kernel(attn_bf16_kernel<kModeCombine>, grid, dim3(kAttnThreads),
                                 (size_t)kAttnSmem, s, 1, a, nchunks, fk, partial, pre);
  if (st != CSA2_OK) return st;
  return launch_kernel(attn_combine_kernel, dim3((unsigned)a.hq, (unsigned)a.nq), dim3(128), 0, s,
                       1, static_cast<const float*>(partial), nchunks, (int)a.hq, a.out);
}

}  // namespace csa2
