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
// attn_tc_kernel     bf16 queries, d = 512: one CTA per (80-key chunk, 16
//                    heads, query).  The chunk's rows are gathered and
//                    dequantised into shared memory as bf16 (exact: every
//                    E2M1 value times a UE8M0 scale is a bf16 value), then
//                    S^T = K Q^T and O^T = V^T P^T run on the tcgen05
//                    tensor cores (bf16 operands, fp32 accumulators in
//                    tensor memory); P is split into two bf16 terms (p = hi
//                    + lo) so the probabilities keep ~16 bits.  Each chunk
//                    writes its (max, sum, unnormalised O) to the
//                    workspace; the chunks of one (query, head group) form
//                    a thread-block cluster and, after one cluster barrier,
//                    each merges a slice of the output.  With more than 8
//                    chunks attn_combine_kernel merges instead.
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
  const int64_t b = qi / a.q_per_seq;
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
// bf16 tensor-core path (d = 512): tcgen05, accumulators in tensor memory
// ---------------------------------------------------------------------------

constexpr int kD = 512;
constexpr int kHG = 16;                  // heads per CTA (MMA N)
constexpr int kKC = 80;                  // keys per chunk (S: MMA M = 128, rows 80.. unused)
constexpr int kAttnWarps = 8;
constexpr int kAttnThreads = 32 * kAttnWarps;
constexpr int kMaxClusterChunks = 8;     // portable cluster size
constexpr int kDBlocks = kD / 64;        // 64-element (128-byte) swizzle atoms along d
constexpr int kKBlockBytes = kKC * 128;  // one d-block of the K tile: kKC rows of 128 bytes
// shared memory (offsets from a 1024-byte aligned base)
constexpr int kOffK = 0;                              // K tile [d-block][key][128 B], swizzled
constexpr int kOffQ = kOffK + kDBlocks * kKBlockBytes;  // Q [d-block][head][128 B]
constexpr int kOffP = kOffQ + kDBlocks * kHG * 128;   // P hi, P lo: [key-block][head][128 B]
constexpr int kPBytes = 2 * kHG * 128;                // keys 0..127 in two 64-key blocks
constexpr int kAttnSmem = kOffP + 2 * kPBytes + 1024;  // + alignment slack
constexpr int kTmemCols = 128;           // S^T: 16 columns; O^T: 4 x 16 columns
constexpr int kTmemO = kHG;              // first O^T column
constexpr int kPieces = kD / 8;          // 16-byte pieces of a bf16 row (8 elements)
constexpr int kBlocks = kD / 32;         // 32-element blocks of a row (16 code bytes each)
constexpr int kBItems = kKC * kBlocks / kAttnThreads;  // K-tile blocks per thread
constexpr int kQItems = kHG * kPieces / kAttnThreads;  // Q-tile pieces per thread
constexpr uint64_t kAttnWaitNs = 2000000000ull;        // far beyond any legal wait
static_assert(kKC * kBlocks % kAttnThreads == 0 && kAttnThreads % kBlocks == 0 &&
                  kHG * kPieces % kAttnThreads == 0,
              "tiles split evenly over the threads, one block column per thread");
static_assert(kKC % 16 == 0 && kKC <= 128 && kKC > 64, "keys per chunk: PV K steps of 16");
static_assert(kKBlockBytes % 1024 == 0 && kOffQ % 1024 == 0 && kOffP % 1024 == 0,
              "swizzle atoms start on 1024-byte boundaries");
static_assert((128 - kKC) * 128 <= kDBlocks * kHG * 128,
              "rows kKC..127 of the last d-block (read by the M = 128 MMA, unused) stay "
              "inside the Q tile");

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

// Byte offset of the 16-byte piece `piece` (0..7) of row `row` inside a
// 128-byte swizzle atom: the piece index is XORed with row % 8.
__device__ __forceinline__ uint32_t swz(int row, int piece) {
  return (uint32_t)(row * 128 + ((piece ^ (row & 7)) << 4));
}

// One CTA = (key chunk, 16 heads, query).  Phases:
//  1. key sources of the chunk (idx reads); Q copied into its swizzled tile;
//  2. K tile: window rows copy with cp.async; FP4 rows load their code and
//     scale bytes into registers (all loads in flight), then dequantise
//     exactly to bf16; keys without a row are zero rows;
//  3. S^T = K Q^T: 32 MMAs (M = 128 keys, N = 16 heads, K = 16) into tensor
//     memory; the chunk's softmax statistics (m, l) per head and P = e^(s-m)
//     split into bf16 hi + lo, written as the K-major B operand of
//  4. O^T = V^T P^T: the K tile read MN-major as V^T (M = 128 dims x 4, K =
//     keys), 2 x 5 MMAs per 128 dims;
//  5. the unnormalised O, m and l go to this chunk's partial in the
//     workspace.  CLUSTER: the chunks of one (query, head group) are a
//     thread-block cluster; after one cluster barrier each CTA merges
//     1/nchunks of the output from every chunk's partial.  Otherwise
//     attn_combine_kernel merges.
// pre: Q may be read before the programmatic-launch wait (the caller knows
// the kernels still running on the stream do not write it).
template <bool CLUSTER>
__global__ void __launch_bounds__(kAttnThreads, 2)
    attn_tc_kernel(const csa2_attn_args a, int nchunks, float* __restrict__ partial, int pre) {
  extern __shared__ uint8_t sm_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t* sK = smem + kOffK;
  uint8_t* sQ = smem + kOffQ;
  uint8_t* sPh = smem + kOffP;
  uint8_t* sPl = sPh + kPBytes;
  __shared__ ChunkRows rows;
  __shared__ __align__(8) uint64_t bar_s, bar_o;
  __shared__ uint32_t tmem_slot;
  __shared__ float red_m[3][kHG], red_l[3][kHG];
  __shared__ float s_m[kHG], s_l[kHG];
  __shared__ int s_abort;

  const int chunk = blockIdx.x, hg = blockIdx.y;
  const int64_t qi = blockIdx.z;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid & 31;
  const int ngroups = a.hq / kHG;

  if (tid == 0) {
    mbar_init(&bar_s, 1);
    mbar_init(&bar_o, 1);
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(&tmem_slot, kTmemCols);
  // Q [16 heads x 512] -> [d-block][head][128 B], swizzled
  const uint8_t* qsrc =
      static_cast<const uint8_t*>(a.q) + ((qi * a.hq + (int64_t)hg * kHG) * kD) * 2;
  auto load_q = [&] {
#pragma unroll
    for (int u = 0; u < kQItems; ++u) {
      const int i = tid + u * kAttnThreads;
      const int h = i / kPieces, c = i % kPieces;
      cp_async16(sQ + (c >> 3) * (kHG * 128) + swz(h, c & 7), qsrc + h * kD * 2 + c * 16);
    }
  };
  if (pre) load_q();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  pdl_wait();
  if (!pre) load_q();

  int32_t ws, wl;
  window_of(a, qi, ws, wl);
  const int64_t nkeys = a.k + wl;

  // ---- 1. key sources
  if (tid < kKC) {
    const int64_t t = (int64_t)chunk * kKC + tid;
    KeySrc src{nullptr, nullptr, nullptr};
    if (t < nkeys) src = key_source(a, qi, t, ws, wl);
    rows.codes[tid] = src.codes;
    rows.scales[tid] = src.scales;
    rows.win[tid] = src.win;
  }
  __syncthreads();

  // ---- 2. K tile: item = (key r, 32-element block c) = 16 code bytes -> 64
  // bf16 bytes = 4 pieces of the d-block c / 2; thread t takes block c = t %
  // 16 of keys t / 16 + 16u.  A thread's four pieces go out in the order
  // (v + rot) % 4 so that the lanes of a warp spread over the bank groups.
  {
    const int c = tid % kBlocks;
    const int rot = (tid >> 1) & 3;
    uint8_t* kblk = sK + (c >> 1) * kKBlockBytes;
    const int p0 = (c & 1) * 4;  // first piece of the block inside its 128-byte row
    uint4 cw[kBItems];
    uint32_t sb[kBItems];
#pragma unroll
    for (int u = 0; u < kBItems; ++u) {
      const int r = tid / kBlocks + u * (kAttnThreads / kBlocks);
      const uint8_t* cp = rows.codes[r];
      cw[u] = cp ? __ldg(reinterpret_cast<const uint4*>(cp) + c) : make_uint4(0, 0, 0, 0);
      sb[u] = cp ? (uint32_t)__ldg(rows.scales[r] + c) : 0u;
    }
#pragma unroll
    for (int u = 0; u < kBItems; ++u) {
      const int r = tid / kBlocks + u * (kAttnThreads / kBlocks);
      const uint16_t* wrow = rows.win[r];
      if (wrow) {
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const int vv = (v + rot) & 3;
          cp_async16(kblk + swz(r, p0 + vv), wrow + c * 32 + vv * 8);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kBItems; ++u) {
      const int r = tid / kBlocks + u * (kAttnThreads / kBlocks);
      if (rows.win[r]) continue;  // copied by cp.async
      const bool fp4 = rows.codes[r] != nullptr;  // else: no key, zero row (P is 0 there)
      // scale 2^(sb - 127) in [2^-119, 2^123]: every product is a normal
      // bf16, so the bf16x2 multiply is exact; other scales take fp32
      const bool fast = sb[u] >= 8 && sb[u] <= 250;
      const float scf = ue8m0_value(sb[u]);
      const __nv_bfloat16 sc1 = __float2bfloat16_rn(fast ? scf : 1.f);
      const __nv_bfloat162 sc2 = __halves2bfloat162(sc1, sc1);
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const int vv = (v + rot) & 3;
        const uint32_t word =
            vv == 0 ? cw[u].x : (vv == 1 ? cw[u].y : (vv == 2 ? cw[u].z : cw[u].w));
        uint32_t packed[4] = {0u, 0u, 0u, 0u};
        if (fast) {
          e2m1x8_to_bf16(word, sc2, packed);
        } else if (fp4) {
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            const uint32_t byte = (word >> (8 * p)) & 0xFFu;
            packed[p] = pack_bf16x2(e2m1_value(byte & 15u) * scf, e2m1_value(byte >> 4) * scf);
          }
        }
        *reinterpret_cast<uint4*>(kblk + swz(r, p0 + vv)) =
            make_uint4(packed[0], packed[1], packed[2], packed[3]);
      }
    }
  }
  cp_async_wait_all();
  fence_proxy_async_smem();
  __syncthreads();

  // ---- 3. S^T = K Q^T (one thread issues; K = 512 in 32 steps of 16)
  if (tid == 0) {
    tc_fence_after();
    constexpr uint32_t idesc = idesc_bf16_f32(128, kHG);
    const uint32_t kb = smem_u32(sK), qb = smem_u32(sQ);
#pragma unroll
    for (int kk = 0; kk < kD / 16; ++kk) {
      const uint32_t in = (uint32_t)(kk & 3) * 32;  // 16 bf16 = 32 bytes along the atom
      tc_mma_bf16(tmem, sdesc_k_sw128(kb + (kk >> 2) * kKBlockBytes + in),
                  sdesc_k_sw128(qb + (kk >> 2) * (kHG * 128) + in), idesc, kk > 0 ? 1u : 0u);
    }
    tc_commit(&bar_s);
  }
  // softmax over the chunk's keys: warps of TMEM lane quarters 0..2 (keys
  // 0..95; keys >= kKC are not in the chunk), warp w takes heads 8 (w / 4) ..
  const int qtr = warp & 3;
  const int h0 = (warp >> 2) * 8;
  const bool smx = qtr < 3;
  const int key = qtr * 32 + lane;
  bool ok = mbar_wait(&bar_s, 0, &s_abort, a.dev_status, kAttnWaitNs);
  ok = __all_sync(0xffffffffu, ok);
  tc_fence_after();
  float sv[8];
  if (smx) {
    if (ok) {
      tmem_ld8(tmem + ((uint32_t)(qtr * 32) << 16) + (uint32_t)h0, sv);
      tmem_ld_wait();
    }
    const bool valid = ok && key < kKC && (rows.codes[key] || rows.win[key]);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      sv[i] = valid ? sv[i] * a.softmax_scale : -INFINITY;
      // max over the warp's 32 keys on order-preserving integer keys
      const uint32_t mk = __reduce_max_sync(0xffffffffu, score_key(sv[i]));
      if (lane == 0) {
        const uint32_t u = (mk & 0x80000000u) ? (mk & 0x7FFFFFFFu) : ~mk;
        red_m[qtr][h0 + i] = __uint_as_float(u);
      }
    }
  }
  __syncthreads();
  if (smx) {
    float l8[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float m = fmaxf(fmaxf(red_m[0][h0 + i], red_m[1][h0 + i]), red_m[2][h0 + i]);
      const float p = (sv[i] == -INFINITY) ? 0.f : expf(sv[i] - m);
      float l = p;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
      l8[i] = l;
      // P = hi + lo with hi = bf16(p), lo = bf16(p - hi): ~16 significant
      // bits.  Element (head h, key t) of the K-major operand.
      if (key < kKC) {
        const __nv_bfloat16 hi = __float2bfloat16_rn(p);
        const __nv_bfloat16 lo = __float2bfloat16_rn(p - __bfloat162float(hi));
        const int h = h0 + i;
        const uint32_t off = (uint32_t)((key >> 6) * (kHG * 128)) + swz(h, (key & 63) >> 3) +
                             (uint32_t)((key & 7) * 2);
        *reinterpret_cast<__nv_bfloat16*>(sPh + off) = hi;
        *reinterpret_cast<__nv_bfloat16*>(sPl + off) = lo;
      }
    }
    if (lane == 0)
#pragma unroll
      for (int i = 0; i < 8; ++i) red_l[qtr][h0 + i] = l8[i];
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  if (tid < kHG) {
    s_m[tid] = fmaxf(fmaxf(red_m[0][tid], red_m[1][tid]), red_m[2][tid]);
    s_l[tid] = red_l[0][tid] + red_l[1][tid] + red_l[2][tid];
  }

  // ---- 4. O^T = V^T P^T: dims 128 mb .. as M (two d-blocks, MN-major), keys as K
  if (tid == 0 && ok) {
    tc_fence_after();
    constexpr uint32_t idesc = idesc_bf16_f32(128, kHG, true);
    const uint32_t kb = smem_u32(sK), ph = smem_u32(sPh), pl = smem_u32(sPl);
#pragma unroll
    for (int mb = 0; mb < kD / 128; ++mb)
#pragma unroll
      for (int ks = 0; ks < kKC / 16; ++ks) {
        const uint64_t ad = sdesc_mn_sw128(kb + (2 * mb) * kKBlockBytes + ks * 2048,
                                           kKBlockBytes, 1024);
        const uint32_t pof = (uint32_t)((ks >> 2) * (kHG * 128) + (ks & 3) * 32);
        const uint32_t dt = tmem + (uint32_t)(kTmemO + kHG * mb);
        tc_mma_bf16(dt, ad, sdesc_k_sw128(ph + pof), idesc, ks > 0 ? 1u : 0u);
        tc_mma_bf16(dt, ad, sdesc_k_sw128(pl + pof), idesc, 1u);
      }
    tc_commit(&bar_o);
  }

  // ---- 5. this chunk's partial: O (unnormalised), m, l
  float* part = partial + ((qi * ngroups + hg) * (int64_t)nchunks + chunk) *
                              PartialLayout::kFloats;
  {
    bool got = ok && mbar_wait(&bar_o, 0, &s_abort, a.dev_status, kAttnWaitNs);
    got = __all_sync(0xffffffffu, got);
    tc_fence_after();
    // warp w: TMEM lane quarter w % 4 (dims 32 (w % 4) + lane of each block
    // of 128), blocks 2 (w / 4) and 2 (w / 4) + 1
#pragma unroll
    for (int bb = 0; bb < 2; ++bb) {
      const int mb = 2 * (warp >> 2) + bb;
      float o[16];
      if (got) {
        tmem_ld16(tmem + ((uint32_t)(qtr * 32) << 16) + (uint32_t)(kTmemO + kHG * mb), o);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) o[i] = 0.f;
      }
      const int dd = mb * 128 + qtr * 32 + lane;
#pragma unroll
      for (int h = 0; h < kHG; ++h) part[h * kD + dd] = o[h];
    }
    __syncthreads();  // s_m / s_l are set
    if (tid < kHG) {
      part[kHG * kD + tid] = ok ? s_m[tid] : -INFINITY;
      part[kHG * kD + kHG + tid] = ok ? s_l[tid] : 0.f;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }

  if constexpr (CLUSTER) {
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
        f[c] = (ml[c].x == -INFINITY) ? 0.f : expf(ml[c].x - M);
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

size_t attn_workspace_bytes(const csa2_attn_args& a) {
  if (a.q_dtype != CSA2_BF16) return 0;
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
    cudaError_t r = cudaFuncSetAttribute(attn_tc_kernel<true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kAttnSmem);
    if (r == cudaSuccess)
      r = cudaFuncSetAttribute(attn_tc_kernel<false>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, kAttnSmem);
    return r;
  });
  if (e != cudaSuccess) return cuda_fail(e);
  const dim3 grid((unsigned)nchunks, (unsigned)(a.hq / kHG), (unsigned)a.nq);
  float* partial = static_cast<float*>(a.workspace);
  const int pre = q_ready ? 1 : 0;
  if (nchunks <= kMaxClusterChunks)
    return launch_kernel(attn_tc_kernel<true>, grid, dim3(kAttnThreads), (size_t)kAttnSmem, s,
                         (unsigned)nchunks, a, nchunks, partial, pre);
  csa2_status st = launch_kernel(attn_tc_kernel<false>, grid, dim3(kAttnThreads),
                                 (size_t)kAttnSmem, s, 1, a, nchunks, partial, pre);
  if (st != CSA2_OK) return st;
  return launch_kernel(attn_combine_kernel, dim3((unsigned)a.hq, (unsigned)a.nq), dim3(128), 0, s,
                       1, static_cast<const float*>(partial), nchunks, (int)a.hq, a.out);
}

}  // namespace csa2
