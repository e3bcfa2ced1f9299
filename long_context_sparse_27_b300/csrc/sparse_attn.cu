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
// attn_bf16_kernel   bf16 queries, d = 512: one CTA per (64-key chunk, 16
//                    heads, query).  The chunk's rows are gathered and
//                    dequantised into shared memory as bf16 (exact: every
//                    E2M1 value times a UE8M0 scale is a bf16 value), then
//                    S = Q K^T and O = P V run as m16n8k16 bf16 MMAs with
//                    fp32 accumulation; P is split into two bf16 terms
//                    (p = hi + lo) so the probabilities keep ~16 bits.
//                    Each CTA writes (max, sum, unnormalised O) for its
//                    chunk; attn_combine_kernel merges the chunks.
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

__device__ __forceinline__ void window_of(const csa2_attn_args& a, int64_t qi, int32_t& ws,
                                          int32_t& wl) {
  ws = a.win_start ? a.win_start[qi] : 0;
  wl = a.win_len ? a.win_len[qi] : a.w_rows;
  if (wl < 0) wl = 0;
}

// ---------------------------------------------------------------------------
// fp32 path
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(128) attn_f32_kernel(const csa2_attn_args a) {
  extern __shared__ float sm[];  // q [d], logits [k + win_max]
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
  if (wl > a.win_max) wl = a.win_max;
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
// bf16 tensor-core path (d = 512, 16 heads per CTA, 64 keys per chunk)
// ---------------------------------------------------------------------------

constexpr int kD = 512;
constexpr int kHG = 16;                  // heads per CTA (MMA M)
constexpr int kKC = 64;                  // keys per chunk
constexpr int kRowBytes = kD * 2 + 16;   // padded bf16 row (breaks ldmatrix bank conflicts)
constexpr int kPRow = kKC * 2 + 16;      // padded P row
constexpr int kAttnThreads = 128;
constexpr int kSmemQ = kHG * kRowBytes;
constexpr int kSmemK = kKC * kRowBytes;
constexpr int kSmemP = 2 * kHG * kPRow;
constexpr int kAttnSmem = kSmemQ + kSmemK + kSmemP;

struct PartialLayout {
  // per (query, head group, chunk): O [16][512] f32, then m [16], l [16]
  static constexpr int64_t kFloats = (int64_t)kHG * kD + 2 * kHG;
};

__global__ void __launch_bounds__(kAttnThreads, 2)
    attn_bf16_kernel(const csa2_attn_args a, int nchunks, float* __restrict__ partial) {
  extern __shared__ __align__(16) uint8_t sm_raw[];
  uint8_t* sQ = sm_raw;
  uint8_t* sK = sm_raw + kSmemQ;
  uint8_t* sPh = sK + kSmemK;
  uint8_t* sPl = sPh + kHG * kPRow;
  __shared__ const uint8_t* row_codes[kKC];
  __shared__ const uint8_t* row_scales[kKC];
  __shared__ const uint16_t* row_win[kKC];
  __shared__ float red_m[4][kHG], red_l[4][kHG];

  const int chunk = blockIdx.x, hg = blockIdx.y;
  const int64_t qi = blockIdx.z;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid & 31;

  int32_t ws, wl;
  window_of(a, qi, ws, wl);
  if (wl > a.win_max) wl = a.win_max;
  const int64_t nkeys = a.k + wl;

  // 1. key sources of this chunk
  if (tid < kKC) {
    const int64_t t = (int64_t)chunk * kKC + tid;
    KeySrc src{nullptr, nullptr, nullptr};
    if (t < nkeys) src = key_source(a, qi, t, ws, wl);
    row_codes[tid] = src.codes;
    row_scales[tid] = src.scales;
    row_win[tid] = src.win;
  }
  // 2. the 16 query heads (bf16 rows of 1024 bytes)
  {
    const uint8_t* qsrc = static_cast<const uint8_t*>(a.q) +
                          ((qi * a.hq + (int64_t)hg * kHG) * kD) * 2;
    for (int i = tid; i < kHG * (kD * 2 / 16); i += kAttnThreads) {
      const int r = i / (kD * 2 / 16), c = i % (kD * 2 / 16);
      *reinterpret_cast<uint4*>(sQ + r * kRowBytes + c * 16) =
          *reinterpret_cast<const uint4*>(qsrc + r * kD * 2 + c * 16);
    }
  }
  __syncthreads();
  // 3. gather + dequantise: item = (row, 32-element block)
  for (int i = tid; i < kKC * (kD / 32); i += kAttnThreads) {
    const int r = i / (kD / 32), blk = i % (kD / 32);
    uint8_t* dst = sK + r * kRowBytes + blk * 64;
    uint4 o[4];
    if (row_codes[r]) {
      const uint4 cw = *reinterpret_cast<const uint4*>(row_codes[r] + blk * 16);
      const float sc = ue8m0_value(row_scales[r][blk]);
      const uint32_t w4[4] = {cw.x, cw.y, cw.z, cw.w};
      uint32_t packed[16];
#pragma unroll
      for (int wi = 0; wi < 4; ++wi)
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const uint32_t byte = (w4[wi] >> (8 * p)) & 0xFFu;
          packed[wi * 4 + p] =
              pack_bf16x2(e2m1_value(byte & 15u) * sc, e2m1_value(byte >> 4) * sc);
        }
#pragma unroll
      for (int v = 0; v < 4; ++v)
        o[v] = make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2], packed[4 * v + 3]);
    } else if (row_win[r]) {
      const uint4* src = reinterpret_cast<const uint4*>(row_win[r] + blk * 32);
#pragma unroll
      for (int v = 0; v < 4; ++v) o[v] = src[v];
    } else {
#pragma unroll
      for (int v = 0; v < 4; ++v) o[v] = make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int v = 0; v < 4; ++v) *reinterpret_cast<uint4*>(dst + v * 16) = o[v];
  }
  __syncthreads();

  // 4. S = Q K^T for this warp's 16 keys (two n-tiles of 8)
  float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  {
    const uint32_t qbase = smem_u32(sQ) + (lane & 15) * kRowBytes + (lane >> 4) * 16;
    const int krow = warp * 16 + (lane & 7) + ((lane >> 4) << 3);
    const uint32_t kbase = smem_u32(sK) + krow * kRowBytes + ((lane >> 3) & 1) * 16;
#pragma unroll 8
    for (int ks = 0; ks < kD / 16; ++ks) {
      uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
      ldmatrix_x4(qbase + ks * 32, a0, a1, a2, a3);
      ldmatrix_x4(kbase + ks * 32, b0, b1, b2, b3);
      mma_bf16_16816(s[0], a0, a1, a2, a3, b0, b1);
      mma_bf16_16816(s[1], a0, a1, a2, a3, b2, b3);
    }
  }
  // 5. chunk softmax: rows r0 = lane/4 and r0 + 8; keys 16*warp + 8*nt + 2*(lane%4) + {0,1}
  const int r0 = lane >> 2;
  float x[2][4];
  float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int key = warp * 16 + nt * 8 + 2 * (lane & 3) + (e & 1);
      const bool valid = row_codes[key] || row_win[key];
      x[nt][e] = valid ? s[nt][e] * a.softmax_scale : -INFINITY;
      if (e < 2)
        m0 = fmaxf(m0, x[nt][e]);
      else
        m1 = fmaxf(m1, x[nt][e]);
    }
#pragma unroll
  for (int o = 1; o < 4; o <<= 1) {
    m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, o));
    m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, o));
  }
  if ((lane & 3) == 0) {
    red_m[warp][r0] = m0;
    red_m[warp][r0 + 8] = m1;
  }
  __syncthreads();
  m0 = fmaxf(fmaxf(red_m[0][r0], red_m[1][r0]), fmaxf(red_m[2][r0], red_m[3][r0]));
  m1 = fmaxf(fmaxf(red_m[0][r0 + 8], red_m[1][r0 + 8]),
             fmaxf(red_m[2][r0 + 8], red_m[3][r0 + 8]));
  float l0 = 0.f, l1 = 0.f;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    float p[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float m = e < 2 ? m0 : m1;
      p[e] = (x[nt][e] == -INFINITY) ? 0.f : expf(x[nt][e] - m);
    }
    l0 += p[0] + p[1];
    l1 += p[2] + p[3];
    const int col = warp * 16 + nt * 8 + 2 * (lane & 3);
    // hi / lo bf16 split of p
    const __nv_bfloat162 h01 = __floats2bfloat162_rn(p[0], p[1]);
    const __nv_bfloat162 h23 = __floats2bfloat162_rn(p[2], p[3]);
    const float2 f01 = __bfloat1622float2(h01), f23 = __bfloat1622float2(h23);
    const uint32_t lo01 = pack_bf16x2(p[0] - f01.x, p[1] - f01.y);
    const uint32_t lo23 = pack_bf16x2(p[2] - f23.x, p[3] - f23.y);
    *reinterpret_cast<__nv_bfloat162*>(sPh + r0 * kPRow + col * 2) = h01;
    *reinterpret_cast<__nv_bfloat162*>(sPh + (r0 + 8) * kPRow + col * 2) = h23;
    *reinterpret_cast<uint32_t*>(sPl + r0 * kPRow + col * 2) = lo01;
    *reinterpret_cast<uint32_t*>(sPl + (r0 + 8) * kPRow + col * 2) = lo23;
  }
#pragma unroll
  for (int o = 1; o < 4; o <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, o);
    l1 += __shfl_xor_sync(0xffffffffu, l1, o);
  }
  if ((lane & 3) == 0) {
    red_l[warp][r0] = l0;
    red_l[warp][r0 + 8] = l1;
  }
  __syncthreads();

  // 6. O = P V for this warp's 128 dims (16 n-tiles), keys as the K dimension
  float o[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  {
    const uint32_t pbase_h = smem_u32(sPh) + (lane & 15) * kPRow + (lane >> 4) * 16;
    const uint32_t pbase_l = smem_u32(sPl) + (lane & 15) * kPRow + (lane >> 4) * 16;
    const int vrow = (lane & 7) + ((lane >> 3) & 1) * 8;
    const uint32_t vbase = smem_u32(sK) + vrow * kRowBytes + (warp * 128 + (lane >> 4) * 8) * 2;
#pragma unroll
    for (int ks = 0; ks < kKC / 16; ++ks) {
      uint32_t h0, h1, h2, h3, l0r, l1r, l2r, l3r;
      ldmatrix_x4(pbase_h + ks * 32, h0, h1, h2, h3);
      ldmatrix_x4(pbase_l + ks * 32, l0r, l1r, l2r, l3r);
#pragma unroll
      for (int np = 0; np < 8; ++np) {
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4_trans(vbase + ks * 16 * kRowBytes + np * 32, b0, b1, b2, b3);
        mma_bf16_16816(o[2 * np], h0, h1, h2, h3, b0, b1);
        mma_bf16_16816(o[2 * np], l0r, l1r, l2r, l3r, b0, b1);
        mma_bf16_16816(o[2 * np + 1], h0, h1, h2, h3, b2, b3);
        mma_bf16_16816(o[2 * np + 1], l0r, l1r, l2r, l3r, b2, b3);
      }
    }
  }
  // 7. partial results
  float* part = partial + ((qi * (a.hq / kHG) + hg) * (int64_t)nchunks + chunk) *
                              PartialLayout::kFloats;
#pragma unroll
  for (int nt = 0; nt < 16; ++nt) {
    const int col = warp * 128 + nt * 8 + 2 * (lane & 3);
    *reinterpret_cast<float2*>(part + r0 * kD + col) = make_float2(o[nt][0], o[nt][1]);
    *reinterpret_cast<float2*>(part + (r0 + 8) * kD + col) = make_float2(o[nt][2], o[nt][3]);
  }
  if (tid < kHG) {
    part[kHG * kD + tid] = fmaxf(fmaxf(red_m[0][tid], red_m[1][tid]),
                                 fmaxf(red_m[2][tid], red_m[3][tid]));
    part[kHG * kD + kHG + tid] = red_l[0][tid] + red_l[1][tid] + red_l[2][tid] + red_l[3][tid];
  }
}

// out[q, h, :] = sum_c e^(m_c - M) O_c / sum_c e^(m_c - M) l_c
__global__ void __launch_bounds__(128)
    attn_combine_kernel(const float* __restrict__ partial, int nchunks, int hq,
                        float* __restrict__ out) {
  const int h = blockIdx.x;
  const int64_t qi = blockIdx.y;
  const int hg = h / kHG, hr = h % kHG;
  const float* base =
      partial + ((qi * (hq / kHG) + hg) * (int64_t)nchunks) * PartialLayout::kFloats;
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

}  // namespace

size_t attn_workspace_bytes(const csa2_attn_args& a) {
  if (a.q_dtype != CSA2_BF16) return 0;
  const int64_t nchunks = (a.k + win_bound(a) + kKC - 1) / kKC;
  return (size_t)a.nq * (a.hq / kHG) * nchunks * PartialLayout::kFloats * sizeof(float);
}

csa2_status launch_sparse_attn(const csa2_attn_args& in, cudaStream_t s) {
  if (in.nq == 0) return CSA2_OK;
  csa2_attn_args a = in;
  a.win_max = win_bound(in);
  if (a.q_dtype == CSA2_F32) {
    const size_t smem = sizeof(float) * ((size_t)a.d + a.k + a.win_max);
    if (smem > 48 * 1024) return CSA2_ERR_UNSUPPORTED;
    attn_f32_kernel<<<dim3((unsigned)a.hq, (unsigned)a.nq), 128, smem, s>>>(a);
    return check_launch();
  }
  const int nchunks = (int)((a.k + a.win_max + kKC - 1) / kKC);
  if (nchunks == 0) {
    cudaError_t e = cudaMemsetAsync(a.out, 0, (size_t)a.nq * a.hq * kD * sizeof(float), s);
    return e == cudaSuccess ? CSA2_OK : cuda_fail(e);
  }
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(attn_bf16_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kAttnSmem);
    if (e != cudaSuccess) return cuda_fail(e);
    attr_set = true;
  }
  float* partial = static_cast<float*>(a.workspace);
  attn_bf16_kernel<<<dim3((unsigned)nchunks, (unsigned)(a.hq / kHG), (unsigned)a.nq),
                     kAttnThreads, kAttnSmem, s>>>(a, nchunks, partial);
  csa2_status st = check_launch();
  if (st != CSA2_OK) return st;
  attn_combine_kernel<<<dim3((unsigned)a.hq, (unsigned)a.nq), 128, 0, s>>>(partial, nchunks,
                                                                         a.hq, a.out);
  return check_launch();
}

}  // namespace csa2
