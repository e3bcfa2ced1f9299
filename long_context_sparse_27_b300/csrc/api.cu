// api.cu -- the C ABI of libcsa2 (declared in include/csa2.h): argument
// checks, workspace sizing, status codes, host-side fault injection and the
// static Full / Reindex / Reuse layer schedule.
//
// The three layer modes are those of "Unlocking Extreme Context Scaling with
// DeepSeek-V4.1-Flash", section "Compressed Sparse Attention 2 (CSA2)": Full
// computes main KV and indexer K afresh and selects new top-k entries;
// Reindex uses the main KV and indexer K of the last Full layer with a new
// indexer Q; Reuse takes both the main KV and the top-k indices of an
// earlier layer.  The modes are fixed per layer ("static layer modes",
// aiany.app DeepSeek-V4.1-Flash page, "What Sets It Apart").
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>

#include "internal.h"

namespace csa2 {

static thread_local int32_t g_last_cuda_error = 0;

csa2_status cuda_fail(cudaError_t e) {
  g_last_cuda_error = (int32_t)e;
  return CSA2_ERR_CUDA;
}

csa2_status check_launch() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? CSA2_OK : cuda_fail(e);
}

bool pdl_enabled() {
  static const bool on = [] {
    const char* e = std::getenv("CSA2_PDL");
    return !(e && e[0] == '0');
  }();
  return on;
}

int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (dev < 0 || dev >= 64) return 148;
  if (!cached[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

// CSA2_FAULT_INJECT="<call>:<status>" makes the named entry point return
// <status> before it enqueues anything (host-side failure injection for
// tests of the callers' error paths).  <call> is the entry point's name
// without the "csa2_" prefix, e.g. "topk:4".
csa2_status injected(const char* call) {
  const char* env = std::getenv("CSA2_FAULT_INJECT");
  if (!env || !*env) return CSA2_OK;
  const char* colon = std::strchr(env, ':');
  if (!colon) return CSA2_OK;
  const size_t len = (size_t)(colon - env);
  if (std::strlen(call) != len || std::strncmp(env, call, len) != 0) return CSA2_OK;
  const int v = std::atoi(colon + 1);
  return (v > 0 && v <= CSA2_ERR_DEVICE_CAPACITY) ? (csa2_status)v : CSA2_OK;
}

namespace {

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// A paged layout for rows of n entries: pages of a positive multiple of 64
// entries, a pool of at least one page addressable with 32-bit row numbers,
// and block-table rows that cover n entries.
bool pages_ok(const csa2_pages& pg, int64_t n) {
  if (!pg.block_table) return true;
  if (pg.page_rows < 64 || pg.page_rows % 64 != 0 || pg.num_pages < 1) return false;
  if ((int64_t)pg.num_pages * pg.page_rows > ((int64_t)1 << 31) - 1) return false;
  return pg.bt_ld >= (n + pg.page_rows - 1) / pg.page_rows;
}

csa2_status check_quant(const csa2_quant_args* a) {
  if (!a || a->rows < 0 || a->d <= 0 || a->d % 32 != 0) return CSA2_ERR_INVALID_ARG;
  if (a->rows == 0) return CSA2_OK;
  if (!a->x || !a->codes || !a->scales) return CSA2_ERR_INVALID_ARG;
  if (a->x_ld < a->d || a->codes_ld < a->d / 2 || a->scales_ld < a->d / 32)
    return CSA2_ERR_INVALID_ARG;
  if (!aligned(a->x, 16) || a->x_ld % 8 != 0 || !aligned(a->codes, 4) || a->codes_ld % 4 != 0)
    return CSA2_ERR_ALIGNMENT;
  if ((a->idxk == nullptr) != (a->idxk_e4m3 == nullptr)) return CSA2_ERR_INVALID_ARG;
  if (a->pages.block_table &&
      (!pages_ok(a->pages, 0) || a->rows_per_seq < 1 || a->entry0 < 0 ||
       a->pages.bt_ld < (a->entry0 + a->rows_per_seq + a->pages.page_rows - 1) /
                            a->pages.page_rows))
    return CSA2_ERR_INVALID_ARG;
  if (a->idxk) {
    if (a->di <= 0 || a->di % 8 != 0 || a->idxk_ld < a->di || a->idxk_e4m3_ld < a->di)
      return CSA2_ERR_INVALID_ARG;
    if (!aligned(a->idxk, 16) || a->idxk_ld % 8 != 0 || !aligned(a->idxk_e4m3, 8) ||
        a->idxk_e4m3_ld % 8 != 0)
      return CSA2_ERR_ALIGNMENT;
  }
  return CSA2_OK;
}

csa2_status check_index_q(const void* q, const float* w, int64_t nq, int32_t hi, int32_t di,
                          const uint8_t* q8, const float* c) {
  if (nq < 0 || hi < 1) return CSA2_ERR_INVALID_ARG;
  if (di != 32 && di != 64 && di != 128 && di != 256) return CSA2_ERR_INVALID_ARG;
  if (nq == 0) return CSA2_OK;
  if (!q || !w || !q8 || !c) return CSA2_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(q8, 16)) return CSA2_ERR_ALIGNMENT;
  return CSA2_OK;
}

bool fp8_path(const csa2_index_args* a) {
  return (a->q_dtype == CSA2_BF16 || a->q_dtype == CSA2_E4M3) && a->k_dtype == CSA2_E4M3;
}

size_t index_ws(const csa2_index_args* a) {
  if (!fp8_path(a) || a->q_dtype == CSA2_E4M3) return 0;
  const int64_t nq = a->B * a->q_per_seq;
  return align256((size_t)nq * a->hi * a->di) + align256((size_t)nq * a->hi * sizeof(float));
}

csa2_status check_index(const csa2_index_args* a) {
  if (!a || a->B < 0 || a->q_per_seq < 1 || a->n < 0 || a->hi < 1 || a->di < 1)
    return CSA2_ERR_INVALID_ARG;
  const int64_t nq = a->B * a->q_per_seq;
  if (nq == 0 || a->n == 0) return CSA2_OK;
  if (!a->q || !a->w || !a->k || !a->scores) return CSA2_ERR_INVALID_ARG;
  if (a->k_ld < a->di || a->k_seq_stride < 0 || a->scores_ld < a->n) return CSA2_ERR_INVALID_ARG;
  if (!pages_ok(a->pages, a->n)) return CSA2_ERR_INVALID_ARG;
  const bool paged = a->pages.block_table != nullptr;
  if (!paged && a->B > 1 && a->k_seq_stride < a->k_ld * a->n) return CSA2_ERR_INVALID_ARG;
  if (fp8_path(a)) {
    if (a->hi != 64 || a->di != 128) return CSA2_ERR_UNSUPPORTED;
    if (!aligned(a->k, 16) || a->k_ld % 16 != 0 || a->k_seq_stride % 16 != 0)
      return CSA2_ERR_ALIGNMENT;
    if (!aligned(a->q, 16)) return CSA2_ERR_ALIGNMENT;
    if (a->n > (int64_t)1 << 30 || nq * a->hi > (int64_t)1 << 31 ||
        nq * ((a->n + 127) / 128) >= (int64_t)1 << 31)
      return CSA2_ERR_UNSUPPORTED;
    if (a->q_dtype == CSA2_E4M3) return aligned(a->w, 16) ? CSA2_OK : CSA2_ERR_ALIGNMENT;
    if (!a->workspace || a->workspace_bytes < index_ws(a)) return CSA2_ERR_WORKSPACE;
    if (!aligned(a->workspace, 256)) return CSA2_ERR_ALIGNMENT;
    return CSA2_OK;
  }
  if (a->q_dtype == CSA2_F32 && a->k_dtype == CSA2_F32) {
    if (a->hi > 64 || a->di > 256) return CSA2_ERR_UNSUPPORTED;
    return CSA2_OK;
  }
  return CSA2_ERR_UNSUPPORTED;
}

// hist1 (nullable): first-level top-k histograms the decode FP8 kernel adds
// the scores' keys to (index_fuses_topk_hist).
csa2_status run_index(const csa2_index_args& a, uint32_t* hist1, IndexTuning tune,
                      cudaStream_t s) {
  if (a.B * a.q_per_seq == 0 || a.n == 0) return CSA2_OK;
  if (!fp8_path(&a)) return launch_index_score_f32(a, s);
  if (a.q_dtype == CSA2_E4M3)
    return launch_index_score_fp8(a, static_cast<const uint8_t*>(a.q), a.w, hist1, tune, s);
  // decode: the indexer kernel quantises its queries itself (one launch)
  const csa2_status fused = launch_index_score_bf16q(a, hist1, tune, s);
  if (fused != CSA2_ERR_UNSUPPORTED) return fused;
  const int64_t nq = a.B * a.q_per_seq;
  uint8_t* q8 = static_cast<uint8_t*>(a.workspace);
  float* c = reinterpret_cast<float*>(q8 + align256((size_t)nq * a.hi * a.di));
  csa2_status st = launch_quantize_index_q(a.q, a.w, nq, a.hi, a.di, q8, c, s);
  if (st != CSA2_OK) return st;
  return launch_index_score_fp8(a, q8, c, hist1, tune, s);
}

csa2_status check_topk(const float* scores, int64_t rows, int64_t n, int64_t ld, int32_t k,
                       int32_t* idx_out, int64_t idx_ld, void* ws, size_t ws_bytes) {
  if (rows < 0 || n < 0 || k < 1 || idx_ld < k || ld < n) return CSA2_ERR_INVALID_ARG;
  if (k > 2048) return CSA2_ERR_UNSUPPORTED;
  if (n >= ((int64_t)1 << 31)) return CSA2_ERR_UNSUPPORTED;
  if (rows == 0) return CSA2_OK;
  if (!idx_out || (n > 0 && !scores)) return CSA2_ERR_INVALID_ARG;
  if (!ws || ws_bytes < topk_workspace_bytes(rows, n, k)) return CSA2_ERR_WORKSPACE;
  if (!aligned(ws, 256)) return CSA2_ERR_ALIGNMENT;
  return CSA2_OK;
}

csa2_status check_attn(const csa2_attn_args* a) {
  if (!a || a->nq < 0 || a->q_per_seq < 1 || a->hq < 1 || a->d < 32 || a->d % 32 != 0 ||
      a->n < 0 || a->k < 0 || a->w_rows < 0 || a->win_max < 0)
    return CSA2_ERR_INVALID_ARG;
  if (a->nq == 0) return CSA2_OK;
  if (!a->q || !a->out) return CSA2_ERR_INVALID_ARG;
  if (a->k > 0 && (!a->idx || !a->codes || !a->scales || a->idx_ld < a->k))
    return CSA2_ERR_INVALID_ARG;
  if (a->w_rows > 0 && !a->window) return CSA2_ERR_INVALID_ARG;
  if (a->codes_ld < a->d / 2 || a->scales_ld < a->d / 32) return CSA2_ERR_INVALID_ARG;
  if (!pages_ok(a->pages, a->n)) return CSA2_ERR_INVALID_ARG;
  if (a->window && a->win_ld < a->d) return CSA2_ERR_INVALID_ARG;
  if (a->q_dtype == CSA2_F32) {
    if (a->hq > 65535 || a->d > 256) return CSA2_ERR_UNSUPPORTED;
    const int64_t wm = a->win_max > 0 ? a->win_max : a->w_rows;
    if (sizeof(float) * ((size_t)a->d + a->k + wm) > 48 * 1024) return CSA2_ERR_UNSUPPORTED;
    return CSA2_OK;
  }
  if (a->q_dtype != CSA2_BF16) return CSA2_ERR_UNSUPPORTED;
  if (a->d != 512 || a->hq % 16 != 0) return CSA2_ERR_UNSUPPORTED;
  if (a->nq > 65535) return CSA2_ERR_UNSUPPORTED;
  if (!aligned(a->q, 16)) return CSA2_ERR_ALIGNMENT;
  if (a->k > 0 && (!aligned(a->codes, 16) || a->codes_ld % 16 != 0 ||
                   a->codes_seq_stride % 16 != 0 || !aligned(a->scales, 16) ||
                   a->scales_ld % 16 != 0 || a->scales_seq_stride % 16 != 0))
    return CSA2_ERR_ALIGNMENT;
  if (a->window && (!aligned(a->window, 16) || a->win_ld % 8 != 0 || a->win_seq_stride % 8 != 0))
    return CSA2_ERR_ALIGNMENT;
  const size_t need = attn_workspace_bytes(*a);
  if (need > 0 && (!a->workspace || a->workspace_bytes < need)) return CSA2_ERR_WORKSPACE;
  if (need > 0 && !aligned(a->workspace, 16)) return CSA2_ERR_ALIGNMENT;
  return CSA2_OK;
}

// ---- layer stack ----

struct StackPieces {
  size_t scores, ix, tk, pl, at, sel;
  size_t total() const { return scores + tk + pl + sel + std::max(ix, at); }
};

// The selection of a prefill chunk without its score matrix (see
// IndexSelect): a sample of every kSampleStride-th tile of 128 entries gives
// each query a threshold no entry of its top k lies below; the full pass then
// keeps only the entries at or above it, at most kCandCap per query.
constexpr int kSampleStride = 8;
constexpr int64_t kCandCap = 8192;

bool prefill_select(const csa2_stack_args& s) {
  return s.q_per_seq > 1 && s.q_per_seq % 4 == 0 && s.n > kTopkShortRow && s.pool == 0 &&
         s.block == 0 && s.idx_k_dtype == CSA2_E4M3 &&
         (s.idx_q_dtype == CSA2_BF16 || s.idx_q_dtype == CSA2_E4M3) && s.hi == 64 &&
         s.di == 128 && s.k <= kCandCap && topk_cand_fits(kCandCap, s.n);
}

// compact sample columns of a prefill selection
int64_t sample_cols(const csa2_stack_args& s) {
  const int64_t ktiles = (s.n + 127) / 128;
  return (ktiles + kSampleStride - 1) / kSampleStride * 128;
}

// slots of the Hierarchical Sparse Indexer's candidate pool (0 = off): the
// top-P pool, or the entries of the kept blocks under block-level pruning
int64_t pool_slots(const csa2_stack_args& s) {
  if (s.block > 0) return (int64_t)s.blocks_kept * s.block;
  return s.pool > 0 ? std::min<int64_t>(s.pool, s.n) : 0;
}

int64_t stack_blocks(const csa2_stack_args& s) {
  return s.block > 0 ? (s.n + s.block - 1) / s.block : 0;
}

csa2_index_args stack_index_args(const csa2_stack_args& s, const csa2_layer_desc& L,
                                 const csa2_layer_desc& src, float* scores, void* ws,
                                 size_t ws_bytes) {
  csa2_index_args a;
  std::memset(&a, 0, sizeof(a));
  a.q = L.idx_q;
  a.q_dtype = s.idx_q_dtype;
  a.w = L.idx_w;
  a.k = src.idxk;
  a.k_dtype = s.idx_k_dtype;
  a.B = s.B;
  a.q_per_seq = s.q_per_seq;
  a.hi = s.hi;
  a.di = s.di;
  a.n = s.n;
  a.k_ld = s.di;
  a.k_seq_stride = s.n * s.di;
  a.n_valid = s.n_valid;
  a.scores = scores;
  a.scores_ld = s.n;
  a.workspace = ws;
  a.workspace_bytes = ws_bytes;
  a.dev_status = s.dev_status;
  a.pages = s.pages;
  return a;
}

csa2_attn_args stack_attn_args(const csa2_stack_args& s, const csa2_layer_desc& L,
                               const csa2_layer_desc& kv, const int32_t* idx, void* ws,
                               size_t ws_bytes) {
  csa2_attn_args a;
  std::memset(&a, 0, sizeof(a));
  a.q = L.attn_q;
  a.q_dtype = s.attn_q_dtype;
  a.nq = s.B * s.q_per_seq;
  a.q_per_seq = s.q_per_seq;
  a.hq = s.hq;
  a.d = s.d;
  a.codes = kv.codes;
  a.scales = kv.scales;
  a.n = s.n;
  a.codes_ld = s.d / 2;
  a.codes_seq_stride = s.n * (s.d / 2);
  a.scales_ld = s.d / 32;
  a.scales_seq_stride = s.n * (s.d / 32);
  a.idx = idx;
  a.k = s.k;
  a.idx_ld = s.k;
  a.window = L.window;
  a.w_rows = s.w_rows;
  a.win_ld = s.d;
  a.win_seq_stride = (int64_t)s.w_rows * s.d;
  a.win_start = s.win_start;
  a.win_len = s.win_len;
  a.win_max = s.win_max;
  a.softmax_scale = s.softmax_scale;
  a.out = L.out;
  a.workspace = ws;
  a.workspace_bytes = ws_bytes;
  a.dev_status = s.dev_status;
  a.pages = s.pages;
  return a;
}

// Quantise a Full layer's new rows into its caches: new_kv [B, nr, d] goes
// to rows new_row .. new_row + nr - 1 of every sequence.  With one new row
// per sequence a single launch covers all sequences (the sequence stride is
// the row stride); otherwise one launch per sequence.
csa2_status quantize_new_rows(const csa2_stack_args& s, const csa2_layer_desc& d,
                              cudaStream_t cs) {
  const int64_t nr = d.new_rows > 0 ? d.new_rows : 1;
  const bool e4m3 = s.idx_k_dtype == CSA2_E4M3;
  if (s.pages.block_table) {
    // paged caches: one launch writes every sequence's new rows through the
    // block table (the fp32 indexer keys are not paged: checked before)
    csa2_quant_args q;
    std::memset(&q, 0, sizeof(q));
    q.x = d.new_kv;
    q.rows = s.B * nr;
    q.d = s.d;
    q.x_ld = s.d;
    q.codes = d.codes;
    q.codes_ld = s.d / 2;
    q.scales = d.scales;
    q.scales_ld = s.d / 32;
    q.idxk = d.new_idxk;
    q.di = s.di;
    q.idxk_ld = s.di;
    q.idxk_e4m3 = static_cast<uint8_t*>(d.idxk);
    q.idxk_e4m3_ld = s.di;
    q.pages = s.pages;
    q.rows_per_seq = nr;
    q.entry0 = d.new_row;
    csa2_status st = check_quant(&q);
    if (st != CSA2_OK) return st;
    return launch_quantize_fp4(q, cs, s.dev_status);
  }
  const int64_t per_call = nr == 1 ? 1 : s.B;  // number of calls
  for (int64_t b = 0; b < per_call; ++b) {
    csa2_quant_args q;
    std::memset(&q, 0, sizeof(q));
    const int64_t row0 = b * s.n + d.new_row;  // in rows of the [B, n] cache
    q.x = static_cast<const uint16_t*>(d.new_kv) + b * nr * s.d;
    q.rows = nr == 1 ? s.B : nr;
    q.d = s.d;
    q.x_ld = s.d;
    q.codes = d.codes + row0 * (s.d / 2);
    q.codes_ld = nr == 1 ? s.n * (s.d / 2) : s.d / 2;
    q.scales = d.scales + row0 * (s.d / 32);
    q.scales_ld = nr == 1 ? s.n * (s.d / 32) : s.d / 32;
    if (e4m3) {
      q.idxk = static_cast<const uint16_t*>(d.new_idxk) + b * nr * s.di;
      q.di = s.di;
      q.idxk_ld = s.di;
      q.idxk_e4m3 = static_cast<uint8_t*>(d.idxk) + row0 * s.di;
      q.idxk_e4m3_ld = nr == 1 ? s.n * s.di : s.di;
    }
    csa2_status st = check_quant(&q);
    if (st != CSA2_OK) return st;
    if ((st = launch_quantize_fp4(q, cs, s.dev_status)) != CSA2_OK) return st;
    if (!e4m3) {
      // fp32 indexer keys are stored as given
      const size_t row_bytes = (size_t)s.di * sizeof(float);
      cudaError_t e = cudaMemcpy2DAsync(
          static_cast<float*>(d.idxk) + row0 * s.di, nr == 1 ? (size_t)s.n * row_bytes : row_bytes,
          static_cast<const float*>(d.new_idxk) + b * nr * s.di, row_bytes, row_bytes,
          (size_t)q.rows, cudaMemcpyDeviceToDevice, cs);
      if (e != cudaSuccess) return cuda_fail(e);
    }
  }
  return CSA2_OK;
}

StackPieces stack_pieces(const csa2_stack_args& s) {
  StackPieces p;
  const int64_t nq = s.B * s.q_per_seq;
  const bool psel = prefill_select(s);
  // scores: the whole [nq, n] matrix, or a prefill selection's sample of it
  p.scores = align256((size_t)nq * (psel ? sample_cols(s) : s.n) * sizeof(float));
  // a prefill selection's thresholds, candidate counters and candidates
  p.sel = psel ? align256((size_t)nq * 8) + align256((size_t)nq * kCandCap * sizeof(uint2)) : 0;
  csa2_layer_desc dummy;
  std::memset(&dummy, 0, sizeof(dummy));
  csa2_index_args ia = stack_index_args(s, dummy, dummy, nullptr, nullptr, 0);
  p.ix = align256(index_ws(&ia));
  p.tk = align256(topk_workspace_bytes(nq, s.n, s.k));
  p.pl = align256((size_t)nq * pool_slots(s) * sizeof(int32_t));
  csa2_attn_args aa = stack_attn_args(s, dummy, dummy, nullptr, nullptr, 0);
  p.at = align256(attn_workspace_bytes(aa));
  return p;
}

}  // namespace
}  // namespace csa2

using namespace csa2;

extern "C" {

const char* csa2_version(void) { return "0.1.0"; }

const char* csa2_status_string(int32_t st) {
  switch (st) {
    case CSA2_OK: return "CSA2_OK";
    case CSA2_ERR_INVALID_ARG: return "CSA2_ERR_INVALID_ARG";
    case CSA2_ERR_UNSUPPORTED: return "CSA2_ERR_UNSUPPORTED";
    case CSA2_ERR_ALIGNMENT: return "CSA2_ERR_ALIGNMENT";
    case CSA2_ERR_CUDA: return "CSA2_ERR_CUDA";
    case CSA2_ERR_WORKSPACE: return "CSA2_ERR_WORKSPACE";
    case CSA2_ERR_DEVICE_TIMEOUT: return "CSA2_ERR_DEVICE_TIMEOUT";
    case CSA2_ERR_DEVICE_BOUNDS: return "CSA2_ERR_DEVICE_BOUNDS";
    case CSA2_ERR_DEVICE_CAPACITY: return "CSA2_ERR_DEVICE_CAPACITY";
    default: return "CSA2_ERR_UNKNOWN";
  }
}

int32_t csa2_last_cuda_error(void) { return g_last_cuda_error; }

csa2_status csa2_status_from_device(int32_t w) {
  if (w & CSA2_DEVFLAG_TIMEOUT) return CSA2_ERR_DEVICE_TIMEOUT;
  if (w & CSA2_DEVFLAG_BOUNDS) return CSA2_ERR_DEVICE_BOUNDS;
  if (w & CSA2_DEVFLAG_CAPACITY) return CSA2_ERR_DEVICE_CAPACITY;
  return CSA2_OK;
}

csa2_status csa2_quantize_fp4(const csa2_quant_args* args, csa2_stream_t stream) {
  csa2_status st = check_quant(args);
  if (st != CSA2_OK) return st;
  if ((st = injected("quantize_fp4")) != CSA2_OK) return st;
  return launch_quantize_fp4(*args, reinterpret_cast<cudaStream_t>(stream));
}

csa2_status csa2_quantize_index_q(const void* q, const float* w, int64_t nq, int32_t hi,
                                  int32_t di, uint8_t* q8, float* c, csa2_stream_t stream) {
  csa2_status st = check_index_q(q, w, nq, hi, di, q8, c);
  if (st != CSA2_OK) return st;
  if ((st = injected("quantize_index_q")) != CSA2_OK) return st;
  return launch_quantize_index_q(q, w, nq, hi, di, q8, c, reinterpret_cast<cudaStream_t>(stream));
}

size_t csa2_index_score_workspace_bytes(const csa2_index_args* args) {
  return args ? index_ws(args) : 0;
}

csa2_status csa2_index_score(const csa2_index_args* args, csa2_stream_t stream) {
  csa2_status st = check_index(args);
  if (st != CSA2_OK) return st;
  if ((st = injected("index_score")) != CSA2_OK) return st;
  return run_index(*args, nullptr, IndexTuning{}, reinterpret_cast<cudaStream_t>(stream));
}

csa2_status csa2_index_score_pool(const csa2_index_args* args, const int32_t* pool,
                                  int64_t pool_ld, int32_t pool_n, csa2_stream_t stream) {
  if (!args) return CSA2_ERR_INVALID_ARG;
  // the checks of csa2_index_score, with rows of pool_n scores
  csa2_index_args chk = *args;
  chk.scores_ld = std::max(chk.scores_ld, chk.n);
  csa2_status st = check_index(&chk);
  if (st != CSA2_OK) return st;
  if (!fp8_path(args)) return CSA2_ERR_UNSUPPORTED;
  if (pool_n < 1 || pool_ld < pool_n || args->scores_ld < pool_n) return CSA2_ERR_INVALID_ARG;
  if (pool_n > 2048) return CSA2_ERR_UNSUPPORTED;
  const int64_t nq = args->B * args->q_per_seq;
  if (nq == 0 || args->n == 0) return CSA2_OK;
  if (!pool) return CSA2_ERR_INVALID_ARG;
  if ((st = injected("index_score_pool")) != CSA2_OK) return st;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const uint8_t* q8 = static_cast<const uint8_t*>(args->q);
  const float* c = args->w;
  if (args->q_dtype != CSA2_E4M3) {
    uint8_t* wq = static_cast<uint8_t*>(args->workspace);
    float* wc = reinterpret_cast<float*>(wq + align256((size_t)nq * args->hi * args->di));
    if ((st = launch_quantize_index_q(args->q, args->w, nq, args->hi, args->di, wq, wc, cs)) !=
        CSA2_OK)
      return st;
    q8 = wq;
    c = wc;
  }
  return launch_index_score_pool(*args, q8, c, pool, pool_ld, pool_n, args->scores,
                                 args->scores_ld, cs);
}

csa2_status csa2_index_candidates(const csa2_index_args* args, const uint32_t* theta,
                                  uint32_t* cand_cnt, uint64_t* cand, int64_t cand_cap,
                                  csa2_stream_t stream) {
  if (!args) return CSA2_ERR_INVALID_ARG;
  // the checks of csa2_index_score (no score matrix is written)
  csa2_index_args chk = *args;
  chk.scores = reinterpret_cast<float*>(cand);
  chk.scores_ld = std::max(chk.scores_ld, chk.n);
  csa2_status st = check_index(&chk);
  if (st != CSA2_OK) return st;
  if (!fp8_path(args) || args->q_per_seq % 4 != 0) return CSA2_ERR_UNSUPPORTED;
  const int64_t nq = args->B * args->q_per_seq;
  if (nq == 0 || args->n == 0) return CSA2_OK;
  if (!theta || !cand_cnt || !cand || cand_cap < 1) return CSA2_ERR_INVALID_ARG;
  if (!aligned(cand, 8)) return CSA2_ERR_ALIGNMENT;
  if ((st = injected("index_candidates")) != CSA2_OK) return st;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const uint8_t* q8 = static_cast<const uint8_t*>(args->q);
  const float* c = args->w;
  if (args->q_dtype != CSA2_E4M3) {
    uint8_t* wq = static_cast<uint8_t*>(args->workspace);
    float* wc = reinterpret_cast<float*>(wq + align256((size_t)nq * args->hi * args->di));
    if ((st = launch_quantize_index_q(args->q, args->w, nq, args->hi, args->di, wq, wc, cs)) !=
        CSA2_OK)
      return st;
    q8 = wq;
    c = wc;
  }
  IndexSelect emit;
  emit.theta = theta;
  emit.cand_cnt = cand_cnt;
  emit.cand = reinterpret_cast<uint2*>(cand);
  emit.cand_cap = cand_cap;
  return launch_index_select_prefill(*args, q8, c, emit, cs);
}

csa2_status csa2_project_fp4(const csa2_project_args* a, csa2_stream_t stream) {
  if (!a || a->rows < 0 || a->hidden < 32 || a->hidden % 32 != 0 || a->d < 64 || a->d % 64 != 0)
    return CSA2_ERR_INVALID_ARG;
  if (a->rows == 0) return CSA2_OK;
  if (!a->h || !a->w || !a->codes || !a->scales) return CSA2_ERR_INVALID_ARG;
  if (a->h_ld < a->hidden || a->w_ld < a->hidden || a->codes_ld < a->d / 2 ||
      a->scales_ld < a->d / 32 || (a->out && a->out_ld < a->d))
    return CSA2_ERR_INVALID_ARG;
  if (!aligned(a->h, 16) || !aligned(a->w, 16) || a->h_ld % 8 != 0 || a->w_ld % 8 != 0)
    return CSA2_ERR_ALIGNMENT;
  if (a->out && (!aligned(a->out, 8) || a->out_ld % 2 != 0)) return CSA2_ERR_ALIGNMENT;
  if (a->rows > (int64_t)65535 * 64 * 1024) return CSA2_ERR_UNSUPPORTED;
  csa2_status st = injected("project_fp4");
  if (st != CSA2_OK) return st;
  return launch_project_fp4(*a, reinterpret_cast<cudaStream_t>(stream));
}

csa2_status csa2_index_block_keys(const uint8_t* k8, int64_t B, int64_t n, int64_t k_ld,
                                  int64_t k_seq_stride, const csa2_pages* pages, int32_t G,
                                  int64_t blk0, int64_t nblk, uint8_t* out, int64_t out_ld,
                                  int64_t out_seq_stride, int32_t* dev_status,
                                  csa2_stream_t stream) {
  if (B < 0 || n < 0 || G < 1 || G > 65536 || (G & (G - 1)) != 0 || blk0 < 0 || nblk < 0)
    return CSA2_ERR_INVALID_ARG;
  const csa2_pages pg = pages ? *pages : csa2_pages{nullptr, 0, 0, 0};
  if (!pages_ok(pg, n)) return CSA2_ERR_INVALID_ARG;
  if (blk0 + nblk > (n + G - 1) / G) return CSA2_ERR_INVALID_ARG;
  if (B == 0 || nblk == 0) return CSA2_OK;
  if (!k8 || !out || k_ld < 128 || out_ld < 128) return CSA2_ERR_INVALID_ARG;
  if (!pg.block_table && B > 1 && (k_seq_stride < k_ld * n || out_seq_stride < out_ld * nblk))
    return CSA2_ERR_INVALID_ARG;
  csa2_status st = injected("index_block_keys");
  if (st != CSA2_OK) return st;
  return launch_block_keys(k8, B, n, k_ld, k_seq_stride, pg, G, blk0, nblk, out, out_ld,
                           out_seq_stride, dev_status, reinterpret_cast<cudaStream_t>(stream));
}

size_t csa2_topk_workspace_bytes(int64_t rows, int64_t n, int32_t k) {
  if (rows < 0 || k < 1) return 0;
  return topk_workspace_bytes(rows, n, k);
}

csa2_status csa2_topk(const float* scores, int64_t rows, int64_t n, int64_t ld,
                      const int32_t* n_valid, int32_t k, int32_t* idx_out, int64_t idx_ld,
                      void* workspace, size_t workspace_bytes, int32_t* dev_status,
                      csa2_stream_t stream) {
  csa2_status st = check_topk(scores, rows, n, ld, k, idx_out, idx_ld, workspace, workspace_bytes);
  if (st != CSA2_OK) return st;
  if ((st = injected("topk")) != CSA2_OK) return st;
  return launch_topk(scores, rows, n, ld, n_valid, k, idx_out, idx_ld, workspace, dev_status,
                     reinterpret_cast<cudaStream_t>(stream));
}

size_t csa2_sparse_attn_workspace_bytes(const csa2_attn_args* args) {
  return args ? attn_workspace_bytes(*args) : 0;
}

csa2_status csa2_sparse_attn(const csa2_attn_args* args, csa2_stream_t stream) {
  csa2_status st = check_attn(args);
  if (st != CSA2_OK) return st;
  if ((st = injected("sparse_attn")) != CSA2_OK) return st;
  return launch_sparse_attn(*args, reinterpret_cast<cudaStream_t>(stream));
}

csa2_status csa2_validate_plan(const csa2_layer_desc* L, int32_t n_layers, int32_t* bad_layer) {
  if (bad_layer) *bad_layer = -1;
  if (!L || n_layers < 1) return CSA2_ERR_INVALID_ARG;
  int32_t last_full = -1;
  for (int32_t l = 0; l < n_layers; ++l) {
    const csa2_layer_desc& d = L[l];
    bool ok = true;
    switch (d.mode) {
      case CSA2_MODE_FULL:
        ok = d.kv_src == l && d.idx_src == l;
        if (ok) last_full = l;
        break;
      case CSA2_MODE_REINDEX:
        // the last Full layer's main KV and indexer K, a fresh selection
        ok = last_full >= 0 && d.kv_src == last_full && d.idx_src == l;
        break;
      case CSA2_MODE_REUSE:
        ok = d.kv_src >= 0 && d.kv_src < l && L[d.kv_src].mode == CSA2_MODE_FULL &&
             d.idx_src >= 0 && d.idx_src < l &&
             (L[d.idx_src].mode == CSA2_MODE_FULL || L[d.idx_src].mode == CSA2_MODE_REINDEX) &&
             L[d.idx_src].kv_src == d.kv_src;
        break;
      default:
        ok = false;
    }
    if (!ok) {
      if (bad_layer) *bad_layer = l;
      return CSA2_ERR_INVALID_ARG;
    }
  }
  return CSA2_OK;
}

size_t csa2_layer_stack_workspace_bytes(const csa2_stack_args* s) {
  if (!s) return 0;
  return stack_pieces(*s).total();
}

csa2_status csa2_layer_stack(const csa2_layer_desc* L, int32_t n_layers,
                             const csa2_stack_args* s, csa2_stream_t stream) {
  csa2_status st = csa2_validate_plan(L, n_layers, nullptr);
  if (st != CSA2_OK) return st;
  if (!s || s->B < 1 || s->q_per_seq < 1 || s->n < 1 || s->k < 1 || s->pool < 0 ||
      s->win_max < 0)
    return CSA2_ERR_INVALID_ARG;
  if (s->pool > 0) {
    if (s->pool < s->k) return CSA2_ERR_INVALID_ARG;
    if (s->pool > 2048 || s->idx_k_dtype != CSA2_E4M3) return CSA2_ERR_UNSUPPORTED;
  }
  if (!pages_ok(s->pages, s->n)) return CSA2_ERR_INVALID_ARG;
  // paged caches hold E4M3 indexer keys (the new rows are cast into them)
  if (s->pages.block_table && s->idx_k_dtype != CSA2_E4M3) return CSA2_ERR_UNSUPPORTED;
  if (s->block < 0 || s->blocks_kept < 0) return CSA2_ERR_INVALID_ARG;
  if (s->block > 0) {
    if ((s->block & (s->block - 1)) != 0 || s->block > 65536 || s->blocks_kept < 1 ||
        s->pool > 0 || (int64_t)s->blocks_kept * s->block < s->k)
      return CSA2_ERR_INVALID_ARG;
    if (s->idx_k_dtype != CSA2_E4M3 || s->q_per_seq != 1 || s->n_valid ||
        (int64_t)s->blocks_kept * s->block > 2048 || stack_blocks(*s) > kTopkShortRow ||
        s->blocks_kept > 2048)
      return CSA2_ERR_UNSUPPORTED;
  }
  // workspace: scores | per-row top-k histograms | the candidate pool |
  // scratch of the index (quantised Q) or attention (chunk partials) step
  const StackPieces p = stack_pieces(*s);
  if (!s->workspace || s->workspace_bytes < p.total()) return CSA2_ERR_WORKSPACE;
  if (!aligned(s->workspace, 256)) return CSA2_ERR_ALIGNMENT;
  float* scores = static_cast<float*>(s->workspace);
  uint32_t* hist = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(s->workspace) + p.scores);
  int32_t* pool = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(s->workspace) + p.scores +
                                             p.tk);
  uint8_t* selw = static_cast<uint8_t*>(s->workspace) + p.scores + p.tk + p.pl;
  uint32_t* theta = reinterpret_cast<uint32_t*>(selw);
  uint32_t* cand_cnt = theta + s->B * s->q_per_seq;
  uint2* cand = reinterpret_cast<uint2*>(selw + align256((size_t)s->B * s->q_per_seq * 8));
  void* scratch = selw + p.sel;
  const size_t scratch_bytes = s->workspace_bytes - p.scores - p.tk - p.pl - p.sel;
  const bool psel = prefill_select(*s);
  const int64_t nq = s->B * s->q_per_seq;
  const int64_t P = pool_slots(*s);
  // check every call's arguments before anything is enqueued
  for (int32_t l = 0; l < n_layers; ++l) {
    const csa2_layer_desc& d = L[l];
    const csa2_layer_desc& kv = L[d.kv_src];
    if (d.mode == CSA2_MODE_FULL) {
      if (!d.codes || !d.scales || !d.idxk) return CSA2_ERR_INVALID_ARG;
      if (s->block > 0 && !d.block_keys) return CSA2_ERR_INVALID_ARG;
      if ((d.new_kv == nullptr) != (d.new_idxk == nullptr)) return CSA2_ERR_INVALID_ARG;
      const int64_t nr = d.new_rows > 0 ? d.new_rows : 1;
      if (d.new_kv && (d.new_row < 0 || d.new_rows < 0 || d.new_row + nr > s->n))
        return CSA2_ERR_INVALID_ARG;
    }
    if (d.mode != CSA2_MODE_REUSE) {
      if (!d.topk_idx) return CSA2_ERR_INVALID_ARG;
      csa2_index_args ia = stack_index_args(*s, d, kv, scores, scratch, scratch_bytes);
      if ((st = check_index(&ia)) != CSA2_OK) return st;
      if ((st = check_topk(scores, nq, s->n, s->n, s->k, d.topk_idx, s->k, hist, p.tk)) !=
          CSA2_OK)
        return st;
      if (P > 0 && (st = check_topk(scores, nq, s->n, s->n, (int32_t)P, pool, P, hist, p.tk)) !=
                       CSA2_OK)
        return st;
    }
    const int32_t* idx = L[d.mode == CSA2_MODE_REUSE ? d.idx_src : l].topk_idx;
    csa2_attn_args aa = stack_attn_args(*s, d, kv, idx, scratch, scratch_bytes);
    if ((st = check_attn(&aa)) != CSA2_OK) return st;
  }
  if ((st = injected("layer_stack")) != CSA2_OK) return st;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  // indexer-key traffic: a Full layer's keys are read again by the Reindex
  // layers that take that Full layer as their source.  A read that has a
  // later re-read keeps its keys in L2 (normal policy); each re-read walks
  // the tiles in the opposite direction to the previous read, so it starts
  // on the tiles that read touched last -- the ones still in L2.
  bool reverse_next[64] = {false};  // per Full layer (by index, plans of <= 64 layers)
  auto read_again = [&](int32_t from, int32_t src) {
    if (P > 0) return false;  // pooled Reindex layers read only the pool's rows
    for (int32_t m = from + 1; m < n_layers; ++m)
      if (L[m].mode == CSA2_MODE_REINDEX && L[m].kv_src == src) return true;
    return false;
  };
  // the top-k histograms start at zero; every selection leaves them zeroed,
  // so one clear serves the whole stack (and keeps the launches back to back)
  if ((st = clear_topk_hist(hist, nq, s->n, cs)) != CSA2_OK) return st;
  for (int32_t l = 0; l < n_layers; ++l) {
    const csa2_layer_desc& d = L[l];
    const csa2_layer_desc& kv = L[d.kv_src];
    // a decode Full layer on the plain path quantises its new rows inside its
    // indexer launch (the CTA that loads a new row's tile writes it first)
    NewRows nrows;
    bool fuse_new = false;
    if (d.mode == CSA2_MODE_FULL && d.new_kv && s->block == 0 && !psel) {
      nrows.kv = static_cast<const uint16_t*>(d.new_kv);
      nrows.idxk = static_cast<const uint16_t*>(d.new_idxk);
      nrows.row0 = d.new_row;
      nrows.rows = (int32_t)(d.new_rows > 0 ? d.new_rows : 1);
      nrows.d = s->d;
      nrows.codes = d.codes;
      nrows.scales = d.scales;
      nrows.k8 = static_cast<uint8_t*>(d.idxk);
      const csa2_index_args ia = stack_index_args(*s, d, kv, scores, scratch, scratch_bytes);
      fuse_new = index_bf16q_supported(ia, &nrows);
    }
    if (d.mode == CSA2_MODE_FULL && d.new_kv && !fuse_new) {
      if ((st = quantize_new_rows(*s, d, cs)) != CSA2_OK) return st;
      if (s->block > 0) {
        // the block keys of the blocks the new rows fall in
        const int64_t nr = d.new_rows > 0 ? d.new_rows : 1;
        const int64_t b0 = d.new_row / s->block, b1 = (d.new_row + nr - 1) / s->block;
        const bool paged = s->pages.block_table != nullptr;
        if ((st = launch_block_keys(static_cast<const uint8_t*>(d.idxk), s->B, s->n, s->di,
                                    paged ? 0 : s->n * s->di, s->pages, s->block, b0,
                                    b1 - b0 + 1, d.block_keys, 128, stack_blocks(*s) * 128,
                                    s->dev_status, cs)) != CSA2_OK)
          return st;
      }
    }
    if (d.mode == CSA2_MODE_FULL && s->block > 0) {
      // block-level pruning: score the block keys, keep the best blocks, score
      // only their entries at token level and select the top-k among them
      csa2_index_args ia = stack_index_args(*s, d, kv, scores, scratch, scratch_bytes);
      uint8_t* wq = static_cast<uint8_t*>(scratch);
      float* wc = reinterpret_cast<float*>(wq + align256((size_t)nq * s->hi * s->di));
      if ((st = launch_quantize_index_q(ia.q, ia.w, nq, s->hi, s->di, wq, wc, cs)) != CSA2_OK)
        return st;
      const int64_t nb = stack_blocks(*s);
      csa2_index_args ib = ia;
      ib.k = d.block_keys;
      ib.n = nb;
      ib.k_ld = 128;
      ib.k_seq_stride = nb * 128;
      ib.scores_ld = nb;
      ib.n_valid = nullptr;
      std::memset(&ib.pages, 0, sizeof(ib.pages));  // block keys are contiguous
      if ((st = launch_index_score_fp8(ib, wq, wc, nullptr, IndexTuning{}, cs)) != CSA2_OK)
        return st;
      if ((st = launch_topk_small(scores, nb, nullptr, 0, nq, (int32_t)nb, nullptr,
                                  s->blocks_kept, nullptr, 0, pool, P, cs, s->block, s->n)) !=
          CSA2_OK)
        return st;
      if ((st = launch_index_score_pool(ia, wq, wc, pool, P, (int32_t)P, scores, P, cs)) !=
          CSA2_OK)
        return st;
      if ((st = launch_topk_small(scores, P, nullptr, 0, nq, (int32_t)P, nullptr, s->k, pool, P,
                                  d.topk_idx, s->k, cs)) != CSA2_OK)
        return st;
    } else if (d.mode != CSA2_MODE_REUSE && psel) {
      // a prefill chunk: sampled scores -> thresholds -> candidates -> top-k
      csa2_index_args ia = stack_index_args(*s, d, kv, scores, scratch, scratch_bytes);
      const uint8_t* q8 = static_cast<const uint8_t*>(ia.q);
      const float* c = ia.w;
      if (ia.q_dtype != CSA2_E4M3) {
        uint8_t* wq = static_cast<uint8_t*>(scratch);
        float* wc = reinterpret_cast<float*>(wq + align256((size_t)nq * s->hi * s->di));
        if ((st = launch_quantize_index_q(ia.q, ia.w, nq, s->hi, s->di, wq, wc, cs)) != CSA2_OK)
          return st;
        q8 = wq;
        c = wc;
      }
      const int64_t ns = sample_cols(*s);
      csa2_index_args is = ia;
      is.scores_ld = ns;
      IndexSelect sample;
      sample.tile_stride = kSampleStride;
      if ((st = launch_index_select_prefill(is, q8, c, sample, cs)) != CSA2_OK) return st;
      // the sample's k-th largest key to 24 bits: its level-1 bin, then the
      // next 12 bits within that bin
      if ((st = launch_topk_hist(scores, nq, ns, ns, nullptr, hist, cs)) != CSA2_OK) return st;
      if ((st = launch_topk_theta(hist, nq, s->k, theta, cand_cnt, 0, cs)) != CSA2_OK) return st;
      if ((st = launch_topk_hist(scores, nq, ns, ns, nullptr, hist, cs, theta)) != CSA2_OK)
        return st;
      if ((st = launch_topk_theta(hist, nq, s->k, theta, cand_cnt, 1, cs)) != CSA2_OK) return st;
      IndexSelect emit;
      emit.theta = theta;
      emit.cand_cnt = cand_cnt;
      emit.cand = cand;
      emit.cand_cap = kCandCap;
      if ((st = launch_index_select_prefill(ia, q8, c, emit, cs)) != CSA2_OK) return st;
      if ((st = launch_topk_cand(cand, cand_cnt, kCandCap, nq, s->n, s->n_valid, s->k, d.topk_idx,
                                 s->k, s->dev_status, cs)) != CSA2_OK)
        return st;
    } else if (d.mode == CSA2_MODE_REINDEX && P > 0) {
      // Hierarchical Sparse Indexer: score the last Full layer's pool only,
      // then its top-k (pool positions mapped back to entry indices)
      csa2_index_args ia = stack_index_args(*s, d, kv, scores, scratch, scratch_bytes);
      const uint8_t* q8 = static_cast<const uint8_t*>(ia.q);
      const float* c = ia.w;
      if (ia.q_dtype != CSA2_E4M3) {
        uint8_t* wq = static_cast<uint8_t*>(scratch);
        float* wc = reinterpret_cast<float*>(wq + align256((size_t)nq * s->hi * s->di));
        if ((st = launch_quantize_index_q(ia.q, ia.w, nq, s->hi, s->di, wq, wc, cs)) != CSA2_OK)
          return st;
        q8 = wq;
        c = wc;
      }
      if ((st = launch_index_score_pool(ia, q8, c, pool, P, (int32_t)P, scores, P, cs)) !=
          CSA2_OK)
        return st;
      if ((st = launch_topk_small(scores, P, nullptr, 0, nq, (int32_t)P, nullptr, s->k, pool, P,
                                  d.topk_idx, s->k, cs)) != CSA2_OK)
        return st;
    } else if (d.mode != CSA2_MODE_REUSE) {
      csa2_index_args ia = stack_index_args(*s, d, kv, scores, scratch, scratch_bytes);
      // long rows: the indexer kernel also builds the top-k's first-level
      // histograms in decode, a histogram pass over the scores otherwise;
      // short rows are selected with every key in shared memory (no
      // histogram, so none is accumulated)
      const bool long_rows = s->n > kTopkShortRow;
      const bool fused = long_rows && index_fuses_topk_hist(ia);
      IndexTuning tune;
      if (d.kv_src < 64) {
        tune.reverse = reverse_next[d.kv_src];
        tune.keep_in_l2 = read_again(l, d.kv_src);
        reverse_next[d.kv_src] = !tune.reverse;
      }
      st = fuse_new ? launch_index_score_bf16q(ia, fused ? hist : nullptr, tune, cs, &nrows)
                    : run_index(ia, fused ? hist : nullptr, tune, cs);
      if (st != CSA2_OK) return st;
      if (long_rows && !fused &&
          (st = launch_topk_hist(scores, nq, s->n, s->n, s->n_valid, hist, cs)) != CSA2_OK)
        return st;
      // the k (or, for the pool, P) best of each row
      auto select = [&](int32_t kk, int32_t* out, int64_t out_ld) {
        return long_rows ? launch_topk_select(scores, nq, s->n, s->n, s->n_valid, kk, hist, out,
                                              out_ld, cs)
                         : launch_topk_small(scores, s->n, nullptr, 0, nq, (int32_t)s->n,
                                             s->n_valid, kk, nullptr, 0, out, out_ld, cs);
      };
      if (P > 0 && d.mode == CSA2_MODE_FULL) {
        // a Full layer of the Hierarchical Sparse Indexer keeps its top-P as
        // the pool, then takes its top-k inside the pool (the same entries
        // as the top-k of the whole row: the pool holds them)
        if ((st = select((int32_t)P, pool, P)) != CSA2_OK) return st;
        if ((st = launch_topk_small(scores, s->n, pool, P, nq, (int32_t)P, nullptr, s->k, pool,
                                    P, d.topk_idx, s->k, cs)) != CSA2_OK)
          return st;
      } else if ((st = select(s->k, d.topk_idx, s->k)) != CSA2_OK) {
        return st;
      }
    }
    const int32_t* idx = L[d.mode == CSA2_MODE_REUSE ? d.idx_src : l].topk_idx;
    csa2_attn_args aa = stack_attn_args(*s, d, kv, idx, scratch, scratch_bytes);
    // the attention queries are inputs of the call: the kernels before this
    // one in the stack never write them, so they may load before its wait
    if ((st = launch_sparse_attn(aa, cs, true)) != CSA2_OK) return st;
  }
  return CSA2_OK;
}

}  // extern "C"
