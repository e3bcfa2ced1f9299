// internal.h -- launchers shared between the C-ABI layer and the kernels.
#pragma once

#include <cuda.h>  // CUtensorMap (type only)
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>

#include "../../include/csa2.h"

namespace csa2 {

// cuTensorMapEncodeTiled, fetched from the driver at run time (null if absent).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn tensor_map_encoder();
// Limit of a tensor-core pipeline's waits: CSA2_WAIT_LIMIT_NS, else 2 s.
uint64_t wait_limit_ns();

// Round up to a multiple of 256 bytes (every workspace region starts aligned).
inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Host-side failure injection: the status CSA2_FAULT_INJECT names for the
// entry point `call` (its name without "csa2_"), else CSA2_OK.
csa2_status injected(const char* call);
// Records a failed CUDA call for csa2_last_cuda_error() and maps it to a status.
csa2_status cuda_fail(cudaError_t e);
// cudaGetLastError() after a launch, mapped to a status.
csa2_status check_launch();

// a1 (dev_status: where a paged destination outside the pool is reported)
csa2_status launch_quantize_fp4(const csa2_quant_args& a, cudaStream_t s,
                                int32_t* dev_status = nullptr);
// a2
csa2_status launch_quantize_index_q(const void* q, const float* w, int64_t nq, int32_t hi,
                                    int32_t di, uint8_t* q8, float* c, cudaStream_t s);
// a3, fp32 CUDA-core path
csa2_status launch_index_score_f32(const csa2_index_args& a, cudaStream_t s);
// How one FP8 indexer launch walks the keys.  Each CTA owns a contiguous
// range of 128-entry tiles; `reverse` walks it from its end (so a launch
// that follows another reader of the same keys starts on the tiles that
// reader left in L2), `keep_in_l2` loads with the normal L2 policy instead of
// evict-first (when a later layer reads the same keys again).
struct IndexTuning {
  bool reverse = false;
  bool keep_in_l2 = false;
};

// The forms of a prefill indexer launch (q_per_seq a multiple of 4) that
// feed a selection without the full score matrix:
//   sampled  (tile_stride = R > 1, theta null): only every R-th tile of 128
//            entries is scored, its scores written compactly (tile t of the
//            sample to columns 128 t ..) into a.scores / a.scores_ld;
//   emitting (theta set, tile_stride 1): every tile is scored, nothing is
//            stored but the (key, entry) pairs of the visible entries whose
//            order-preserving key is >= theta[q], appended to cand[q *
//            cand_cap ..] through the counter cand_cnt[q] (zero before).
struct IndexSelect {
  int tile_stride = 1;
  const uint32_t* theta = nullptr;
  uint32_t* cand_cnt = nullptr;
  uint2* cand = nullptr;
  int64_t cand_cap = 0;
};
csa2_status launch_index_select_prefill(const csa2_index_args& a, const uint8_t* q8,
                                        const float* c, const IndexSelect& sel, cudaStream_t s);
// a3, FP8 tensor-core path: q8 / c already quantised.  hist1 (nullable):
// [nq][4096] first-level top-k histograms the decode kernel adds its scores'
// keys to (see index_fuses_topk_hist).
csa2_status launch_index_score_fp8(const csa2_index_args& a, const uint8_t* q8, const float* c,
                                   uint32_t* hist1, IndexTuning tune, cudaStream_t s);
// A decode Full layer's new cache rows (a1), quantised inside the indexer
// launch that reads them: the CTA whose tiles hold a new row writes its FP4
// codes and scales and its E4M3 indexer key before that CTA loads the tile.
// Row j of sequence b goes to cache row b * n + j, or through the block
// table when the caches are paged.
struct NewRows {
  const uint16_t* kv = nullptr;    // bf16 [B, rows, d]
  const uint16_t* idxk = nullptr;  // bf16 [B, rows, 128]
  int64_t row0 = 0;                // first new entry of every sequence
  int32_t rows = 0;
  int32_t d = 0;                   // a multiple of 256
  uint8_t* codes = nullptr;        // FP4 codes [B * n (or pool rows), d / 2]
  uint8_t* scales = nullptr;       // UE8M0 scales [.., d / 32]
  uint8_t* k8 = nullptr;           // E4M3 indexer keys [.., 128]
};
// The same with bf16 queries and raw weights (a.q, a.w), quantised inside
// the indexer kernel (decode shapes: hi 64, di 128, q_per_seq not a
// multiple of 4); CSA2_ERR_UNSUPPORTED (nothing launched) when the launch
// cannot take that form, and the caller quantises separately.  nr
// (optional, one query per sequence): new rows quantised in the launch.
csa2_status launch_index_score_bf16q(const csa2_index_args& a, uint32_t* hist1, IndexTuning tune,
                                     cudaStream_t s, const NewRows* nr = nullptr);
// Whether launch_index_score_bf16q takes this launch, and also its new rows
// when nr is given.
bool index_bf16q_supported(const csa2_index_args& a, const NewRows* nr = nullptr);
// Scores of a candidate pool (the Hierarchical Sparse Indexer): for every
// query q and slot i < pool_n, scores[q * scores_ld + i] = the FP8 indexer
// score of entry pool[q * pool_ld + i] of q's sequence (-inf for a slot
// holding -1).  a.k / k_ld / k_seq_stride / B / q_per_seq / dev_status as
// for launch_index_score_fp8 (hi == 64, di == 128); q8 / c quantised Q.
csa2_status launch_index_score_pool(const csa2_index_args& a, const uint8_t* q8, const float* c,
                                    const int32_t* pool, int64_t pool_ld, int32_t pool_n,
                                    float* scores, int64_t scores_ld, cudaStream_t s);
// whether launch_index_score_fp8 builds the top-k histograms for `a`
bool index_fuses_topk_hist(const csa2_index_args& a);
// a4: rows of at most kTopkShortRow entries are selected by
// launch_topk_small (every key in shared memory, no histogram); longer rows
// by launch_topk_select from their level-1 histograms.
constexpr int64_t kTopkShortRow = 4096;
// the workspace holds one first-level histogram per row (the first rows *
// kTopkHistStride words: 4096 fine and 64 coarse bins), then for rows longer
// than 4096 a counter and the slices' candidate slots per row
size_t topk_workspace_bytes(int64_t rows, int64_t n, int32_t k);
csa2_status launch_topk(const float* scores, int64_t rows, int64_t n, int64_t ld,
                        const int32_t* n_valid, int32_t k, int32_t* idx_out, int64_t idx_ld,
                        void* ws, int32_t* dev_status, cudaStream_t s);
// the pieces of launch_topk: zero the histograms (and the counters of a
// long-row workspace for rows of n); select from scores whose histograms are
// complete (the selection leaves histograms and counters zeroed)
csa2_status clear_topk_hist(uint32_t* hist1, int64_t rows, int64_t n, cudaStream_t s);
// The selection of a prefill chunk without its score matrix: theta[r], the
// lowest key of the 24-bit key prefix holding the k-th largest key of a
// sample of row r's scores (so no entry of the row's top k lies below it),
// in two levels over the row's histogram: level 0 reads the 12-bit
// histogram, sets theta[r] = T1 << 20 and keeps in cand_cnt[r] how many of
// the k fall in bin T1; level 1 reads the histogram of the next 12 bits of
// the keys in bin T1, completes theta[r] and zeroes cand_cnt[r].  Each level
// clears the histogram.  Then the exact top k of each row among its
// candidates (see IndexSelect), written ascending, -1 padded (more than cap
// candidates: CSA2_DEVFLAG_CAPACITY).
csa2_status launch_topk_theta(uint32_t* hist1, int64_t rows, int32_t k, uint32_t* theta,
                              uint32_t* cand_cnt, int level, cudaStream_t s);
size_t topk_cand_smem(int64_t cap, int64_t n);
// whether a candidate selection of `cap` slots over rows of n entries fits a CTA
bool topk_cand_fits(int64_t cap, int64_t n);
csa2_status launch_topk_cand(const uint2* cand, const uint32_t* cand_cnt, int64_t cap,
                             int64_t rows, int64_t n, const int32_t* n_valid, int32_t k,
                             int32_t* out, int64_t out_ld, int32_t* dev_status, cudaStream_t s);
// within (optional, per row): count only the keys in level-1 bin
// within[r] >> 20, binned by their next 12 bits
csa2_status launch_topk_hist(const float* scores, int64_t rows, int64_t n, int64_t ld,
                             const int32_t* n_valid, uint32_t* hist1, cudaStream_t s,
                             const uint32_t* within = nullptr);
// Block keys of the Hierarchical Sparse Indexer's first level: for blocks
// blk0 .. blk0 + nblk - 1 of every sequence b < B, out[b * out_seq_stride +
// blk * out_ld + i] = E4M3((sum of the di = 128 key bytes i of the block's
// entries, decoded) / G) (G a power of two, entries past n count as zero).
csa2_status launch_block_keys(const uint8_t* k8, int64_t B, int64_t n, int64_t k_ld,
                              int64_t k_seq_stride, const csa2_pages& pages, int32_t G,
                              int64_t blk0, int64_t nblk, uint8_t* out, int64_t out_ld,
                              int64_t out_seq_stride, int32_t* dev_status, cudaStream_t s);
// The decoder's global KV: h [rows, hidden] x w [d, hidden]^T quantised to
// FP4 (codes / scales), the fp32 projection optionally to out.
csa2_status launch_project_fp4(const csa2_project_args& a, cudaStream_t s);
// Top-k of short rows (n <= 4096, one CTA per row; n_valid optional): value i of row r is
// scores[r * ld + i], or with gather scores[r * ld + gather[r * gather_ld +
// i]] (an index < 0 is an empty slot, below every value); positions are
// written ascending as remap[r * remap_ld + i] (or i), padded with -1.
// expand = G > 0: position p (a block) written at output slot s is written
// as the G entries p * G .. p * G + G - 1 into slots s * G .., those at or
// past expand_n as -1 (the row then holds k * G slots).
csa2_status launch_topk_small(const float* scores, int64_t ld, const int32_t* gather,
                              int64_t gather_ld, int64_t rows, int32_t n, const int32_t* n_valid,
                              int32_t k, const int32_t* remap, int64_t remap_ld, int32_t* idx_out,
                              int64_t idx_ld, cudaStream_t s, int32_t expand = 0,
                              int64_t expand_n = 0);
// remap (optional): entry j of row r is written as remap[r * remap_ld + j]
// (positions in a candidate pool -> entry indices); clear_hist = false
// leaves the histograms for another selection from the same scores.
csa2_status launch_topk_select(const float* scores, int64_t rows, int64_t n, int64_t ld,
                               const int32_t* n_valid, int32_t k, uint32_t* hist1,
                               int32_t* idx_out, int64_t idx_ld, cudaStream_t s,
                               const int32_t* remap = nullptr, int64_t remap_ld = 0,
                               bool clear_hist = true);
// a5
// q_ready: the attention queries, the window rows and the window ranges may
// be read before the kernel's programmatic-launch wait (no kernel still
// running on the stream writes them); set by the layer stack, whose
// preceding kernels never do.
size_t attn_workspace_bytes(const csa2_attn_args& a);
csa2_status launch_sparse_attn(const csa2_attn_args& a, cudaStream_t s, bool q_ready = false);

// number of SMs of the current device (cached per device)
int sm_count();

// Kernel attributes (the dynamic shared-memory limit) are per device: runs
// `set` once for each device the calling thread makes current (bit d of
// `done` records device d; devices past 63 run it every time).  Host threads
// may call concurrently: the mask is atomic, and two threads that both see
// the bit clear both run `set`, which is harmless (the attributes are
// idempotent).
template <class F>
cudaError_t once_per_device(std::atomic<uint64_t>& done, F&& set) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = (dev >= 0 && dev < 64) ? (uint64_t)1 << dev : 0;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = set();
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
  return e;
}

// Whether launches use programmatic dependent launch: CSA2_PDL=0 turns it
// off (read once per process; default on).
bool pdl_enabled();

// Launch with programmatic dependent launch (see pdl_trigger / pdl_wait in
// common.cuh) and, if cluster_x > 1, thread-block clusters of cluster_x CTAs
// along x.
template <typename... KArgs, typename... Args>
csa2_status launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t s, unsigned cluster_x, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  if (pdl_enabled()) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster_x > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster_x;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
  return e == cudaSuccess ? check_launch() : cuda_fail(e);
}

}  // namespace csa2
