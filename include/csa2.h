/*
 * csa2.h -- C ABI of libcsa2, the CSA2 global-attention step over an FP4
 * (E2M1) main KV cache on B300 (sm_103a).
 *
 * Pages cited (the method is described in prose only):
 *   [P3] "Unlocking Extreme Context Scaling with DeepSeek-V4.1-Flash",
 *        sections "Compressed Sparse Attention 2 (CSA2)" (the three layer
 *        modes, Top-512, indexer Q / indexer K) and "Deployment and
 *        Infrastructure" (FP4 main KV cache).
 *   [P4] aiany.app item page on DeepSeek-V4.1-Flash, section "What Sets It
 *        Apart" (static layer modes, E2M1 FP4 KV format).
 *   [P5] "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression"
 *        (Daily Paper Cast transcript), Introduction (global branch beside a
 *        local sliding window) and Method (Full / Reindex / Reuse modes).
 *   [MX] OCP Microscaling Formats (MX) v1.0: E2M1 elements with a shared
 *        power-of-two (UE8M0) scale per 32 elements.
 *
 * Conventions shared by every call
 *   - Pointers marked "device" are CUDA device (or managed) addresses; the
 *     argument structs themselves live in host memory and are read before
 *     the call returns.
 *   - Calls are asynchronous on `stream` (NULL = the legacy default stream):
 *     they validate arguments on the host, enqueue kernels and return.
 *   - The caller owns all memory.  The library never allocates device or
 *     pinned memory and keeps no per-call state between calls; scratch comes
 *     from a caller-provided workspace sized by the *_workspace_bytes calls.
 *     Two calls in flight at the same time must not share a workspace.
 *   - No C++ exception crosses the ABI.  A non-zero csa2_status means
 *     nothing was enqueued, except CSA2_ERR_CUDA, where a launch failed and
 *     earlier kernels of the same call may have been enqueued.
 *   - `dev_status` (optional, device int32) collects errors that only the
 *     GPU can see: kernels OR CSA2_DEVFLAG_* bits into it.  The caller
 *     zeroes it and reads it after synchronising.  Every wait of the
 *     tensor-core indexer's pipeline gives up after a limit (2 s, or the
 *     environment variable CSA2_WAIT_LIMIT_NS in nanoseconds, read at each
 *     launch), raises CSA2_DEVFLAG_TIMEOUT and ends the kernel cleanly (no
 *     copy or MMA left in flight; the context stays usable).  Test hook:
 *     CSA2_TEST_STALL_LOADS=1 makes that kernel issue no key loads, so its
 *     waits run out.
 *   - Strides ("_ld" = between rows, "_seq_stride" = between sequences) are
 *     in elements of the tensor's own type (bytes for 8-bit tensors).
 *   - Query q belongs to sequence b = q / q_per_seq.  In decode q_per_seq is
 *     1; a prefill chunk is one sequence with q_per_seq queries.
 */
#ifndef CSA2_H
#define CSA2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t. */
typedef struct CUstream_st* csa2_stream_t;

typedef enum csa2_status {
  CSA2_OK = 0,
  CSA2_ERR_INVALID_ARG = 1,    /* NULL / negative / inconsistent argument */
  CSA2_ERR_UNSUPPORTED = 2,    /* shape or dtype combination not built */
  CSA2_ERR_ALIGNMENT = 3,      /* pointer or stride not 16-byte aligned */
  CSA2_ERR_CUDA = 4,           /* a CUDA call failed: csa2_last_cuda_error() */
  CSA2_ERR_WORKSPACE = 5,      /* workspace NULL or smaller than required */
  CSA2_ERR_DEVICE_TIMEOUT = 6, /* reported through dev_status only */
  CSA2_ERR_DEVICE_BOUNDS = 7,  /* reported through dev_status only */
  CSA2_ERR_DEVICE_CAPACITY = 8 /* reported through dev_status only */
} csa2_status;

/* Bits a kernel ORs into *dev_status. */
#define CSA2_DEVFLAG_TIMEOUT 0x1 /* a pipeline wait gave up (kernel returned early) */
#define CSA2_DEVFLAG_BOUNDS 0x2  /* an index outside [-1, n) was skipped */
#define CSA2_DEVFLAG_CAPACITY 0x4 /* a bounded candidate buffer overflowed: the
                                     selection of that row is not exact */

typedef enum csa2_dtype {
  CSA2_F32 = 0,
  CSA2_BF16 = 1,
  CSA2_E4M3 = 2
} csa2_dtype;

typedef enum csa2_mode {
  CSA2_MODE_FULL = 0,    /* fresh main KV + indexer K, fresh top-k      [P3][P5] */
  CSA2_MODE_REINDEX = 1, /* last Full layer's KV + indexer K, fresh Q and top-k */
  CSA2_MODE_REUSE = 2    /* an earlier layer's KV and top-k indices          */
} csa2_mode;

/* "major.minor.patch" of the library. */
const char* csa2_version(void);
/* Human-readable name of a status code. */
const char* csa2_status_string(int32_t status);
/* The cudaError_t of the most recent CSA2_ERR_CUDA on the calling thread. */
int32_t csa2_last_cuda_error(void);
/* Turns a dev_status word read back by the caller into a status:
 * CSA2_OK, CSA2_ERR_DEVICE_TIMEOUT, CSA2_ERR_DEVICE_BOUNDS or
 * CSA2_ERR_DEVICE_CAPACITY (in that order of precedence). */
csa2_status csa2_status_from_device(int32_t dev_status_word);

/* ------------------------------------------------------------------------ */
/* Paged caches (the serving layout)                                         */
/* ------------------------------------------------------------------------ */
/*
 * The pages name serving stacks that run the model (vLLM, SGLang) ["Unlocking
 * Extreme Context Scaling with DeepSeek-V4.1-Flash", "Deployment and
 * Infrastructure"] but no cache layout.  This library's paged layout: the
 * rows of a cache (FP4 codes, scales, indexer K) live in one pool of
 * fixed-size pages of page_rows consecutive entries of one sequence; entry
 * j of sequence b is pool row
 *   block_table[b * bt_ld + j / page_rows] * page_rows + j % page_rows
 * (a row of the pool is addressed with the cache's own row stride, *_ld).
 * Every step computes exactly what it computes on the contiguous layout;
 * only where rows live changes.
 *
 * block_table  device int32; NULL = not paged (the call's own layout)
 * bt_ld        block-table row stride (>= ceil(n / page_rows) pages)
 * page_rows    entries per page: a multiple of 64, >= 64
 * num_pages    pages in the pool (the pool holds num_pages * page_rows rows)
 * A page id outside [0, num_pages) reached by a step raises
 * CSA2_DEVFLAG_BOUNDS, and its rows read as empty (a gathered row is
 * skipped; an indexer tile reads zeros); a new row aimed at such a page is
 * not written (csa2_quantize_fp4 has no dev_status: there it is only not
 * written; the layer stack reports it).
 */
typedef struct csa2_pages {
  const int32_t* block_table;
  int64_t bt_ld;
  int32_t page_rows;
  int32_t num_pages;
} csa2_pages;

/* ------------------------------------------------------------------------ */
/* a1: FP4 quantiser                                                         */
/* ------------------------------------------------------------------------ */
/*
 * Writes new main-KV rows into the FP4 cache [P3 "Deployment and
 * Infrastructure": FP4 main KV; P4 "What Sets It Apart": E2M1 format], and
 * optionally casts the matching indexer-K rows to E4M3.
 *
 * Per row and 32-element block (d % 32 == 0):
 *   amax = max |x|;  amax == 0 -> scale byte 0, all codes 0;
 *   else e = clamp(floor(log2 amax) - 2, -127, 127), scale byte = e + 127,
 *   code_i = E2M1(x_i / 2^e): nearest, ties to even, |.| > 6 -> 6, sign kept.
 *   Element 2i of a row goes in the low nibble of code byte i.  [MX]
 * Indexer K: e4m3_i = E4M3(k_i): nearest, ties to even, |.| > 448 -> 448.
 *
 * x       device bf16, row r at x + r * x_ld (x_ld >= d)
 * codes   device u8, row r at codes + r * codes_ld (codes_ld >= d / 2)
 * scales  device u8, row r at scales + r * scales_ld (scales_ld >= d / 32)
 * idxk    optional device bf16 [rows, di] (row r at idxk + r * idxk_ld);
 * idxk_e4m3 device u8, row r at idxk_e4m3 + r * idxk_e4m3_ld; both NULL to skip.
 * A strided destination lets one call write one new row per sequence of a
 * [B, N, ...] cache: pass the address of row N-1 of sequence 0 and the
 * sequence stride as the row stride.
 * Errors: INVALID_ARG (NULL, rows < 0, d % 32 != 0, strides too small;
 *         paged: page_rows not a positive multiple of 64, num_pages < 1,
 *         rows_per_seq < 1, entry0 < 0),
 *         ALIGNMENT (x, x_ld not multiples of 8 elements; codes, codes_ld
 *         not multiples of 4 bytes; idxk / idxk_e4m3 rows not 8 / 4 aligned).
 */
typedef struct csa2_quant_args {
  const void* x;
  int64_t rows;
  int32_t d;
  int64_t x_ld;
  uint8_t* codes;
  int64_t codes_ld;
  uint8_t* scales;
  int64_t scales_ld;
  const void* idxk;
  int32_t di;
  int64_t idxk_ld;
  uint8_t* idxk_e4m3;
  int64_t idxk_e4m3_ld;
  /* Paged destination (pages.block_table != NULL): codes / scales /
   * idxk_e4m3 are pools, and row r of x is entry entry0 + r % rows_per_seq
   * of sequence r / rows_per_seq, written through the block table. */
  csa2_pages pages;
  int64_t rows_per_seq;
  int64_t entry0;
} csa2_quant_args;

csa2_status csa2_quantize_fp4(const csa2_quant_args* args, csa2_stream_t stream);

/* ------------------------------------------------------------------------ */
/* a2: indexer-Q quantiser (FP8 indexer path)                                */
/* ------------------------------------------------------------------------ */
/*
 * The pages name a per-layer indexer Q scored against FP8 indexer keys [P3
 * "CSA2"] but not the precision of Q.  This library casts Q to E4M3 per
 * (row, head) with the smallest power-of-two scale sigma = 2^e (e >= -126)
 * such that max|q| / sigma <= 448, and folds sigma into the head weight:
 *   q8[r, h, :] = E4M3(q[r, h, :] / sigma),  c[r, h] = w[r, h] * sigma.
 * A head whose values are all zero gets sigma = 1 and zero codes.
 *
 * q  device bf16 [nq, hi, di] contiguous;  w  device f32 [nq, hi]
 * q8 device u8 [nq, hi, di];  c  device f32 [nq, hi]
 * Errors: INVALID_ARG (NULL, nq < 0, hi < 1, di not in {32, 64, 128, 256}),
 *         ALIGNMENT (q / q8 not 16-byte aligned).
 */
csa2_status csa2_quantize_index_q(const void* q, const float* w, int64_t nq, int32_t hi,
                                  int32_t di, uint8_t* q8, float* c, csa2_stream_t stream);

/* ------------------------------------------------------------------------ */
/* a3: indexer score                                                         */
/* ------------------------------------------------------------------------ */
/*
 * scores[q, j] = sum_h w'[q,h] * max(0, <q_h, k_j>) for j < n_valid[q],
 * -inf for n_valid[q] <= j < n.  [P3 "CSA2": Full mode computes indexer K
 * afresh; Reindex scores with a local indexer Q; the weighted ReLU head sum
 * is this library's definition of the indexer.]
 *
 * Two paths:
 *   q F32 + k F32: w' = w, fp32 CUDA-core kernel (hi <= 64, di <= 256).
 *   q BF16 + k E4M3: q is first quantised as in csa2_quantize_index_q
 *     (w' = c, into the workspace), then scored by an FP8 tcgen05
 *     tensor-core kernel (hi == 64, di == 128).
 *   q E4M3 + k E4M3: q is already quantised (the q8 of
 *     csa2_quantize_index_q) and w holds the folded weights c (16-byte
 *     aligned); only the tensor-core kernel runs (no workspace).
 *
 * k       device, row j of sequence b at k + b * k_seq_stride + j * k_ld
 *         (elements); E4M3 needs k, k_ld, k_seq_stride 16-byte aligned.
 * n_valid optional device int32 [nq] (NULL = every entry visible).
 * scores  device f32, row q at scores + q * scores_ld.
 * Errors: INVALID_ARG, UNSUPPORTED (other shapes / dtypes; on the E4M3
 *         path also n > 2^30 or nq * ceil(n / 128) >= 2^31), ALIGNMENT,
 *         WORKSPACE (csa2_index_score_workspace_bytes), CUDA.
 * Device: CSA2_DEVFLAG_TIMEOUT if the tensor-core pipeline stalled.
 */
typedef struct csa2_index_args {
  const void* q;
  int32_t q_dtype;
  const float* w;
  const void* k;
  int32_t k_dtype;
  int64_t B;
  int64_t q_per_seq;
  int32_t hi;
  int32_t di;
  int64_t n;
  int64_t k_ld;
  int64_t k_seq_stride;
  const int32_t* n_valid;
  float* scores;
  int64_t scores_ld;
  void* workspace;
  size_t workspace_bytes;
  int32_t* dev_status;
  /* Paged keys (pages.block_table != NULL): k is a pool of rows k_ld
   * apart; k_seq_stride is not used. */
  csa2_pages pages;
} csa2_index_args;

size_t csa2_index_score_workspace_bytes(const csa2_index_args* args);
csa2_status csa2_index_score(const csa2_index_args* args, csa2_stream_t stream);

/*
 * The restricted step of the Hierarchical Sparse Indexer: score only a
 * candidate pool chosen by an earlier indexer [P5 Method: indexers
 * restricted to a shared candidate pool selected by an earlier indexer].
 * For query q and slot i < pool_n:
 *   scores[q, i] = sum_h w'[q,h] * max(0, <q_h, k_pool[q,i]>)
 * (the FP8 path of csa2_index_score at entry pool[q, i] of q's sequence),
 * -inf for a slot holding -1.  Only the FP8 path (q BF16 or E4M3, k E4M3,
 * hi == 64, di == 128); n_valid is not read (pool entries are visible by
 * construction); scores / scores_ld hold [nq, pool_n], scores_ld >= pool_n.
 * pool    device int32, row q at pool + q * pool_ld, entries in [-1, n)
 * pool_n  1 <= pool_n <= 2048
 * Workspace: csa2_index_score_workspace_bytes(args) (the quantised Q).
 * Errors: as csa2_index_score; UNSUPPORTED for another path or pool_n.
 * Device: CSA2_DEVFLAG_BOUNDS for a pool entry outside [-1, n) (the slot is
 *         scored as empty).
 */
csa2_status csa2_index_score_pool(const csa2_index_args* args, const int32_t* pool,
                                  int64_t pool_ld, int32_t pool_n, csa2_stream_t stream);

/*
 * The scoring pass of a prefill chunk's fused score -> top-k step, which
 * stores no score matrix (the pass the layer stack runs after its sampled
 * threshold; the threshold reading is the library's, see csa2_layer_stack).
 * For every query q, every visible entry j whose score s[q, j] (exactly as
 * csa2_index_score computes it) has an order-preserving key >= theta[q] is
 * appended to q's candidates as cand[q * cand_cap + i] = key | (uint64_t)j
 * << 32.  The kernel reserves slots through cand_cnt[q], 32 at a time (or,
 * when a query's tiles spread over many CTAs, exactly as needed); a
 * reserved slot it does not fill holds 0xFFFFFFFF00000000 (entry
 * 0xFFFFFFFF).  Candidates are in no particular order.  The key of a float
 * x with bits u is u ^ 0x80000000 for x >= 0 (-0 counts as +0) and ~u
 * otherwise, so a larger score has a larger key.
 * Only the prefill form of the FP8 path: q_per_seq a multiple of 4, q BF16
 * or E4M3, k E4M3, hi == 64, di == 128.  scores / scores_ld are not read.
 * theta    device uint32 [nq]
 * cand_cnt device uint32 [nq], zero on entry; on exit the slots reserved
 *          (above cand_cap: the candidates past cand_cap were dropped)
 * cand     device uint64 [nq, cand_cap], 8-byte aligned
 * Workspace: csa2_index_score_workspace_bytes(args) (the quantised Q).
 * Errors: as csa2_index_score; UNSUPPORTED for another path or form.
 */
csa2_status csa2_index_candidates(const csa2_index_args* args, const uint32_t* theta,
                                  uint32_t* cand_cnt, uint64_t* cand, int64_t cand_cap,
                                  csa2_stream_t stream);

/*
 * Block keys, the first level of the Hierarchical Sparse Indexer [P5
 * Method: indexers restricted to a candidate pool selected by an earlier
 * indexer; P5 Related Work: scoring token-level entries and pruning them on
 * block-level representations].  This library's definition: the entries of
 * a sequence form blocks of G consecutive entries, and block blk's key is
 *   out[blk, i] = E4M3( (sum over the block's entries j < n of E4M3^-1(k8[j, i])) / G )
 * (entries past n count as zero; E4M3 cast as everywhere: nearest, ties to
 * even, saturating).  The sum is exact, so the cast is the only rounding.
 * Computes blocks blk0 .. blk0 + nblk - 1 of every sequence b < B.
 *
 * k8     device E4M3 [B, n, 128]: row j of sequence b at k8 + b*k_seq_stride
 *        + j*k_ld; or (pages non-NULL with a block table) a page pool of rows
 *        k_ld apart.
 * out    device u8: block blk of sequence b at out + b*out_seq_stride + blk*out_ld
 * G      a power of two, 1 <= G <= 65536
 * Errors: INVALID_ARG (NULL, negative sizes, G not a power of two, blocks
 *         past ceil(n / G), strides below 128, a bad paged layout), CUDA.
 * Device: CSA2_DEVFLAG_BOUNDS for a page outside the pool (its rows count
 *         as zero).
 */
csa2_status csa2_index_block_keys(const uint8_t* k8, int64_t B, int64_t n, int64_t k_ld,
                                  int64_t k_seq_stride, const csa2_pages* pages, int32_t G,
                                  int64_t blk0, int64_t nblk, uint8_t* out, int64_t out_ld,
                                  int64_t out_seq_stride, int32_t* dev_status,
                                  csa2_stream_t stream);

/* ------------------------------------------------------------------------ */
/* a4: top-k                                                                 */
/* ------------------------------------------------------------------------ */
/*
 * Per row r: the min(k, n_valid[r]) entries j < n_valid[r] that are largest
 * by (score descending, index ascending), written ascending by index to
 * idx_out[r, 0..), the rest of the row set to -1.  [P3 "CSA2": Full mode
 * selects new Top-512 indices; the tie rule and order are this library's.]
 * +0 and -0 compare equal.  NaN scores are outside the contract.
 *
 * scores  device f32, row r at scores + r * ld;  n_valid optional [rows]
 * idx_out device int32, row r at idx_out + r * idx_ld
 * 1 <= k <= 2048.  Workspace: csa2_topk_workspace_bytes(rows, n, k): one
 * histogram per row of 4096 fine and 64 coarse bins (rows * 16,640 bytes)
 * and, for rows longer than 4096,
 * a counter per row and S candidate slots of 8 KiB per row (S = about 296 /
 * rows, at most 64, at most one per 4096 entries); the call clears what must
 * start at zero.
 * Kernels: rows of at most 4096 entries run one CTA per row with every key
 * in shared memory; longer rows a histogram pass over the scores, then one
 * selection kernel with S CTAs per row: each scans its slice once and keeps
 * the entries of the histogram's threshold bin and above, and the row's
 * last CTA to finish resolves the threshold among the kept entries (or, when
 * a slice kept more than its slot holds, over the whole row again).
 * Errors: INVALID_ARG, UNSUPPORTED (k > 2048), WORKSPACE, CUDA.
 */
size_t csa2_topk_workspace_bytes(int64_t rows, int64_t n, int32_t k);
csa2_status csa2_topk(const float* scores, int64_t rows, int64_t n, int64_t ld,
                      const int32_t* n_valid, int32_t k, int32_t* idx_out, int64_t idx_ld,
                      void* workspace, size_t workspace_bytes, int32_t* dev_status,
                      csa2_stream_t stream);

/*
 * csa2_topk_noalloc: the same selection as csa2_topk, for callers that
 * cannot allocate device memory -- for example code running inside an
 * allocator callback, a plugin whose host framework owns every device
 * allocation, or a process that must not grow its memory footprint after
 * start-up.  The pages have no counterpart to this entry point; it exists
 * only for those callers.
 *
 * The caller still passes the scores and idx_out buffers; the selector's
 * scratch comes from one fixed 4 MiB array compiled into the library, which
 * every GPU that loads the library keeps until the process exits.  Limit:
 * csa2_topk_workspace_bytes(rows, n, k) must not exceed 4 MiB (252 rows of
 * at most 4096 entries; 8 rows of 262144); larger calls return
 * CSA2_ERR_WORKSPACE and enqueue nothing.  The call allocates nothing (no cudaMalloc / cudaFree).
 * The first call on a device looks up the array's device address for that
 * device (with that device current), so make that first call before any
 * stream capture.  The address is looked up again whenever a call runs in
 * another CUDA context than the lookup did (after cudaDeviceReset, or from a
 * non-primary context), since the array may then sit elsewhere; make such a
 * first call in a new context before any capture too.  CSA2_FAULT_INJECT
 * reaches it as "topk_noalloc".  Every call shares the one array: calls that may overlap
 * on the GPU (different streams, or different host threads) race and give
 * wrong results; serialise them.  The parts of the array that must start at
 * zero are cleared by each call, so a call never sees a previous call's data.
 * Other arguments and errors as for csa2_topk.
 */
csa2_status csa2_topk_noalloc(const float* scores, int64_t rows, int64_t n, int64_t ld,
                              const int32_t* n_valid, int32_t k, int32_t* idx_out,
                              int64_t idx_ld, int32_t* dev_status, csa2_stream_t stream);

/* ------------------------------------------------------------------------ */
/* a5: sparse attention over gathered FP4 rows + the bf16 sliding window     */
/* ------------------------------------------------------------------------ */
/*
 * For query q (sequence b) and head h, with the key set
 *   K = { dequant(row idx[q, t] of sequence b) : idx[q, t] >= 0 }
 *     U { window row win_start[q] + u of sequence b : 0 <= u < win_len[q] },
 *   out[q, h, :] = sum_{x in K} softmax_x(softmax_scale * <q_h, x>) x.
 * One latent row is both key and value; the two sets are not de-duplicated;
 * an empty K gives zeros.  [P4 "What Sets It Apart": FP4 E2M1 main KV;
 * P5 Introduction: global branch beside local sliding-window attention.]
 * dequant(row)[i] = E2M1(code_i) * 2^(scale_byte(i/32) - 127).
 *
 * Paths: q F32 (hq <= 64, d <= 256; CUDA cores) or q BF16 (hq % 16 == 0,
 * d == 512; tcgen05 bf16 tensor-core MMA, fp32 accumulation in tensor
 * memory, probabilities split into two bf16 terms).  The BF16 path cuts the
 * k + win_max keys of a query into chunks of 80; each chunk writes its
 * partial result (max, sum, unnormalised output per head) to the workspace,
 * csa2_sparse_attn_workspace_bytes of it (nq * ceil(hq/32) * chunks * 65.8 KB).
 * With at most 8 chunks (k + win_max <= 640) the chunks of a query form a
 * thread-block cluster that merges the partials itself; with more, a second
 * kernel merges them.
 * q        device [nq, hq, d] contiguous
 * codes    device u8: row j of sequence b at codes + b*codes_seq_stride + j*codes_ld
 * scales   device u8: likewise with scales_seq_stride / scales_ld
 * idx      device int32, row q at idx + q * idx_ld, k entries, -1 = none
 * window   device bf16: row u of sequence b at window + b*win_seq_stride + u*win_ld
 * win_start / win_len  optional device int32 [nq] (NULL: 0 / w_rows)
 * win_max  host upper bound on win_len (0: w_rows); sizes the launch
 * out      device f32 [nq, hq, d]
 * An index outside [-1, n) is skipped and raises CSA2_DEVFLAG_BOUNDS; a
 * window range outside [0, w_rows), or a win_len above the bound win_max,
 * is clipped the same way (and raises the same flag).
 * Errors: INVALID_ARG, UNSUPPORTED, ALIGNMENT (BF16 path: codes, scales
 *         and window rows 16-byte aligned), WORKSPACE, CUDA.
 */
typedef struct csa2_attn_args {
  const void* q;
  int32_t q_dtype;
  int64_t nq;
  int64_t q_per_seq;
  int32_t hq;
  int32_t d;
  const uint8_t* codes;
  const uint8_t* scales;
  int64_t n;
  int64_t codes_ld;
  int64_t codes_seq_stride;
  int64_t scales_ld;
  int64_t scales_seq_stride;
  const int32_t* idx;
  int32_t k;
  int64_t idx_ld;
  const void* window;
  int32_t w_rows;
  int64_t win_ld;
  int64_t win_seq_stride;
  const int32_t* win_start;
  const int32_t* win_len;
  int32_t win_max;
  float softmax_scale;
  float* out;
  void* workspace;
  size_t workspace_bytes;
  int32_t* dev_status;
  /* Paged main KV (pages.block_table != NULL): codes / scales are pools of
   * rows codes_ld / scales_ld apart; the *_seq_stride fields are not used. */
  csa2_pages pages;
} csa2_attn_args;

size_t csa2_sparse_attn_workspace_bytes(const csa2_attn_args* args);
csa2_status csa2_sparse_attn(const csa2_attn_args* args, csa2_stream_t stream);

/* ------------------------------------------------------------------------ */
/* the decoder's global KV: projection of the encoder state + FP4 quantise   */
/* ------------------------------------------------------------------------ */
/*
 * out[r, c] = sum_k h[r, k] * w[c, k] (fp32 accumulation of bf16 products),
 * quantised per 32-element block of each row exactly as csa2_quantize_fp4
 * into codes / scales.  [P3 "Causal Encoder-Decoder (CED) Efficiency": the
 * decoder derives its global KV cache from the final encoder hidden state
 * using per-layer projections; P3 "Deployment and Infrastructure": FP4 main
 * KV.]  The codes are decided on the fp32 projection, which is also written
 * to `out` when out is not NULL.
 *
 * h      device bf16 [rows, hidden], row r at h + r * h_ld (elements)
 * w      device bf16 [d, hidden]: row c holds the weights of output column c
 * codes  device u8 [rows, d/2] (even column in the low nibble), codes_ld
 * scales device u8 [rows, d/32] (UE8M0), scales_ld
 * out    optional device f32 [rows, d], out_ld
 * dev_status optional device int32 (see CSA2_DEVFLAG_*)
 * hidden a multiple of 32; d a multiple of 64.  From 64 rows on, when hidden
 * is a multiple of 256, the product runs on tcgen05 tensor cores; up to 16
 * rows (hidden <= 16384) every CTA loads its whole share at once; other
 * sizes stream through a ring.  Every path sums each output in fp32 in a
 * fixed order (the result does not depend on the launch).
 * Errors: INVALID_ARG, ALIGNMENT (h, w 16-byte aligned with h_ld, w_ld
 *         multiples of 8; out 8-byte aligned with out_ld even), CUDA.
 */
typedef struct csa2_project_args {
  const void* h;
  const void* w;
  int64_t rows;
  int32_t hidden;
  int32_t d;
  int64_t h_ld;
  int64_t w_ld;
  uint8_t* codes;
  int64_t codes_ld;
  uint8_t* scales;
  int64_t scales_ld;
  float* out;
  int64_t out_ld;
  int32_t* dev_status; /* optional: CSA2_DEVFLAG_TIMEOUT if a pipeline wait gave up */
} csa2_project_args;

csa2_status csa2_project_fp4(const csa2_project_args* args, csa2_stream_t stream);

/* ------------------------------------------------------------------------ */
/* a6: the static Full / Reindex / Reuse layer schedule                      */
/* ------------------------------------------------------------------------ */
/*
 * Runs one step of a stack of CSA2 layers in order on `stream` [P3 "CSA2";
 * P4 "static layer modes"; P5 Method]:
 *   Full    quantise this step's new rows into the layer's own caches
 *           (optional), score its own indexer K with its indexer Q, top-k
 *           into its own topk_idx, attend over its own FP4 KV.
 *   Reindex score the indexer K of layer kv_src (a Full layer) with its own
 *           indexer Q, top-k into its own topk_idx, attend over kv_src's KV.
 *   Reuse   attend over kv_src's KV with the indices of layer idx_src (a
 *           Full or Reindex layer); no indexer work.
 * Validation before anything is enqueued: layer 0 is Full; a Full layer
 * names itself; kv_src names an earlier Full layer; a Reindex layer's
 * idx_src is itself; a Reuse layer's idx_src names an earlier Full or
 * Reindex layer whose kv_src equals its own kv_src.
 *
 * Layouts (per layer, all device, contiguous):
 *   codes [B, n, d/2] u8, scales [B, n, d/32] u8, idxk [B, n, di]
 *   (E4M3 or F32 per idx_k_dtype); new_kv bf16 [B, new_rows, d] and
 *   new_idxk [B, new_rows, di] (bf16 for E4M3 idxk, f32 for F32 idxk) are
 *   quantised into rows new_row .. new_row + new_rows - 1 of every sequence
 *   (decode: one new compressed entry per sequence; a prefill chunk: the
 *   entries it completes); new_rows = 0 is read as 1;
 *   idx_q [nq, hi, di] (idx_q_dtype), idx_w f32 [nq, hi];
 *   attn_q [nq, hq, d] (attn_q_dtype); window bf16 [B, w_rows, d];
 *   topk_idx int32 [nq, k]; out f32 [nq, hq, d].
 * Workspace: csa2_layer_stack_workspace_bytes (scores, selector and
 * attention scratch, reused layer after layer).
 * Windows: win_start / win_len (optional, per query) select each query's
 * rows of its layer's window buffer as in csa2_sparse_attn; win_max, a host
 * upper bound on win_len (0: w_rows), sizes the attention launch (a prefill
 * chunk's buffer holds T + W - 1 rows, each query sees W of them).
 * Errors: INVALID_ARG (a plan or argument check, pool < k, win_max < 0),
 *         UNSUPPORTED, ALIGNMENT, WORKSPACE -- found before any launch;
 *         CUDA from a launch.
 *
 * Hierarchical Sparse Indexer (args->pool = P > 0) [P5 Method]: every Full
 * layer's indexer, which scores all entries, also keeps its top-P entries
 * (the top-k order) as the candidate pool, and every Reindex layer scores
 * only the pool of its kv_src (the last Full layer, so one pool lives in
 * the workspace) and takes its top-k inside it.  A Full layer's own top-k
 * is unchanged.  Needs the FP8 indexer (idx_k_dtype E4M3) and
 * k <= P <= 2048; P >= n restricts nothing.
 */
typedef struct csa2_layer_desc {
  int32_t mode;
  int32_t kv_src;
  int32_t idx_src;
  const void* new_kv;
  const void* new_idxk;
  int64_t new_row;
  int64_t new_rows;
  const void* idx_q;
  const float* idx_w;
  const void* attn_q;
  const void* window;
  uint8_t* codes;
  uint8_t* scales;
  void* idxk;
  int32_t* topk_idx;
  float* out;
  /* Full layers with block-level pruning (args->block > 0): the block keys
   * of the layer's indexer K, [B, ceil(n / block), 128] E4M3 contiguous,
   * kept current by the stack for the blocks its new rows touch. */
  uint8_t* block_keys;
} csa2_layer_desc;

typedef struct csa2_stack_args {
  int64_t B;
  int64_t q_per_seq;
  int64_t n;
  int32_t hi;
  int32_t di;
  int32_t hq;
  int32_t d;
  int32_t k;
  int32_t w_rows;
  int32_t idx_q_dtype;
  int32_t idx_k_dtype;
  int32_t attn_q_dtype;
  const int32_t* n_valid;
  const int32_t* win_start;
  const int32_t* win_len;
  float softmax_scale;
  void* workspace;
  size_t workspace_bytes;
  int32_t* dev_status;
  int32_t pool;  /* candidate pool size P of the Hierarchical Sparse Indexer; 0 = off */
  int32_t win_max; /* host upper bound on win_len (0: w_rows); sizes the attention launch */
  /* Paged caches: every Full layer's codes, scales and idxk are pools
   * ([num_pages * page_rows] rows of d/2, d/32 and di) shared through this
   * one block table; new rows are written through it. */
  csa2_pages pages;
  /* Block-level pruning of the Hierarchical Sparse Indexer (0 = off): blocks
   * of `block` entries (a power of two); a Full layer scores the block keys,
   * keeps its best blocks_kept blocks and scores at token level only their
   * entries (the candidate pool, blocks_kept * block <= 2048 slots), taking
   * its top-k there; Reindex layers score the same pool.  Decode shapes only
   * (q_per_seq == 1, n_valid NULL), ceil(n / block) <= 4096, no `pool`. */
  int32_t block;
  int32_t blocks_kept;
} csa2_stack_args;

/* Checks a schedule (see above) without touching the GPU.  Returns CSA2_OK
 * or CSA2_ERR_INVALID_ARG and, if bad_layer is not NULL, the first layer
 * that breaks a rule (-1 if the arguments themselves are bad). */
csa2_status csa2_validate_plan(const csa2_layer_desc* layers, int32_t n_layers,
                               int32_t* bad_layer);
size_t csa2_layer_stack_workspace_bytes(const csa2_stack_args* args);
csa2_status csa2_layer_stack(const csa2_layer_desc* layers, int32_t n_layers,
                             const csa2_stack_args* args, csa2_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* CSA2_H */
