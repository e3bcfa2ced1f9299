"""ctypes view of the CSA2 oracle plus the layer-mode semantics.

TEST INFRASTRUCTURE ONLY: imported by tests/, by the package smoke check and
by the CPU-baseline leg of bench.py; never by the product path.

Pages cited:
  [P3] "Unlocking Extreme Context Scaling with DeepSeek-V4.1-Flash",
       section "Compressed Sparse Attention 2 (CSA2)".
  [P4] aiany.app item page on DeepSeek-V4.1-Flash, "What Sets It Apart".
  [P5] "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression"
       (Daily Paper Cast transcript), Method.

All arrays are numpy; float inputs are float64 holding the exact bf16 /
fp32 values the product consumed.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None

FULL, REINDEX, REUSE = 0, 1, 2

_D = ctypes.POINTER(ctypes.c_double)
_U8 = ctypes.POINTER(ctypes.c_uint8)
_I32 = ctypes.POINTER(ctypes.c_int32)
_I64 = ctypes.c_int64


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        L.oracle_e2m1_value.restype = ctypes.c_double
        L.oracle_e2m1_value.argtypes = [ctypes.c_int]
        L.oracle_ue8m0_value.restype = ctypes.c_double
        L.oracle_ue8m0_value.argtypes = [ctypes.c_int]
        L.oracle_e4m3_value.restype = ctypes.c_double
        L.oracle_e4m3_value.argtypes = [ctypes.c_int]
        L.oracle_e2m1_encode.restype = ctypes.c_int
        L.oracle_e2m1_encode.argtypes = [ctypes.c_double]
        L.oracle_e4m3_encode.restype = ctypes.c_int
        L.oracle_e4m3_encode.argtypes = [ctypes.c_double]
        L.oracle_floor_log2.restype = ctypes.c_int
        L.oracle_floor_log2.argtypes = [ctypes.c_double]
        L.oracle_quantize_fp4.restype = ctypes.c_int
        L.oracle_quantize_fp4.argtypes = [_D, _I64, ctypes.c_int32, _U8, _U8]
        L.oracle_dequantize_fp4.restype = None
        L.oracle_dequantize_fp4.argtypes = [_U8, _U8, _I64, ctypes.c_int32, _D]
        L.oracle_cast_e4m3.restype = None
        L.oracle_cast_e4m3.argtypes = [_D, _I64, _U8]
        L.oracle_quantize_index_q.restype = None
        L.oracle_quantize_index_q.argtypes = [_D, _D, _I64, ctypes.c_int32,
                                              ctypes.c_int32, _U8, _D]
        L.oracle_index_score.restype = None
        L.oracle_index_score.argtypes = [_D, _D, _D, _I64, _I64, ctypes.c_int32,
                                         ctypes.c_int32, _I64, _I32, _D]
        L.oracle_topk.restype = None
        L.oracle_topk.argtypes = [_D, _I64, _I64, _I32, ctypes.c_int32, _I32]
        L.oracle_sparse_attn.restype = ctypes.c_int
        L.oracle_sparse_attn.argtypes = [_D, _I64, _I64, ctypes.c_int32, ctypes.c_int32,
                                         _U8, _U8, _I64, _I32, ctypes.c_int32,
                                         _D, ctypes.c_int32, _I32, _I32,
                                         ctypes.c_double, _D]
        _lib = L
    return _lib


def _p(a, typ):
    return a.ctypes.data_as(typ)


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _opt_i32(a):
    if a is None:
        return None, None
    a = np.ascontiguousarray(a, dtype=np.int32)
    return a, _p(a, _I32)


# ---- number formats -------------------------------------------------------

def e2m1_value(code):
    return lib().oracle_e2m1_value(int(code))


def ue8m0_value(s):
    return lib().oracle_ue8m0_value(int(s))


def e4m3_value(b):
    return lib().oracle_e4m3_value(int(b))


def e2m1_encode(y):
    return lib().oracle_e2m1_encode(float(y))


def e4m3_encode(x):
    return lib().oracle_e4m3_encode(float(x))


def floor_log2(a):
    return lib().oracle_floor_log2(float(a))


def e4m3_table():
    """float64 [256]: the value of every E4M3 byte (NaN at 0x7f and 0xff)."""
    return np.array([e4m3_value(b) for b in range(256)], dtype=np.float64)


def e4m3_decode(codes):
    return e4m3_table()[np.asarray(codes, dtype=np.uint8)]


# ---- a1 / a2 ---------------------------------------------------------------

def quantize_fp4(x):
    """x [rows, d] -> (codes uint8 [rows, d/2], scales uint8 [rows, d/32])."""
    x = _f64(x)
    rows, d = x.shape
    codes = np.zeros((rows, d // 2), dtype=np.uint8)
    scales = np.zeros((rows, d // 32), dtype=np.uint8)
    rc = lib().oracle_quantize_fp4(_p(x, _D), rows, d, _p(codes, _U8), _p(scales, _U8))
    if rc != 0:
        raise ValueError("oracle_quantize_fp4: bad arguments")
    return codes, scales


def gather_pages(pool, block_table, n):
    """The logical per-sequence view of a paged cache: row j of sequence b
    is row j % page_rows of physical page block_table[b, j // page_rows].

    pool [num_pages, page_rows, ...] (codes, scales or indexer K rows);
    block_table int [B, pages_per_seq]; n rows per sequence
    (n <= pages_per_seq * page_rows).  Returns [B, n, ...].
    Reading (the serving layout the pages' inference stacks use, "Unlocking
    ...", Deployment and Infrastructure): fixed-size pages in one shared
    pool and one block table per sequence; every other step reads the
    logical view, so paging changes where rows live, not what is computed.
    """
    pool = np.asarray(pool)
    bt = np.asarray(block_table, dtype=np.int64)
    page_rows = pool.shape[1]
    j = np.arange(n)
    pages = bt[:, j // page_rows]                  # [B, n] physical page of each row
    return pool[pages, (j % page_rows)[None, :]]


def project_kv(h, w):
    """The decoder's global KV of one layer: h [rows, hidden] (the final
    encoder hidden state) times that layer's projection w [d, hidden]
    (row c: the weights of output column c), in fp64: out [rows, d].
    ["Unlocking...", Causal Encoder-Decoder (CED) Efficiency: the decoder
    derives its global KV cache from the final encoder hidden state using
    per-layer projections.]  Reading: a plain linear map, no bias."""
    return _f64(h) @ _f64(w).T


def project_quantize_fp4(h, w):
    """project_kv, then the FP4 main-KV quantiser (a1) of its rows."""
    return quantize_fp4(project_kv(h, w))


def dequantize_fp4(codes, scales, d):
    codes = np.ascontiguousarray(codes, dtype=np.uint8).reshape(-1, d // 2)
    scales = np.ascontiguousarray(scales, dtype=np.uint8).reshape(-1, d // 32)
    out = np.zeros((codes.shape[0], d), dtype=np.float64)
    lib().oracle_dequantize_fp4(_p(codes, _U8), _p(scales, _U8), codes.shape[0], d, _p(out, _D))
    return out


def cast_e4m3(x):
    x = _f64(x)
    out = np.zeros(x.shape, dtype=np.uint8)
    lib().oracle_cast_e4m3(_p(x, _D), x.size, _p(out, _U8))
    return out


def quantize_index_q(q, w):
    """q [nq, hi, di], w [nq, hi] -> (q8 uint8 [nq, hi, di], c float64 [nq, hi])."""
    q = _f64(q)
    w = _f64(w)
    nq, hi, di = q.shape
    q8 = np.zeros(q.shape, dtype=np.uint8)
    c = np.zeros((nq, hi), dtype=np.float64)
    lib().oracle_quantize_index_q(_p(q, _D), _p(w, _D), nq, hi, di, _p(q8, _U8), _p(c, _D))
    return q8, c


# ---- a3 / a4 / a5 ------------------------------------------------------------

def index_score(qv, c, kv, q_per_seq=1, n_valid=None):
    """qv [nq, hi, di], c [nq, hi], kv [B, n, di] (decoded values) -> [nq, n]."""
    qv, c, kv = _f64(qv), _f64(c), _f64(kv)
    nq, hi, di = qv.shape
    n = kv.shape[1]
    nvarr, nvp = _opt_i32(n_valid)
    out = np.zeros((nq, n), dtype=np.float64)
    lib().oracle_index_score(_p(qv, _D), _p(c, _D), _p(kv, _D), nq, q_per_seq, hi, di, n,
                             nvp, _p(out, _D))
    return out


def index_score_fp8(q, w, k8, q_per_seq=1, n_valid=None):
    """FP8 path: q [nq, hi, di] (bf16 values), w, k8 uint8 E4M3 [B, n, di]."""
    q8, c = quantize_index_q(q, w)
    return index_score(e4m3_decode(q8), c, e4m3_decode(k8), q_per_seq, n_valid)


def topk(scores, k, n_valid=None):
    scores = _f64(scores)
    rows, n = scores.shape
    nvarr, nvp = _opt_i32(n_valid)
    out = np.zeros((rows, k), dtype=np.int32)
    lib().oracle_topk(_p(scores, _D), rows, n, nvp, k, _p(out, _I32))
    return out


def sparse_attn(q, codes, scales, idx, window, scale, q_per_seq=1,
                win_start=None, win_len=None):
    """q [nq, hq, d]; codes [B, n, d/2]; scales [B, n, d/32]; idx [nq, k];
    window [B, w_rows, d] -> out float64 [nq, hq, d]."""
    q = _f64(q)
    nq, hq, d = q.shape
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    n = codes.shape[1]
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    k = idx.shape[1]
    window = _f64(window)
    w_rows = window.shape[1]
    ws, wsp = _opt_i32(win_start)
    wl, wlp = _opt_i32(win_len)
    out = np.zeros((nq, hq, d), dtype=np.float64)
    rc = lib().oracle_sparse_attn(_p(q, _D), nq, q_per_seq, hq, d, _p(codes, _U8),
                                  _p(scales, _U8), n, _p(idx, _I32), k, _p(window, _D),
                                  w_rows, wsp, wlp, float(scale), _p(out, _D))
    if rc != 0:
        raise ValueError(f"oracle_sparse_attn: bad arguments ({rc})")
    return out


# ---- a6: layer modes -----------------------------------------------------------

def default_sources(modes):
    """Resolve (kv_src, idx_src) for a static schedule of layer modes.

    [P3 "CSA2"]: Reindex uses the main KV and indexer K of the last Full
    layer; Reuse reuses the main KV and top-K indices of an earlier layer.
    Reading for Reuse: both come from the most recent Full layer.
    Raises ValueError for a schedule that has no Full layer before a
    Reindex or Reuse layer.
    """
    out = []
    last_full = -1
    for l, m in enumerate(modes):
        if m == FULL:
            last_full = l
            out.append((l, l))
        elif m in (REINDEX, REUSE):
            if last_full < 0:
                raise ValueError(f"layer {l}: no earlier Full layer")
            out.append((last_full, last_full if m == REUSE else l))
        else:
            raise ValueError(f"layer {l}: unknown mode {m}")
    return out


def default_plan(modes):
    """[(mode, kv_src, idx_src)] for a static schedule (see default_sources)."""
    return [(m, kv, ix) for m, (kv, ix) in zip(modes, default_sources(modes))]


def pool_restrict(scores, pool):
    """Scores of the entries outside each row's candidate pool set to -inf.

    [P5 Method; P3 "CSA2"] Hierarchical Sparse Indexer: an indexer restricted
    to a shared candidate pool chosen by an earlier indexer scores only the
    pool's entries.  Reading: an entry outside the pool is no candidate at all
    (its score is -inf, below every scored entry); pool rows hold entry
    indices, -1 for an empty slot.
    """
    scores = np.array(scores, dtype=np.float64)
    rows, n = scores.shape
    keep = np.zeros((rows, n), dtype=bool)
    for r in range(rows):
        p = pool[r][pool[r] >= 0]
        keep[r, p] = True
    scores[~keep] = -np.inf
    return scores


def block_summaries(k8, G):
    """Block-level representations of the indexer keys, the first level of
    the Hierarchical Sparse Indexer [P5 Method; P5 Related Work: hierarchical
    approaches score token-level entries and prune them on block-level
    representations].  Reading (the pages give no rule): the entries of each
    sequence form blocks of G consecutive entries; a block's key is the sum
    of its entries' decoded E4M3 keys divided by G (entries past the end of
    the sequence count as zero), cast back to E4M3 like any indexer key.
    k8 uint8 [B, n, di] -> uint8 [B, ceil(n / G), di]."""
    kv = e4m3_decode(np.asarray(k8, dtype=np.uint8))
    B, n, di = kv.shape
    nb = -(-n // G)
    padded = np.zeros((B, nb * G, di), dtype=np.float64)
    padded[:, :n] = kv
    return cast_e4m3(padded.reshape(B, nb, G, di).sum(axis=2) / G)


def block_pool(blocks, G, n):
    """The candidate pool of the chosen blocks: blocks int [rows, Bk]
    (ascending block indices, -1 padded) -> pool int32 [rows, Bk * G], the
    entries of block i in slots i*G .. i*G + G - 1 (ascending), -1 for a
    padded block or an entry past n."""
    blocks = np.asarray(blocks, dtype=np.int64)
    rows, bk = blocks.shape
    ent = blocks[:, :, None] * G + np.arange(G)[None, None, :]
    ok = (blocks[:, :, None] >= 0) & (ent < n)
    return np.where(ok, ent, -1).reshape(rows, bk * G).astype(np.int32)


def layer_stack(plan, layers, k, scale, q_per_seq=1, n_valid=None, pool=0, block=0,
                blocks_kept=0):
    """Run a static CSA2 schedule.

    plan: list of (mode, kv_src, idx_src).
    layers: list of dicts.  A Full layer holds its own cache 'codes',
    'scales' (FP4 main KV) and 'k8' (E4M3 indexer K).  Full and Reindex
    layers hold 'idx_q' and 'idx_w'; every layer holds 'attn_q' and
    'window'.  An optional 'k_f32' in place of 'k8' (and fp32 'idx_q')
    selects the fp32 indexer.
    pool > 0 runs the Hierarchical Sparse Indexer [P5 Method]: a Full layer's
    indexer, which scores every entry, also chooses the candidate pool, its
    top-`pool` entries (the same order as top-k); a Reindex layer scores only
    the pool of the Full layer whose KV it reads.  Readings: the pool is the
    earlier indexer's top-P under the top-k order; a Full layer's own top-k
    is unchanged (it lies inside its pool).
    block > 0 (with blocks_kept = Bk) runs the Hierarchical Sparse Indexer
    with block-level pruning first: a Full layer scores the block summaries
    of its indexer keys (block_summaries, blocks of `block` entries) with
    the same indexer formula, keeps its top-Bk blocks (the top-k order on
    block indices), and scores at token level only the entries of those
    blocks (block_pool), taking its top-k inside them; the Reindex layers
    that read its KV score the same pool.  Readings as for the pool, plus
    block_summaries.
    Returns (idx per layer, out per layer).
    """
    idx_of, out_of, pool_of = [], [], {}
    for l, (mode, kv_src, idx_src) in enumerate(plan):
        L = layers[l]
        src = layers[kv_src]
        if mode in (FULL, REINDEX):
            if "k8" in src:
                s = index_score_fp8(L["idx_q"], L["idx_w"], src["k8"], q_per_seq, n_valid)
            else:
                s = index_score(L["idx_q"], L["idx_w"], src["k_f32"], q_per_seq, n_valid)
            if block > 0 and mode == FULL:
                summ = block_summaries(src["k8"], block)
                sb = index_score_fp8(L["idx_q"], L["idx_w"], summ, q_per_seq)
                pool_of[l] = block_pool(topk(sb, blocks_kept), block, src["k8"].shape[1])
            elif pool > 0 and mode == FULL:
                pool_of[l] = topk(s, pool, n_valid)
            if (pool > 0 and mode == REINDEX) or block > 0:
                s = pool_restrict(s, pool_of[kv_src])
            idx = topk(s, k, n_valid)
        else:
            idx = idx_of[idx_src].copy()
        out = sparse_attn(L["attn_q"], src["codes"], src["scales"], idx, L["window"], scale,
                          q_per_seq)
        idx_of.append(idx)
        out_of.append(out)
    return idx_of, out_of
