"""Python binding of libcsa2 (include/csa2.h): argument marshalling only.

Every function takes torch CUDA tensors, passes their device pointers and
the current CUDA stream to the C ABI, and raises Csa2Error on a non-zero
status.  Output tensors are allocated with torch when not given (torch is
used for device memory and streams only; all arithmetic runs in the
library's kernels).  There is no fallback: if libcsa2.so is missing or
fails to load, importing this module raises.
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcsa2.so")

F32, BF16, E4M3 = 0, 1, 2
FULL, REINDEX, REUSE = 0, 1, 2
DEVFLAG_TIMEOUT, DEVFLAG_BOUNDS, DEVFLAG_CAPACITY = 0x1, 0x2, 0x4

_c_i32, _c_i64, _c_p, _c_f, _c_sz = (ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p,
                                     ctypes.c_float, ctypes.c_size_t)


class Pages(ctypes.Structure):
    """csa2_pages: a paged cache's block table (block_table None = not paged)."""
    _fields_ = [("block_table", _c_p), ("bt_ld", _c_i64), ("page_rows", _c_i32),
                ("num_pages", _c_i32)]


def pages(block_table=None, page_rows=0, num_pages=0):
    """csa2_pages of a block table int32 [B, pages per sequence] (or none)."""
    if block_table is None:
        return Pages()
    if block_table.dtype != torch.int32 or block_table.stride(1) != 1:
        raise ValueError("pages: the block table must be int32 with contiguous rows")
    return Pages(block_table=block_table.data_ptr(), bt_ld=block_table.stride(0),
                 page_rows=page_rows, num_pages=num_pages)


class QuantArgs(ctypes.Structure):
    _fields_ = [("x", _c_p), ("rows", _c_i64), ("d", _c_i32), ("x_ld", _c_i64),
                ("codes", _c_p), ("codes_ld", _c_i64), ("scales", _c_p), ("scales_ld", _c_i64),
                ("idxk", _c_p), ("di", _c_i32), ("idxk_ld", _c_i64), ("idxk_e4m3", _c_p),
                ("idxk_e4m3_ld", _c_i64), ("pages", Pages), ("rows_per_seq", _c_i64),
                ("entry0", _c_i64)]


class IndexArgs(ctypes.Structure):
    _fields_ = [("q", _c_p), ("q_dtype", _c_i32), ("w", _c_p), ("k", _c_p), ("k_dtype", _c_i32),
                ("B", _c_i64), ("q_per_seq", _c_i64), ("hi", _c_i32), ("di", _c_i32),
                ("n", _c_i64), ("k_ld", _c_i64), ("k_seq_stride", _c_i64), ("n_valid", _c_p),
                ("scores", _c_p), ("scores_ld", _c_i64), ("workspace", _c_p),
                ("workspace_bytes", _c_sz), ("dev_status", _c_p), ("pages", Pages)]


class AttnArgs(ctypes.Structure):
    _fields_ = [("q", _c_p), ("q_dtype", _c_i32), ("nq", _c_i64), ("q_per_seq", _c_i64),
                ("hq", _c_i32), ("d", _c_i32), ("codes", _c_p), ("scales", _c_p), ("n", _c_i64),
                ("codes_ld", _c_i64), ("codes_seq_stride", _c_i64), ("scales_ld", _c_i64),
                ("scales_seq_stride", _c_i64), ("idx", _c_p), ("k", _c_i32), ("idx_ld", _c_i64),
                ("window", _c_p), ("w_rows", _c_i32), ("win_ld", _c_i64),
                ("win_seq_stride", _c_i64), ("win_start", _c_p), ("win_len", _c_p),
                ("win_max", _c_i32), ("softmax_scale", _c_f), ("out", _c_p), ("workspace", _c_p),
                ("workspace_bytes", _c_sz), ("dev_status", _c_p), ("pages", Pages)]


class LayerDesc(ctypes.Structure):
    _fields_ = [("mode", _c_i32), ("kv_src", _c_i32), ("idx_src", _c_i32), ("new_kv", _c_p),
                ("new_idxk", _c_p), ("new_row", _c_i64), ("new_rows", _c_i64), ("idx_q", _c_p),
                ("idx_w", _c_p),
                ("attn_q", _c_p), ("window", _c_p), ("codes", _c_p), ("scales", _c_p),
                ("idxk", _c_p), ("topk_idx", _c_p), ("out", _c_p), ("block_keys", _c_p)]


class ProjectArgs(ctypes.Structure):
    _fields_ = [("h", _c_p), ("w", _c_p), ("rows", _c_i64), ("hidden", _c_i32), ("d", _c_i32),
                ("h_ld", _c_i64), ("w_ld", _c_i64), ("codes", _c_p), ("codes_ld", _c_i64),
                ("scales", _c_p), ("scales_ld", _c_i64), ("out", _c_p), ("out_ld", _c_i64),
                ("dev_status", _c_p)]


class StackArgs(ctypes.Structure):
    _fields_ = [("B", _c_i64), ("q_per_seq", _c_i64), ("n", _c_i64), ("hi", _c_i32),
                ("di", _c_i32), ("hq", _c_i32), ("d", _c_i32), ("k", _c_i32), ("w_rows", _c_i32),
                ("idx_q_dtype", _c_i32), ("idx_k_dtype", _c_i32), ("attn_q_dtype", _c_i32),
                ("n_valid", _c_p), ("win_start", _c_p), ("win_len", _c_p),
                ("softmax_scale", _c_f), ("workspace", _c_p), ("workspace_bytes", _c_sz),
                ("dev_status", _c_p), ("pool", _c_i32), ("win_max", _c_i32),
                ("pages", Pages), ("block", _c_i32), ("blocks_kept", _c_i32)]


EXPORTS = {
    "csa2_version": (ctypes.c_char_p, []),
    "csa2_status_string": (ctypes.c_char_p, [_c_i32]),
    "csa2_last_cuda_error": (_c_i32, []),
    "csa2_status_from_device": (_c_i32, [_c_i32]),
    "csa2_quantize_fp4": (_c_i32, [ctypes.POINTER(QuantArgs), _c_p]),
    "csa2_quantize_index_q": (_c_i32, [_c_p, _c_p, _c_i64, _c_i32, _c_i32, _c_p, _c_p, _c_p]),
    "csa2_index_score_workspace_bytes": (_c_sz, [ctypes.POINTER(IndexArgs)]),
    "csa2_index_score": (_c_i32, [ctypes.POINTER(IndexArgs), _c_p]),
    "csa2_index_score_pool": (_c_i32, [ctypes.POINTER(IndexArgs), _c_p, _c_i64, _c_i32, _c_p]),
    "csa2_index_candidates": (_c_i32, [ctypes.POINTER(IndexArgs), _c_p, _c_p, _c_p, _c_i64,
                                       _c_p]),
    "csa2_project_fp4": (_c_i32, [ctypes.POINTER(ProjectArgs), _c_p]),
    "csa2_index_block_keys": (_c_i32, [_c_p, _c_i64, _c_i64, _c_i64, _c_i64,
                                       ctypes.POINTER(Pages), _c_i32, _c_i64, _c_i64, _c_p,
                                       _c_i64, _c_i64, _c_p, _c_p]),
    "csa2_topk_workspace_bytes": (_c_sz, [_c_i64, _c_i64, _c_i32]),
    "csa2_topk": (_c_i32, [_c_p, _c_i64, _c_i64, _c_i64, _c_p, _c_i32, _c_p, _c_i64, _c_p, _c_sz,
                           _c_p, _c_p]),
    "csa2_topk_noalloc": (_c_i32, [_c_p, _c_i64, _c_i64, _c_i64, _c_p, _c_i32, _c_p, _c_i64,
                                   _c_p, _c_p]),
    "csa2_sparse_attn_workspace_bytes": (_c_sz, [ctypes.POINTER(AttnArgs)]),
    "csa2_sparse_attn": (_c_i32, [ctypes.POINTER(AttnArgs), _c_p]),
    "csa2_validate_plan": (_c_i32, [ctypes.POINTER(LayerDesc), _c_i32, ctypes.POINTER(_c_i32)]),
    "csa2_layer_stack_workspace_bytes": (_c_sz, [ctypes.POINTER(StackArgs)]),
    "csa2_layer_stack": (_c_i32, [ctypes.POINTER(LayerDesc), _c_i32, ctypes.POINTER(StackArgs),
                                  _c_p]),
}


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libcsa2.so not built ({LIB_PATH}); run "
                          "python -m long_context_sparse_27_b300.build")
    L = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in EXPORTS.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    return L


lib = _load()


class Csa2Error(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        msg = lib.csa2_status_string(status).decode()
        if status == 4:
            msg += f" (cudaError {lib.csa2_last_cuda_error()})"
        super().__init__(f"{where}: {msg}")


def _check(st, where):
    if st != 0:
        raise Csa2Error(st, where)


def version():
    return lib.csa2_version().decode()


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _dtype_code(t):
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype in (torch.uint8, torch.float8_e4m3fn):
        return E4M3
    raise TypeError(f"unsupported dtype {t.dtype}")


def _workspace(nbytes, device):
    # 256-byte aligned scratch from torch's allocator
    return torch.empty(max(int(nbytes), 1) + 256, dtype=torch.uint8, device=device)


def _aligned_ptr(ws):
    p = ws.data_ptr()
    return (p + 255) & ~255


# ---- a1 / a2 ----------------------------------------------------------------

def quantize_fp4(x, codes=None, scales=None, idxk=None, idxk_e4m3=None, pages=None,
                 rows_per_seq=1, entry0=0):
    """x bf16 [rows, d] -> codes u8 [rows, d/2], scales u8 [rows, d/32];
    optional idxk bf16 [rows, di] -> idxk_e4m3 u8 [rows, di].  Row strides
    of the given tensors are honoured (views into a cache work).  pages (a
    Pages): codes / scales / idxk_e4m3 are page pools and row r goes to
    entry entry0 + r % rows_per_seq of sequence r // rows_per_seq."""
    rows, d = x.shape
    dev = x.device
    if codes is None:
        codes = torch.empty(rows, d // 2, dtype=torch.uint8, device=dev)
    if scales is None:
        scales = torch.empty(rows, d // 32, dtype=torch.uint8, device=dev)
    a = QuantArgs(x=_ptr(x), rows=rows, d=d, x_ld=x.stride(0), codes=_ptr(codes),
                  codes_ld=codes.stride(0), scales=_ptr(scales), scales_ld=scales.stride(0))
    if pages is not None:
        a.pages, a.rows_per_seq, a.entry0 = pages, rows_per_seq, entry0
    if idxk is not None:
        if idxk_e4m3 is None:
            idxk_e4m3 = torch.empty(rows, idxk.shape[1], dtype=torch.uint8, device=dev)
        a.idxk, a.di, a.idxk_ld = _ptr(idxk), idxk.shape[1], idxk.stride(0)
        a.idxk_e4m3, a.idxk_e4m3_ld = _ptr(idxk_e4m3), idxk_e4m3.stride(0)
    _check(lib.csa2_quantize_fp4(ctypes.byref(a), _stream()), "csa2_quantize_fp4")
    return (codes, scales) if idxk is None else (codes, scales, idxk_e4m3)


def quantize_index_q(q, w, q8=None, c=None):
    nq, hi, di = q.shape
    if q8 is None:
        q8 = torch.empty(nq, hi, di, dtype=torch.uint8, device=q.device)
    if c is None:
        c = torch.empty(nq, hi, dtype=torch.float32, device=q.device)
    _check(lib.csa2_quantize_index_q(_ptr(q), _ptr(w), nq, hi, di, _ptr(q8), _ptr(c), _stream()),
           "csa2_quantize_index_q")
    return q8, c


# ---- a3 ----------------------------------------------------------------------

def index_args(q, w, k, q_per_seq=1, n_valid=None, scores=None, dev_status=None, pages=None,
               n=None):
    """q: f32, bf16, or uint8 / float8_e4m3fn (already quantised; w = c).
    k [B, n, di]; or, with pages, the pool [rows, di] and n given."""
    nq, hi, di = q.shape
    if pages is None:
        B, n = k.shape[0], k.shape[1]
        k_ld, k_seq = k.stride(1), k.stride(0)
    else:
        B, k_ld, k_seq = nq // q_per_seq, k.stride(0), 0
    a = IndexArgs(q=_ptr(q), q_dtype=_dtype_code(q), w=_ptr(w), k=_ptr(k),
                  k_dtype=_dtype_code(k), B=B, q_per_seq=q_per_seq, hi=hi, di=di, n=n,
                  k_ld=k_ld, k_seq_stride=k_seq, n_valid=_ptr(n_valid),
                  scores=_ptr(scores), scores_ld=(scores.stride(0) if scores is not None else n),
                  dev_status=_ptr(dev_status))
    if pages is not None:
        a.pages = pages
    return a


def index_score(q, w, k, q_per_seq=1, n_valid=None, scores=None, dev_status=None, pages=None,
                n=None):
    """q [nq, hi, di] (f32 with f32 k, or bf16 with E4M3 k as uint8),
    w f32 [nq, hi], k [B, n, di] -> scores f32 [nq, n].  pages: k is a page
    pool [rows, di] and n the entries per sequence."""
    nq = q.shape[0]
    n = k.shape[1] if pages is None else n
    if scores is None:
        scores = torch.empty(nq, n, dtype=torch.float32, device=q.device)
    a = index_args(q, w, k, q_per_seq, n_valid, scores, dev_status, pages, n)
    need = lib.csa2_index_score_workspace_bytes(ctypes.byref(a))
    ws = _workspace(need, q.device) if need else None
    if ws is not None:
        a.workspace, a.workspace_bytes = _aligned_ptr(ws), need
    _check(lib.csa2_index_score(ctypes.byref(a), _stream()), "csa2_index_score")
    return scores


def index_score_pool(q, w, k, pool, q_per_seq=1, scores=None, dev_status=None, pages=None,
                     n=None):
    """The Hierarchical Sparse Indexer's restricted scoring: q bf16 [nq, 64,
    128] (or its E4M3 quantisation with w = c), w f32 [nq, 64], k E4M3 [B, n,
    128] as uint8, pool int32 [nq, P] (entry indices, -1 = empty slot) ->
    scores f32 [nq, P] (-inf at empty slots)."""
    nq, P = pool.shape
    if pool.stride(1) != 1:
        raise ValueError("index_score_pool: rows of pool must be contiguous")
    if scores is None:
        scores = torch.empty(nq, P, dtype=torch.float32, device=q.device)
    a = index_args(q, w, k, q_per_seq, None, scores, dev_status, pages, n)
    need = lib.csa2_index_score_workspace_bytes(ctypes.byref(a))
    ws = _workspace(need, q.device) if need else None
    if ws is not None:
        a.workspace, a.workspace_bytes = _aligned_ptr(ws), need
    _check(lib.csa2_index_score_pool(ctypes.byref(a), _ptr(pool), pool.stride(0), P, _stream()),
           "csa2_index_score_pool")
    return scores


def index_candidates(q, w, k, theta, cand_cap, q_per_seq, n_valid=None, cand=None,
                     cand_cnt=None, dev_status=None, pages=None, n=None):
    """The prefill chunk's scoring pass that stores no scores: q [nq, 64, 128]
    (bf16, or its E4M3 quantisation with w = c), k E4M3 [B, n, 128] as uint8,
    theta uint32 [nq] (order-preserving keys, as int32) -> (cand int64 [nq,
    cand_cap]: key | entry << 32, cand_cnt int32 [nq]: slots reserved)."""
    nq = q.shape[0]
    n = k.shape[1] if pages is None else n
    if theta.dtype != torch.int32 or theta.numel() != nq:
        raise ValueError("index_candidates: theta must be int32 [nq]")
    if cand is None:
        cand = torch.empty(nq, cand_cap, dtype=torch.int64, device=q.device)
    if cand_cnt is None:
        cand_cnt = torch.zeros(nq, dtype=torch.int32, device=q.device)
    a = index_args(q, w, k, q_per_seq, n_valid, None, dev_status, pages, n)
    need = lib.csa2_index_score_workspace_bytes(ctypes.byref(a))
    ws = _workspace(need, q.device) if need else None
    if ws is not None:
        a.workspace, a.workspace_bytes = _aligned_ptr(ws), need
    _check(lib.csa2_index_candidates(ctypes.byref(a), _ptr(theta), _ptr(cand_cnt), _ptr(cand),
                                     cand_cap, _stream()), "csa2_index_candidates")
    return cand, cand_cnt


def project_fp4(h, w, with_out=False, dev_status=None):
    """The decoder's global KV of one layer: h bf16 [rows, hidden] (final
    encoder hidden state), w bf16 [d, hidden] (the layer's projection, one
    row per output column) -> (codes u8 [rows, d/2], scales u8 [rows, d/32],
    out f32 [rows, d] or None)."""
    rows, hidden = h.shape
    d = w.shape[0]
    if h.stride(1) != 1 or w.stride(1) != 1:
        raise ValueError("project_fp4: rows of h and w must be contiguous")
    codes = torch.empty(rows, d // 2, dtype=torch.uint8, device=h.device)
    scales = torch.empty(rows, d // 32, dtype=torch.uint8, device=h.device)
    out = torch.empty(rows, d, dtype=torch.float32, device=h.device) if with_out else None
    a = ProjectArgs(h=_ptr(h), w=_ptr(w), rows=rows, hidden=hidden, d=d, h_ld=h.stride(0),
                    w_ld=w.stride(0), codes=_ptr(codes), codes_ld=codes.stride(0),
                    scales=_ptr(scales), scales_ld=scales.stride(0), out=_ptr(out),
                    out_ld=(out.stride(0) if out is not None else 0),
                    dev_status=_ptr(dev_status))
    _check(lib.csa2_project_fp4(ctypes.byref(a), _stream()), "csa2_project_fp4")
    return codes, scales, out


def index_block_keys(k8, G, n=None, pages=None, B=None, blk0=0, nblk=None, out=None,
                     dev_status=None):
    """Block keys of the Hierarchical Sparse Indexer: k8 E4M3 [B, n, 128] as
    uint8 (or, with pages, the pool [rows, 128] and B, n given) -> uint8
    [B, ceil(n / G), 128]; blocks blk0 .. blk0 + nblk - 1 are computed."""
    if pages is None:
        B, n = k8.shape[0], k8.shape[1]
        k_ld, k_seq = k8.stride(1), k8.stride(0)
    else:
        k_ld, k_seq = k8.stride(0), 0
    nb = -(-n // G)
    if out is None:
        out = torch.zeros(B, nb, 128, dtype=torch.uint8, device=k8.device)
    nblk = nb - blk0 if nblk is None else nblk
    _check(lib.csa2_index_block_keys(_ptr(k8), B, n, k_ld, k_seq,
                                     ctypes.byref(pages if pages is not None else Pages()), G,
                                     blk0, nblk, _ptr(out), out.stride(1), out.stride(0),
                                     _ptr(dev_status), _stream()), "csa2_index_block_keys")
    return out


# ---- a4 ----------------------------------------------------------------------

def topk_workspace_bytes(rows, n, k):
    return lib.csa2_topk_workspace_bytes(rows, n, k)


def _check_topk_tensors(where, scores, out, n_valid):
    # the C ABI takes one row stride per tensor: rows must be contiguous
    if scores.dtype != torch.float32 or scores.stride(1) != 1:
        raise ValueError(f"{where}: scores must be float32 with contiguous rows")
    if out.dtype != torch.int32 or out.stride(1) != 1:
        raise ValueError(f"{where}: out must be int32 with contiguous rows")
    if n_valid is not None and (n_valid.dtype != torch.int32 or not n_valid.is_contiguous()):
        raise ValueError(f"{where}: n_valid must be a contiguous int32 tensor")


def topk(scores, k, n_valid=None, out=None, workspace=None, dev_status=None):
    """scores f32 [rows, n] -> int32 [rows, k], ascending indices, -1 padded."""
    rows, n = scores.shape
    if out is None:
        out = torch.empty(rows, k, dtype=torch.int32, device=scores.device)
    _check_topk_tensors("topk", scores, out, n_valid)
    need = lib.csa2_topk_workspace_bytes(rows, n, k)
    ws = workspace if workspace is not None else _workspace(need, scores.device)
    _check(lib.csa2_topk(_ptr(scores), rows, n, scores.stride(0), _ptr(n_valid), k, _ptr(out),
                         out.stride(0), _aligned_ptr(ws), need, _ptr(dev_status), _stream()),
           "csa2_topk")
    return out


def topk_noalloc(scores, k, n_valid=None, out=None, dev_status=None):
    """As topk(), for callers that cannot allocate device memory: the scratch
    is a fixed array inside the library (see csa2_topk_noalloc); only `out`
    is allocated here when not given."""
    rows, n = scores.shape
    if out is None:
        out = torch.empty(rows, k, dtype=torch.int32, device=scores.device)
    _check_topk_tensors("topk_noalloc", scores, out, n_valid)
    _check(lib.csa2_topk_noalloc(_ptr(scores), rows, n, scores.stride(0), _ptr(n_valid), k,
                                 _ptr(out), out.stride(0), _ptr(dev_status), _stream()),
           "csa2_topk_noalloc")
    return out


# ---- a5 ----------------------------------------------------------------------

def attn_args(q, codes, scales, idx, window, softmax_scale, q_per_seq=1, win_start=None,
              win_len=None, win_max=0, out=None, dev_status=None, pages=None, n=None):
    nq, hq, d = q.shape
    if pages is None:
        n = codes.shape[1]
        c_ld, c_seq, s_ld, s_seq = codes.stride(1), codes.stride(0), scales.stride(1), \
            scales.stride(0)
    else:
        c_ld, c_seq, s_ld, s_seq = codes.stride(0), 0, scales.stride(0), 0
    a = AttnArgs(q=_ptr(q), q_dtype=_dtype_code(q), nq=nq, q_per_seq=q_per_seq, hq=hq, d=d,
                 codes=_ptr(codes), scales=_ptr(scales), n=n,
                 codes_ld=c_ld, codes_seq_stride=c_seq, scales_ld=s_ld, scales_seq_stride=s_seq,
                 idx=_ptr(idx), k=idx.shape[1], idx_ld=idx.stride(0), window=_ptr(window),
                 w_rows=window.shape[1], win_ld=window.stride(1),
                 win_seq_stride=window.stride(0), win_start=_ptr(win_start),
                 win_len=_ptr(win_len), win_max=win_max, softmax_scale=softmax_scale,
                 out=_ptr(out), dev_status=_ptr(dev_status))
    if pages is not None:
        a.pages = pages
    return a


def sparse_attn(q, codes, scales, idx, window, softmax_scale, q_per_seq=1, win_start=None,
                win_len=None, win_max=0, out=None, dev_status=None, pages=None, n=None):
    """q [nq, hq, d] f32 or bf16; codes u8 [B, n, d/2]; scales u8 [B, n, d/32];
    idx int32 [nq, k]; window bf16 [B, w_rows, d] -> out f32 [nq, hq, d].
    pages: codes / scales are page pools [rows, d/2] / [rows, d/32] and n
    the entries per sequence."""
    nq, hq, d = q.shape
    if out is None:
        out = torch.empty(nq, hq, d, dtype=torch.float32, device=q.device)
    a = attn_args(q, codes, scales, idx, window, softmax_scale, q_per_seq, win_start, win_len,
                  win_max, out, dev_status, pages, n)
    need = lib.csa2_sparse_attn_workspace_bytes(ctypes.byref(a))
    ws = _workspace(need, q.device) if need else None
    if ws is not None:
        a.workspace, a.workspace_bytes = _aligned_ptr(ws), need
    _check(lib.csa2_sparse_attn(ctypes.byref(a), _stream()), "csa2_sparse_attn")
    return out


# ---- a6 ----------------------------------------------------------------------

_DESC_KEYS = ("new_kv", "new_idxk", "idx_q", "idx_w", "attn_q", "window", "codes", "scales",
              "idxk", "topk_idx", "out", "block_keys")


def layer_descs(layers):
    """layers: list of dicts with 'mode', 'kv_src', 'idx_src', 'new_row' and
    tensors under the names of csa2_layer_desc's fields."""
    arr = (LayerDesc * len(layers))()
    for i, L in enumerate(layers):
        arr[i].mode, arr[i].kv_src, arr[i].idx_src = L["mode"], L["kv_src"], L["idx_src"]
        arr[i].new_row = L.get("new_row", 0)
        arr[i].new_rows = L.get("new_rows", 0)
        for key in _DESC_KEYS:
            setattr(arr[i], key, _ptr(L.get(key)))
    return arr


def validate_plan(layers):
    """Returns (status, first bad layer or -1)."""
    arr = layer_descs(layers)
    bad = _c_i32(-1)
    st = lib.csa2_validate_plan(arr, len(layers), ctypes.byref(bad))
    return st, bad.value


def stack_args(B, q_per_seq, n, hi, di, hq, d, k, w_rows, idx_q_dtype, idx_k_dtype,
               attn_q_dtype, softmax_scale, n_valid=None, win_start=None, win_len=None,
               dev_status=None, pool=0, win_max=0, pages=None, block=0, blocks_kept=0):
    a = StackArgs(B=B, q_per_seq=q_per_seq, n=n, hi=hi, di=di, hq=hq, d=d, k=k,
                  w_rows=w_rows, idx_q_dtype=idx_q_dtype, idx_k_dtype=idx_k_dtype,
                  attn_q_dtype=attn_q_dtype, n_valid=_ptr(n_valid),
                  win_start=_ptr(win_start), win_len=_ptr(win_len),
                  softmax_scale=softmax_scale, dev_status=_ptr(dev_status), pool=pool,
                  win_max=win_max, block=block, blocks_kept=blocks_kept)
    if pages is not None:
        a.pages = pages
    return a


def layer_stack_workspace_bytes(sargs):
    return lib.csa2_layer_stack_workspace_bytes(ctypes.byref(sargs))


def layer_stack(descs, sargs, workspace):
    """Enqueue one step of the layer schedule on the current stream.
    descs: a LayerDesc array (layer_descs); sargs: StackArgs; workspace: a
    uint8 CUDA tensor of at least layer_stack_workspace_bytes(sargs) + 256."""
    need = lib.csa2_layer_stack_workspace_bytes(ctypes.byref(sargs))
    sargs.workspace, sargs.workspace_bytes = _aligned_ptr(workspace), need
    _check(lib.csa2_layer_stack(descs, len(descs), ctypes.byref(sargs), _stream()),
           "csa2_layer_stack")
