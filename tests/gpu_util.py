"""Helpers shared by the GPU parity tests: device checks, comparisons."""
import numpy as np
import pytest
import torch


def need_gpu():
    if not torch.cuda.is_available():
        pytest.fail("GPU test selected but no CUDA device is visible")
    from long_context_sparse_27_b300 import csa2  # raises if libcsa2.so is missing
    return csa2


def f64(t):
    """Exact float64 copy of a bf16 / fp32 tensor, as numpy."""
    return t.detach().cpu().double().numpy()


def score_close(gpu, ref, rtol=1e-3, floor_frac=1e-2):
    """|g - o| <= rtol * max(|o|, floor_frac * max_j |o|) per row; -inf must
    match -inf exactly.  Returns the worst ratio (<= 1 passes)."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    ninf = np.isneginf(ref)
    assert np.array_equal(np.isneginf(gpu), ninf), "masked entries differ"
    g = np.where(ninf, 0.0, gpu)
    o = np.where(ninf, 0.0, ref)
    rowmax = np.abs(o).max(axis=1, keepdims=True)
    tol = rtol * np.maximum(np.abs(o), floor_frac * rowmax)
    tol = np.where(tol == 0, 1e-30, tol)
    return float((np.abs(g - o) / tol).max())


def rel_l2(gpu, ref):
    """max over (query, head) of ||g - o|| / ||o||."""
    g = np.asarray(gpu, dtype=np.float64)
    o = np.asarray(ref, dtype=np.float64)
    num = np.sqrt(((g - o) ** 2).sum(-1))
    den = np.sqrt((o ** 2).sum(-1))
    den = np.where(den == 0, 1.0, den)
    return float((num / den).max())


def recall(gpu_idx, ref_idx):
    g = np.asarray(gpu_idx)
    r = np.asarray(ref_idx)
    hit = tot = 0
    for a, b in zip(g, r):
        sb = set(int(x) for x in b if x >= 0)
        sa = set(int(x) for x in a if x >= 0)
        hit += len(sa & sb)
        tot += len(sb)
    return hit / max(tot, 1)


def topk_valid(scores_row, sel, k, nv):
    """The selection is a valid top-k of scores_row[:nv] under (score desc,
    index asc), written ascending and padded with -1."""
    s = np.asarray(scores_row[:nv], dtype=np.float64)
    sel = np.asarray(sel)
    m = min(k, nv)
    if not (np.all(sel[m:] == -1) and np.all(np.diff(sel[:m]) > 0)):
        return False
    chosen = sel[:m]
    if m == 0:
        return True
    if chosen.min() < 0 or chosen.max() >= nv:
        return False
    mask = np.zeros(nv, bool)
    mask[chosen] = True
    if m == nv:
        return True
    lo = s[mask].min()
    hi = s[~mask].max()
    if lo > hi:
        return True
    if lo < hi:
        return False
    # equal at the boundary: chosen equal-score entries must precede unchosen ones
    eq_chosen = np.where(mask & (s == lo))[0]
    eq_rest = np.where(~mask & (s == lo))[0]
    return eq_chosen.max() < eq_rest.min()
