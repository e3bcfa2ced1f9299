"""csa2_topk_noalloc through the C ABI, against the oracle and csa2_topk.

csa2_topk_noalloc serves callers that cannot allocate device memory (code
running inside an allocator callback, a plugin whose host owns every device
allocation, a process that must keep its footprint fixed after start-up):
its scratch is a fixed array inside the library.  It must select exactly what
the oracle's top-k selects on the same float32 scores, and what csa2_topk
selects -- indices are compared bit for bit, the tolerance the other top-k
tests use -- on two calls in a row (the second call must not see the first
call's leftovers in the shared array), and it must refuse a problem larger
than its fixed scratch.  This file is collected last so that a run stopping
at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from gpu_util import need_gpu
from long_context_sparse_27_b300 import synth

pytestmark = pytest.mark.gpu


def call_noalloc(csa2, scores, k, n_valid=None):
    rows, n = scores.shape
    out = torch.full((rows, k), -7, dtype=torch.int32, device=scores.device)
    st = csa2.lib.csa2_topk_noalloc(
        ctypes.c_void_p(scores.data_ptr()), rows, n, scores.stride(0),
        None if n_valid is None else ctypes.c_void_p(n_valid.data_ptr()), k,
        ctypes.c_void_p(out.data_ptr()), out.stride(0), None,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st, out


def test_noalloc_matches_topk_twice(orc):
    csa2 = need_gpu()
    # first call: the 1M-context decode shape (8 rows of 262144 scores)
    s1 = synth.scores_with_ties(8, 262144, seed=901).cuda()
    st, got1 = call_noalloc(csa2, s1, 512)
    assert st == 0
    ref1 = csa2.topk(s1, 512)
    torch.cuda.synchronize()
    assert np.array_equal(got1.cpu().numpy(), orc.topk(s1.cpu().double().numpy(), 512))
    assert torch.equal(got1, ref1)
    # second call: other scores, many ties and ragged visibility; the shared
    # scratch still holds the first call's histograms and candidates
    s2 = synth.scores_with_ties(20, 30000, seed=902, levels=50).cuda()
    nv = torch.randint(0, 30001, (20,), generator=torch.Generator().manual_seed(903)).int().cuda()
    st, got2 = call_noalloc(csa2, s2, 512, nv)
    assert st == 0
    ref2 = csa2.topk(s2, 512, n_valid=nv)
    torch.cuda.synchronize()
    assert np.array_equal(got2.cpu().numpy(),
                          orc.topk(s2.cpu().double().numpy(), 512, nv.cpu().numpy()))
    assert torch.equal(got2, ref2)
    assert not np.array_equal(got1.cpu().numpy()[:1], got2.cpu().numpy()[:1])


def test_noalloc_refuses_oversized_problem():
    csa2 = need_gpu()
    k = 512
    per_row = csa2.topk_workspace_bytes(1, 1000, k)
    rows = (4 << 20) // per_row + 1  # one row more than the fixed scratch holds
    s = torch.zeros(rows, 1000, device="cuda")
    st, out = call_noalloc(csa2, s, k)
    torch.cuda.synchronize()
    assert st == 5  # CSA2_ERR_WORKSPACE
    assert int((out != -7).sum()) == 0  # nothing was enqueued
    st, _ = call_noalloc(csa2, s[: rows - 1], k)
    assert st == 0
