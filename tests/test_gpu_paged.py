"""Paged caches (the serving layout) on the GPU, through the C ABI.

Entry j of sequence b lives in row j % page_rows of page block_table[b, j //
page_rows] of one shared pool (reading of "Unlocking Extreme Context Scaling
with DeepSeek-V4.1-Flash", Deployment and Infrastructure: serving stacks run
the model; the pages give no layout).  Paging changes where rows live, not
what is computed, so every step over a paged pool must give, bit for bit,
what it gives over the contiguous cache holding the same rows (the oracle's
gather_pages view); a small layer stack is also checked against the fp64
oracle through that view.  Block tables are seeded permutations with spare
pages that no sequence uses.
"""
import math

import numpy as np
import pytest
import torch

from gpu_util import f64, need_gpu, recall, rel_l2, score_close
from long_context_sparse_27_b300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def csa2():
    return need_gpu()


def dev(t):
    return t.to("cuda")


def to_pool(contig, bt, page_rows, num_pages):
    """The pool holding contiguous rows [B, n, ...] at the block table's
    pages (unused rows hold a junk byte pattern)."""
    B, n = contig.shape[:2]
    pool = torch.full((num_pages * page_rows,) + tuple(contig.shape[2:]), 0x5A,
                      dtype=contig.dtype, device=contig.device)
    j = torch.arange(n, device=contig.device)
    for b in range(B):
        rows = bt[b, j // page_rows].long() * page_rows + j % page_rows
        pool[rows] = contig[b]
    return pool


def paged(csa2, B, n, page_rows, seed):
    bt, num_pages = synth.block_table(B, n, page_rows, seed, "cuda")
    return bt, num_pages, csa2.pages(bt, page_rows, num_pages)


@pytest.mark.parametrize("B,n,page_rows", [(3, 1000, 64), (2, 4096, 256), (8, 262144, 256),
                                           (1, 200, 128)])
def test_paged_index_score_equals_contiguous(csa2, orc, B, n, page_rows):
    wl = synth.scaled(synth.C128K, B=B, N=n)
    q = synth.index_q(wl, 300 + n, "cuda")
    w = synth.index_w(wl, 301 + n, "cuda")
    k8 = torch.randint(0, 0x7F, (B, n, 128), dtype=torch.uint8, device="cuda",
                       generator=torch.Generator(device="cuda").manual_seed(302 + n))
    bt, num_pages, pg = paged(csa2, B, n, page_rows, 303 + n)
    pool = to_pool(k8, bt, page_rows, num_pages)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = csa2.index_score(q, w, pool, pages=pg, n=n, dev_status=st)
    ref = csa2.index_score(q, w, k8)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(got.view(torch.int32), ref.view(torch.int32))
    if n <= 4096:  # and the fp64 oracle through the logical view of the pool
        view = orc.gather_pages(pool.cpu().numpy().reshape(num_pages, page_rows, 128),
                                bt.cpu().numpy(), n)
        o = orc.index_score_fp8(f64(q), f64(w), view)
        assert score_close(got.cpu().numpy(), o) <= 1.0


def test_paged_prefill_index_score_equals_contiguous(csa2):
    # a prefill chunk (4 queries per MMA group) with causal visibility
    T, n, page_rows = 16, 1500, 64
    wl = synth.scaled(synth.PREFILL, q_per_seq=T, N=n, pos0=4 * n - T)
    q = synth.index_q(wl, 310, "cuda")
    w = synth.index_w(wl, 311, "cuda")
    nv = synth.prefill_n_valid(wl, "cuda")
    k8 = torch.randint(0, 0x7F, (1, n, 128), dtype=torch.uint8, device="cuda",
                       generator=torch.Generator(device="cuda").manual_seed(312))
    bt, num_pages, pg = paged(csa2, 1, n, page_rows, 313)
    pool = to_pool(k8, bt, page_rows, num_pages)
    got = csa2.index_score(q, w, pool, q_per_seq=T, n_valid=nv, pages=pg, n=n)
    ref = csa2.index_score(q, w, k8, q_per_seq=T, n_valid=nv)
    torch.cuda.synchronize()
    assert torch.equal(got.view(torch.int32), ref.view(torch.int32))


def test_paged_f32_index_score_equals_contiguous(csa2):
    wl = synth.scaled(synth.TINY, B=2, N=700)
    q = synth.index_q(wl, 320, "cuda")
    w = synth.index_w(wl, 321, "cuda")
    k = synth.index_k_rows(wl, 322, "cuda")
    bt, num_pages, pg = paged(csa2, 2, 700, 64, 323)
    pool = to_pool(k, bt, 64, num_pages)
    got = csa2.index_score(q, w, pool, pages=pg, n=700)
    ref = csa2.index_score(q, w, k)
    torch.cuda.synchronize()
    assert torch.equal(got.view(torch.int32), ref.view(torch.int32))


def test_paged_pool_score_equals_contiguous(csa2):
    B, n, P, page_rows = 3, 5000, 700, 128
    wl = synth.scaled(synth.C128K, B=B, N=n)
    q = synth.index_q(wl, 330, "cuda")
    w = synth.index_w(wl, 331, "cuda")
    k8 = torch.randint(0, 0x7F, (B, n, 128), dtype=torch.uint8, device="cuda",
                       generator=torch.Generator(device="cuda").manual_seed(332))
    pool_idx = synth.random_indices(B, P, n, 333, pad=9).cuda()
    bt, num_pages, pg = paged(csa2, B, n, page_rows, 334)
    kpool = to_pool(k8, bt, page_rows, num_pages)
    got = csa2.index_score_pool(q, w, kpool, pool_idx, pages=pg, n=n)
    ref = csa2.index_score_pool(q, w, k8, pool_idx)
    torch.cuda.synchronize()
    assert torch.equal(got.view(torch.int32), ref.view(torch.int32))


@pytest.mark.parametrize("nq,n,k,W,page_rows", [(3, 2000, 512, 128, 64), (2, 3000, 1024, 128, 256)])
def test_paged_attention_equals_contiguous(csa2, orc, nq, n, k, W, page_rows):
    d, hq = 512, 64
    x = synth.normal((nq * n, d), 340 + n)
    codes, scales = csa2.quantize_fp4(dev(x))
    codes, scales = codes.reshape(nq, n, d // 2), scales.reshape(nq, n, d // 32)
    q = dev(synth.normal((nq, hq, d), 341))
    idx = dev(synth.random_indices(nq, k, n, 342, pad=11))
    win = dev(synth.normal((nq, W, d), 343))
    bt, num_pages, pg = paged(csa2, nq, n, page_rows, 344)
    cpool = to_pool(codes, bt, page_rows, num_pages)
    spool = to_pool(scales, bt, page_rows, num_pages)
    got = csa2.sparse_attn(q, cpool, spool, idx, win, 1 / math.sqrt(d), pages=pg, n=n)
    ref = csa2.sparse_attn(q, codes, scales, idx, win, 1 / math.sqrt(d))
    torch.cuda.synchronize()
    assert torch.equal(got, ref)
    rc, rs = orc.quantize_fp4(f64(x))
    o = orc.sparse_attn(f64(q), rc.reshape(nq, n, -1), rs.reshape(nq, n, -1), idx.cpu().numpy(),
                        f64(win), 1 / math.sqrt(d))
    assert rel_l2(got.cpu().numpy(), o) <= 2e-3


def test_paged_quantiser_writes_through_the_block_table(csa2, orc):
    # rows of 3 sequences written at entries 5..9 of each, through the table;
    # every other pool row keeps its junk pattern
    B, n, d, di, page_rows, nr = 3, 300, 512, 128, 64, 5
    bt, num_pages, pg = paged(csa2, B, n, page_rows, 350)
    codes = torch.full((num_pages * page_rows, d // 2), 0x5A, dtype=torch.uint8, device="cuda")
    scales = torch.full((num_pages * page_rows, d // 32), 0x5A, dtype=torch.uint8, device="cuda")
    k8 = torch.full((num_pages * page_rows, di), 0x5A, dtype=torch.uint8, device="cuda")
    x = synth.normal((B * nr, d), 351)
    kx = synth.normal((B * nr, di), 352) * 50
    csa2.quantize_fp4(dev(x), codes, scales, dev(kx), k8, pages=pg, rows_per_seq=nr, entry0=5)
    rc, rs = orc.quantize_fp4(f64(x))
    rk = orc.cast_e4m3(f64(kx))
    written = np.zeros(num_pages * page_rows, bool)
    btn = bt.cpu().numpy()
    for r in range(B * nr):
        b, j = r // nr, 5 + r % nr
        row = btn[b, j // page_rows] * page_rows + j % page_rows
        written[row] = True
        assert np.array_equal(codes[row].cpu().numpy(), rc[r])
        assert np.array_equal(scales[row].cpu().numpy(), rs[r])
        assert np.array_equal(k8[row].cpu().numpy(), rk[r])
    rest = torch.from_numpy(~written).cuda()
    assert bool((codes[rest] == 0x5A).all()) and bool((k8[rest] == 0x5A).all())


def test_paged_page_outside_the_pool_is_flagged(csa2):
    # a block table naming a page past the pool: the attention gather skips
    # the row and raises the bounds flag; nothing faults
    B, n, d, page_rows = 1, 256, 512, 64
    x = synth.normal((n, d), 360)
    codes, scales = csa2.quantize_fp4(dev(x))
    bt, num_pages, _ = paged(csa2, B, n, page_rows, 361)
    bt[0, 2] = num_pages + 7
    pg = csa2.pages(bt, page_rows, num_pages)
    cpool = torch.zeros(num_pages * page_rows, d // 2, dtype=torch.uint8, device="cuda")
    spool = torch.zeros(num_pages * page_rows, d // 32, dtype=torch.uint8, device="cuda")
    idx = torch.tensor([[3, 130, 140, 200]], dtype=torch.int32, device="cuda")  # 130, 140: page 2
    q = dev(synth.normal((1, 16, d), 362))
    win = dev(synth.normal((1, 4, d), 363))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = csa2.sparse_attn(q, cpool, spool, idx, win, 0.04, pages=pg, n=n, dev_status=st)
    torch.cuda.synchronize()
    assert csa2.lib.csa2_status_from_device(int(st.item())) == 7
    assert torch.isfinite(out).all()


def run_stack(wl, seed):
    from long_context_sparse_27_b300.workload import StackWorkload
    W = StackWorkload(wl, seed=seed, gen_device="cpu", keep_bf16=True)
    W.run()
    torch.cuda.synchronize()
    return W


@pytest.mark.parametrize("pool", [0, 1024])
def test_paged_stack_equals_contiguous(csa2, orc, pool):
    # a (Full, Reindex, Reuse, Reuse) group over 2 sequences of 6000 entries,
    # with and without the candidate pool; the Full layers' new rows are
    # written through the block table by the stack itself
    base = synth.scaled(synth.C1M, B=2, N=6000, modes=synth.C1M.modes[:4], pool=pool)
    Wc = run_stack(base, 7)
    Wp = run_stack(synth.scaled(base, page_rows=64), 7)
    assert int(Wp.dev_status.item()) == 0 and int(Wc.dev_status.item()) == 0
    for Lc, Lp in zip(Wc.layers, Wp.layers):
        if "topk_idx" in Lc:
            assert torch.equal(Lc["topk_idx"], Lp["topk_idx"])
        assert torch.equal(Lc["out"], Lp["out"])
    # the stack's new rows landed in the pool: entry N - 1 of every sequence
    btn = Wp.block_table.cpu().numpy()
    L0c, L0p = Wc.layers[0], Wp.layers[0]
    for b in range(base.B):
        j = base.N - 1
        row = btn[b, j // 64] * 64 + j % 64
        assert torch.equal(L0p["codes"][row], L0c["codes"][b, j])
        assert torch.equal(L0p["idxk"][row], L0c["idxk"][b, j])
    # the oracle quantises the same bf16 rows itself; the pools' logical view
    # (every entry, the stack's new rows included) must hold its bytes, and
    # the stack's selections and outputs must match its schedule
    plan = [(m, kv, ix) for m, (kv, ix) in zip(base.modes, Wp.plan)]
    layers = []
    for L, host in zip(Wp.layers, Wp.bf16):
        O = {"attn_q": f64(L["attn_q"]), "window": f64(L["window"])}
        if "idx_q" in L:
            O["idx_q"], O["idx_w"] = f64(L["idx_q"]), f64(L["idx_w"])
        if host:
            c, sc = orc.quantize_fp4(host["kv"].double().numpy().reshape(-1, base.D))
            O["codes"] = c.reshape(base.B, base.N, -1)
            O["scales"] = sc.reshape(base.B, base.N, -1)
            O["k8"] = orc.cast_e4m3(host["kk"].double().numpy())
            views = [orc.gather_pages(L[key].cpu().numpy().reshape(-1, 64, w), btn, base.N)
                     for key, w in (("codes", base.D // 2), ("scales", base.D // 32),
                                    ("idxk", base.Di))]
            assert np.array_equal(views[0], O["codes"])
            assert np.array_equal(views[1], O["scales"])
            assert np.array_equal(views[2], O["k8"])
        layers.append(O)
    ref_idx, ref_out = orc.layer_stack(plan, layers, base.k, 1 / math.sqrt(base.D), pool=pool)
    for l, (m, kv, ix) in enumerate(plan):
        g_idx = Wp.layers[l if m != synth.REUSE else ix]["topk_idx"].cpu().numpy()
        assert recall(g_idx, ref_idx[l]) >= 0.999
        g = Wp.layers[l]["out"].cpu().numpy()
        same = [q for q in range(base.nq) if np.array_equal(g_idx[q], ref_idx[l][q])]
        assert len(same) >= 1
        assert rel_l2(g[same], ref_out[l][same]) <= 2e-3
