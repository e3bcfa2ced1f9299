"""GPU parity of the whole CSA2 step (csa2_layer_stack) against the oracle.

Scaled-down versions of every workload run end to end through the static
Full / Reindex / Reuse schedule; the oracle runs the same schedule on the
same generator bytes.  Checks: index recall >= 0.999 against the oracle's
fp64 scores, attention within 2e-3 relative L2 wherever the two selections
agree (and agreement on >= 99% of the queries), the mode identities, and a
full-size (1M-context, 20-layer) step checked on sampled outputs.
"""
import math

import numpy as np
import pytest
import torch

from gpu_util import f64, need_gpu, recall, rel_l2, score_close, topk_valid
from long_context_sparse_27_b300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def csa2():
    return need_gpu()


def oracle_layers(orc, W):
    """The oracle's view of a StackWorkload: its own quantisation of the same
    bf16 rows; every other input is a generator tensor."""
    wl = W.wl
    out = []
    for L, host in zip(W.layers, W.bf16):
        O = {"attn_q": f64(L["attn_q"]), "window": f64(L["window"])}
        if "idx_q" in L:
            O["idx_q"] = f64(L["idx_q"])
            O["idx_w"] = f64(L["idx_w"])
        if host:
            kv = f64(host["kv"]).reshape(wl.B * wl.N, wl.D)
            c, s = orc.quantize_fp4(kv)
            O["codes"] = c.reshape(wl.B, wl.N, wl.D // 2)
            O["scales"] = s.reshape(wl.B, wl.N, wl.D // 32)
            if wl.fp32_indexer:
                O["k_f32"] = f64(host["kk"])
            else:
                O["k8"] = orc.cast_e4m3(f64(host["kk"]))
        out.append(O)
    return out


def run_stack(W):
    W.dev_status.zero_()
    W.run()
    torch.cuda.synchronize()
    assert int(W.dev_status.item()) == 0


def compare(orc, W, min_agree=0.99):
    wl = W.wl
    plan = [(m, kv, ix) for m, (kv, ix) in zip(wl.modes, W.plan)]
    nv = None if W.n_valid is None else W.n_valid.cpu().numpy()
    ref_idx, ref_out = oracle_stack(orc, W, plan, nv)
    agree = total = 0
    for l, (m, kv, ix) in enumerate(plan):
        gidx = W.layers[l if m != synth.REUSE else ix]["topk_idx"].cpu().numpy()
        assert recall(gidx, ref_idx[l]) >= 0.999, l
        gout = W.layers[l]["out"].cpu().numpy()
        same = [q for q in range(wl.nq) if np.array_equal(gidx[q], ref_idx[l][q])]
        agree += len(same)
        total += wl.nq
        if same:
            assert rel_l2(gout[same], ref_out[l][same]) <= 2e-3, l
    assert agree >= min_agree * total


def oracle_stack(orc, W, plan, nv):
    wl = W.wl
    layers = oracle_layers(orc, W)
    if wl.q_per_seq == 1:
        return orc.layer_stack(plan, layers, wl.k, 1 / math.sqrt(wl.D), q_per_seq=1, n_valid=nv,
                               pool=wl.pool)
    # prefill: per-query windows (rows t .. t + W - 1)
    idx_of, out_of = [], []
    for l, (m, kv, ix) in enumerate(plan):
        L, src = layers[l], layers[kv]
        if m != synth.REUSE:
            s = orc.index_score_fp8(L["idx_q"], L["idx_w"], src["k8"], wl.q_per_seq, nv)
            idx = orc.topk(s, wl.k, nv)
        else:
            idx = idx_of[ix].copy()
        out = orc.sparse_attn(L["attn_q"], src["codes"], src["scales"], idx, L["window"],
                              1 / math.sqrt(wl.D), q_per_seq=wl.q_per_seq,
                              win_start=W.win_start.cpu().numpy(),
                              win_len=W.win_len.cpu().numpy())
        idx_of.append(idx)
        out_of.append(out)
    return idx_of, out_of


def build(wl, seed):
    from long_context_sparse_27_b300.workload import StackWorkload
    return StackWorkload(wl, seed=seed, gen_device="cpu", keep_bf16=True)


def test_stack_tiny(csa2, orc):
    W = build(synth.TINY, 1)
    run_stack(W)
    compare(orc, W, min_agree=1.0)


def test_stack_group3_scaled(csa2, orc):
    W = build(synth.scaled(synth.GROUP3, B=3, N=3000), 2)
    run_stack(W)
    compare(orc, W)


def test_stack_1m_pattern_scaled(csa2, orc):
    W = build(synth.scaled(synth.C1M, B=2, N=2500, modes=synth.C1M.modes[:8]), 3)
    run_stack(W)
    compare(orc, W)


def test_stack_128k_scaled(csa2, orc):
    W = build(synth.scaled(synth.C128K, B=4, N=4096), 4)
    run_stack(W)
    compare(orc, W)


def test_stack_prefill_scaled(csa2, orc):
    wl = synth.scaled(synth.PREFILL, q_per_seq=16, N=1000, pos0=4 * 1000 - 16)
    W = build(wl, 5)
    run_stack(W)
    compare(orc, W)


@pytest.mark.parametrize("N", [1000, 20000])
def test_stack_prefill_reindex_scaled(csa2, orc, N):
    # a prefill chunk through Full, Reindex and Reuse layers: the Reindex
    # layer's indexer walks its tiles from the end over the Full layer's keys;
    # long rows (20000) select from the scoring pass's candidates
    wl = synth.scaled(synth.PREFILL, q_per_seq=16, N=N, pos0=4 * N - 16,
                      modes=(synth.FULL, synth.REINDEX, synth.REUSE))
    W = build(wl, 6)
    run_stack(W)
    compare(orc, W)


def test_stack_1m_pool_scaled(csa2, orc):
    # the Hierarchical Sparse Indexer: Reindex layers score only the top-1024
    # pool of their Full layer (pool < N, so the restriction matters)
    W = build(synth.scaled(synth.C1M_POOL, B=2, N=2500, modes=synth.C1M.modes[:8], pool=1024), 8)
    run_stack(W)
    compare(orc, W)


def test_stack_pool_covering_every_entry(csa2):
    # a pool as large as the sequence restricts nothing: same selections and
    # outputs as the plain schedule, bit for bit
    from long_context_sparse_27_b300.workload import StackWorkload
    wl = synth.scaled(synth.C1M, B=2, N=1500, modes=(synth.FULL, synth.REINDEX, synth.REUSE))
    A = StackWorkload(wl, seed=9, gen_device="cuda")
    B = StackWorkload(synth.scaled(wl, pool=2048), seed=9, gen_device="cuda")
    run_stack(A)
    run_stack(B)
    for La, Lb in zip(A.layers, B.layers):
        if "topk_idx" in La:
            assert torch.equal(La["topk_idx"], Lb["topk_idx"])
        assert torch.equal(La["out"], Lb["out"])


@pytest.mark.parametrize("pool", [0, 512])
def test_stack_sequences_shorter_than_k(csa2, orc, pool):
    # N = 300 < k = 512: every selection is all 300 entries padded with -1,
    # the pool (P = min(512, N)) holds every entry, attention sees 300 FP4
    # keys and the window
    wl = synth.scaled(synth.C1M, B=2, N=300, modes=(synth.FULL, synth.REINDEX, synth.REUSE),
                      pool=pool)
    W = build(wl, 16)
    run_stack(W)
    for L in W.layers[:2]:
        idx = L["topk_idx"].cpu().numpy()
        assert np.array_equal(idx[:, :300], np.tile(np.arange(300, dtype=np.int32), (2, 1)))
        assert np.all(idx[:, 300:] == -1)
    compare(orc, W, min_agree=1.0)


def test_stack_mode_identities(csa2):
    from long_context_sparse_27_b300.workload import StackWorkload
    wl = synth.scaled(synth.C1M, B=2, N=3000, modes=(synth.FULL, synth.REINDEX, synth.REUSE))
    W = StackWorkload(wl, seed=6, gen_device="cuda")
    # Reindex with the Full layer's indexer Q and w selects what Full selected
    W.layers[1]["idx_q"].copy_(W.layers[0]["idx_q"])
    W.layers[1]["idx_w"].copy_(W.layers[0]["idx_w"])
    # Reuse with the Full layer's query and window reproduces its output
    W.layers[2]["attn_q"].copy_(W.layers[0]["attn_q"])
    W.layers[2]["window"].copy_(W.layers[0]["window"])
    run_stack(W)
    assert torch.equal(W.layers[1]["topk_idx"], W.layers[0]["topk_idx"])
    assert torch.equal(W.layers[2]["out"], W.layers[0]["out"])


def test_stack_rejects_bad_plans(csa2):
    from long_context_sparse_27_b300.workload import StackWorkload
    wl = synth.scaled(synth.C1M, B=1, N=512, modes=(synth.FULL, synth.REINDEX, synth.REUSE))
    W = StackWorkload(wl, seed=7, gen_device="cuda")
    bad = [dict(L) for L in W.layers]
    bad[1]["kv_src"] = 1  # Reindex must read the last Full layer
    st, where = csa2.validate_plan(bad)
    assert st == 1 and where == 1
    with pytest.raises(csa2.Csa2Error):
        csa2.layer_stack(csa2.layer_descs(bad), W.stack_args(), W.workspace)


# ------------------------------------------------------------------ full size

def sampled_full_check(csa2, orc, wl, seed, queries, index_layers=(0,)):
    """A full-size step as the benchmark runs it (device-drawn inputs, the
    same launch configuration), checked on sampled queries: for each index
    layer in `index_layers` and each sampled query, the GPU's scores at
    sampled entries against the oracle, the GPU selection as a valid top-k
    of the GPU's own scores, recall >= 0.999 against the oracle's fp64
    selection, and the attention output of that layer (and of the Reuse
    layers that take its indices) wherever the two selections agree."""
    from long_context_sparse_27_b300.workload import StackWorkload
    W = StackWorkload(wl, seed=seed, gen_device="cuda", keep_bf16=False)
    run_stack(W)
    nv_all = None if W.n_valid is None else W.n_valid.cpu().numpy()
    rng = np.random.default_rng(seed)
    checked_attn = 0
    for l in index_layers:
        m, (kvs, _) = wl.modes[l], W.plan[l]
        assert m in (synth.FULL, synth.REINDEX)
        L, src = W.layers[l], W.layers[kvs]
        # the source Full layer's rows, drawn again (the draws are seeded)
        s0 = seed * 1000 + 20 * kvs
        kk = synth.index_k_rows(wl, s0 + 6, "cuda")
        kv = synth.kv_rows(wl, s0 + 5, "cuda")
        scores = csa2.index_score(L["idx_q"], L["idx_w"], src["idxk"], q_per_seq=wl.q_per_seq,
                                  n_valid=W.n_valid)
        torch.cuda.synchronize()
        g_idx_all = L["topk_idx"].cpu().numpy()
        for q in queries:
            b = q // wl.q_per_seq
            nvq = wl.N if nv_all is None else int(nv_all[q])
            g_s = scores[q:q + 1].cpu().numpy()
            g_idx = g_idx_all[q:q + 1]
            assert topk_valid(g_s[0], g_idx[0], wl.k, nvq), (l, q)
            k8 = orc.cast_e4m3(f64(kk[b]))[None]
            ref_s = orc.index_score_fp8(f64(L["idx_q"][q:q + 1]), f64(L["idx_w"][q:q + 1]), k8,
                                        1, None if nv_all is None else nv_all[q:q + 1])
            cols = rng.choice(wl.N, min(4096, wl.N), replace=False)
            sel = g_idx[0][g_idx[0] >= 0]
            cols[: len(sel)] = sel  # include the selected entries
            assert score_close(g_s[:, cols], ref_s[:, cols]) <= 1.0, (l, q)
            ref_idx = orc.topk(ref_s, wl.k, None if nv_all is None else nv_all[q:q + 1])
            assert recall(g_idx, ref_idx) >= 0.999, (l, q)
            if not np.array_equal(g_idx, ref_idx):
                continue
            rows = ref_idx[0][ref_idx[0] >= 0]
            c, sc = orc.quantize_fp4(f64(kv[b, rows]))
            codes = np.zeros((1, wl.N, wl.D // 2), np.uint8)
            scl = np.zeros((1, wl.N, wl.D // 32), np.uint8)
            codes[0, rows], scl[0, rows] = c, sc
            # this layer and every Reuse layer that takes its indices
            for l2 in [l] + [j for j, (mm, (kv2, ix2)) in enumerate(zip(wl.modes, W.plan))
                             if mm == synth.REUSE and ix2 == l]:
                L2 = W.layers[l2]
                kw = {}
                if W.win_start is not None:  # prefill: query t attends window rows t .. t+W-1
                    kw = dict(win_start=W.win_start.cpu().numpy()[q:q + 1],
                              win_len=W.win_len.cpu().numpy()[q:q + 1])
                win = f64(L2["window"][b:b + 1])
                ref = orc.sparse_attn(f64(L2["attn_q"][q:q + 1]), codes, scl, ref_idx, win,
                                      1 / math.sqrt(wl.D), **kw)
                assert rel_l2(L2["out"][q:q + 1].cpu().numpy(), ref) <= 2e-3, (l2, q)
                checked_attn += 1
    assert checked_attn > 0


def test_full_size_1m_sampled(csa2, orc):
    """The 1M-context, 20-layer decode step as the benchmark runs it: the
    first group's Full and Reindex layers (and the Reuse layers after them)
    for the first and last sequence."""
    sampled_full_check(csa2, orc, synth.C1M, 11, queries=(0, 7), index_layers=(0, 1))


def test_full_size_128k_sampled(csa2, orc):
    sampled_full_check(csa2, orc, synth.C128K, 12, queries=(0, 9, 15))


def test_full_size_group3_sampled(csa2, orc):
    sampled_full_check(csa2, orc, synth.GROUP3, 13, queries=(0, 31), index_layers=(0, 1))


def test_full_size_prefill_sampled(csa2, orc):
    """The 4096-query prefill chunk at N = 262144: the first, a middle and the
    last query (their causal visibility differs)."""
    sampled_full_check(csa2, orc, synth.PREFILL, 14, queries=(0, 2047, 4095))


def test_full_size_1m_pool_sampled(csa2, orc):
    """The pooled 1M-context step (Reindex layers score only the top-2048 pool
    of their Full layer) at full size, checked for the first Reindex layer on
    the first and last sequence: the GPU pool is the top-2048 of the GPU's
    Full-layer scores; the pooled scores against the oracle at every pool
    entry; the GPU selection a valid top-k of its pooled scores; recall
    against the oracle's selection inside the oracle's own pool; the
    attention output where the two selections agree."""
    from long_context_sparse_27_b300.workload import StackWorkload
    wl, seed = synth.C1M_POOL, 15
    W = StackWorkload(wl, seed=seed, gen_device="cuda", keep_bf16=False)
    run_stack(W)
    F0, R1 = W.layers[0], W.layers[1]
    P = wl.pool
    kk = synth.index_k_rows(wl, seed * 1000 + 6, "cuda")
    kv = synth.kv_rows(wl, seed * 1000 + 5, "cuda")
    g_full = csa2.index_score(F0["idx_q"], F0["idx_w"], F0["idxk"])
    g_pool = orc.topk(g_full.cpu().numpy(), P)                 # the GPU's pool, decided on its scores
    g_ps = csa2.index_score_pool(R1["idx_q"], R1["idx_w"], F0["idxk"],
                                 torch.from_numpy(g_pool).cuda()).cpu().numpy()
    g_idx_all = R1["topk_idx"].cpu().numpy()
    checked = 0
    for q in (0, 7):
        k8 = orc.cast_e4m3(f64(kk[q]))[None]
        ref_full = orc.index_score_fp8(f64(F0["idx_q"][q:q + 1]), f64(F0["idx_w"][q:q + 1]), k8)
        ref_re = orc.index_score_fp8(f64(R1["idx_q"][q:q + 1]), f64(R1["idx_w"][q:q + 1]), k8)
        assert score_close(g_ps[q:q + 1], ref_re[:, g_pool[q]]) <= 1.0, q
        restricted = np.full((1, wl.N), -np.inf)
        restricted[0, g_pool[q]] = g_ps[q]
        g_idx = g_idx_all[q:q + 1]
        assert topk_valid(restricted[0], g_idx[0], wl.k, wl.N), q
        ref_pool = orc.topk(ref_full, P)
        ref_idx = orc.topk(orc.pool_restrict(ref_re, ref_pool), wl.k)
        assert recall(g_idx, ref_idx) >= 0.999, q
        if not np.array_equal(g_idx, ref_idx):
            continue
        rows = ref_idx[0]
        c, sc = orc.quantize_fp4(f64(kv[q, rows]))
        codes = np.zeros((1, wl.N, wl.D // 2), np.uint8)
        scl = np.zeros((1, wl.N, wl.D // 32), np.uint8)
        codes[0, rows], scl[0, rows] = c, sc
        ref = orc.sparse_attn(f64(R1["attn_q"][q:q + 1]), codes, scl, ref_idx,
                              f64(R1["window"][q:q + 1]), 1 / math.sqrt(wl.D))
        assert rel_l2(R1["out"][q:q + 1].cpu().numpy(), ref) <= 2e-3, q
        checked += 1
    assert checked > 0


def test_stack_prefill_selection_without_the_score_matrix(csa2, orc):
    # a prefill chunk of 64 queries over 20000 entries (long rows): the stack
    # scores a sample of the tiles, derives each query's threshold, keeps
    # the entries at or above it and selects among them; the result must be,
    # bit for bit, the top-k of the full score matrix of the same kernel
    wl = synth.scaled(synth.PREFILL, q_per_seq=64, N=20000, pos0=4 * 20000 - 64)
    W = build(wl, 6)
    run_stack(W)
    assert int(W.dev_status.item()) == 0
    L = W.layers[0]
    scores = csa2.index_score(L["idx_q"], L["idx_w"], L["idxk"], q_per_seq=wl.q_per_seq,
                              n_valid=W.n_valid)
    ref = csa2.topk(scores, wl.k, n_valid=W.n_valid)
    torch.cuda.synchronize()
    assert torch.equal(L["topk_idx"], ref)
    assert np.array_equal(L["topk_idx"].cpu().numpy(),
                          orc.topk(scores.cpu().double().numpy(), wl.k, W.n_valid.cpu().numpy()))
    compare(orc, W)


def test_stack_prefill_candidate_overflow_is_flagged(csa2):
    # every indexer key equal: every visible entry reaches the sample's
    # threshold, far more than a query's candidate buffer holds; the
    # selection reports CSA2_DEVFLAG_CAPACITY instead of failing silently
    wl = synth.scaled(synth.PREFILL, q_per_seq=8, N=20000, pos0=4 * 20000 - 8)
    W = build(wl, 7)
    W.layers[0]["idxk"][:] = 0x38                    # E4M3 1.0 everywhere
    W.layers[0]["new_idxk"][:] = 1.0
    W.dev_status.zero_()
    W.run()
    torch.cuda.synchronize()
    assert int(W.dev_status.item()) & csa2.DEVFLAG_CAPACITY
    assert csa2.lib.csa2_status_from_device(int(W.dev_status.item())) == 8


@pytest.mark.parametrize("page_rows", [0, 64])
def test_stack_new_rows_quantised_before_they_are_scored(csa2, orc, page_rows):
    # a decode Full layer quantises the step's new rows inside its indexer
    # launch, in the CTA that loads their tile and before that load.  Each
    # new indexer key is made its sequence's best entry (200 x the direction
    # of the query's weighted head sum), so a load that ran ahead of the
    # write (a zero key, score 0) would drop entry N - 1 from the selection
    wl = synth.scaled(synth.C1M, B=3, N=9000, modes=synth.C1M.modes[:4], page_rows=page_rows)
    W = build(wl, 23)
    N = wl.N
    for L, host in zip(W.layers, W.bf16):
        if L["mode"] != synth.FULL:
            continue
        v = (L["idx_w"].float()[:, :, None] * L["idx_q"].float()).sum(1)
        k = (v / v.abs().amax(1, keepdim=True) * 200).to(torch.bfloat16)
        L["new_idxk"].copy_(k[:, None, :])
        host["kk"][:, N - 1] = k.cpu()
    run_stack(W)
    for L, host in zip(W.layers, W.bf16):
        if L["mode"] != synth.FULL:
            continue
        idx = L["topk_idx"].cpu().numpy()
        assert all(N - 1 in idx[b] for b in range(wl.B))
        # the rows the launch wrote: the oracle's quantisation of the same bf16 rows
        if page_rows:
            bt = W.block_table.cpu().numpy()
            rows = [int(bt[b, (N - 1) // page_rows]) * page_rows + (N - 1) % page_rows
                    for b in range(wl.B)]
        else:
            rows = [b * N + N - 1 for b in range(wl.B)]
        codes = L["codes"].reshape(-1, wl.D // 2)[rows].cpu().numpy()
        scales = L["scales"].reshape(-1, wl.D // 32)[rows].cpu().numpy()
        k8 = L["idxk"].reshape(-1, wl.Di)[rows].cpu().numpy()
        c, s = orc.quantize_fp4(f64(host["kv"][:, N - 1]))
        assert np.array_equal(codes, c) and np.array_equal(scales, s)
        assert np.array_equal(k8, orc.cast_e4m3(f64(host["kk"][:, N - 1])))
    compare(orc, W)
