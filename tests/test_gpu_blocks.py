"""Block-level pruning of the Hierarchical Sparse Indexer on the GPU.

Reading ("DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression",
Method and Related Work): a block of G consecutive entries is represented by
the E4M3 cast of the sum of its entries' indexer keys divided by G; a Full
layer scores the block keys with the indexer formula, keeps its best blocks
and scores at token level only their entries.  Checks: block keys bit-exact
against the oracle (contiguous and paged caches, a partial last block), a
stack with pruning against the oracle's pruned schedule (index recall,
attention), and keeping every block equal, bit for bit, to the plain stack.
"""
import math

import numpy as np
import pytest
import torch

from gpu_util import f64, need_gpu, recall, rel_l2
from long_context_sparse_27_b300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def csa2():
    return need_gpu()


def keys8(B, n, seed):
    # E4M3 codes of N(0,1) * 3 values, with a few saturated (+-448) and zero rows
    x = synth.normal((B, n, 128), seed, dtype=torch.float32) * 3
    x[:, ::37] *= 1000
    x[:, ::53] = 0
    return x


@pytest.mark.parametrize("B,n,G", [(2, 1000, 64), (3, 130, 8), (1, 64, 64), (2, 5, 1)])
def test_block_keys_bit_exact(csa2, orc, B, n, G):
    x = keys8(B, n, 400 + n)
    z = torch.zeros(B * n, 32, dtype=torch.bfloat16, device="cuda")
    _, _, k8 = csa2.quantize_fp4(z, idxk=x.reshape(B * n, 128).to(torch.bfloat16).cuda())
    k8 = k8.reshape(B, n, 128)
    got = csa2.index_block_keys(k8, G)
    want = orc.block_summaries(orc.cast_e4m3(f64(x.to(torch.bfloat16))), G)
    assert np.array_equal(got.cpu().numpy(), want)
    # a sub-range of blocks leaves the others untouched
    nb = -(-n // G)
    if nb > 2:
        part = torch.full_like(got, 0x5A)
        csa2.index_block_keys(k8, G, blk0=1, nblk=nb - 2, out=part)
        assert torch.equal(part[:, 1:nb - 1], got[:, 1:nb - 1])
        assert bool((part[:, 0] == 0x5A).all()) and bool((part[:, nb - 1] == 0x5A).all())


def test_block_keys_paged(csa2, orc):
    B, n, G, page_rows = 2, 700, 16, 64
    x = keys8(B, n, 410)
    z = torch.zeros(B * n, 32, dtype=torch.bfloat16, device="cuda")
    _, _, k8 = csa2.quantize_fp4(z, idxk=x.reshape(B * n, 128).to(torch.bfloat16).cuda())
    k8 = k8.reshape(B, n, 128)
    bt, num_pages = synth.block_table(B, n, page_rows, 411, "cuda")
    pool = torch.zeros(num_pages * page_rows, 128, dtype=torch.uint8, device="cuda")
    j = torch.arange(n, device="cuda")
    for b in range(B):
        pool[bt[b, j // page_rows].long() * page_rows + j % page_rows] = k8[b]
    got = csa2.index_block_keys(pool, G, n=n, pages=csa2.pages(bt, page_rows, num_pages), B=B)
    assert torch.equal(got, csa2.index_block_keys(k8, G))


def run_stack(wl, seed):
    from long_context_sparse_27_b300.workload import StackWorkload
    W = StackWorkload(wl, seed=seed, gen_device="cpu", keep_bf16=True)
    W.run()
    torch.cuda.synchronize()
    return W


def oracle_layers(orc, W):
    wl = W.wl
    layers = []
    for L, host in zip(W.layers, W.bf16):
        O = {"attn_q": f64(L["attn_q"]), "window": f64(L["window"])}
        if "idx_q" in L:
            O["idx_q"], O["idx_w"] = f64(L["idx_q"]), f64(L["idx_w"])
        if host:
            c, sc = orc.quantize_fp4(host["kv"].double().numpy().reshape(-1, wl.D))
            O["codes"] = c.reshape(wl.B, wl.N, -1)
            O["scales"] = sc.reshape(wl.B, wl.N, -1)
            O["k8"] = orc.cast_e4m3(host["kk"].double().numpy())
        layers.append(O)
    return layers


@pytest.mark.parametrize("page_rows", [0, 64])
def test_block_pruned_stack_matches_the_oracle(csa2, orc, page_rows):
    # (Full, Reindex, Reuse, Reuse) over 2 sequences of 6000 entries, blocks
    # of 64, 8 kept (a 512-entry pool, top-64): the Full layer's new row
    # changes its block's key, which the stack recomputes before scoring
    wl = synth.scaled(synth.C1M_BLOCK, B=2, N=6000, modes=synth.C1M.modes[:4], k=64,
                      blocks_kept=8, page_rows=page_rows)
    W = run_stack(wl, 11)
    assert int(W.dev_status.item()) == 0
    layers = oracle_layers(orc, W)
    # the stack kept the Full layer's block keys current (its new row included)
    bk = orc.block_summaries(layers[0]["k8"], wl.block)
    assert np.array_equal(W.layers[0]["block_keys"].cpu().numpy(), bk)
    plan = [(m, kv, ix) for m, (kv, ix) in zip(wl.modes, W.plan)]
    ref_idx, ref_out = orc.layer_stack(plan, layers, wl.k, 1 / math.sqrt(wl.D), block=wl.block,
                                       blocks_kept=wl.blocks_kept)
    for l, (m, kv, ix) in enumerate(plan):
        g_idx = W.layers[l if m != synth.REUSE else ix]["topk_idx"].cpu().numpy()
        assert recall(g_idx, ref_idx[l]) >= 0.999
        g = W.layers[l]["out"].cpu().numpy()
        same = [q for q in range(wl.nq) if np.array_equal(g_idx[q], ref_idx[l][q])]
        assert len(same) >= 1
        assert rel_l2(g[same], ref_out[l][same]) <= 2e-3


def test_keeping_every_block_is_the_plain_stack(csa2):
    # 2048 entries in 32 blocks of 64, all kept (a pool holds at most 2048
    # slots): pruning removes nothing, so selections and outputs equal the
    # plain schedule's
    base = synth.scaled(synth.C1M, B=2, N=2048, modes=synth.C1M.modes[:4], k=128)
    Wp = run_stack(base, 12)
    Wb = run_stack(synth.scaled(base, block=64, blocks_kept=32), 12)
    assert int(Wb.dev_status.item()) == 0
    for Lp, Lb in zip(Wp.layers, Wb.layers):
        if "topk_idx" in Lp:
            assert torch.equal(Lp["topk_idx"], Lb["topk_idx"])
        assert torch.equal(Lp["out"], Lb["out"])
