"""Pins for the oracle's indexer score, top-k, sparse attention and modes.

Independent witnesses: numpy einsum (score brute force), Python's sorted()
(top-k brute force), torch's float64 scaled_dot_product_attention on CPU
(attention), closed forms and invariants.
"""
import numpy as np
import pytest
import torch

from long_context_sparse_27_b300 import synth


# ---- indexer score --------------------------------------------------------

def test_score_against_einsum(orc):
    rng = np.random.default_rng(10)
    nq, hi, di, B, n = 6, 5, 16, 3, 40
    qv = rng.standard_normal((nq, hi, di))
    c = rng.random((nq, hi))
    kv = rng.standard_normal((B, n, di))
    s = orc.index_score(qv, c, kv, q_per_seq=2)
    kq = kv[np.arange(nq) // 2]                          # [nq, n, di]
    dots = np.einsum("qhd,qnd->qhn", qv, kq)
    ref = np.einsum("qh,qhn->qn", c, np.maximum(dots, 0))
    assert np.allclose(s, ref, rtol=1e-12, atol=1e-12)


def test_score_negative_weights_relu_first(orc):
    # the ReLU acts on each head's dot product before weighting
    qv = np.array([[[1.0], [1.0]]])          # 1 query, 2 heads, dim 1
    c = np.array([[1.0, -2.0]])
    kv = np.array([[[3.0], [-1.0]]])         # entries: +3, -1
    s = orc.index_score(qv, c, kv)
    assert s[0, 0] == 3.0 - 6.0              # both heads active
    assert s[0, 1] == 0.0                    # both heads clipped


def test_score_single_head_closed_form(orc):
    rng = np.random.default_rng(11)
    q = rng.standard_normal((1, 1, 1))
    kv = rng.standard_normal((1, 50, 1))
    s = orc.index_score(q, np.ones((1, 1)), kv)
    assert np.array_equal(s[0], np.maximum(q[0, 0, 0] * kv[0, :, 0], 0))


def test_score_visibility(orc):
    rng = np.random.default_rng(12)
    qv = rng.standard_normal((3, 2, 4))
    kv = rng.standard_normal((1, 10, 4))
    s = orc.index_score(qv, np.ones((3, 2)), kv, q_per_seq=3, n_valid=[0, 4, 10])
    assert np.isneginf(s[0]).all()
    assert np.isneginf(s[1, 4:]).all() and np.isfinite(s[1, :4]).all()
    assert np.isfinite(s[2]).all()


def test_score_fp8_path_exact_dot(orc):
    # the fp8 path decodes q8 / k8 and scales by c = w * sigma; its
    # inner products of E4M3 values are exact in fp64, so it equals an
    # einsum over the decoded values
    rng = np.random.default_rng(13)
    q = torch.randn(2, 4, 128, dtype=torch.float64).to(torch.bfloat16).double().numpy()
    w = rng.random((2, 4)) / 64
    kb = torch.randn(2, 30, 128, dtype=torch.float64).to(torch.bfloat16).double().numpy()
    k8 = orc.cast_e4m3(kb)
    s = orc.index_score_fp8(q, w, k8)
    q8, c = orc.quantize_index_q(q, w)
    qd = orc.e4m3_decode(q8)
    kd = orc.e4m3_decode(k8)
    dots = np.einsum("qhd,qnd->qhn", qd, kd)
    assert np.array_equal(s, np.einsum("qh,qhn->qn", c, np.maximum(dots, 0)))
    # and it approximates the unquantised score
    exact = np.einsum("qh,qhn->qn", w, np.maximum(np.einsum("qhd,qnd->qhn", q, kb), 0))
    assert np.allclose(s, exact, rtol=0.15, atol=0.05 * np.abs(exact).max())


# ---- top-k ------------------------------------------------------------------

def brute_topk(row, k, nv):
    order = sorted(range(nv), key=lambda j: (-row[j], j))[:k]
    out = sorted(order)
    return out + [-1] * (k - len(out))


@pytest.mark.parametrize("levels", [0, 3, 50])
def test_topk_brute_force(orc, levels):
    s = synth.scores_with_ties(7, 300, seed=20 + levels, levels=levels).double().numpy()
    nv = np.array([300, 299, 128, 5, 0, 64, 1], dtype=np.int32)
    got = orc.topk(s, 64, nv)
    for r in range(7):
        assert list(got[r]) == brute_topk(list(s[r]), 64, int(nv[r])), r


def test_topk_invariants(orc):
    s = synth.scores_with_ties(4, 5000, seed=21).double().numpy()
    k = 512
    got = orc.topk(s, k)
    for r in range(4):
        sel = got[r]
        assert (np.diff(sel) > 0).all() and len(sel) == k
        mask = np.zeros(5000, bool)
        mask[sel] = True
        assert s[r, mask].min() >= s[r, ~mask].max()


def test_topk_ties_lowest_index(orc):
    s = np.zeros((1, 20))
    s[0, [3, 7, 11, 15]] = 1.0
    got = orc.topk(s, 6)
    # the four ones, then the two lowest-index zeros
    assert list(got[0]) == [0, 1, 3, 7, 11, 15]


def test_topk_signed_zero_equal(orc):
    s = np.array([[-0.0, 0.0, -0.0, 0.0]])
    assert list(orc.topk(s, 2)[0]) == [0, 1]


def test_topk_k_at_least_n(orc):
    s = synth.scores_with_ties(2, 10, seed=22).double().numpy()
    got = orc.topk(s, 16)
    assert list(got[0]) == list(range(10)) + [-1] * 6


# ---- sparse attention --------------------------------------------------------

def sdpa_ref(q, keys, scale):
    """torch float64 SDPA with keys as values; q [hq, d], keys [m, d]."""
    qt = torch.from_numpy(q)[None, :, None, :]                   # [1, hq, 1, d]
    kt = torch.from_numpy(keys)[None, None].expand(1, q.shape[0], -1, -1)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, kt, scale=scale)
    return o[0, :, 0, :].numpy()


def make_cache(orc, B, n, d, seed):
    x = synth.normal((B, n, d), seed).double().numpy()
    codes, scales = orc.quantize_fp4(x.reshape(B * n, d))
    return codes.reshape(B, n, d // 2), scales.reshape(B, n, d // 32)


def test_attn_against_sdpa(orc):
    B, n, d, hq, k, W = 2, 200, 64, 4, 16, 8
    codes, scales = make_cache(orc, B, n, d, 30)
    q = synth.normal((2 * B, hq, d), 31).double().numpy()
    idx = synth.random_indices(2 * B, k, n, 32, pad=3).numpy()
    win = synth.normal((B, W + 5, d), 33).double().numpy()
    ws = np.array([0, 5, 2, 3], np.int32)
    wl = np.array([W, W, 3, 0], np.int32)
    scale = 1 / np.sqrt(d)
    out = orc.sparse_attn(q, codes, scales, idx, win, scale, q_per_seq=2,
                          win_start=ws, win_len=wl)
    for qi in range(2 * B):
        b = qi // 2
        sel = idx[qi][idx[qi] >= 0]
        keys = np.concatenate([orc.dequantize_fp4(codes[b, sel], scales[b, sel], d),
                               win[b, ws[qi]:ws[qi] + wl[qi]]])
        assert np.allclose(out[qi], sdpa_ref(q[qi], keys, scale), rtol=1e-10, atol=1e-12)


def test_attn_k_covers_all_equals_dense(orc):
    # k >= N: the sparse step sees every entry, so it equals dense attention
    # over the whole dequantised cache plus the window
    B, n, d, hq, W = 1, 48, 32, 3, 4
    codes, scales = make_cache(orc, B, n, d, 34)
    q = synth.normal((1, hq, d), 35).double().numpy()
    win = synth.normal((1, W, d), 36).double().numpy()
    x = synth.normal((B, n, d), 37).double().numpy()
    s = orc.index_score(x[:, :, :8][:, None, 0], np.ones((1, 1)), x[:, :, :8])  # any scores
    idx = orc.topk(s, 64)                       # k = 64 >= n = 48 -> all + padding
    assert (idx[0, :n] == np.arange(n)).all() and (idx[0, n:] == -1).all()
    out = orc.sparse_attn(q, codes, scales, idx, win, 0.3)
    dense = np.concatenate([orc.dequantize_fp4(codes[0], scales[0], d), win[0]])
    assert np.allclose(out[0], sdpa_ref(q[0], dense, 0.3), rtol=1e-10, atol=1e-12)


def test_attn_zero_query_is_mean(orc):
    B, n, d = 1, 30, 32
    codes, scales = make_cache(orc, B, n, d, 38)
    win = synth.normal((1, 4, d), 39).double().numpy()
    idx = np.array([[2, 5, 9, -1]], np.int32)
    out = orc.sparse_attn(np.zeros((1, 2, d)), codes, scales, idx, win, 1.0)
    keys = np.concatenate([orc.dequantize_fp4(codes[0, [2, 5, 9]], scales[0, [2, 5, 9]], d), win[0]])
    assert np.allclose(out[0, 0], keys.mean(0), rtol=0, atol=1e-14)
    assert np.allclose(out[0, 1], keys.mean(0), rtol=0, atol=1e-14)


def test_attn_dominant_logit_picks_row(orc):
    B, n, d = 1, 30, 32
    codes, scales = make_cache(orc, B, n, d, 40)
    row = orc.dequantize_fp4(codes[0, 7:8], scales[0, 7:8], d)[0]
    win = np.zeros((1, 2, d))
    q = (row * 1e3)[None, None, :]
    out = orc.sparse_attn(q, codes, scales, np.array([[7, 1, 3]], np.int32), win, 1.0)
    assert np.allclose(out[0, 0], row, rtol=0, atol=1e-12)


def test_attn_no_keys_zero(orc):
    codes, scales = make_cache(orc, 1, 4, 32, 41)
    out = orc.sparse_attn(np.ones((1, 1, 32)), codes, scales, np.array([[-1, -1]], np.int32),
                          np.zeros((1, 0, 32)), 1.0)
    assert (out == 0).all()


def test_attn_rejects_bad_index(orc):
    codes, scales = make_cache(orc, 1, 4, 32, 42)
    with pytest.raises(ValueError):
        orc.sparse_attn(np.ones((1, 1, 32)), codes, scales, np.array([[4]], np.int32),
                        np.zeros((1, 1, 32)), 1.0)


# ---- layer modes --------------------------------------------------------------

F, RI, RU = synth.FULL, synth.REINDEX, synth.REUSE


def test_default_sources():
    from oracle import oracle as o
    assert o.default_sources([F, RI, RU]) == [(0, 0), (0, 1), (0, 0)]
    assert o.default_sources([F, RI, RU, RU, F, RI, RU, RU]) == [
        (0, 0), (0, 1), (0, 0), (0, 0), (4, 4), (4, 5), (4, 4), (4, 4)]
    with pytest.raises(ValueError):
        o.default_sources([RI, F])
    with pytest.raises(ValueError):
        o.default_sources([RU])


def small_stack_layers(orc, modes, seed, B=2, n=300, hi=4, di=128, hq=2, d=64, W=8,
                       same_q=False):
    layers = []
    base_q = synth.normal((B, hi, di), seed).double().numpy()
    for l, m in enumerate(modes):
        L = {"attn_q": synth.normal((B, hq, d), seed + 10 * l + 1).double().numpy(),
             "window": synth.normal((B, W, d), seed + 10 * l + 2).double().numpy()}
        if m in (F, RI):
            L["idx_q"] = base_q if same_q else synth.normal((B, hi, di), seed + 10 * l + 3).double().numpy()
            L["idx_w"] = np.full((B, hi), 1.0 / 64)
        if m == F:
            x = synth.normal((B, n, d), seed + 10 * l + 4).double().numpy()
            c, s = orc.quantize_fp4(x.reshape(B * n, d))
            L["codes"], L["scales"] = c.reshape(B, n, d // 2), s.reshape(B, n, d // 32)
            kb = synth.normal((B, n, di), seed + 10 * l + 5).double().numpy()
            L["k8"] = orc.cast_e4m3(kb)
        layers.append(L)
    return layers


def test_modes_reuse_copies_indices(orc):
    modes = [F, RI, RU]
    layers = small_stack_layers(orc, modes, 50)
    idx, out = orc.layer_stack(orc.default_plan(modes), layers, k=32, scale=0.125)
    assert np.array_equal(idx[2], idx[0])
    # Reindex draws a fresh Q: its selection differs from the Full layer's
    assert not np.array_equal(idx[1], idx[0])


def test_modes_reindex_same_q_reproduces_full(orc):
    modes = [F, RI]
    layers = small_stack_layers(orc, modes, 60, same_q=True)
    idx, out = orc.layer_stack(orc.default_plan(modes), layers, k=32, scale=0.125)
    assert np.array_equal(idx[1], idx[0])


def test_modes_reuse_same_query_same_output(orc):
    modes = [F, RU]
    layers = small_stack_layers(orc, modes, 70)
    layers[1]["attn_q"] = layers[0]["attn_q"]
    layers[1]["window"] = layers[0]["window"]
    idx, out = orc.layer_stack(orc.default_plan(modes), layers, k=32, scale=0.125)
    assert np.array_equal(out[1], out[0])


def test_modes_reindex_uses_full_layer_kv(orc):
    # the Reindex layer's attention reads the Full layer's cache: swapping
    # in another cache for layer 1 changes nothing
    modes = [F, RI]
    layers = small_stack_layers(orc, modes, 80)
    idx_a, out_a = orc.layer_stack(orc.default_plan(modes), layers, k=32, scale=0.125)
    other = small_stack_layers(orc, [F], 81)[0]
    layers[1].update({"codes": other["codes"], "scales": other["scales"], "k8": other["k8"]})
    idx_b, out_b = orc.layer_stack(orc.default_plan(modes), layers, k=32, scale=0.125)
    assert np.array_equal(idx_a[1], idx_b[1]) and np.array_equal(out_a[1], out_b[1])


# ---- Hierarchical Sparse Indexer (candidate pool shared by a Full layer) ----

def test_pool_covering_every_entry_is_the_plain_schedule(orc):
    # a pool as large as the sequence restricts nothing: the hierarchical
    # schedule reduces to the plain one
    modes = [F, RI, RU, RI]
    layers = small_stack_layers(orc, modes, 90, n=300)
    plain = orc.layer_stack(orc.default_plan(modes), layers, k=32, scale=0.125)
    pooled = orc.layer_stack(orc.default_plan(modes), layers, k=32, scale=0.125, pool=300)
    for a, b in zip(plain[0], pooled[0]):
        assert np.array_equal(a, b)
    for a, b in zip(plain[1], pooled[1]):
        assert np.array_equal(a, b)


def test_pool_same_q_reproduces_full(orc):
    # the Full layer's top-k lies inside its own pool, so a Reindex layer with
    # the Full layer's queries still selects exactly the Full layer's entries
    modes = [F, RI]
    layers = small_stack_layers(orc, modes, 91, same_q=True)
    idx, _ = orc.layer_stack(orc.default_plan(modes), layers, k=32, scale=0.125, pool=64)
    assert np.array_equal(idx[1], idx[0])


def test_pool_selection_by_sorting(orc):
    # brute force: score every entry with the Reindex queries, keep the pool
    # members of the Full layer's 64 best (by sorting), sort those by (score
    # descending, index ascending) and take 32
    modes = [F, RI]
    layers = small_stack_layers(orc, modes, 92, B=3, n=200)
    idx, _ = orc.layer_stack(orc.default_plan(modes), layers, k=32, scale=0.125, pool=64)
    full = orc.index_score_fp8(layers[0]["idx_q"], layers[0]["idx_w"], layers[0]["k8"])
    re = orc.index_score_fp8(layers[1]["idx_q"], layers[1]["idx_w"], layers[0]["k8"])
    plain, _ = orc.layer_stack(orc.default_plan(modes), layers, k=32, scale=0.125)
    left_pool = 0
    for q in range(3):
        pool = sorted(range(200), key=lambda j: (-full[q, j], j))[:64]
        best = sorted(pool, key=lambda j: (-re[q, j], j))[:32]
        assert list(idx[1][q]) == sorted(best)
        left_pool += not set(plain[1][q]) <= set(pool)
    # the case is not trivial: the plain Reindex selection leaves the pool
    assert left_pool > 0


def test_pool_with_short_rows(orc):
    # fewer visible entries than the pool: the pool is every visible entry and
    # the Reindex layer selects as in the plain schedule; -1 pads a row with
    # fewer visible entries than k
    modes = [F, RI]
    layers = small_stack_layers(orc, modes, 93, B=3, n=120)
    nv = np.array([120, 50, 20], dtype=np.int32)
    plain, _ = orc.layer_stack(orc.default_plan(modes), layers, k=32, scale=0.125, n_valid=nv)
    pooled, _ = orc.layer_stack(orc.default_plan(modes), layers, k=32, scale=0.125, n_valid=nv,
                                pool=64)
    assert np.array_equal(plain[0], pooled[0])
    assert np.array_equal(plain[1][1:], pooled[1][1:])   # rows with nv <= pool
    assert list(pooled[1][2][20:]) == [-1] * 12


# ---- paged caches (the serving layout) --------------------------------------

def test_pages_identity_table_is_the_contiguous_layout(orc):
    B, n, page_rows = 3, 40, 16
    cache = synth.normal((B, 48, 32), 300).double().numpy()  # 3 pages of 16 rows per sequence
    pool = cache.reshape(B * 3, page_rows, 32)
    table = np.arange(B * 3).reshape(B, 3)
    assert np.array_equal(orc.gather_pages(pool, table, n), cache[:, :n])


def test_pages_permuted_pool_gives_the_same_view(orc):
    # moving physical pages (and updating the table) changes no logical row
    B, page_rows = 2, 8
    cache = synth.normal((B, 32, 4), 301).double().numpy()
    pool = cache.reshape(B * 4, page_rows, 4)
    table = np.arange(B * 4).reshape(B, 4)
    perm = np.random.default_rng(302).permutation(B * 4)   # new position of each page
    moved = np.empty_like(pool)
    moved[perm] = pool
    assert np.array_equal(orc.gather_pages(moved, perm[table], 30),
                          orc.gather_pages(pool, table, 30))


def test_pages_feed_the_selection_unchanged(orc):
    # the stack on a paged indexer-K cache, read through its logical view,
    # selects what the contiguous cache selects
    B, n, page_rows = 2, 200, 64
    kb = synth.normal((B, 256, 128), 303).double().numpy()
    k8 = orc.cast_e4m3(kb)
    q = synth.normal((B, 4, 128), 304).double().numpy()
    w = np.full((B, 4), 0.25)
    pool = k8.reshape(B * 4, page_rows, 128)[::-1].copy()   # pages stored in reverse order
    table = (B * 4 - 1 - np.arange(B * 4)).reshape(B, 4)
    ref = orc.topk(orc.index_score_fp8(q, w, k8[:, :n]), 16)
    got = orc.topk(orc.index_score_fp8(q, w, orc.gather_pages(pool, table, n)), 16)
    assert np.array_equal(got, ref)


# ---- Hierarchical Sparse Indexer: block-level pruning ------------------------

def test_block_summaries_hand_worked(orc):
    # blocks of 2 entries over 5 entries (the last block has one entry and a
    # zero): block key = E4M3((sum of the decoded keys) / 2).  Input codes:
    # 1 = 0x38, 3 = 0x44, 2 = 0x40, 0.5 = 0x30, 448 = 0x7E, -1 = 0xB8,
    # 1.125 = 0x39, -2 = 0xC0, -3 = 0xC4, 6 = 0x4C (E4M3: bias 7, 3 mantissa
    # bits).  Expected: (1+3)/2 = 2 -> 0x40; (1+2)/2 = 1.5 -> 0x3C; (0.5+0)/2
    # = 0.25 -> 0x28; 448 -> 0x7E; (-1+1)/2 = 0 -> 0x00; 1/2 -> 0x30;
    # (1+1.125)/2 = 1.0625, halfway between 1 (0x38) and 1.125 (0x39): ties
    # to the even mantissa -> 0x38; (-2-3)/2 = -2.5 -> 0xC2; 6/2 = 3 -> 0x44.
    cols = [[0x38, 0x44, 0x38, 0x40, 0x30],
            [0x7E, 0x7E, 0xB8, 0x38, 0x38],
            [0x38, 0x39, 0xC0, 0xC4, 0x4C],
            [0x00, 0x00, 0x00, 0x00, 0x00]]
    k8 = np.array(cols, dtype=np.uint8).T[None]           # [1, 5, 4]
    got = orc.block_summaries(k8, 2)
    want = np.array([[0x40, 0x7E, 0x38, 0x00],
                     [0x3C, 0x00, 0xC2, 0x00],
                     [0x28, 0x30, 0x44, 0x00]], dtype=np.uint8)[None]
    assert np.array_equal(got, want)


def test_block_pool_expands_ascending_blocks(orc):
    pool = orc.block_pool(np.array([[0, 2, -1], [1, 3, 4]]), 4, 18)
    assert pool[0].tolist() == [0, 1, 2, 3, 8, 9, 10, 11, -1, -1, -1, -1]
    assert pool[1].tolist() == [4, 5, 6, 7, 12, 13, 14, 15, 16, 17, -1, -1]


def test_blocks_keeping_every_block_is_the_plain_schedule(orc):
    modes = [F, RI, RU, RI]
    layers = small_stack_layers(orc, modes, 94, n=300)
    plain = orc.layer_stack(orc.default_plan(modes), layers, k=32, scale=0.125)
    blocked = orc.layer_stack(orc.default_plan(modes), layers, k=32, scale=0.125, block=16,
                              blocks_kept=19)   # 19 blocks of 16 cover 300 entries
    for a, b in zip(plain[0] + plain[1], blocked[0] + blocked[1]):
        assert np.array_equal(a, b)


def test_single_entry_blocks_keep_the_full_top_k(orc):
    # blocks of one entry: a block's key is the entry's own key, so the top-k
    # blocks are the top-k entries and the Full layer selects as in the plain
    # schedule; the Reindex layer then chooses inside those k entries
    modes = [F, RI]
    layers = small_stack_layers(orc, modes, 95, n=200)
    plain, _ = orc.layer_stack(orc.default_plan(modes), layers, k=32, scale=0.125)
    blocked, _ = orc.layer_stack(orc.default_plan(modes), layers, k=32, scale=0.125, block=1,
                                 blocks_kept=32)
    assert np.array_equal(plain[0], blocked[0])
    assert all(set(blocked[1][q]) == set(plain[0][q]) for q in range(2))


def test_block_selection_by_sorting(orc):
    # brute force with loops: block keys as means of decoded keys (cast by
    # the E4M3 rule), block scores, the 3 best blocks by (score desc, block
    # asc), then the 16 best entries of those blocks by (score desc, index asc)
    modes = [F]
    layers = small_stack_layers(orc, modes, 96, B=2, n=100)
    G, Bk, k = 8, 3, 16
    idx, _ = orc.layer_stack(orc.default_plan(modes), layers, k=k, scale=0.125, block=G,
                             blocks_kept=Bk)
    L = layers[0]
    dec = orc.e4m3_decode(L["k8"])
    nb = -(-100 // G)
    summ = np.zeros((2, nb, 128))
    for b in range(2):
        for blk in range(nb):
            for j in range(blk * G, min(100, blk * G + G)):
                summ[b, blk] += dec[b, j]
    summ = orc.cast_e4m3(summ / G)
    sb = orc.index_score_fp8(L["idx_q"], L["idx_w"], summ)
    s = orc.index_score_fp8(L["idx_q"], L["idx_w"], L["k8"])
    for q in range(2):
        keep = sorted(range(nb), key=lambda t: (-sb[q, t], t))[:Bk]
        ents = [j for t in keep for j in range(t * G, min(100, t * G + G))]
        best = sorted(ents, key=lambda j: (-s[q, j], j))[:k]
        assert list(idx[0][q]) == sorted(best)
