"""GPU parity of each CSA2 step against the fp64 oracle (through the C ABI).

Inputs come from the seeded generators in long_context_sparse_27_b300.synth
(drawn on the CPU, copied to the GPU); the oracle consumes the same bytes and
never any output of the CUDA path.  Bars: quantisers bit-exact, top-k
bit-exact on the same float32 scores, indexer scores within 1e-3 relative,
attention within 2e-3 relative L2 per (query, head).
"""
import math

import numpy as np
import pytest
import torch

from gpu_util import f64, need_gpu, rel_l2, score_close
from long_context_sparse_27_b300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def csa2():
    return need_gpu()


def dev(t):
    return t.to("cuda")


# ---------------------------------------------------------------- a1 quantiser

def fp4_inputs(rows, d, seed):
    x = synth.normal((rows, d), seed, dtype=torch.float32)
    # blocks across magnitudes, zero blocks, tiny and huge blocks, ties
    scale = torch.exp2(torch.randint(-130, 120, (rows, d // 32),
                                     generator=torch.Generator().manual_seed(seed + 1)).float())
    x = (x.view(rows, d // 32, 32) * scale[:, :, None]).view(rows, d)
    x[0, :32] = 0.0
    x[1, :32] = -0.0
    x[2, :8] = torch.tensor([6.0, 7.0, -5.0, 2.5, 0.25, 0.75, 1.25, 3.5])
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("rows,d", [(1000, 512), (37, 128), (5, 32)])
def test_quantize_fp4_bit_exact(csa2, orc, rows, d):
    x = fp4_inputs(rows, d, 100 + d)
    codes, scales = csa2.quantize_fp4(dev(x))
    rc, rs = orc.quantize_fp4(f64(x))
    assert np.array_equal(codes.cpu().numpy(), rc)
    assert np.array_equal(scales.cpu().numpy(), rs)


def test_quantize_fp4_every_bf16_pattern(csa2, orc):
    # all 65536 bf16 bit patterns (finite ones) as elements of 32-blocks
    bits = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    v = bits[torch.isfinite(bits.float())]
    v = v[: (v.numel() // 512) * 512].reshape(-1, 512)
    codes, scales = csa2.quantize_fp4(dev(v))
    rc, rs = orc.quantize_fp4(f64(v))
    assert np.array_equal(scales.cpu().numpy(), rs)
    assert np.array_equal(codes.cpu().numpy(), rc)


def test_quantize_fp4_strided_rows_and_idxk(csa2, orc):
    # one new row per sequence written at row N-1 of a [B, N, ...] cache
    B, N, d, di = 4, 10, 512, 128
    cache_c = torch.zeros(B, N, d // 2, dtype=torch.uint8, device="cuda")
    cache_s = torch.zeros(B, N, d // 32, dtype=torch.uint8, device="cuda")
    cache_k = torch.zeros(B, N, di, dtype=torch.uint8, device="cuda")
    x = synth.normal((B, d), 7)
    kx = synth.normal((B, di), 8) * 100  # reach the E4M3 saturation
    csa2.quantize_fp4(dev(x), cache_c[:, N - 1], cache_s[:, N - 1], dev(kx), cache_k[:, N - 1])
    rc, rs = orc.quantize_fp4(f64(x))
    assert np.array_equal(cache_c[:, N - 1].cpu().numpy(), rc)
    assert np.array_equal(cache_s[:, N - 1].cpu().numpy(), rs)
    assert np.array_equal(cache_k[:, N - 1].cpu().numpy(), orc.cast_e4m3(f64(kx)))
    assert int(cache_c[:, : N - 1].sum()) == 0 and int(cache_k[:, : N - 1].sum()) == 0


def test_cast_e4m3_every_bf16_pattern(csa2, orc):
    bits = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    v = bits[torch.isfinite(bits.float())]
    v = v[: (v.numel() // 128) * 128].reshape(-1, 128)
    x = torch.zeros(v.shape[0], 32, dtype=torch.bfloat16)
    _, _, k8 = csa2.quantize_fp4(dev(x), idxk=dev(v))
    assert np.array_equal(k8.cpu().numpy(), orc.cast_e4m3(f64(v)))


# ---------------------------------------------------------- a2 indexer-Q quant

def test_quantize_index_q_bit_exact(csa2, orc):
    nq, hi, di = 12, 64, 128
    q = synth.normal((nq, hi, di), 11, dtype=torch.float32)
    mag = torch.exp2(torch.randint(-140, 100, (nq, hi, 1),
                                   generator=torch.Generator().manual_seed(12)).float())
    q = (q * mag).to(torch.bfloat16)
    q[0, 0] = 0.0
    q[0, 1, 3] = 448.0
    q[0, 2, 3] = 450.0
    w = synth.uniform((nq, hi), 13, scale=1 / 64)
    q8, c = csa2.quantize_index_q(dev(q), dev(w))
    rq8, rc = orc.quantize_index_q(f64(q), f64(w))
    assert np.array_equal(q8.cpu().numpy(), rq8)
    # c is an fp32 output: the oracle's exact w * sigma rounded to fp32 (they
    # differ from the exact value only where w * sigma is an fp32 subnormal)
    assert np.array_equal(c.cpu().numpy(), rc.astype(np.float32))


# ------------------------------------------------------------- a3 index score

def test_index_score_f32_tiny(csa2, orc):
    w_ = synth.TINY
    q = synth.index_q(w_, 20)
    w = synth.index_w(w_, 21)
    k = synth.index_k_rows(w_, 22)
    s = csa2.index_score(dev(q), dev(w), dev(k))
    ref = orc.index_score(f64(q), f64(w), f64(k))
    assert score_close(s.cpu().numpy(), ref) <= 1.0


@pytest.mark.parametrize("B,n", [(2, 1000), (3, 4096), (1, 128), (1, 77)])
def test_index_score_fp8_decode(csa2, orc, B, n):
    wl = synth.scaled(synth.C128K, B=B, N=n)
    q = synth.index_q(wl, 30 + n)
    w = synth.index_w(wl, 31 + n)
    kb = synth.index_k_rows(wl, 32 + n)
    x = torch.zeros(B * n, 32, dtype=torch.bfloat16, device="cuda")
    _, _, k8 = csa2.quantize_fp4(x, idxk=dev(kb.reshape(B * n, 128)))
    k8 = k8.reshape(B, n, 128)
    s = csa2.index_score(dev(q), dev(w), k8)
    ref = orc.index_score_fp8(f64(q), f64(w), orc.cast_e4m3(f64(kb)))
    assert score_close(s.cpu().numpy(), ref) <= 1.0


@pytest.mark.parametrize("B,n", [(8, 262144), (3, 1000), (2, 130), (600, 128)])
def test_index_score_fused_q_matches_separate_quantiser(csa2, orc, B, n):
    # decode launches quantise the bf16 indexer queries inside the indexer
    # kernel; the scores must equal, bit for bit, those of the same kernel
    # fed the separately quantised q8 and c (csa2_quantize_index_q, itself
    # bit-exact against the oracle).  600 queries of 128 entries give CTAs
    # spanning more than two queries: that launch takes the separate path.
    wl = synth.scaled(synth.C128K, B=B, N=n)
    q = synth.index_q(wl, 34 + n, "cuda")
    q[0, 5] = 0.0                              # an all-zero head
    q[min(1, B - 1), 7, 3] = 3.0e38            # saturating magnitudes
    w = synth.index_w(wl, 35 + n, "cuda")
    k8 = torch.randint(0, 0x7F, (B, n, 128), dtype=torch.uint8, device="cuda",
                       generator=torch.Generator(device="cuda").manual_seed(36 + n))
    fused = csa2.index_score(q, w, k8)
    q8, c = csa2.quantize_index_q(q, w)
    sep = csa2.index_score(q8, c, k8)
    torch.cuda.synchronize()
    assert torch.equal(fused.view(torch.int32), sep.view(torch.int32))
    rq8, rc = orc.quantize_index_q(f64(q), f64(w))
    assert np.array_equal(q8.cpu().numpy(), rq8)


def test_index_score_fp8_prefill_causal(csa2, orc):
    # 8 queries of one sequence at the end of a 4x-compressed context
    wl = synth.scaled(synth.PREFILL, q_per_seq=8, N=700, pos0=4 * 700 - 8)
    q = synth.index_q(wl, 40)
    w = synth.index_w(wl, 41)
    kb = synth.index_k_rows(wl, 42)
    nv = synth.prefill_n_valid(wl)
    assert int(nv.min()) < 700 and int(nv.max()) == 700
    x = torch.zeros(700, 32, dtype=torch.bfloat16, device="cuda")
    _, _, k8 = csa2.quantize_fp4(x, idxk=dev(kb.reshape(700, 128)))
    s = csa2.index_score(dev(q), dev(w), k8.reshape(1, 700, 128), q_per_seq=8, n_valid=dev(nv))
    ref = orc.index_score_fp8(f64(q), f64(w), orc.cast_e4m3(f64(kb)), q_per_seq=8,
                              n_valid=nv.numpy())
    assert score_close(s.cpu().numpy(), ref) <= 1.0


def test_index_score_prefill_relu_scalings_agree(csa2, orc):
    # the prefill epilogue takes ReLU as a saturating multiply by 2^-25 and
    # undoes the scale on the head weights, or, where a weight reaches 2^100,
    # on the head sums; queries 4..7 repeat queries 0..3 with weights scaled
    # by 2^110, so they take the second form and must give the same scores
    # times 2^110, bit for bit (both are exact up to power-of-two scalings).
    # Keys of magnitude <= 1 keep the scaled scores below the fp32 range.
    n = 1000
    g = torch.Generator().manual_seed(61)

    def e4m3_bytes(shape, top):
        b = torch.randint(0, top + 1, shape, generator=g, dtype=torch.int32)
        return (b | (torch.randint(0, 2, shape, generator=g, dtype=torch.int32) << 7)).to(
            torch.uint8)

    q8 = e4m3_bytes((4, 64, 128), 0x7E).repeat(2, 1, 1)
    c = (torch.rand(4, 64, generator=g, dtype=torch.float64) * 2 - 1) / 64
    c = torch.cat([c, c * 2.0 ** 110]).float()
    k8 = e4m3_bytes((1, n, 128), 0x38)
    s = csa2.index_score(dev(q8), dev(c), dev(k8), q_per_seq=8).cpu()
    assert torch.isfinite(s).all()
    assert torch.equal((s[:4].double() * 2.0 ** 110).float().view(torch.int32),
                       s[4:].view(torch.int32))
    ref = orc.index_score(orc.e4m3_decode(q8.numpy()), c.double().numpy(),
                          orc.e4m3_decode(k8.numpy()), q_per_seq=8)
    assert score_close(s.numpy(), ref) <= 1.0


def _score_keys(s):
    """Order-preserving uint32 keys of float32 scores (-0 counts as +0)."""
    u = np.ascontiguousarray(s, dtype=np.float32).view(np.uint32).copy()
    u[u == 0x80000000] = 0
    return np.where(u & 0x80000000, ~u, u | 0x80000000).astype(np.uint32)


def test_index_candidates_are_the_scores_at_or_above_theta(csa2):
    # the prefill scoring pass that stores no scores keeps exactly the
    # visible entries whose score key is >= theta[q], with the keys of
    # csa2_index_score's scores; reserved slots left unused hold entry
    # 0xFFFFFFFF (slots are reserved 32 at a time, or exactly when a query's
    # tiles spread over many CTAs, as here); a buffer too small for a query's
    # candidates reports more slots than it holds
    T, n = 16, 5000
    wl = synth.scaled(synth.PREFILL, q_per_seq=T, N=n, pos0=4 * n - T)
    q = synth.index_q(wl, 320, "cuda")
    w = synth.index_w(wl, 321, "cuda")
    k8 = torch.randint(0, 0x7F, (1, n, 128), dtype=torch.uint8, device="cuda",
                       generator=torch.Generator(device="cuda").manual_seed(322))
    nv = synth.prefill_n_valid(wl, "cuda")
    s = csa2.index_score(q, w, k8, q_per_seq=T, n_valid=nv).cpu().numpy()
    keys = _score_keys(s)
    nvh = nv.cpu().numpy()
    theta = np.zeros(T, np.uint32)
    for t in range(T):
        theta[t] = np.sort(keys[t, :nvh[t]])[::-1][min(299, nvh[t] - 1)]
    theta[3] = 0            # every visible entry
    theta[5] = 0xFFFFFFFF   # none (no score reaches the largest key)
    th = torch.from_numpy(theta.view(np.int32)).cuda()
    cap = n + 1024
    cand, cnt = csa2.index_candidates(q, w, k8, th, cap, T, n_valid=nv)
    cand, cnt = cand.cpu().numpy().view(np.uint64), cnt.cpu().numpy().view(np.uint32)
    for t in range(T):
        assert cnt[t] <= cap
        c = cand[t, :cnt[t]]
        ent = (c >> np.uint64(32)).astype(np.uint32)
        key = (c & np.uint64(0xFFFFFFFF)).astype(np.uint32)
        filled = ent != 0xFFFFFFFF
        assert np.all(key[~filled] == 0)
        want = np.nonzero(keys[t, :nvh[t]] >= theta[t])[0]
        got = np.sort(ent[filled])
        assert np.array_equal(got, want), t
        assert np.array_equal(key[filled], keys[t, ent[filled]]), t
    assert cnt[5] == 0 and (cnt[3] >= nvh[3])
    # a buffer of 64 slots: the counter still counts every reservation
    cand2, cnt2 = csa2.index_candidates(q, w, k8, th, 64, T, n_valid=nv)
    assert int(cnt2.cpu().numpy().view(np.uint32)[3]) >= nvh[3] > 64


def test_index_score_fp8_exact_small_integers(csa2, orc):
    # q and k with small-integer E4M3 values (q8 in {0, +-64, 448}, k in
    # {0, +-1}): every product and partial sum is an integer below 2^14, so
    # the tensor-core path must reproduce the oracle exactly
    B, n = 1, 256
    g = torch.Generator().manual_seed(50)
    q = torch.randint(-1, 2, (1, 64, 128), generator=g).to(torch.bfloat16)
    q[0, :, 0] = 7  # fixes every head's scale at 2^-6 (amax 7)
    w = torch.full((1, 64), 1.0 / 64)
    kb = torch.randint(-1, 2, (n, 128), generator=g).to(torch.bfloat16)
    x = torch.zeros(n, 32, dtype=torch.bfloat16, device="cuda")
    _, _, k8 = csa2.quantize_fp4(x, idxk=dev(kb))
    s = csa2.index_score(dev(q), dev(w), k8.reshape(1, n, 128))
    ref = orc.index_score_fp8(f64(q), f64(w), orc.cast_e4m3(f64(kb)).reshape(1, n, 128))
    assert np.array_equal(s.cpu().double().numpy(), ref)


@pytest.mark.parametrize("B,n,P", [(2, 3000, 2048), (3, 1000, 300), (1, 200, 77)])
def test_index_score_pool(csa2, orc, B, n, P):
    # the Hierarchical Sparse Indexer's restricted scoring: each query's pool
    # is a random set of its sequence's entries (some slots empty, -1); ragged
    # pool sizes leave a partial 128-slot tile
    wl = synth.scaled(synth.C128K, B=B, N=n)
    q = synth.index_q(wl, 35 + n)
    w = synth.index_w(wl, 36 + n)
    kb = synth.index_k_rows(wl, 37 + n)
    x = torch.zeros(B * n, 32, dtype=torch.bfloat16, device="cuda")
    _, _, k8 = csa2.quantize_fp4(x, idxk=dev(kb.reshape(B * n, 128)))
    k8 = k8.reshape(B, n, 128)
    g = torch.Generator().manual_seed(38 + n)
    pool = torch.stack([torch.randperm(n, generator=g)[:P] for _ in range(B)]).to(torch.int32)
    pool[:, -5:] = -1
    s = csa2.index_score_pool(dev(q), dev(w), k8, dev(pool)).cpu().numpy()
    ref = orc.index_score_fp8(f64(q), f64(w), orc.cast_e4m3(f64(kb)))
    for b in range(B):
        keep = pool[b].numpy() >= 0
        assert np.all(np.isneginf(s[b, ~keep]))
        assert score_close(s[b:b + 1, keep], ref[b:b + 1, pool[b].numpy()[keep]]) <= 1.0


def test_index_score_pool_exact_small_integers(csa2, orc):
    # the exact case of the full indexer, through the pooled kernel: small
    # integer E4M3 values make every product and sum exact
    n, P = 256, 256
    g = torch.Generator().manual_seed(51)
    q = torch.randint(-1, 2, (1, 64, 128), generator=g).to(torch.bfloat16)
    q[0, :, 0] = 7
    w = torch.full((1, 64), 1.0 / 64)
    kb = torch.randint(-1, 2, (n, 128), generator=g).to(torch.bfloat16)
    x = torch.zeros(n, 32, dtype=torch.bfloat16, device="cuda")
    _, _, k8 = csa2.quantize_fp4(x, idxk=dev(kb))
    pool = torch.randperm(n, generator=g)[None, :P].to(torch.int32)
    s = csa2.index_score_pool(dev(q), dev(w), k8.reshape(1, n, 128), dev(pool))
    ref = orc.index_score_fp8(f64(q), f64(w), orc.cast_e4m3(f64(kb)).reshape(1, n, 128))
    assert np.array_equal(s.cpu().double().numpy()[0], ref[0, pool[0].numpy()])


# ------------------------------------ the decoder's global KV (projection + a1)

@pytest.mark.parametrize("rows,hidden,d", [(8, 4096, 512), (100, 256, 128), (1, 64, 64),
                                           (1024, 512, 512), (5, 416, 64), (65, 4096, 64),
                                           (300, 1024, 512), (64, 768, 192),
                                           # at most 16 rows: one round of loads per CTA,
                                           # uneven and empty shares of the hidden features,
                                           # the largest hidden size of that path and past it
                                           (16, 4096, 512), (3, 96, 128), (16, 16384, 64),
                                           (12, 16416, 64), (17, 512, 64)])
def test_project_fp4(csa2, orc, rows, hidden, d):
    h = synth.normal((rows, hidden), 210 + rows)
    w = synth.normal((d, hidden), 211 + rows) * 0.05
    w = w.to(torch.bfloat16)
    h[0] = 0  # an all-zero row: scale byte 0, zero codes
    codes, scales, out = csa2.project_fp4(dev(h), dev(w), with_out=True)
    g = out.cpu().double().numpy()
    ref = orc.project_kv(f64(h), f64(w))
    # fp32 summation of exact bf16 products: |error| <= hidden * 2^-23 * sum |terms| (the
    # recursive-summation bound with the unit of a truncating adder)
    bound = hidden * 2.0 ** -23 * (np.abs(f64(h)) @ np.abs(f64(w)).T)
    assert np.all(np.abs(g - ref) <= bound + 1e-30)
    # the codes: the oracle's quantiser on the kernel's own fp32 projection
    rc, rs = orc.quantize_fp4(g)
    assert np.array_equal(codes.cpu().numpy(), rc) and np.array_equal(scales.cpu().numpy(), rs)
    assert int(scales[0].abs().sum()) == 0 and int(codes[0].sum()) == 0


@pytest.mark.parametrize("rows", [70, 9])
def test_project_fp4_exact_small_integers(csa2, orc, rows):
    # integer inputs keep every product and partial sum exact in fp32: the
    # projection and its codes match the oracle's fp64 path bit for bit
    g = torch.Generator().manual_seed(212)
    h = torch.randint(-3, 4, (rows, 256), generator=g).to(torch.bfloat16)
    w = torch.randint(-2, 3, (128, 256), generator=g).to(torch.bfloat16)
    codes, scales, out = csa2.project_fp4(dev(h), dev(w), with_out=True)
    assert np.array_equal(out.cpu().double().numpy(), orc.project_kv(f64(h), f64(w)))
    rc, rs = orc.project_quantize_fp4(f64(h), f64(w))
    assert np.array_equal(codes.cpu().numpy(), rc) and np.array_equal(scales.cpu().numpy(), rs)


# -------------------------------------------------------------------- a4 top-k

@pytest.mark.parametrize("rows,n,k,levels", [
    (3, 5000, 64, 0), (4, 4096, 512, 0), (5, 3000, 512, 40), (2, 262144, 512, 0),
    (2, 70000, 512, 3), (6, 1000, 2048, 0), (1, 100, 512, 0), (9, 1, 1, 0),
    (4, 8000, 512, 1), (300, 5000, 256, 0), (37, 40000, 512, 0), (3, 262144, 2048, 5),
    # rows of an odd length: the histogram pass and the slices take scalar loads
    (3, 30001, 512, 0), (1, 4097, 64, 2)])
def test_topk_bit_exact(csa2, orc, rows, n, k, levels):
    s = synth.scores_with_ties(rows, n, seed=60 + rows + k, levels=levels)
    g = torch.Generator().manual_seed(61)
    nv = torch.randint(0, n + 1, (rows,), generator=g).int()
    nv[0] = n
    got = csa2.topk(dev(s), k, n_valid=dev(nv))
    ref = orc.topk(f64(s), k, nv.numpy())
    assert np.array_equal(got.cpu().numpy(), ref)


@pytest.mark.parametrize("n", [20000, 4000])   # cluster selector; one CTA per short row
def test_topk_degenerate_rows(csa2, orc, n):
    k = 512
    s = torch.zeros(6, n)
    s[1] = 1.0                                   # all equal: lowest indices win
    s[2, ::2] = -0.0                             # signed zeros compare equal
    s[3, n // 4:] = 2.0                          # a long run of equal maxima
    s[4] = torch.arange(n).float().flip(0)       # strictly decreasing
    s[5] = -torch.inf
    s[5, 17] = 3.0
    got = csa2.topk(dev(s), k)
    ref = orc.topk(f64(s), k)
    assert np.array_equal(got.cpu().numpy(), ref)


def test_topk_long_equal_runs(csa2, orc):
    # rows long enough that one warp's share of a row holds more entries in
    # the top bins than its ordered list keeps, so the selector re-reads them
    n, k = 200000, 512
    s = torch.zeros(4, n)
    s[0] = 0.5                                    # all equal
    s[1, 100000:] = 1.0                           # a long run of equal maxima
    s[2] = synth.scores_with_ties(1, n, seed=71, levels=3)[0]  # three values
    s[3, ::3] = 7.0
    s[3, 150000:150010] = 8.0                     # a few above a long tie run
    got = csa2.topk(dev(s), k)
    ref = orc.topk(f64(s), k)
    assert np.array_equal(got.cpu().numpy(), ref)


def test_topk_strided_rows(csa2, orc):
    s = synth.scores_with_ties(4, 3000, seed=70)
    big = torch.full((4, 3100), 99.0)
    big[:, :3000] = s
    out = torch.full((4, 600), -7, dtype=torch.int32, device="cuda")
    csa2.topk(dev(big)[:, :3000], 512, out=out[:, :512])
    assert np.array_equal(out[:, :512].cpu().numpy(), orc.topk(f64(s), 512))
    assert int((out[:, 512:] != -7).sum()) == 0


# -------------------------------------------------------- a5 sparse attention

def make_cache(csa2, B, n, d, seed):
    x = synth.normal((B * n, d), seed)
    codes, scales = csa2.quantize_fp4(dev(x))
    return (codes.reshape(B, n, d // 2), scales.reshape(B, n, d // 32))


def oracle_cache(orc, B, n, d, seed):
    x = synth.normal((B * n, d), seed)
    c, s = orc.quantize_fp4(f64(x))
    return c.reshape(B, n, d // 2), s.reshape(B, n, d // 32)


def test_attn_f32_tiny(csa2, orc):
    wl = synth.TINY
    codes, scales = make_cache(csa2, 1, wl.N, wl.D, 80)
    rc, rs = oracle_cache(orc, 1, wl.N, wl.D, 80)
    q = synth.attn_q(wl, 81)
    idx = synth.random_indices(1, wl.k, wl.N, 82, pad=5)
    win = synth.window_rows(wl, 83)
    scale = 1 / math.sqrt(wl.D)
    out = csa2.sparse_attn(dev(q), codes, scales, dev(idx), dev(win), scale)
    ref = orc.sparse_attn(f64(q), rc, rs, idx.numpy(), f64(win), scale)
    assert rel_l2(out.cpu().numpy(), ref) <= 2e-3


# (3, 64, 2000, 512, 128): 640 keys = 8 chunks of 80, merged on chip (the
# 128K / 1M decode shape); (2, 16, 3000, 1024, 128): 15 chunks, merged
# through the workspace; the others are ragged single / few-chunk cases.
@pytest.mark.parametrize("nq,hq,n,k,W", [(3, 64, 2000, 512, 128), (2, 16, 300, 64, 7),
                                          (1, 32, 50, 8, 0), (2, 16, 600, 512, 128),
                                          (2, 16, 3000, 1024, 128), (1, 16, 700, 560, 80)])
def test_attn_bf16(csa2, orc, nq, hq, n, k, W):
    d = 512
    codes, scales = make_cache(csa2, nq, n, d, 90 + n)
    rc, rs = oracle_cache(orc, nq, n, d, 90 + n)
    q = synth.normal((nq, hq, d), 91)
    idx = synth.random_indices(nq, k, n, 92, pad=min(k, 13))
    win = synth.normal((nq, max(W, 1), d), 93)[:, :W]
    scale = 1 / math.sqrt(d)
    out = csa2.sparse_attn(dev(q), codes, scales, dev(idx), dev(win).contiguous(), scale)
    ref = orc.sparse_attn(f64(q), rc, rs, idx.numpy(), f64(win), scale)
    assert rel_l2(out.cpu().numpy(), ref) <= 2e-3


def test_attn_bf16_single_key_is_the_dequantised_row(csa2, orc):
    # one selected entry, no window and q = 0: its softmax weight is exactly
    # 1, so the output is the dequantised FP4 row itself, bit for bit.  The
    # rows hold every code byte, with scale bytes 0..252 -- every byte the
    # quantiser writes for bf16 input (the fast bf16 path for 8..250, the
    # fp32 path outside it; 253 and 254 would overflow bf16).
    d, n, hq = 512, 253, 48
    codes = torch.arange(n * d // 2, dtype=torch.int64).remainder(256).to(torch.uint8)
    codes = codes.reshape(n, d // 2)
    codes = codes[:, torch.randperm(d // 2, generator=torch.Generator().manual_seed(124))]
    scales = torch.arange(n * d // 32, dtype=torch.int64).remainder(253).to(torch.uint8)
    scales = scales.reshape(n, d // 32)
    ref_rows = orc.dequantize_fp4(codes.numpy(), scales.numpy(), d)      # [n, d]
    # n queries of one sequence; query j selects entry j
    q = torch.zeros((n, hq, d), dtype=torch.bfloat16)
    idx = torch.arange(n, dtype=torch.int32).reshape(n, 1)
    win = torch.zeros((1, 0, d), dtype=torch.bfloat16)
    out = csa2.sparse_attn(dev(q), dev(codes)[None], dev(scales)[None], dev(idx), dev(win), 0.01,
                           q_per_seq=n)
    got = out.cpu().double().numpy()
    assert np.array_equal(got, np.broadcast_to(ref_rows[:, None, :], got.shape))


def test_attn_bf16_empty_chunks(csa2, orc):
    # 200 selected entries then 312 x -1: chunks 3..5 hold no key at all and
    # must drop out of the merge (their max is -inf)
    d, n, k, W, hq = 512, 400, 512, 128, 32
    codes, scales = make_cache(csa2, 2, n, d, 120)
    rc, rs = oracle_cache(orc, 2, n, d, 120)
    q = synth.normal((2, hq, d), 121)
    idx = synth.random_indices(2, k, n, 122, pad=312)
    win = synth.normal((2, W, d), 123)
    out = csa2.sparse_attn(dev(q), codes, scales, dev(idx), dev(win), 1 / math.sqrt(d))
    ref = orc.sparse_attn(f64(q), rc, rs, idx.numpy(), f64(win), 1 / math.sqrt(d))
    assert rel_l2(out.cpu().numpy(), ref) <= 2e-3


def test_attn_bf16_prefill_windows(csa2, orc):
    # 6 queries of one sequence; query t attends window rows t .. t + W - 1
    T, W, n, k, d, hq = 6, 5, 400, 64, 512, 16
    codes, scales = make_cache(csa2, 1, n, d, 95)
    rc, rs = oracle_cache(orc, 1, n, d, 95)
    q = synth.normal((T, hq, d), 96)
    idx = synth.random_indices(T, k, n, 97, pad=3)
    win = synth.normal((1, T + W - 1, d), 98)
    ws = torch.arange(T, dtype=torch.int32)
    wl = torch.tensor([W, W, 2, 0, W, 1], dtype=torch.int32)
    out = csa2.sparse_attn(dev(q), codes, scales, dev(idx), dev(win), 0.05, q_per_seq=T,
                           win_start=dev(ws), win_len=dev(wl), win_max=W)
    ref = orc.sparse_attn(f64(q), rc, rs, idx.numpy(), f64(win), 0.05, q_per_seq=T,
                          win_start=ws.numpy(), win_len=wl.numpy())
    assert rel_l2(out.cpu().numpy(), ref) <= 2e-3


def test_attn_bf16_many_queries_walk_their_chunks(csa2, orc):
    # 160 queries x 64 heads: 640 CTAs of 16 heads, enough to fill the GPU,
    # so each CTA takes one (query, head group) and walks its 8 chunks with a
    # running softmax (no partials); per-query windows (some short, one
    # empty) and ragged selections.  The same queries launched 8 at a time
    # (one CTA per chunk, merged in a cluster) meet the same bar.
    T, W, n, k, d, hq = 160, 128, 2000, 512, 512, 64
    codes, scales = make_cache(csa2, 1, n, d, 130)
    rc, rs = oracle_cache(orc, 1, n, d, 130)
    q = synth.normal((T, hq, d), 131)
    idx = synth.random_indices(T, k, n, 132, pad=37)
    win = synth.normal((1, T + W - 1, d), 133)
    ws = torch.arange(T, dtype=torch.int32)
    wl = torch.full((T,), W, dtype=torch.int32)
    wl[::7] = 3
    wl[5] = 0
    scale = 1 / math.sqrt(d)
    out = csa2.sparse_attn(dev(q), codes, scales, dev(idx), dev(win), scale, q_per_seq=T,
                           win_start=dev(ws), win_len=dev(wl), win_max=W)
    ref = orc.sparse_attn(f64(q), rc, rs, idx.numpy(), f64(win), scale, q_per_seq=T,
                          win_start=ws.numpy(), win_len=wl.numpy())
    assert rel_l2(out.cpu().numpy(), ref) <= 2e-3
    sub = slice(40, 48)
    out8 = csa2.sparse_attn(dev(q[sub]), codes, scales, dev(idx[sub]), dev(win), scale,
                            q_per_seq=8, win_start=dev(ws[sub]), win_len=dev(wl[sub]), win_max=W)
    assert rel_l2(out8.cpu().numpy(), ref[sub]) <= 2e-3


def test_attn_bounds_flag(csa2):
    d, n = 512, 100
    codes, scales = make_cache(csa2, 1, n, d, 99)
    q = dev(synth.normal((1, 16, d), 100))
    idx = torch.tensor([[3, 5, n, -2, 7, -1]], dtype=torch.int32, device="cuda")
    win = dev(synth.normal((1, 4, d), 101))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = csa2.sparse_attn(q, codes, scales, idx, win, 0.04, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & csa2.DEVFLAG_BOUNDS
    assert torch.isfinite(out).all()


def test_attn_window_longer_than_bound_flags(csa2):
    # a win_len above the launch bound win_max is clipped to win_max and
    # reported, like any other window range the launch cannot hold
    T, W, n, k, d, hq = 3, 4, 200, 16, 512, 16
    codes, scales = make_cache(csa2, 1, n, d, 130)
    q = dev(synth.normal((T, hq, d), 131))
    idx = dev(synth.random_indices(T, k, n, 132))
    win = dev(synth.normal((1, T + W, d), 133))
    ws = dev(torch.arange(T, dtype=torch.int32))
    for wl, flagged in (([W, W, W], False), ([W, W + 1, W], True)):
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = csa2.sparse_attn(q, codes, scales, idx, win, 0.04, q_per_seq=T, win_start=ws,
                               win_len=dev(torch.tensor(wl, dtype=torch.int32)), win_max=W,
                               dev_status=st)
        torch.cuda.synchronize()
        assert bool(int(st.item()) & csa2.DEVFLAG_BOUNDS) == flagged
        assert csa2.lib.csa2_status_from_device(int(st.item())) == (7 if flagged else 0)
        assert torch.isfinite(out).all()


def test_index_wait_timeout_returns_a_status(csa2, monkeypatch):
    # the device-side failure path: the indexer's producer issues no loads
    # (test hook), its MMA and epilogue waits run out after 1 ms, the kernel
    # returns with CSA2_DEVFLAG_TIMEOUT, and the context stays usable: the
    # same launch without the hook gives the scores of a clean run
    B, n = 4, 20000
    wl = synth.scaled(synth.C128K, B=B, N=n)
    q8, c = csa2.quantize_index_q(synth.index_q(wl, 140, "cuda"), synth.index_w(wl, 141, "cuda"))
    k8 = torch.randint(0, 0x7F, (B, n, 128), dtype=torch.uint8, device="cuda",
                       generator=torch.Generator(device="cuda").manual_seed(142))
    ref = csa2.index_score(q8, c, k8)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    monkeypatch.setenv("CSA2_TEST_STALL_LOADS", "1")
    monkeypatch.setenv("CSA2_WAIT_LIMIT_NS", "1000000")
    csa2.index_score(q8, c, k8, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & csa2.DEVFLAG_TIMEOUT
    assert csa2.lib.csa2_status_from_device(int(st.item())) == 6
    monkeypatch.delenv("CSA2_TEST_STALL_LOADS")
    monkeypatch.delenv("CSA2_WAIT_LIMIT_NS")
    st.zero_()
    again = csa2.index_score(q8, c, k8, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(again.view(torch.int32), ref.view(torch.int32))
