"""Seeded synthetic inputs for the CSA2 step.

This module only draws random tensors with the shapes and distributions of
the workloads; it holds none of the method's arithmetic (no quantisation,
no scoring, no selection).  Both the CUDA path and the oracle consume what
it produces.

Workload recipes (decode unless stated; N = compressed entries per sequence,
one entry per 4 tokens):

  tiny      B=1, N=4096, indexer 8 heads x 64 (fp32 q/k), top-64, 8 query
            heads, latent 128, window 32; q/k/attention-q ~ N(0,1) fp32,
            w ~ U(0,1)/8, KV ~ N(0,1) bf16; 1% of indexer-K rows x3.
  128k      B=16, N=32768, indexer 64 x 128 (bf16 q, K cast to E4M3),
            w ~ U(0,1)/64, top-512, 64 heads x 512 FP4 KV, window 128 bf16;
            all N(0,1); 1% of indexer-K rows x3.
  group3    B=32, N=65536, 128k shapes, Full -> Reindex -> Reuse; Gaussian,
            nothing planted; Reindex draws a fresh indexer Q and w.
  1m        B=8, N=262144, 128k shapes, 20 layers (Full, Reindex, Reuse,
            Reuse) x 5; Gaussian with 0.5% of indexer-K rows x3.
  prefill   4096 queries at positions 1,044,480..1,048,575 of one sequence,
            N=262144, 128k shapes, one Full layer; 1024 new KV rows.

"Planted" rows are indexer-K rows scaled by 3 before any cast, so that the
top-k set is well separated; the main KV is never planted.
"""
from dataclasses import dataclass, replace

import torch

FULL, REINDEX, REUSE = 0, 1, 2


@dataclass(frozen=True)
class Workload:
    name: str
    B: int            # sequences
    q_per_seq: int    # queries per sequence (1 in decode)
    N: int            # compressed entries per sequence
    Hi: int           # indexer heads
    Di: int           # indexer dim
    Hq: int           # attention heads
    D: int            # shared K = V latent dim
    k: int            # top-k
    W: int            # sliding-window rows
    fp32_indexer: bool
    attn_q_fp32: bool
    w_div: float      # w ~ U(0,1) / w_div
    plant_frac: float
    modes: tuple      # static layer schedule
    pos0: int = -1    # prefill: absolute token position of the first query
    pool: int = 0     # Hierarchical Sparse Indexer candidate pool (0 = off)
    page_rows: int = 0  # paged caches: entries per page (0 = contiguous caches)
    block: int = 0        # block-level pruning: entries per block (0 = off)
    blocks_kept: int = 0  # blocks a Full layer keeps

    @property
    def nq(self):
        return self.B * self.q_per_seq


TINY = Workload("tiny", B=1, q_per_seq=1, N=4096, Hi=8, Di=64, Hq=8, D=128, k=64, W=32,
                fp32_indexer=True, attn_q_fp32=True, w_div=8.0, plant_frac=0.01,
                modes=(FULL,))
C128K = Workload("128k", B=16, q_per_seq=1, N=32768, Hi=64, Di=128, Hq=64, D=512, k=512,
                 W=128, fp32_indexer=False, attn_q_fp32=False, w_div=64.0, plant_frac=0.01,
                 modes=(FULL,))
GROUP3 = Workload("group3", B=32, q_per_seq=1, N=65536, Hi=64, Di=128, Hq=64, D=512, k=512,
                  W=128, fp32_indexer=False, attn_q_fp32=False, w_div=64.0, plant_frac=0.0,
                  modes=(FULL, REINDEX, REUSE))
C1M = Workload("1m", B=8, q_per_seq=1, N=262144, Hi=64, Di=128, Hq=64, D=512, k=512, W=128,
               fp32_indexer=False, attn_q_fp32=False, w_div=64.0, plant_frac=0.005,
               modes=(FULL, REINDEX, REUSE, REUSE) * 5)
PREFILL = Workload("prefill", B=1, q_per_seq=4096, N=262144, Hi=64, Di=128, Hq=64, D=512,
                   k=512, W=128, fp32_indexer=False, attn_q_fp32=False, w_div=64.0,
                   plant_frac=0.0, modes=(FULL,), pos0=1048576 - 4096)

# one (Full, Reindex, Reuse, Reuse) group of the 1m stack: the same kernels
# and launch shapes with a fifth of the device memory (profiling captures)
C1M_GROUP = replace(C1M, name="1m4", modes=C1M.modes[:4])

# the 1m stack with the Hierarchical Sparse Indexer: every Reindex layer
# scores only the top-2048 pool of its Full layer
C1M_POOL = replace(C1M, name="1m-pool", pool=2048)

C1M_POOL_GROUP = replace(C1M_POOL, name="1m4-pool", modes=C1M.modes[:4])

# the 1m stack over paged caches: pages of 256 entries (1024 tokens), the
# pages of every sequence scattered over one pool in a seeded random order
C1M_PAGED = replace(C1M, name="1m-paged", page_rows=256)
C1M_PAGED_GROUP = replace(C1M_PAGED, name="1m4-paged", modes=C1M.modes[:4])

# the 1m stack with the Hierarchical Sparse Indexer's block-level pruning:
# blocks of 64 entries, a Full layer keeps its 32 best blocks (a 2048-entry
# pool) and scores only their entries
C1M_BLOCK = replace(C1M, name="1m-block", block=64, blocks_kept=32)
C1M_BLOCK_GROUP = replace(C1M_BLOCK, name="1m4-block", modes=C1M.modes[:4])
# a quarter of the prefill chunk (1024 queries): the same kernels with a
# quarter of the score scratch (profiling captures)
PREFILL_1K = replace(PREFILL, name="prefill1k", q_per_seq=1024, pos0=1048576 - 1024)

WORKLOADS = {w.name: w for w in (TINY, C128K, GROUP3, C1M, C1M_GROUP, PREFILL, C1M_POOL,
                                 C1M_POOL_GROUP, PREFILL_1K, C1M_PAGED, C1M_PAGED_GROUP,
                                 C1M_BLOCK, C1M_BLOCK_GROUP)}


def block_table(B, n, page_rows, seed, device="cpu", spare=None):
    """A paged layout's block table int32 [B, ceil(n / page_rows)]: every
    sequence's pages drawn without repetition, in a seeded random order, from
    a pool with `spare` (default B) pages no sequence uses.  Returns (table,
    pages in the pool)."""
    pps = (n + page_rows - 1) // page_rows
    spare = B if spare is None else spare
    num_pages = B * pps + spare
    g = _gen(seed, "cpu")
    perm = torch.randperm(num_pages, generator=g)[: B * pps]
    return perm.reshape(B, pps).to(torch.int32).to(device), num_pages


def scaled(w: Workload, **kw) -> Workload:
    """The same recipe at other sizes (parity cases the oracle finishes quickly)."""
    return replace(w, **kw)


def _gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal(shape, seed, device="cpu", dtype=torch.bfloat16):
    g = _gen(seed, device)
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(dtype)


def uniform(shape, seed, device="cpu", scale=1.0):
    g = _gen(seed, device)
    return torch.rand(shape, generator=g, device=device, dtype=torch.float32) * scale


def planted_rows(n_rows, frac, seed, device="cpu"):
    """Boolean mask over n_rows with round(frac * n_rows) seeded rows set."""
    m = torch.zeros(n_rows, dtype=torch.bool, device=device)
    cnt = int(round(frac * n_rows))
    if cnt > 0:
        g = _gen(seed, device)
        perm = torch.randperm(n_rows, generator=g, device=device)
        m[perm[:cnt]] = True
    return m


def index_k_rows(w: Workload, seed, device="cpu", n=None):
    """Indexer-K rows [B, n, Di] (bf16, or fp32 for the fp32 indexer), with
    the planted rows of each sequence scaled by 3."""
    n = w.N if n is None else n
    dt = torch.float32 if w.fp32_indexer else torch.bfloat16
    k = normal((w.B, n, w.Di), seed, device, torch.float32)
    if w.plant_frac > 0:
        for b in range(w.B):
            m = planted_rows(n, w.plant_frac, seed * 7919 + b + 1, device)
            k[b, m] *= 3.0
    return k.to(dt)


def index_q(w: Workload, seed, device="cpu"):
    dt = torch.float32 if w.fp32_indexer else torch.bfloat16
    return normal((w.nq, w.Hi, w.Di), seed, device, dt)


def index_w(w: Workload, seed, device="cpu"):
    return uniform((w.nq, w.Hi), seed, device, 1.0 / w.w_div)


def kv_rows(w: Workload, seed, device="cpu", n=None):
    """Main-KV latent rows [B, n, D] in bf16, before FP4 quantisation."""
    n = w.N if n is None else n
    return normal((w.B, n, w.D), seed, device, torch.bfloat16)


def attn_q(w: Workload, seed, device="cpu"):
    dt = torch.float32 if w.attn_q_fp32 else torch.bfloat16
    return normal((w.nq, w.Hq, w.D), seed, device, dt)


def window_rows(w: Workload, seed, device="cpu"):
    """Sliding-window rows: [B, W, D] in decode; [B, q_per_seq + W - 1, D] in
    prefill, where query t uses rows t .. t + W - 1."""
    rows = w.W if w.q_per_seq == 1 else w.q_per_seq + w.W - 1
    return normal((w.B, rows, w.D), seed, device, torch.bfloat16)


def prefill_n_valid(w: Workload, device="cpu"):
    """Causal visibility over compressed positions: a query at absolute
    position p sees the entries completed by then, floor((p + 1) / 4)."""
    p = torch.arange(w.q_per_seq, dtype=torch.int64, device=device) + w.pos0
    nv = torch.div(p + 1, 4, rounding_mode="floor").clamp(max=w.N)
    return nv.repeat(w.B).to(torch.int32)


def scores_with_ties(rows, n, seed, device="cpu", levels=0):
    """Synthetic score rows for exercising the selector on its own:
    N(0,1) fp32, or (levels > 0) integers in [0, levels) so ties abound."""
    if levels > 0:
        g = _gen(seed, device)
        return torch.randint(0, levels, (rows, n), generator=g, device=device).float()
    return normal((rows, n), seed, device, torch.float32)


def random_indices(rows, k, n, seed, device="cpu", pad=0):
    """rows x k distinct ascending indices in [0, n), the last `pad` of each
    row set to -1 (the selector's output format)."""
    g = _gen(seed, device)
    out = torch.full((rows, k), -1, dtype=torch.int32)
    for r in range(rows):
        sel = torch.randperm(n, generator=g, device=device)[: k - pad]
        out[r, : k - pad] = torch.sort(sel).values.to(torch.int32).cpu()
    return out.to(device)
