"""Device-resident inputs for one step of a CSA2 layer schedule.

Draws every tensor with the seeded generators of `synth`, fills each Full
layer's FP4 main-KV cache and E4M3 indexer-K cache for entries 0 .. N-2 with
the library's own quantiser, and keeps entry N-1 (the compressed entry that
completes in this decode step) as the step's new rows, which the layer
schedule quantises itself.  Also builds the descriptor array and stack
arguments for csa2_layer_stack.

Schedule sources: a Reindex layer reads the most recent Full layer's caches;
a Reuse layer reads the most recent Full layer's caches and top-k indices.
"""
import math
from dataclasses import dataclass

import torch

from . import csa2, synth

FULL, REINDEX, REUSE = synth.FULL, synth.REINDEX, synth.REUSE


def default_sources(modes):
    out, last_full = [], -1
    for l, m in enumerate(modes):
        if m == FULL:
            last_full = l
            out.append((l, l))
        elif m == REINDEX:
            out.append((last_full, l))
        else:
            out.append((last_full, last_full))
    return out


@dataclass
class StepIO:
    dev_in: torch.Tensor    # uint8: every per-step input of the step, packed
    dev_out: torch.Tensor   # uint8: every output of the step, packed
    layers: list            # the workload's layer dicts with inputs / outputs in the blocks
    descs: object           # csa2 layer descriptors of `layers`
    in_bytes: int           # payload bytes of dev_in (without alignment padding)
    out_bytes: int


class StackWorkload:
    """All tensors of one decode (or prefill) step, on `device`.

    gen_device: where the random draws happen ("cpu" keeps them reproducible
    for the oracle; "cuda" is fast for the large workloads).
    keep_bf16: keep the unquantised KV / indexer-K rows (on the host) so an
    oracle can quantise them itself.
    """

    def __init__(self, wl: synth.Workload, seed=0, device="cuda", gen_device=None,
                 keep_bf16=False, sources=None):
        self.wl = wl
        self.device = device
        gen = gen_device or device
        self.plan = sources or default_sources(wl.modes)
        self.pages = None
        if wl.page_rows:
            # one block table shared by every Full layer's pools
            self.block_table, self.num_pages = synth.block_table(
                wl.B, wl.N, wl.page_rows, seed * 1000 + 999, device)
            self.pages = csa2.pages(self.block_table, wl.page_rows, self.num_pages)
        self.layers = []
        self.bf16 = []
        B, N = wl.B, wl.N
        nq = wl.nq
        for l, m in enumerate(wl.modes):
            s = seed * 1000 + 20 * l
            kv_src, idx_src = self.plan[l]
            L = {"mode": m, "kv_src": kv_src, "idx_src": idx_src,
                 "attn_q": synth.attn_q(wl, s + 1, gen).to(device),
                 "window": synth.window_rows(wl, s + 2, gen).to(device),
                 "out": torch.empty(nq, wl.Hq, wl.D, dtype=torch.float32, device=device)}
            host = {}
            if m in (FULL, REINDEX):
                L["idx_q"] = synth.index_q(wl, s + 3, gen).to(device)
                L["idx_w"] = synth.index_w(wl, s + 4, gen).to(device)
                L["topk_idx"] = torch.full((nq, wl.k), -1, dtype=torch.int32, device=device)
            if m == FULL:
                kv = synth.kv_rows(wl, s + 5, gen)
                kk = synth.index_k_rows(wl, s + 6, gen)
                if keep_bf16:
                    host["kv"] = kv.cpu()
                    host["kk"] = kk.cpu()
                self._fill_cache(L, kv.to(device), kk.to(device))
                del kv, kk
                if wl.block:
                    # block keys of the cache as filled (the step refreshes the
                    # block its new row falls in)
                    if self.pages is not None:
                        L["block_keys"] = csa2.index_block_keys(
                            L["idxk"], wl.block, n=N, pages=self.pages, B=B)
                    else:
                        L["block_keys"] = csa2.index_block_keys(L["idxk"], wl.block)
            self.layers.append(L)
            self.bf16.append(host)
        self.n_valid = None
        self.win_start = self.win_len = None
        if wl.q_per_seq > 1:
            self.n_valid = synth.prefill_n_valid(wl, device)
            self.win_start = torch.arange(wl.q_per_seq, dtype=torch.int32,
                                          device=device).repeat(wl.B)
            self.win_len = torch.full((nq,), wl.W, dtype=torch.int32, device=device)
        self.dev_status = torch.zeros(1, dtype=torch.int32, device=device)
        self.descs = csa2.layer_descs(self.layers)
        self.sargs = self.stack_args()
        need = csa2.layer_stack_workspace_bytes(self.sargs)
        self.workspace = torch.empty(need + 256, dtype=torch.uint8, device=device)

    def _fill_cache(self, L, kv, kk):
        wl = self.wl
        B, N = wl.B, wl.N
        if self.pages is not None:
            return self._fill_pages(L, kv, kk)
        L["codes"] = torch.zeros(B, N, wl.D // 2, dtype=torch.uint8, device=self.device)
        L["scales"] = torch.zeros(B, N, wl.D // 32, dtype=torch.uint8, device=self.device)
        if wl.fp32_indexer:
            L["idxk"] = torch.zeros(B, N, wl.Di, dtype=torch.float32, device=self.device)
            L["idxk"][:, : N - (1 if wl.q_per_seq == 1 else wl.q_per_seq // 4)] = \
                kk[:, : N - (1 if wl.q_per_seq == 1 else wl.q_per_seq // 4)].float()
        else:
            L["idxk"] = torch.zeros(B, N, wl.Di, dtype=torch.uint8, device=self.device)
        # decode completes one compressed entry per sequence; a prefill chunk
        # of T tokens completes T / 4 entries (4 tokens per entry)
        rows_new = 1 if wl.q_per_seq == 1 else wl.q_per_seq // 4
        old = N - rows_new
        for b in range(B):
            if wl.fp32_indexer:
                csa2.quantize_fp4(kv[b, :old], L["codes"][b, :old], L["scales"][b, :old])
            else:
                csa2.quantize_fp4(kv[b, :old], L["codes"][b, :old], L["scales"][b, :old],
                                  kk[b, :old], L["idxk"][b, :old])
        L["new_kv"] = kv[:, old:].contiguous()
        L["new_idxk"] = (kk[:, old:].float() if wl.fp32_indexer else kk[:, old:]).contiguous()
        L["new_row"] = old
        L["new_rows"] = rows_new

    def _fill_pages(self, L, kv, kk):
        """Paged caches: pools of num_pages * page_rows rows, entries 0 ..
        N - 2 of every sequence quantised into them through the block table
        (one launch of the paged quantiser); entry N - 1 is the step's new
        row, as in the contiguous layout."""
        wl = self.wl
        B, N = wl.B, wl.N
        rows = self.num_pages * wl.page_rows
        L["codes"] = torch.zeros(rows, wl.D // 2, dtype=torch.uint8, device=self.device)
        L["scales"] = torch.zeros(rows, wl.D // 32, dtype=torch.uint8, device=self.device)
        L["idxk"] = torch.zeros(rows, wl.Di, dtype=torch.uint8, device=self.device)
        rows_new = 1 if wl.q_per_seq == 1 else wl.q_per_seq // 4
        old = N - rows_new
        csa2.quantize_fp4(kv[:, :old].reshape(B * old, wl.D), L["codes"], L["scales"],
                          kk[:, :old].reshape(B * old, wl.Di), L["idxk"], pages=self.pages,
                          rows_per_seq=old, entry0=0)
        L["new_kv"] = kv[:, old:].contiguous()
        L["new_idxk"] = kk[:, old:].contiguous()
        L["new_row"] = old
        L["new_rows"] = rows_new

    def stack_args(self):
        wl = self.wl
        return csa2.stack_args(
            B=wl.B, q_per_seq=wl.q_per_seq, n=wl.N, hi=wl.Hi, di=wl.Di, hq=wl.Hq, d=wl.D,
            k=wl.k, w_rows=self.layers[0]["window"].shape[1],
            idx_q_dtype=csa2.F32 if wl.fp32_indexer else csa2.BF16,
            idx_k_dtype=csa2.F32 if wl.fp32_indexer else csa2.E4M3,
            attn_q_dtype=csa2.F32 if wl.attn_q_fp32 else csa2.BF16,
            softmax_scale=1.0 / math.sqrt(wl.D), n_valid=self.n_valid,
            win_start=self.win_start, win_len=self.win_len, dev_status=self.dev_status,
            pool=wl.pool, win_max=wl.W if self.win_len is not None else 0, pages=self.pages,
            block=wl.block, blocks_kept=wl.blocks_kept)

    def run(self):
        """Enqueue one step on the current stream."""
        csa2.layer_stack(self.descs, self.sargs, self.workspace)

    IO_IN = ("new_kv", "new_idxk", "idx_q", "idx_w", "attn_q")

    def make_io(self):
        """A copy of the step's per-step inputs (new KV and indexer-K rows,
        indexer Q and weights, attention Q) packed into one device block and
        of its outputs (the attention results) in another, with layer
        descriptors that read and write those blocks; every other tensor
        (caches, windows, selected indices) is shared with this workload.
        A host copy of `dev_in`, then one run of `descs`, then a copy of
        `dev_out` to the host is one end-to-end step: one transfer each way."""
        align = 256

        def pack(keys):
            slots, off = [], 0
            for l, L in enumerate(self.layers):
                for key in keys:
                    if key in L:
                        t = L[key]
                        slots.append((l, key, off, t))
                        off += (t.numel() * t.element_size() + align - 1) // align * align
            return slots, off

        in_slots, in_bytes = pack(self.IO_IN)
        out_slots, out_bytes = pack(("out",))
        dev_in = torch.empty(max(in_bytes, align), dtype=torch.uint8, device=self.device)
        dev_out = torch.empty(max(out_bytes, align), dtype=torch.uint8, device=self.device)
        layers = [dict(L) for L in self.layers]
        for buf, slots in ((dev_in, in_slots), (dev_out, out_slots)):
            for l, key, off, t in slots:
                nb = t.numel() * t.element_size()
                view = buf[off:off + nb].view(t.dtype).view(t.shape)
                view.copy_(t)
                layers[l][key] = view
        payload_in = sum(t.numel() * t.element_size() for _, _, _, t in in_slots)
        payload_out = sum(t.numel() * t.element_size() for _, _, _, t in out_slots)
        return StepIO(dev_in, dev_out, layers, csa2.layer_descs(layers), payload_in, payload_out)

    # bytes the method must move per step (the roofline numerator); the
    # scores scratch is excluded.
    def algorithmic_bytes(self):
        wl = self.wl
        nq = wl.nq
        queries = (nq * wl.Hi * wl.Di * (4 if wl.fp32_indexer else 2)
                   + nq * wl.Hi * 4 + nq * wl.k * 4)
        full_index = wl.B * wl.N * wl.Di * (4 if wl.fp32_indexer else 1) + queries
        if wl.page_rows:
            # paged caches: the indexer reads each sequence's block table (and
            # every selected entry looks up its page, below)
            full_index += wl.B * (-(-wl.N // wl.page_rows)) * 4
        # a pooled Reindex layer reads its pool and the pool's indexer-K rows
        P = wl.blocks_kept * wl.block if wl.block else min(wl.pool, wl.N)
        reindex = full_index if P == 0 else nq * P * (wl.Di + 4) + queries
        if wl.block:
            # block-level pruning: a Full layer reads the block keys and the
            # kept blocks' indexer-K rows instead of every entry
            full_index = (wl.B * (-(-wl.N // wl.block)) * wl.Di + nq * P * (wl.Di + 4)
                          + queries)
        n_full = sum(1 for m in wl.modes if m == FULL)
        n_re = sum(1 for m in wl.modes if m == REINDEX)
        per_layer = (nq * wl.k * (wl.D // 2 + wl.D // 32) + nq * wl.W * wl.D * 2
                     + nq * wl.Hq * wl.D * (4 if wl.attn_q_fp32 else 2) + nq * wl.Hq * wl.D * 4)
        if wl.page_rows:
            per_layer += nq * wl.k * 4
        return n_full * full_index + n_re * reindex + len(wl.modes) * per_layer

    def visible_pairs(self):
        """(query, entry) pairs the indexer scores: nq * N in decode, the
        causal count in a prefill chunk."""
        if self.n_valid is None:
            return self.wl.nq * self.wl.N
        return int(self.n_valid.to(torch.int64).sum().item())

    def indexer_bytes_per_layer(self):
        wl = self.wl
        return wl.B * wl.N * wl.Di * (4 if wl.fp32_indexer else 1)
