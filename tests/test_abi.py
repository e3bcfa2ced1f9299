"""Host-only checks of the C ABI (no GPU work is ever enqueued here).

The library loads without a GPU (the CUDA runtime is linked statically).
Calls below either fail argument validation or are stopped by the host
fault injection before any launch, so they never touch a device.
"""
import ctypes
import os
import re
import subprocess

import pytest
import torch

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "csa2.h")

# These tests pass fake device pointers; on a machine with a GPU a wrong
# branch could launch with them, so they run only where no GPU is visible.
no_gpu = pytest.mark.skipif(torch.cuda.is_available(), reason="host-only test")


@pytest.fixture(scope="module")
def csa2():
    from long_context_sparse_27_b300 import build
    build.build()
    from long_context_sparse_27_b300 import csa2 as m
    return m


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = set(re.findall(r"\b(csa2_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_every_declared_symbol_is_exported(csa2):
    names = declared_functions()
    assert len(names) >= 15
    out = subprocess.check_output(["nm", "-D", "--defined-only", csa2.LIB_PATH], text=True)
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    # and the binding describes every one of them
    assert set(names) <= set(csa2.EXPORTS)


def test_struct_layouts_match_c(csa2, tmp_path):
    structs = {"csa2_quant_args": csa2.QuantArgs, "csa2_index_args": csa2.IndexArgs,
               "csa2_attn_args": csa2.AttnArgs, "csa2_layer_desc": csa2.LayerDesc,
               "csa2_stack_args": csa2.StackArgs, "csa2_project_args": csa2.ProjectArgs}
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "csa2.h"', "int main(void){"]
    for cname, py in structs.items():
        lines.append(f'printf("{cname} %zu\\n", sizeof({cname}));')
        for f, _ in py._fields_:
            lines.append(f'printf("{cname}.{f} %zu\\n", offsetof({cname}, {f}));')
    lines.append("return 0;}")
    src = tmp_path / "probe.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "probe"
    subprocess.check_call(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o",
                           str(exe)])
    got = dict(l.split() for l in subprocess.check_output([str(exe)], text=True).splitlines())
    for cname, py in structs.items():
        assert int(got[cname]) == ctypes.sizeof(py), cname
        for f, _ in py._fields_:
            assert int(got[f"{cname}.{f}"]) == getattr(py, f).offset, (cname, f)


def test_status_strings(csa2):
    assert csa2.lib.csa2_status_string(0) == b"CSA2_OK"
    assert csa2.lib.csa2_status_string(5) == b"CSA2_ERR_WORKSPACE"
    assert csa2.lib.csa2_status_string(99) == b"CSA2_ERR_UNKNOWN"
    assert csa2.lib.csa2_status_from_device(0) == 0
    assert csa2.lib.csa2_status_from_device(csa2.DEVFLAG_BOUNDS) == 7
    assert csa2.lib.csa2_status_from_device(csa2.DEVFLAG_TIMEOUT | csa2.DEVFLAG_BOUNDS) == 6
    assert csa2.lib.csa2_status_from_device(csa2.DEVFLAG_CAPACITY) == 8
    assert csa2.lib.csa2_status_from_device(csa2.DEVFLAG_CAPACITY | csa2.DEVFLAG_BOUNDS) == 7
    assert csa2.lib.csa2_status_string(8) == b"CSA2_ERR_DEVICE_CAPACITY"
    assert csa2.version().count(".") == 2


def topk_ws(rows, n):
    # one u32 histogram of 4096 fine and 64 coarse bins per row; rows longer
    # than 4096 add a 16-byte counter per row (from a 256-byte boundary) and,
    # per row, S slices of a 16-byte count + 1024 (key, index) pairs, S =
    # about 296 CTAs per launch, at most 64, at most one slice per 4096 entries
    hist = rows * 4160 * 4
    if n <= 4096:
        return hist
    S = max(1, min(-(-296 // rows), 64, -(-n // 4096)))
    return -(-(hist + rows * 16) // 256) * 256 + rows * S * (16 + 1024 * 8)


def test_workspace_sizes(csa2):
    for rows, n, k in ((8, 262144, 512), (3, 100, 2048), (4096, 262144, 512), (20, 30000, 512),
                       (1, 4097, 1)):
        assert csa2.topk_workspace_bytes(rows, n, k) == topk_ws(rows, n)
    assert topk_ws(8, 262144) == 133376 + 8 * 37 * 8208
    a = csa2.IndexArgs(q_dtype=csa2.BF16, k_dtype=csa2.E4M3, B=8, q_per_seq=1, hi=64, di=128,
                       n=262144)
    assert csa2.lib.csa2_index_score_workspace_bytes(ctypes.byref(a)) == 8 * 64 * 128 + 8 * 64 * 4
    a.q_dtype = a.k_dtype = csa2.F32
    assert csa2.lib.csa2_index_score_workspace_bytes(ctypes.byref(a)) == 0


# ---- plan validation (pure host logic) ----

def plan(*triples):
    return [{"mode": m, "kv_src": kv, "idx_src": ix} for m, kv, ix in triples]


F, RI, RU = 0, 1, 2


@pytest.mark.parametrize("layers,ok,bad", [
    (plan((F, 0, 0), (RI, 0, 1), (RU, 0, 0)), True, -1),
    (plan((F, 0, 0), (RI, 0, 1), (RU, 0, 1)), True, -1),      # Reuse of the Reindex indices
    (plan((F, 0, 0), (RI, 0, 1), (RU, 0, 0), (RU, 0, 0), (F, 4, 4), (RI, 4, 5), (RU, 4, 4)),
     True, -1),
    (plan((RI, 0, 0)), False, 0),                              # no Full first
    (plan((F, 0, 0), (F, 0, 1)), False, 1),                    # Full must name itself
    (plan((F, 0, 0), (F, 1, 1), (RI, 0, 2)), False, 2),        # Reindex: the LAST Full layer
    (plan((F, 0, 0), (RU, 1, 0)), False, 1),                   # KV from a later layer
    (plan((F, 0, 0), (F, 1, 1), (RU, 1, 0)), False, 2),        # indices of another cache
    (plan((F, 0, 0), (RU, 0, 0), (RU, 0, 1)), False, 2),       # indices of a Reuse layer
    (plan((F, 0, 0), (3, 0, 0)), False, 1),                    # unknown mode
])
def test_validate_plan(csa2, layers, ok, bad):
    st, where = csa2.validate_plan(layers)
    assert (st == 0) == ok
    assert where == bad


# ---- argument validation and host fault injection (never launches) ----

FAKE = 1 << 20  # 16-byte aligned, never dereferenced


@no_gpu
def test_topk_validation(csa2):
    L = csa2.lib
    ws = csa2.topk_workspace_bytes(4, 1000, 64)
    assert L.csa2_topk(FAKE, 4, 1000, 1000, None, 0, FAKE, 64, FAKE, ws, None, None) == 1
    assert L.csa2_topk(FAKE, 4, 1000, 1000, None, 4096, FAKE, 4096, FAKE, ws, None, None) == 2
    assert L.csa2_topk(FAKE, 4, 1000, 1000, None, 64, FAKE, 64, FAKE, ws - 1, None, None) == 5
    assert L.csa2_topk(FAKE, 4, 1000, 1000, None, 64, FAKE, 64, FAKE + 8, ws, None, None) == 3
    assert L.csa2_topk(FAKE, 4, 1000, 999, None, 64, FAKE, 64, FAKE, ws, None, None) == 1


@no_gpu
def test_fault_injection_stops_before_launch(csa2, monkeypatch):
    L = csa2.lib
    ws = csa2.topk_workspace_bytes(4, 1000, 64)
    monkeypatch.setenv("CSA2_FAULT_INJECT", "topk:4")
    assert L.csa2_topk(FAKE, 4, 1000, 1000, None, 64, FAKE, 64, FAKE, ws, None, None) == 4
    monkeypatch.setenv("CSA2_FAULT_INJECT", "topk:6")
    assert L.csa2_topk(FAKE, 4, 1000, 1000, None, 64, FAKE, 64, FAKE, ws, None, None) == 6
    # a bad argument is reported before the injected failure
    assert L.csa2_topk(FAKE, 4, 1000, 1000, None, 0, FAKE, 64, FAKE, ws, None, None) == 1
    # the entry point without allocation takes its own injection name
    monkeypatch.setenv("CSA2_FAULT_INJECT", "topk_noalloc:4")
    assert L.csa2_topk_noalloc(FAKE, 4, 1000, 1000, None, 64, FAKE, 64, None, None) == 4
    assert L.csa2_topk_noalloc(FAKE, 4, 1000, 1000, None, 0, FAKE, 64, None, None) == 1


@no_gpu
def test_index_validation(csa2, monkeypatch):
    L = csa2.lib
    a = csa2.IndexArgs(q=FAKE, q_dtype=csa2.BF16, w=FAKE, k=FAKE, k_dtype=csa2.E4M3, B=2,
                       q_per_seq=1, hi=64, di=128, n=1000, k_ld=128, k_seq_stride=128 * 1000,
                       scores=FAKE, scores_ld=1000)
    assert L.csa2_index_score(ctypes.byref(a), None) == 5          # no workspace
    a.workspace, a.workspace_bytes = FAKE, L.csa2_index_score_workspace_bytes(ctypes.byref(a))
    a.hi = 32
    assert L.csa2_index_score(ctypes.byref(a), None) == 2          # only 64 x 128 is built
    a.hi = 64
    a.k = FAKE + 8
    assert L.csa2_index_score(ctypes.byref(a), None) == 3          # TMA needs 16-byte rows
    a.k = FAKE
    a.k_seq_stride = 100
    assert L.csa2_index_score(ctypes.byref(a), None) == 1          # overlapping sequences
    a.k_seq_stride = 128 * 1000
    # the tensor-core kernel's per-tile arithmetic is 32-bit: at most 2^30
    # entries, fewer than 2^31 (query, 128-entry tile) pairs
    a.n, a.scores_ld, a.k_seq_stride = (1 << 30) + 1, (1 << 30) + 1, 128 * ((1 << 30) + 1)
    assert L.csa2_index_score(ctypes.byref(a), None) == 2
    a.B, a.q_per_seq, a.n, a.scores_ld, a.k_seq_stride = 1, 1 << 20, 1 << 18, 1 << 18, 0
    a.workspace_bytes = L.csa2_index_score_workspace_bytes(ctypes.byref(a))
    assert L.csa2_index_score(ctypes.byref(a), None) == 2     # 2^20 queries x 2^11 tiles
    a.B, a.q_per_seq, a.n, a.scores_ld, a.k_seq_stride = 2, 1, 1000, 1000, 128 * 1000
    monkeypatch.setenv("CSA2_FAULT_INJECT", "index_score:4")
    assert L.csa2_index_score(ctypes.byref(a), None) == 4


@no_gpu
def test_attn_and_quant_validation(csa2, monkeypatch):
    L = csa2.lib
    a = csa2.AttnArgs(q=FAKE, q_dtype=csa2.BF16, nq=2, q_per_seq=1, hq=64, d=512, codes=FAKE,
                      scales=FAKE, n=100, codes_ld=256, codes_seq_stride=25600, scales_ld=16,
                      scales_seq_stride=1600, idx=FAKE, k=64, idx_ld=64, window=FAKE, w_rows=8,
                      win_ld=512, win_seq_stride=4096, softmax_scale=0.04, out=FAKE)
    # 64 + 8 keys: one 80-key chunk; every chunk's partial (32 heads x 512
    # + max and sum per head, f32) goes through the workspace
    assert L.csa2_sparse_attn_workspace_bytes(ctypes.byref(a)) == 2 * 4 * 1 * (16 * 512 + 32) * 4
    assert L.csa2_sparse_attn(ctypes.byref(a), None) == 5
    a.k = a.idx_ld = 1024  # 1032 keys = 13 chunks > 8: merged by a second kernel
    assert L.csa2_sparse_attn(ctypes.byref(a), None) == 5
    need = L.csa2_sparse_attn_workspace_bytes(ctypes.byref(a))
    assert need == 2 * 4 * 13 * (16 * 512 + 32) * 4  # 2 queries x 4 head groups x 13 chunks
    a.workspace, a.workspace_bytes = FAKE, need
    a.hq = 24
    assert L.csa2_sparse_attn(ctypes.byref(a), None) == 2
    a.hq = 64
    a.codes_ld = 264
    assert L.csa2_sparse_attn(ctypes.byref(a), None) == 3
    a.codes_ld = 256
    monkeypatch.setenv("CSA2_FAULT_INJECT", "sparse_attn:4")
    assert L.csa2_sparse_attn(ctypes.byref(a), None) == 4
    q = csa2.QuantArgs(x=FAKE, rows=4, d=48, x_ld=48, codes=FAKE, codes_ld=24, scales=FAKE,
                       scales_ld=2)
    assert L.csa2_quantize_fp4(ctypes.byref(q), None) == 1      # d % 32 != 0
    q.d, q.x_ld, q.codes_ld, q.scales_ld = 64, 64, 32, 2
    q.x = FAKE + 2
    assert L.csa2_quantize_fp4(ctypes.byref(q), None) == 3
    q.x = FAKE
    monkeypatch.setenv("CSA2_FAULT_INJECT", "quantize_fp4:4")
    assert L.csa2_quantize_fp4(ctypes.byref(q), None) == 4


@no_gpu
def test_pooled_index_validation(csa2, monkeypatch):
    L = csa2.lib
    a = csa2.IndexArgs(q=FAKE, q_dtype=csa2.BF16, w=FAKE, k=FAKE, k_dtype=csa2.E4M3, B=2,
                       q_per_seq=1, hi=64, di=128, n=100000, k_ld=128,
                       k_seq_stride=128 * 100000, scores=FAKE, scores_ld=2048)
    ws = L.csa2_index_score_workspace_bytes(ctypes.byref(a))
    a.workspace, a.workspace_bytes = FAKE, ws
    # the pooled scores need rows of pool_n entries only (scores_ld < n)
    monkeypatch.setenv("CSA2_FAULT_INJECT", "index_score_pool:4")
    assert L.csa2_index_score_pool(ctypes.byref(a), FAKE, 2048, 2048, None) == 4
    monkeypatch.delenv("CSA2_FAULT_INJECT")
    assert L.csa2_index_score_pool(ctypes.byref(a), FAKE, 2048, 0, None) == 1     # empty pool
    assert L.csa2_index_score_pool(ctypes.byref(a), FAKE, 1000, 2048, None) == 1  # pool_ld
    assert L.csa2_index_score_pool(ctypes.byref(a), FAKE, 4096, 4096, None) == 1  # > scores_ld
    a.scores_ld = 4096
    assert L.csa2_index_score_pool(ctypes.byref(a), FAKE, 4096, 4096, None) == 2  # > 2048
    assert L.csa2_index_score_pool(ctypes.byref(a), None, 2048, 2048, None) == 1  # no pool
    a.q_dtype = a.k_dtype = csa2.F32
    assert L.csa2_index_score_pool(ctypes.byref(a), FAKE, 2048, 2048, None) == 2  # FP8 only


@no_gpu
def test_stack_pool_validation(csa2, monkeypatch):
    L = csa2.lib
    descs = csa2.layer_descs([{"mode": 0, "kv_src": 0, "idx_src": 0},
                              {"mode": 1, "kv_src": 0, "idx_src": 1}])
    s = csa2.stack_args(B=2, q_per_seq=1, n=10000, hi=64, di=128, hq=64, d=512, k=512, w_rows=128,
                        idx_q_dtype=csa2.BF16, idx_k_dtype=csa2.E4M3, attn_q_dtype=csa2.BF16,
                        softmax_scale=0.04)
    plain = L.csa2_layer_stack_workspace_bytes(ctypes.byref(s))
    s.pool = 2048
    pooled = L.csa2_layer_stack_workspace_bytes(ctypes.byref(s))
    assert pooled == plain + 2 * 2048 * 4      # the pool: nq x P int32 (256-byte multiple)
    s.pool = 20000                              # P >= n: the pool is every entry
    assert L.csa2_layer_stack_workspace_bytes(ctypes.byref(s)) == plain + 2 * 10000 * 4 + 256 - \
        (2 * 10000 * 4) % 256
    s.workspace, s.workspace_bytes = FAKE, 1 << 40
    s.pool = 256                                # smaller than k
    assert L.csa2_layer_stack(descs, 2, ctypes.byref(s), None) == 1
    s.pool = 4096
    assert L.csa2_layer_stack(descs, 2, ctypes.byref(s), None) == 2
    s.pool = -1
    assert L.csa2_layer_stack(descs, 2, ctypes.byref(s), None) == 1
    s.pool = 2048
    s.idx_q_dtype = s.idx_k_dtype = csa2.F32   # the pooled scoring is FP8 only
    assert L.csa2_layer_stack(descs, 2, ctypes.byref(s), None) == 2
    s.pool, s.win_max = 0, -1                  # a negative window bound
    assert L.csa2_layer_stack(descs, 2, ctypes.byref(s), None) == 1


@no_gpu
def test_project_validation(csa2, monkeypatch):
    L = csa2.lib
    a = csa2.ProjectArgs(h=FAKE, w=FAKE, rows=8, hidden=4096, d=512, h_ld=4096, w_ld=4096,
                         codes=FAKE, codes_ld=256, scales=FAKE, scales_ld=16)
    monkeypatch.setenv("CSA2_FAULT_INJECT", "project_fp4:4")
    assert L.csa2_project_fp4(ctypes.byref(a), None) == 4         # valid: stopped by injection
    a.hidden = 100
    assert L.csa2_project_fp4(ctypes.byref(a), None) == 1         # hidden % 32
    a.hidden, a.d = 4096, 96
    assert L.csa2_project_fp4(ctypes.byref(a), None) == 1         # d % 64
    a.d = 512
    a.h = FAKE + 8
    assert L.csa2_project_fp4(ctypes.byref(a), None) == 3         # 16-byte rows
    a.h, a.w_ld = FAKE, 4100
    assert L.csa2_project_fp4(ctypes.byref(a), None) == 3
    a.w_ld, a.codes_ld = 4096, 100
    assert L.csa2_project_fp4(ctypes.byref(a), None) == 1
    a.codes_ld, a.out, a.out_ld = 256, FAKE, 511
    assert L.csa2_project_fp4(ctypes.byref(a), None) == 1         # out_ld < d


def test_bindings_reject_strided_rows(csa2):
    # the bindings pass stride(0) as the row stride: a row must be contiguous
    h = torch.zeros(64, 8, dtype=torch.bfloat16).t()      # [8, 64], column-major
    w = torch.zeros(64, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        csa2.project_fp4(h, w)
    pool = torch.zeros(4, 2, dtype=torch.int32).t()       # [2, 4], column-major
    with pytest.raises(ValueError):
        csa2.index_score_pool(torch.zeros(2, 64, 128, dtype=torch.bfloat16),
                              torch.zeros(2, 64), torch.zeros(1, 10, 128, dtype=torch.uint8), pool)
    # top-k: a column-strided score view, a strided output, n_valid not int32
    s = torch.zeros(3, 40)
    for fn in (csa2.topk, csa2.topk_noalloc):
        with pytest.raises(ValueError):
            fn(s[:, ::2], 4)
        with pytest.raises(ValueError):
            fn(s, 4, out=torch.zeros(3, 8, dtype=torch.int32)[:, ::2])
        with pytest.raises(ValueError):
            fn(s, 4, n_valid=torch.full((3,), 40, dtype=torch.int64))
