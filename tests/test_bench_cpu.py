"""Host-side pieces of bench.py: the kernel-count claim and the workload
names both arms print (no GPU)."""
import sys

from conftest import ROOT

sys.path.insert(0, ROOT)
import bench  # noqa: E402
from long_context_sparse_27_b300 import synth  # noqa: E402


def test_launches_per_step():
    W = synth.WORKLOADS
    # Full: indexer (Q quantiser, new rows and histogram fused), select,
    # attention; Reindex: the same; Reuse: attention
    assert bench.launches_per_step(W["1m"]) == 5 * (3 + 3 + 1 + 1)
    assert bench.launches_per_step(W["group3"]) == 3 + 3 + 1
    # the pool: Full adds the pool's selection (4), a pooled Reindex runs Q
    # quantiser, pooled scores, short-row selection, attention (4)
    assert bench.launches_per_step(W["1m-pool"]) == 5 * (4 + 4 + 1 + 1)
    # block-level pruning: the Full layer quantises its new rows in a kernel
    # of its own (the block keys are refreshed from them)
    assert bench.launches_per_step(W["1m-block"]) == 5 * (8 + 4 + 1 + 1)
    # a prefill chunk over long rows selects without its score matrix: new
    # rows, Q quantiser, sampled scores, histogram, threshold, histogram
    # within the threshold bin, threshold, emitting scores, candidate
    # selection, attention; 8 chunks of 80 keys need no merge kernel
    assert bench.launches_per_step(W["prefill"]) == 10
    # over short rows it runs its Q quantiser and a histogram pass as kernels
    # of their own
    assert bench.launches_per_step(synth.scaled(W["prefill"], N=4096)) == 6
    # the fp32 indexer of a row longer than 4096 adds a histogram pass
    assert bench.launches_per_step(synth.scaled(W["tiny"], N=8192)) == 5


def test_workload_desc_names_the_variant():
    d = bench.workload_desc(synth.WORKLOADS["1m-pool"])
    assert d.startswith("1m-pool: B=8, N=262144") and "candidate pool 2048" in d
    assert "fp32" in bench.workload_desc(synth.WORKLOADS["tiny"])
    assert "4096 queries per sequence" in bench.workload_desc(synth.WORKLOADS["prefill"])
