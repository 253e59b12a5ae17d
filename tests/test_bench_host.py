"""Host-side parts of bench.py that need no GPU: the CPU baseline (the
oracle on one thread and on every host core) on small synthetic cases."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _small_workload():
    from speculative_decoding_verification_56_gb300 import synth
    samp = synth.make_chain_case(B=4, k=2, V=1000, dtype="bf16", recipe="zipf", seed=1)
    greedy = synth.greedy_variant(samp, 0.7)
    tree = synth.make_tree_case(B=2, N=10, V=1000, dtype="bf16", seed=2)
    return samp, greedy, tree


def test_cpu_baseline_single_and_all_cores():
    import bench
    import oracle
    oracle.build()
    samp, greedy, tree = _small_workload()
    r = bench.cpu_baseline(samp, greedy, tree, 0.2)
    assert r["kind"] == "oracle" and r["cores"] == 1 and r["value"] > 0
    a = r["all_cores"]
    assert a["cores"] == (os.cpu_count() or 1) and a["value"] > 0
    # the positions counted per step are the same in both runs
    assert bench.positions(samp, greedy, tree) == 4 * 2 + 4 * 2 + 2 * 9
