"""Host-side arithmetic of bench.py (no GPU): the roofline's algorithmic bytes
and FLOPs follow the measurement rule -- for decode, the K codes and scales of
every key a request can see, read once, plus Q codes, Q scales and w; for the
tensor-bound workloads, 2 * 128 FLOPs per visible (row, head, key)."""
import numpy as np

import bench
import oracle
from fp4_sparse_attention_gb300 import workloads as wl


def test_decode_scorer_bytes_are_inputs_only():
    p = wl.verify_decode_16k()
    want = 16384 * 68 + 4 * 32 * (64 + 4) + 4 * 32 * 4
    assert bench.kernel_algorithmic_bytes(p, "logits_topk", 2048) == want
    assert bench.kernel_algorithmic_bytes(p, "scorer_logits", 0) == want
    # the logits and top-k written are reported apart
    assert bench.kernel_output_bytes(p, "logits_topk", 2048) == 4 * 16384 * 4 + 4 * 2048 * 8 + 4 * 4


def test_pr_call_counts_the_quantised_queries():
    p = wl.p1_paged_16k()
    # the scorer reads MXFP4 query codes + scales (after quantisation), not bf16
    assert bench.kernel_algorithmic_bytes(p, "scorer_logits", 0) == 16384 * 68 + 4 * 32 * 68 + 4 * 32 * 4
    assert bench.kernel_algorithmic_bytes(p, "quantize_q", 0) == 4 * 32 * (256 + 68)


def test_tensor_flops_count_visible_pairs():
    p = wl.make_problem(name="flops", seed=1, fmt=wl.MXFP4, q_lens=[300], k_lens=[300], num_heads=64,
                        visibility="causal")
    vis = oracle.visible_all(p)
    assert bench.kernel_algorithmic_flops(p) == int(vis.sum()) * 64 * 256
    assert int(vis.sum()) == 300 * 301 // 2


def test_roofline_fraction_and_recorded_traffic():
    p = wl.verify_decode_16k()
    peaks = {"hbm_gbs": 1000.0, "bf16_tflops": 1.0, "bf16_tflops_sustained": 1.0, "source": "test"}
    r = bench.roofline(p, bench.WORKLOADS["verify16k"], "logits_topk", 0.01, 0.02, peaks)
    assert r["bound"] == "hbm" and r["algorithmic_bytes"] == 16384 * 68 + 4 * 32 * 72
    assert np.isclose(r["achieved"], r["algorithmic_bytes"] / 1e-5 / 1e9)
    assert np.isclose(r["frac"], r["achieved"] / 1000.0)
    for (workload, kernel), rec in bench.RECORDED_TRAFFIC.items():
        assert workload in bench.WORKLOADS and len(rec["sha"]) == 16 and rec["bytes"] > 0
