"""The bench's algorithmic byte and operation counts (the numerators of its
roofline fractions), checked against direct sums on the workload sizes."""
import bench
from synth.workloads import WORKLOADS, Workload


def _direct_positions(wl):
    return wl.B * sum((wl.N - wl.n_q + j + 1) // wl.m for j in range(wl.n_q))


def test_causal_positions_match_direct_sums():
    for wl in WORKLOADS.values():
        assert bench.causal_positions(wl) == _direct_positions(wl), wl.name
    small = Workload(0, "t", "full", B=3, N=1000, n_q=37, m=2, prefill=True)
    assert bench.causal_positions(small) == 3 * sum((1000 - 37 + j + 1) // 2 for j in range(37))


def test_scan_bytes_count_entries_and_query_side():
    w3 = WORKLOADS[3]
    assert bench.scan_bytes(w3) == 8 * (72 * 1048576 + 32 * 72 + 32 * 4)
    w6 = WORKLOADS[6]  # 2 tokens per entry: half the entries of the same context
    assert bench.scan_bytes(w6) == 8 * (72 * 524288 + 32 * 72 + 32 * 4)
    # the ALU count: a ReLU and a weighted add per head and causal (entry, token)
    assert bench.scan_alu_ops(WORKLOADS[5]) == 64 * _direct_positions(WORKLOADS[5])


def test_attention_bytes_per_query():
    # 512 FP4 entries x 288 B + 128 FP8 window entries x 512 B + q (64 x 512 bf16) + top-k
    assert bench.attn_bytes_per_query() == 147456 + 65536 + 65536 + 2048


def test_dominant_stage_per_mode():
    # Full: the scan; Reindex (and the group, led by a Reindex layer): the pool
    # rescore, one launch per Reindex layer; Reuse: the attention, one launch per layer.
    assert bench.dominant_stage(WORKLOADS[3], ["full"]) == ("indexer_scan", bench.scan_bytes(WORKLOADS[3]), "scan", 1)
    w2 = WORKLOADS[2]
    name, nbytes, stage, per = bench.dominant_stage(w2, ["reindex"])
    assert (name, stage, per) == ("indexer_rescore", "rescore", 1)
    assert nbytes == 64 * (2048 * 576 + 32 * 72 + 32 * 4 + 2048 * 4)
    w4 = WORKLOADS[4]
    assert bench.dominant_stage(w4, list(w4.layers))[2:] == ("rescore", 1)
    w1 = WORKLOADS[1]
    assert bench.dominant_stage(w1, ["reuse"]) == ("sparse_attn", 64 * bench.attn_bytes_per_query(), "attn", 1)


def test_mode_summary_fractions():
    class Args:
        steps, warmup = 20, 5
    w1 = WORKLOADS[1]
    m = {"kinds": ["reuse"], "ms": 0.01, "stage_ms": {"attn": 0.008}, "e2e": None, "clocks": None, "launches": 1}
    s = bench.mode_summary(Args, w1, m, 6800.0)
    assert s["value"] == 64 / 0.01e-3
    want = 64 * bench.attn_bytes_per_query() / 0.008e-3 / 1e9 / 6800.0
    assert abs(s["dominant"]["frac_of_measured_hbm"] - want) < 1e-12
    assert s["gpu_launches"] == 20
