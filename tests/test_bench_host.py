"""Host-side arithmetic of bench.py (no GPU): the roofline's algorithmic
bytes of the headline workload and the percentile helper."""
import pytest

import bench
import workloads


def test_algorithmic_bytes_of_the_headline_workload():
    # 8 agents x 32,768 shared tokens, H_kv = 8, d = 128, rank 16, one query
    # each: bCache 2 * 32768 * 8 * 128 * 2 B + rCache 2 * 8 * 32768 * 16 * 2 B
    # + q and out 8 * 32 * 128 * 2 B each
    w = workloads.make_workload("llama8b_32k")
    ab = bench.algorithmic_bytes(w)
    assert ab["bcache"] == 2 * 32768 * 8 * 128 * 2 == 134217728
    assert ab["rcache"] == 2 * 8 * 32768 * 16 * 2 == 16777216
    assert ab["q"] == ab["out"] == 8 * 32 * 128 * 2
    assert ab["step"] == 151126016
    assert bench.percentiles([1.0, 2.0, 3.0]) == [1.2, 2.0, 2.8]


def test_chunk_workload_flops():
    # the Qwen-72B-shaped chunk: 16 agents x (65536 + 32) keys, 8 kv heads,
    # G = 8, C = 32, d = 128, rank 64; per (agent, key, head) 2 r d (key
    # residual) + G C (4 d + 2 r) (scores, P Vb, P Lv), per row 2 r d
    w = workloads.make_workload("qwen72b_chunk")
    T, G, C, d, r = 65536 + 32, 8, 32, 128, 64
    per_head = T * (2 * r * d + G * C * (4 * d + 2 * r)) + G * C * 2 * r * d
    assert int(w.seq_lens[0]) == T
    assert 16 * 8 * per_head == 1513103556608


def _profile_values(path):
    vals = {}
    for line in open(path):
        if ":" in line and not line.startswith("#"):
            k, v = line.split(":", 1)
            vals[k.strip()] = v.strip()
    return vals


@pytest.mark.parametrize("path,sources,alg", [
    (bench.TRAFFIC_FILE, bench.KERNEL_SOURCES, 151060480),
    (bench.TRAFFIC8_FILE, bench.KERNEL8_SOURCES, 151060480),
    (bench.PREFILL_TRAFFIC_FILE, bench.PREFILL_SOURCES, 270794752),
])
def test_profile_summaries_feed_roofline_traffic(path, sources, alg):
    # each committed ncu summary names the source hash it was taken on, its
    # DRAM bytes per launch and the algorithmic bytes of the same launch
    vals = _profile_values(path)
    assert int(vals["algorithmic_bytes_per_launch"]) == alg
    traffic = int(vals["dram_bytes_per_launch"])
    # measured traffic can only exceed the algorithmic bytes (re-reads,
    # write-backs), and not by much for these kernels
    assert alg <= traffic <= 1.25 * alg
    # the bench reports it only while the sources hash to the recorded value
    got = bench.traffic_per_launch(path, sources)
    assert got in (None, traffic)
    assert (got == traffic) == (vals["kernel_source_sha256"] == bench.kernel_source_hash(sources))
    assert bench.traffic_per_launch(path, ("workloads.py",)) is None


def test_headline_algorithmic_bytes_per_launch():
    # the decode launch moves the step's bytes except the bf16 output, which
    # the combine writes
    ab = bench.algorithmic_bytes(workloads.make_workload("llama8b_32k"))
    assert ab["step"] - ab["out"] == 151060480
