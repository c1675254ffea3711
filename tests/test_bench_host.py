"""Host-side logic of bench.py, on the CPU: the replica timing reduction over
ranks (two gloo processes), clock-sample parsing, layer-set sizing against L2,
and the ncu traffic lookup that must go null when the kernel source changes."""
import json
import os
import socket

import pytest

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(world)
    got = bench.max_over_ranks(1.5 + rank, world)
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump({"max": got}, f)
    dist.destroy_process_group()


def test_max_over_two_gloo_ranks(tmp_path):
    import torch.multiprocessing as mp
    port = _free_port()
    mp.spawn(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    for r in range(2):
        assert json.load(open(tmp_path / f"r{r}.json"))["max"] == 2.5


def test_single_rank_is_identity():
    assert bench.max_over_ranks(3.25, 1) == 3.25


def test_clock_summary_parsing(tmp_path):
    c = bench.Clocks(0)
    c.path = str(tmp_path / "clk.csv")
    with open(c.path, "w") as f:
        f.write("0, 1965, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Active\n")
        f.write("0, 1980, 2070, 950.0, 0x0, Not Active, Not Active, Not Active, Not Active\n")
        f.write("0, 1995, 2070, 910.0, 0x0, Not Active, Active, Not Active, Not Active\n")
    s = c.summary()
    assert s["sm_mhz"] == 1980 and s["sm_max_mhz"] == 2070 and s["samples"] == 3
    assert s["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]


def test_decode_layer_sets_exceed_three_l2():
    from dit_convrot_linear_gb300 import synth
    l2 = 126 * 2 ** 20
    for bits in (8, 4):
        L = bench.decode_layers(bits, l2)
        per = sum(p.N * p.K * bits // 8 + 4 * p.N for p in synth.DECODE.projs)
        assert L >= synth.DECODE.layers and L * per >= 3 * l2


def test_traffic_lookup_goes_null_on_source_change(tmp_path, monkeypatch):
    path = tmp_path / "traffic.json"
    sha = bench.source_sha("k_gemv.cu", "tq_internal.cuh")
    path.write_text(json.dumps({"k_gemv_a16": {"source_sha": sha, "bytes_per_launch": 123}}))
    monkeypatch.setattr(bench, "TRAFFIC_PATH", str(path))
    assert bench.traffic_for("k_gemv_a16", ["k_gemv.cu", "tq_internal.cuh"]) == 123
    path.write_text(json.dumps({"k_gemv_a16": {"source_sha": "stale", "bytes_per_launch": 123}}))
    assert bench.traffic_for("k_gemv_a16", ["k_gemv.cu", "tq_internal.cuh"]) is None


def test_cpu_baseline_sample_bounds_and_threads():
    """The CPU-oracle baseline stops at its call cap or its time budget, cycles
    its 60 seeded inputs past the cap of one pass, and reports the threads it
    ran on (one when the oracle is set to one)."""
    import oracle
    r = bench.cpu_oracle_decode(8, budget_s=60.0, min_calls=3, max_calls=62)
    assert r["sample"].startswith("62 decode calls") and r["kind"] == "oracle"
    assert r["cores"] == oracle.threads() and r["value"] > 0
    oracle.set_threads(1)
    try:
        one = bench.cpu_oracle_decode(8, budget_s=0.0, min_calls=3)
        assert one["cores"] == 1 and one["sample"].startswith("3 decode calls")
    finally:
        oracle.set_threads(None)
    assert oracle.threads() == max(1, os.cpu_count() or 1)
