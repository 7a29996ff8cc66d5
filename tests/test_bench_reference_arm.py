"""The benchmark's reference arm (the CPU oracle timed on the host cores) on
the smallest workload, without a GPU: one JSON line with the contract's keys,
and nothing from ranks other than 0."""

import json


def test_reference_arm_prints_one_contract_line(capsys, monkeypatch):
    import bench
    monkeypatch.delenv("RANK", raising=False)
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "3", "--warmup", "3"])
    lines = [l for l in capsys.readouterr().out.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["value"] > 0 and d["higher_is_better"] is True
    assert d["steps"] == 3 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["dtype"] == "f64" and d["data"] == "synthetic"
    assert d["config"]["workload"] == bench.WORKLOAD_TEXT["tiny"]
    # the same workload description as the library's own arm prints
    from paged_kv_cache_68_gb300 import workloads as wl
    args = bench.parse_args(["--workload", "tiny"])
    w = wl.on_host(bench.make_workload("tiny", 0, None))
    assert d["config"] == bench.decode_config(args, w, None, 1)
    assert d["config"]["global_batch"] == 4 and d["config"]["parallelism"] == "replicas x1"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1
    assert cb["unit"] == d["unit"] and cb["sample"]
    assert isinstance(cb["cpu_model"], str) and cb["cpu_model"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_do_no_work(capsys, monkeypatch):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "3", "--warmup", "3"])
    assert capsys.readouterr().out.strip() == ""
