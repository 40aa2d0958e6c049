"""The bench's reference arm (the fp64 oracle timed on the host cores) prints
one JSON line with the contract's keys; run on CPU with a capped sample."""
import json
import types

import bench


def test_reference_line(monkeypatch, capsys):
    real = bench.oracle_sample
    monkeypatch.setattr(bench, "oracle_sample",
                        lambda wl, seconds, pool, workers, start_head=0:
                        real(wl, 0.05, pool, workers, start_head))
    monkeypatch.setattr(bench, "oracle_workers", lambda: 2)
    args = types.SimpleNamespace(config="tiny", steps=2, warmup=1, gpus=1)
    bench.run_reference(args)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "cpu_baseline", "e2e"):
        assert k in line, k
    assert line["impl"] == "reference" and line["n_gpus"] == 1 and line["steps"] == 2
    assert line["value"] > 0 and line["unit"] == "query-heads/s" and line["higher_is_better"]
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 2 and cb["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"], "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert line["config"]["workload"].startswith("tiny")
    # the same workload description as the GPU arm prints
    from workloads import preset
    assert line["config"] == bench.bench_config(preset("tiny"), 1, bench.kv_copies(preset("tiny")))


def test_default_workload_is_the_largest():
    """With no --config the bench measures the largest single-GPU workload."""
    import sys
    from workloads import PRESETS
    monkey_argv = sys.argv
    try:
        sys.argv = ["bench.py"]
        args = bench.parse_args()
    finally:
        sys.argv = monkey_argv
    assert args.config == "paged_serving" and "paged_serving" in PRESETS
    assert bench.PASSES["paged_serving"] >= 1
