"""bench.py's reference arm (the oracle timed on the host cores) prints the
one JSON line of the benchmark contract, on rank 0 only; runs without a GPU."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(env_extra=None):
    env = dict(os.environ)
    env.update(env_extra or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                           "--warmup", "0"], capture_output=True, text=True, env=env, timeout=600, cwd=ROOT)


def test_reference_arm_json_line():
    r = _run()
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "GB/s"
    assert d["steps"] == 1 and d["warmup"] == 0 and d["n_gpus"] == 1 and d["higher_is_better"] is True
    assert d["vs_baseline"] is None and d["data"] == "synthetic" and "workload" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_print_nothing():
    r = _run({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_e2e_copy_groups_cover_every_layer_once():
    """The end-to-end step's pipelined copies: every layer's inputs and
    outputs are copied exactly once, in layer order; the first input group
    is layer 0 alone (the first layer waits for one layer's inputs) and the
    last output group is the last layer alone (one output left to copy after
    the last layer); input groups double, output groups halve."""
    sys.path.insert(0, ROOT)
    import bench
    for layers in (1, 2, 3, 5, 7, 8, 32, 48, 80):
        ins, outs = bench.copy_groups(layers)
        for groups in (ins, outs):
            assert [l for a, b in groups for l in range(a, b)] == list(range(layers)), (layers, groups)
            assert all(b > a for a, b in groups)
        assert ins[0] == (0, 1) and outs[-1] == (layers - 1, layers)
        assert all(ins[i + 1][1] - ins[i + 1][0] >= ins[i][1] - ins[i][0] for i in range(len(ins) - 2))
        assert all(outs[i][1] - outs[i][0] >= outs[i + 1][1] - outs[i + 1][0] for i in range(1, len(outs) - 1))
        assert len(ins) <= layers.bit_length() + 1 and len(outs) <= layers.bit_length() + 1
