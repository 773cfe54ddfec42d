"""Host-side parts of the benchmark that need no GPU: the reference arm (the oracle on
the host cores) and the workload configs the JSON line reports."""

import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line():
    """`bench.py --impl reference` (the oracle on the host cores) prints one JSON line with
    the contract's keys; its end-to-end number moves no bytes between host and device."""
    import subprocess
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 0
    assert d["value"] > 0 and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["config"]["workload"].startswith("gqa_lognormal")
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["cpu_baseline"]["value"] == d["value"] and d["cpu_baseline"]["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_bench_configs_name_their_workloads():
    """Every decode workload's config names it with its sizes and formats (the JSON line's
    `config`), and the default workload is the GQA decode at 32K keys."""
    sys.path.insert(0, ROOT)
    import bench
    import synth
    for name in bench.DECODE:
        w = synth.WORKLOADS[name]
        c = bench.decode_config(name, w)
        assert c["workload"].startswith(f"{name}: B={w['B']} Hq={w['Hq']} Hkv={w['Hkv']} d={w.get('d', 128)} "
                                        f"L={w['L']}")
        assert c["k_format"] in ("turbo4", "turbo3", "prod3") and c["v_format"] in ("turbo4", "turbo3", "vgroup2")
        # inputs larger than twice the L2 run back to back, the others flush before each step
        big = w["B"] * w["Hkv"] * w["L"] * bench.decode_unit_bytes(bench.DECODE[name]) > 2 * bench.L2_NOMINAL
        assert ("back to back" in c["l2"]) == big and ("flushed" in c["l2"]) != big
    d = bench.decode_config("gqa_lognormal", synth.WORKLOADS["gqa_lognormal"])
    assert (d["B"], d["Hq"], d["Hkv"], d["L"], d["rotation"]) == (8, 32, 8, 32768, "dense")
    p = bench.prefill_config()
    assert p["mask"] == "causal" and p["T"] == synth.WORKLOADS["prefill_chunk"]["T"]


def _bench(*args, timeout=600):
    import subprocess
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                       timeout=timeout, cwd=ROOT, env={k: v for k, v in os.environ.items() if k != "WORLD_SIZE"})
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-3000:]
    return json.loads(lines[0])


def test_gpus_flag_starts_that_many_ranks():
    """`--gpus 2` outside torchrun starts two ranks under torchrun (127.0.0.1); rank 0 alone
    prints the line, which reports n_gpus 2 (the reference arm: no GPU needed)."""
    d = _bench("--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0", "--workload", "single_head")
    assert d["n_gpus"] == 2 and d["impl"] == "reference" and d["warmup"] == 0


def test_context_sweep_flags_set_the_workload():
    """--B / --L override a decode workload's batch and context, and the config says so."""
    d = _bench("--impl", "reference", "--steps", "1", "--warmup", "0", "--workload", "long_context",
               "--B", "2", "--L", "4096")
    assert (d["config"]["B"], d["config"]["L"]) == (2, 4096)
    assert d["config"]["workload"] == "long_context: B=2 Hq=32 Hkv=8 d=128 L=4096"


def test_gpu_arm_and_reference_arm_share_one_config_builder():
    """Both arms report decode_config(name, workload): the same dict for the same flags."""
    sys.path.insert(0, ROOT)
    import argparse

    import bench
    a = argparse.Namespace(workload="long_context", B=16, L=65536)
    assert bench.decode_config("long_context", bench.decode_workload(a)) == \
        bench.decode_config("long_context", bench.decode_workload(a))
    assert "launch" not in bench.decode_config("long_context", bench.decode_workload(a))
