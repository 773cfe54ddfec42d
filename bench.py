"""Benchmark of the compressed-KV decode step on GB300.

One step = one decode step of the whole hot path on the GQA workload
(B=8, Hq=32, Hkv=8, d=128, context 32,768, turbo4 4-bit K and V, dense seeded
rotation, bf16 q, K/V N(0,1) x per-channel lognormal(0, 0.5) with 1% x8 outlier
channels):
  write path : SET_ROWS of the step's new K and V rows (B*Hkv each) into the cache,
  read path  : q rotation + split, split-K fused decode over the packed cache,
               combine + un-rotation.
The metric is effective HBM bandwidth of the decode (algorithmic bytes / time),
with keys/s alongside; the dominant kernel (split-K decode) is also timed alone
for the roofline.  Inputs are synthetic and seeded (see synth.py).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl tq|reference]
Under torchrun every rank runs the same per-GPU workload (weak scaling) and rank 0
prints one JSON line.
"""

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "fused compressed-KV decode attention: effective HBM GB/s (% of peak), keys/s"
WORKLOAD = "gqa_lognormal"
ROT_SEED_K, ROT_SEED_V = 2, 102
ROW_BYTES = 68
L2_FLUSH_BYTES = 256 << 20
PROFILE = os.path.join(ROOT, "profiles", "decode_partial_gqa_lognormal.md")
FALLBACK_HBM_GBS = 6800.0


def algorithmic_bytes(cfg):
    """Packed K + V of every key of every KV head, plus q (bf16) in and out (fp32)."""
    B, Hq, Hkv, L = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["L"]
    kv = B * Hkv * L * 2 * ROW_BYTES
    return kv, kv + B * Hq * 128 * 2 + B * Hq * 128 * 4


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def profiled_traffic():
    """Per-launch DRAM bytes of the decode kernel from the committed ncu summary, or None
    when the kernel source changed since the capture."""
    if not os.path.exists(PROFILE):
        return None
    fields = {}
    for ln in open(PROFILE):
        if ":" in ln and ln.strip().startswith("- "):
            k, v = ln.strip()[2:].split(":", 1)
            fields[k.strip()] = v.strip()
    src = os.path.join(ROOT, "compressed_attention_gb300", "csrc", "tq_decode.cu")
    digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    if fields.get("source_sha256_16") != digest:
        return None
    try:
        return float(fields["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.idx = device_index
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.file, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for ln in f:
                parts = [p.strip() for p in ln.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.file.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------------------- ranks

def max_over_ranks(x, dist, device):
    """Largest value of the scalar x over all ranks (x itself without a process group)."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank, world, ms):
    """Whole-job rate (units/s) when every rank processes units_per_rank in at most ms."""
    return world * units_per_rank / (ms * 1e-3)


# ----------------------------------------------------------------------------- CPU side

def cpu_oracle_sample(cfg, min_seconds=10.0, max_units=64):
    """Time the oracle (fp64 dequantize-then-softmax attention) on whole (b, KV head) units
    of the workload until about ``min_seconds`` of CPU work; returns GB/s and keys/s."""
    import oracle
    from oracle.formats import Codec
    kc = Codec("turbo4", rotation="dense", rot_seed=ROT_SEED_K)
    vc = Codec("turbo4", rotation="dense", rot_seed=ROT_SEED_V)
    q32, _ = synth.queries(cfg)
    L, g = cfg["L"], cfg["Hq"] // cfg["Hkv"]
    elapsed, units = 0.0, 0
    while units < max_units and (elapsed < min_seconds or units == 0):
        b, h = divmod(units, cfg["Hkv"])
        b %= cfg["B"]
        kb = kc.encode(synth.kv_unit(cfg, "K", b, h)[0])[0]  # inputs: packed blocks (untimed)
        vb = vc.encode(synth.kv_unit(cfg, "V", b, h)[0])[0]
        t0 = time.perf_counter()
        kh = kc.dequantize(kb)[None, None]
        vh = vc.dequantize(vb)[None, None]
        oracle.attention_reference(q32[b:b + 1, h * g:(h + 1) * g], kh, vh)
        elapsed += time.perf_counter() - t0
        units += 1
    keys = units * L
    return {"gbs": keys * 2 * ROW_BYTES / elapsed / 1e9, "keys_per_s": keys / elapsed, "units": units,
            "seconds": elapsed}


def run_reference(args, rank, world):
    if rank != 0:
        return
    cfg = synth.WORKLOADS[WORKLOAD]
    import oracle
    from oracle.formats import Codec
    kc = Codec("turbo4", rotation="dense", rot_seed=ROT_SEED_K)
    vc = Codec("turbo4", rotation="dense", rot_seed=ROT_SEED_V)
    q32, _ = synth.queries(cfg)
    g = cfg["Hq"] // cfg["Hkv"]
    blocks = {}
    for u in range(2):
        b, h = divmod(u, cfg["Hkv"])
        blocks[u] = (kc.encode(synth.kv_unit(cfg, "K", b, h)[0])[0], vc.encode(synth.kv_unit(cfg, "V", b, h)[0])[0])

    def step(u):
        b, h = divmod(u, cfg["Hkv"])
        kb, vb = blocks[u % 2]
        oracle.attention_reference(q32[b:b + 1, h * g:(h + 1) * g], kc.dequantize(kb)[None, None],
                                   vc.dequantize(vb)[None, None])

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(i)
    dt = time.perf_counter() - t0
    keys = args.steps * cfg["L"]
    gbs = keys * 2 * ROW_BYTES / dt / 1e9
    sample = f"one (batch, KV head) unit per step: {cfg['L']} keys x {g} q-heads"
    line = {"impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_dict(cfg),
            "keys_per_s": keys / dt,
            "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": os.cpu_count(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def config_dict(cfg):
    return {"workload": f"{WORKLOAD}: B={cfg['B']} Hq={cfg['Hq']} Hkv={cfg['Hkv']} d=128 L={cfg['L']}",
            "B": cfg["B"], "Hq": cfg["Hq"], "Hkv": cfg["Hkv"], "L": cfg["L"], "d": 128,
            "k_format": "turbo4", "v_format": "turbo4", "rotation": "dense",
            "l2": "flushed before every step: 256 MB write then a read of it (no dirty lines left); "
                  "packed K/V 285 MB > 129 MB L2",
            "launch": "each step replayed from CUDA graphs, steps queued back to back"}


# ----------------------------------------------------------------------------- GPU side

def build_workload(tq, torch, cfg, device):
    B, Hq, Hkv, L = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["L"]
    kctx = tq.Ctx("turbo4", "dense", ROT_SEED_K)
    vctx = tq.Ctx("turbo4", "dense", ROT_SEED_V)
    kc = tq.alloc_cache("turbo4", B * Hkv * L, device)
    vc = tq.alloc_cache("turbo4", B * Hkv * L, device)
    for tensor, ctx, cache in (("K", kctx, kc), ("V", vctx, vc)):
        for b in range(B):
            for h in range(Hkv):
                _, bits = synth.kv_unit(cfg, tensor, b, h)
                src = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(device)
                rows = torch.arange((b * Hkv + h) * L, (b * Hkv + h + 1) * L, dtype=torch.int64, device=device)
                tq.tq_quantize_set_rows(ctx, src, cache, row_ids=rows)
    _, qbits = synth.queries(cfg)
    q = torch.from_numpy(qbits.view(np.int16)).view(torch.bfloat16).to(device)
    # the step's new token: one K and one V row per (b, KV head), written to slot L-1
    rng = np.random.default_rng([cfg["seed"], 99])
    new_k = torch.from_numpy(synth.bf16_bits(rng.standard_normal((B * Hkv, 128), dtype=np.float32))
                             .view(np.int16)).view(torch.bfloat16).to(device)
    new_v = torch.from_numpy(synth.bf16_bits(rng.standard_normal((B * Hkv, 128), dtype=np.float32))
                             .view(np.int16)).view(torch.bfloat16).to(device)
    slots = torch.tensor([(u + 1) * L - 1 for u in range(B * Hkv)], dtype=torch.int64, device=device)
    ws = tq.alloc_workspace(tq.tq_decode_workspace_size(kctx, vctx, B, Hq, Hkv, L), device)
    out = torch.empty((B, Hq, 128), dtype=torch.float32, device=device)
    torch.cuda.synchronize()
    return dict(kctx=kctx, vctx=vctx, kc=kc, vc=vc, q=q, new_k=new_k, new_v=new_v, slots=slots, ws=ws, out=out)


def run_tq(args, rank, world, dist):
    import torch

    import compressed_attention_gb300 as tq

    local = int(os.environ.get("LOCAL_RANK", 0))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    cfg = synth.WORKLOADS[WORKLOAD]
    B, Hq, Hkv, L = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["L"]
    w = build_workload(tq, torch, cfg, device)
    stream = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    flush_f32 = flush.view(torch.float32)

    def flush_l2():
        # Write a buffer twice the L2 size, then read it back: the write evicts every line
        # of the inputs, the read leaves the L2 holding clean lines of the flush buffer,
        # so the timed step neither hits cached inputs nor pays for the flush's write-backs.
        flush.zero_()
        flush_f32.sum()

    launches_per_step = 5

    def write_and_prepare():
        tq.tq_quantize_set_rows(w["kctx"], w["new_k"], w["kc"], row_ids=w["slots"])
        tq.tq_quantize_set_rows(w["vctx"], w["new_v"], w["vc"], row_ids=w["slots"])
        tq.tq_decode_prepare_q(w["kctx"], w["vctx"], w["q"], w["ws"], B, Hq, Hkv, L)

    def partial():
        tq.tq_decode_partial(w["kctx"], w["vctx"], w["kc"], w["vc"], w["ws"], B, Hq, Hkv, L)

    def combine():
        tq.tq_decode_combine(w["kctx"], w["vctx"], w["out"], w["ws"], B, Hq, Hkv, L)

    for _ in range(args.warmup):
        flush_l2()
        write_and_prepare()
        partial()
        combine()
    torch.cuda.synchronize()

    # The step is replayed from three CUDA graphs (write + q preparation, split-K decode,
    # combine) so host launch latency stays out of the device-timed region; events between
    # the graphs time the decode kernel alone on the same stream.
    graphs = []
    for fn in (write_and_prepare, partial, combine):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        graphs.append(g)
    for _ in range(args.warmup):
        flush_l2()
        for g in graphs:
            g.replay()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()

    def timed_steps():
        # Every step and its L2 flush are queued without a host synchronisation in between,
        # so the host runs ahead of the device and no enqueue gap enters a timed region.
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
        for e in ev:
            flush_l2()
            e[0].record(stream)
            graphs[0].replay()
            e[1].record(stream)
            graphs[1].replay()
            e[2].record(stream)
            graphs[2].replay()
            e[3].record(stream)
        torch.cuda.synchronize()
        return ([e[0].elapsed_time(e[3]) for e in ev], [e[1].elapsed_time(e[2]) for e in ev])

    with ClockSampler(local) as clocks:
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        step_ms, part_ms = timed_steps()
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
    clk = clocks.summary()
    total_ms = max_over_ranks(sum(step_ms), dist, device)

    # end to end through the public API with host buffers: q and the new K/V rows copied in,
    # the output read back, every step.
    hq = torch.empty(w["q"].shape, dtype=torch.bfloat16, pin_memory=True).copy_(w["q"].cpu())
    hk = torch.empty(w["new_k"].shape, dtype=torch.bfloat16, pin_memory=True).copy_(w["new_k"].cpu())
    hv = torch.empty(w["new_v"].shape, dtype=torch.bfloat16, pin_memory=True).copy_(w["new_v"].cpu())
    hout = torch.empty(w["out"].shape, dtype=torch.float32, pin_memory=True)
    h2d = (hq.numel() + hk.numel() + hv.numel()) * 2
    d2h = hout.numel() * 4
    e2e_ms = []
    for i in range(args.warmup + args.steps):
        flush_l2()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        w["q"].copy_(hq, non_blocking=True)
        w["new_k"].copy_(hk, non_blocking=True)
        w["new_v"].copy_(hv, non_blocking=True)
        tq.tq_quantize_set_rows(w["kctx"], w["new_k"], w["kc"], row_ids=w["slots"])
        tq.tq_quantize_set_rows(w["vctx"], w["new_v"], w["vc"], row_ids=w["slots"])
        tq.tq_decode_attention(w["kctx"], w["vctx"], w["q"], w["kc"], w["vc"], w["out"], w["ws"], B, Hq, Hkv, L)
        hout.copy_(w["out"], non_blocking=True)
        torch.cuda.synchronize()
        if i >= args.warmup:
            e2e_ms.append((time.perf_counter() - t0) * 1e3)
    status = tq.tq_ctx_device_status(w["kctx"]) or tq.tq_ctx_device_status(w["vctx"])
    if status:
        raise RuntimeError(f"device status {status} after the benchmark")

    kv_bytes, alg_bytes = algorithmic_bytes(cfg)
    ms_per_step = total_ms / args.steps
    value = job_rate(alg_bytes, world, ms_per_step) / 1e9
    keys = B * Hkv * L
    part_avg = max_over_ranks(statistics.mean(part_ms), dist, device)
    peak, peak_kind = measured_peak()
    achieved = kv_bytes / (part_avg * 1e-3) / 1e9
    e2e_step_ms = max_over_ranks(statistics.mean(e2e_ms), dist, device)
    e2e_gbs = job_rate(alg_bytes, world, e2e_step_ms) / 1e9
    if rank != 0:
        return
    cpu = cpu_oracle_sample(cfg) if world == 1 else None  # host-core baseline: N=1 only
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": config_dict(cfg),
        "keys_per_s": job_rate(keys, world, ms_per_step),
        "q_head_scores_per_s": job_rate(B * Hq * L, world, ms_per_step),
        "hbm_frac_of_measured_step": value / peak,
        "operands": "4-bit packed K/V decoded in registers to fp16 centroids; fp16 hi+lo q and p; fp32 accumulate",
        "roofline": {"bound": "hbm", "kernel": "k_partial_t4 (split-K decode)", "achieved": achieved,
                     "peak": peak, "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": profiled_traffic(), "algorithmic_bytes_per_launch": kv_bytes,
                     "avg_launch_ms": part_avg},
        "cpu_baseline": None if cpu is None else {
            "value": cpu["gbs"], "unit": "GB/s", "cores": os.cpu_count(), "kind": "oracle",
            "keys_per_s": cpu["keys_per_s"],
            "sample": f"{cpu['units']} whole (batch, KV head) units of {cfg['L']} keys x "
                      f"{Hq // Hkv} q-heads, fp64 dequantize-then-softmax, {cpu['seconds']:.1f} s"},
        "e2e": {"value": e2e_gbs, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_step_ms},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["tq", "reference"], default="tq")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group("nccl")
    try:
        run_tq(args, rank, world, dist)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
