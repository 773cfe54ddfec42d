"""Benchmark of the compressed-KV hot path on GB300.

Default (the headline line): one decode step of the whole path on the GQA workload
(B=8, Hq=32, Hkv=8, d=128, context 32,768, turbo4 4-bit K and V, dense seeded
rotation, bf16 q, K/V N(0,1) x per-channel lognormal(0, 0.5) with 1% x8 outlier
channels):
  write path : SET_ROWS of the step's new K and V rows (B*Hkv each) into the cache,
  read path  : q rotation + split, split-K fused decode over the packed cache,
               combine + un-rotation.
The metric is effective HBM bandwidth of the decode (algorithmic bytes / time), with
keys/s alongside; the dominant kernel (split-K decode) is also timed alone for the
roofline.

--workload picks another workload of the same path:
  gqa_t3k       the gqa_lognormal inputs with turbo3 keys and turbo4 values
  gqa_t3        the gqa_lognormal inputs with turbo3 keys and turbo3 values
  gqa_d256      head dimension 256: B=4, Hq=32, Hkv=8, L=32,768, turbo4 K and V, dense
  prefill_chunk causal attention of the last 512-token chunk of a 32K-token prompt
                (B=1, Hq=32, Hkv=8) over the turbo4 cache, tensor cores; TFLOP/s
  long_context  B=1, Hq=32, Hkv=8, L=131,072, turbo4 K and V, randomized WHT
  prod_vgroup   B=4, Hq=24, Hkv=4, L=30,000, prod3 keys (2-bit + QJL), vgroup2 values
  single_head   B=1, Hq=Hkv=1, L=512, fp32 q, turbo4 K and V, randomized WHT
  write_chunk   SET_ROWS of 16,384 tokens x 8 KV heads of bf16 K and V
                (--write-format turbo4|turbo3, --write-rotation dense|wht)
Inputs are synthetic and seeded (see synth.py).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl tq|reference]
                       [--workload NAME] [--B B] [--L L]
--B / --L override the batch and context of a decode workload (the context sweep:
long_context at L = 4K, 16K, 64K, 128K and B = 1, 16).
Under torchrun every rank runs the same per-GPU workload (weak scaling) and rank 0
prints one JSON line; --gpus N > 1 outside torchrun starts N ranks under torchrun.
"""

import os

# The oracle legs (numpy) run on one host core: their BLAS calls are kept single-threaded
# so that the reported core count is the one used.
os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
os.environ.setdefault("MKL_NUM_THREADS", "1")

import argparse
import hashlib
import re
import json
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

DECODE_METRIC = "fused compressed-KV decode attention: effective HBM GB/s (% of peak), keys/s"
WRITE_METRIC = "quantize / SET_ROWS write path: effective HBM GB/s (% of peak), rows/s"
PREFILL_METRIC = "chunked prefill attention over the compressed cache: effective TFLOP/s (% of tensor peak), tokens/s"
FALLBACK_TENSOR_TFLOPS = 1900.0
L2_FLUSH_BYTES = 256 << 20
FALLBACK_HBM_GBS = 6800.0
ROW_BYTES = {"turbo4": 68, "turbo3": 56, "prod3": 56, "vgroup2": 48}
CSRC = os.path.join(ROOT, "compressed_attention_gb300", "csrc")

# Decode workloads: formats, rotation and seeds of the K and V contexts, and the kernel
# that dominates the step.
DECODE = {
    "gqa_lognormal": dict(k_fmt="turbo4", v_fmt="turbo4", rotation="dense", k_seed=2, v_seed=102, qjl_seed=0,
                          kernel="k_partial_t4", source="tq_decode.cu"),
    "long_context": dict(k_fmt="turbo4", v_fmt="turbo4", rotation="wht", k_seed=5, v_seed=105, qjl_seed=0,
                         kernel="k_partial_t4", source="tq_decode.cu"),
    "prod_vgroup": dict(k_fmt="prod3", v_fmt="vgroup2", rotation="dense", k_seed=3, v_seed=0, qjl_seed=1003,
                        kernel="k_partial_pv", source="tq_decode_pv.cu"),
    "single_head": dict(k_fmt="turbo4", v_fmt="turbo4", rotation="wht", k_seed=0, v_seed=100, qjl_seed=0,
                        kernel="k_partial_t4", source="tq_decode.cu"),
    "gqa_t3k": dict(k_fmt="turbo3", v_fmt="turbo4", rotation="dense", k_seed=6, v_seed=106, qjl_seed=0,
                    kernel="k_partial_t4", source="tq_decode.cu"),
    "gqa_t3": dict(k_fmt="turbo3", v_fmt="turbo3", rotation="dense", k_seed=8, v_seed=108, qjl_seed=0,
                   kernel="k_partial_t4", source="tq_decode.cu"),
    "gqa_d256": dict(k_fmt="turbo4", v_fmt="turbo4", rotation="dense", k_seed=9, v_seed=109, qjl_seed=0,
                     kernel="k_partial_d256", source="tq_d256.cu", d=256),
}
WRITE_KERNEL = {"dense": ("k_write_dense_tc", "tq_write_tc.cu"), "wht": ("k_write_wht", "tq_write.cu")}
PREFILL = {"prefill_chunk": dict(fmt="turbo4", rotation="dense", k_seed=7, v_seed=107,
                                 kernel="k_prefill_t4", source="tq_prefill.cu")}


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def measured_tensor_peak():
    """Dense 16-bit tensor-core peak (TFLOP/s) for a kernel timed alone: the burst cuBLAS
    bf16 figure (fp16 products run at the same nominal rate)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    return FALLBACK_TENSOR_TFLOPS, "fallback"


def source_digest(source):
    """First 16 hex digits of the SHA-256 of a kernel source with its comments and blank
    space removed: what the compiler sees, so a comment edit keeps a profile valid while
    any code change retires it."""
    text = open(os.path.join(CSRC, source), encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return hashlib.sha256(" ".join(text.split()).encode()).hexdigest()[:16]


def profiled_fields(profile_name, source):
    """The "- key: value" fields of a kernel's committed ncu summary
    (profiles/<profile_name>.md), or None when the kernel source changed since the capture
    or there is no summary."""
    path = os.path.join(ROOT, "profiles", profile_name + ".md")
    if not os.path.exists(path):
        return None
    fields = {}
    for ln in open(path):
        if ":" in ln and ln.strip().startswith("- "):
            k, v = ln.strip()[2:].split(":", 1)
            fields[k.strip()] = v.strip()
    if fields.get("source_sha256_16") != source_digest(source):
        return None
    return fields


def profiled_number(profile_name, source, key):
    fields = profiled_fields(profile_name, source)
    try:
        return float(fields[key]) if fields else None
    except (KeyError, ValueError):
        return None


def profiled_traffic(profile_name, source):
    """Per-launch DRAM bytes of a kernel from its committed ncu summary, or None."""
    return profiled_number(profile_name, source, "traffic_bytes_per_launch")


def issue_roofline(profile_name, source, kernel, avg_ms, clk, n_sms):
    """Instruction-issue roofline of a kernel bound by issue rather than by DRAM: its warp
    instructions per launch (ncu's smsp__inst_executed.sum in the committed summary, null
    when the source changed since) over the live launch time, against one warp instruction
    per cycle on each of the four schedulers of every SM at the SM clock sampled during the
    timed region."""
    inst = profiled_number(profile_name, source, "warp_instructions_per_launch")
    mhz = clk.get("sm_mhz") or clk.get("sm_max_mhz")
    peak = 4 * n_sms * mhz * 1e6 / 1e9 if mhz else None  # Ginst/s
    achieved = inst / (avg_ms * 1e-3) / 1e9 if inst else None
    return {"bound": "issue", "kernel": kernel, "achieved": achieved, "peak": peak, "unit": "Gwarp-inst/s",
            "frac": achieved / peak if achieved and peak else None,
            "warp_instructions_per_launch": inst, "sm_mhz": mhz, "sms": n_sms, "avg_launch_ms": avg_ms}


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

def decode_codecs(spec):
    from oracle.formats import Codec

    def make(fmt, seed):
        if fmt == "vgroup2":
            return Codec("vgroup2")
        return Codec(fmt, d=spec.get("d", 128), rotation=spec["rotation"], rot_seed=seed, qjl_seed=spec["qjl_seed"])
    return make(spec["k_fmt"], spec["k_seed"]), make(spec["v_fmt"], spec["v_seed"])


def unit_rows(name, cfg, tensor, b, h):
    """K or V rows of one (batch, KV head) unit: (fp32 values, bf16 bits or None)."""
    if name == "single_head":
        K, V, _ = synth.single_head_inputs()
        return (K if tensor == "K" else V), None
    return synth.kv_unit(cfg, tensor, b, h)


def decode_queries(name, cfg):
    """q [B, Hq, 128]: (fp32 values, bf16 bits or None)."""
    if name == "single_head":
        return synth.single_head_inputs()[2].reshape(1, 1, 128), None
    return synth.queries(cfg)


def decode_unit_bytes(spec):
    return (ROW_BYTES[spec["k_fmt"]] + ROW_BYTES[spec["v_fmt"]]) * spec.get("d", 128) // 128


class OracleDecode:
    """The oracle (fp64 dequantize-then-softmax attention) over whole (batch, KV head)
    units of a decode workload; inputs are encoded once, outside any timing."""

    def __init__(self, name, cfg, n_units=2):
        import oracle
        self.attend = oracle.attention_reference
        self.cfg, self.spec = cfg, DECODE[name]
        self.kc, self.vc = decode_codecs(self.spec)
        self.q32, _ = decode_queries(name, self.cfg)
        self.g = self.cfg["Hq"] // self.cfg["Hkv"]
        self.blocks = []
        for u in range(min(n_units, self.cfg["B"] * self.cfg["Hkv"])):
            b, h = divmod(u, self.cfg["Hkv"])
            self.blocks.append((b, h, self.kc.encode(unit_rows(name, self.cfg, "K", b, h)[0])[0],
                                self.vc.encode(unit_rows(name, self.cfg, "V", b, h)[0])[0]))

    def unit(self, i):
        b, h, kb, vb = self.blocks[i % len(self.blocks)]
        self.attend(self.q32[b:b + 1, h * self.g:(h + 1) * self.g], self.kc.dequantize(kb)[None, None],
                    self.vc.dequantize(vb)[None, None])
        return self.cfg["L"]


def cpu_fp32_loop(leg, min_seconds=3.0):
    """The plain fp32 compressed-domain decode loop (oracle/cpu_decode_fp32.c: rotate q once,
    score from indices, online softmax, one un-rotation) over the oracle's encoded units,
    on one host core and on every host core (OpenMP over units).  turbo4 keys and values
    only; None for other formats or without a C compiler."""
    if leg.spec["k_fmt"] != "turbo4" or leg.spec["v_fmt"] != "turbo4" or leg.spec.get("d", 128) != 128:
        return None
    from oracle import build_cpu_baseline
    f = build_cpu_baseline.load()
    if f is None:
        return None
    L, g, cores = leg.cfg["L"], leg.g, os.cpu_count() or 1
    rk = np.ascontiguousarray(leg.kc.rot.R, np.float32)
    rv = np.ascontiguousarray(leg.vc.rot.R, np.float32)
    ck = np.ascontiguousarray(leg.kc.c32, np.float32)
    cv = np.ascontiguousarray(leg.vc.c32, np.float32)
    scale = np.float32(1.0 / np.sqrt(128.0))
    out = {}
    for threads in sorted({1, cores}):
        n_units = threads * 2  # the encoded units in turn, two per thread
        kb = np.ascontiguousarray(np.concatenate([leg.blocks[u % len(leg.blocks)][2] for u in range(n_units)]))
        vb = np.ascontiguousarray(np.concatenate([leg.blocks[u % len(leg.blocks)][3] for u in range(n_units)]))
        q = np.ascontiguousarray(np.concatenate([
            leg.q32[b:b + 1, h * g:(h + 1) * g] for b, h, _, _ in
            (leg.blocks[u % len(leg.blocks)] for u in range(n_units))], axis=1).reshape(1, n_units * g, 128),
            np.float32)
        o = np.zeros((1, n_units * g, 128), np.float32)
        t0, reps, used = time.perf_counter(), 0, 0
        while reps == 0 or time.perf_counter() - t0 < min_seconds:
            used = f(q.ctypes.data, kb.ctypes.data, vb.ctypes.data, 1, n_units * g, n_units, L, rk.ctypes.data,
                     rv.ctypes.data, ck.ctypes.data, cv.ctypes.data, scale, o.ctypes.data, threads)
            reps += 1
        dt = time.perf_counter() - t0
        keys = reps * n_units * L
        out["cores_1" if threads == 1 else "cores_all"] = {
            "value": keys * decode_unit_bytes(leg.spec) / dt / 1e9, "unit": "GB/s", "keys_per_s": keys / dt,
            "threads": used, "sample": f"{reps} x {n_units} units of {L} keys x {g} q-heads, {dt:.1f} s"}
    out["kind"] = "plain fp32 compressed-domain decode loop (C, OpenMP over units), not the oracle"
    out["host_cores"] = cores
    return out


class OracleWrite:
    """The oracle encoder over a block of rows of the write workload."""

    def __init__(self, fmt, rotation, n_tokens=256):
        from oracle.formats import Codec
        cfg = synth.WORKLOADS["write_chunk"]
        self.codec = Codec(fmt, rotation=rotation, rot_seed=cfg["seed"])
        self.x32, _ = synth.write_rows(cfg, "K", n_tokens=n_tokens)

    def unit(self, i):
        self.codec.encode(self.x32)
        return len(self.x32)


def cpu_sample(oracle_leg, unit_bytes, what, min_seconds=10.0, max_units=64):
    """Time the oracle on whole units until about min_seconds of CPU work."""
    elapsed, units, items = 0.0, 0, 0
    while units < max_units and (elapsed < min_seconds or units == 0):
        t0 = time.perf_counter()
        items += oracle_leg.unit(units)
        elapsed += time.perf_counter() - t0
        units += 1
    return {"value": items * unit_bytes / elapsed / 1e9, "unit": "GB/s", "cores": 1,
            "kind": "oracle", "rate": items / elapsed,
            "sample": f"{units} {what}, {elapsed:.1f} s, one host core (BLAS single-threaded)",
            "host_cores": os.cpu_count()}


def prefill_flops(cfg):
    """Algorithmic FLOPs of the chunk's attention: 2 d per (row, visible key) for the
    scores and 2 d for the PV product, rows = (b, query, q-head), query i seeing
    L - T + i + 1 keys."""
    T, L = cfg["T"], cfg["L"]
    pairs = cfg["B"] * cfg["Hq"] * (T * (L - T) + T * (T + 1) // 2)
    return 4 * 128 * pairs


class OraclePrefill:
    """The oracle's causal attention for a few chunk queries of one (batch, KV head) unit
    (its g q-heads) over the whole dequantized unit; the unit is encoded once, outside
    any timing."""

    def __init__(self, n_queries=64):
        import oracle
        from oracle.formats import Codec
        self.ref = oracle.prefill_reference
        self.cfg, self.spec = synth.WORKLOADS["prefill_chunk"], PREFILL["prefill_chunk"]
        cfg = self.cfg
        kc = Codec("turbo4", rotation=self.spec["rotation"], rot_seed=self.spec["k_seed"])
        vc = Codec("turbo4", rotation=self.spec["rotation"], rot_seed=self.spec["v_seed"])
        self.kh = kc.dequantize(kc.encode(synth.kv_unit(cfg, "K", 0, 0)[0])[0])[None, None]
        self.vh = vc.dequantize(vc.encode(synth.kv_unit(cfg, "V", 0, 0)[0])[0])[None, None]
        g = cfg["Hq"] // cfg["Hkv"]
        q32 = synth.prefill_queries(cfg)[0]
        self.n = n_queries
        self.q = q32[:1, cfg["T"] - n_queries:, :g]          # the chunk's last queries, KV head 0
        self.start = cfg["L"] - n_queries
        self.flops = 4 * 128 * g * sum(self.start + i + 1 for i in range(n_queries))

    def unit(self, i):
        self.ref(self.q, self.kh, self.vh, [self.start])
        return self.flops


def run_reference(args, rank, world):
    """The reference arm: the oracle as it stands on the host cores, one bounded sample of
    the workload per step, on rank 0 only."""
    if rank != 0:
        return
    if args.workload == "prefill_chunk":
        leg = OraclePrefill()
        for i in range(args.warmup):
            leg.unit(i)
        t0 = time.perf_counter()
        flops = sum(leg.unit(i) for i in range(args.steps))
        dt = time.perf_counter() - t0
        tf = flops / dt / 1e12
        sample = (f"per step: the last {leg.n} chunk queries x {leg.q.shape[2]} q-heads of one KV head "
                  f"over {leg.cfg['L']} keys, fp64 dequantize-then-softmax")
        line = {"impl": "reference", "metric": PREFILL_METRIC, "value": tf, "unit": "TFLOP/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": prefill_config(), "flops_per_step": leg.flops,
                "cpu_baseline": {"value": tf, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                                 "sample": sample + ", one host core (BLAS single-threaded)",
                                 "host_cores": os.cpu_count()},
                "e2e": {"value": tf, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return
    if args.workload == "write_chunk":
        leg = OracleWrite(args.write_format, args.write_rotation)
        unit_bytes = 256 + ROW_BYTES[args.write_format]
        metric, what = WRITE_METRIC, f"blocks of {len(leg.x32)} bf16 rows encoded by the oracle"
        config = write_config(args)
    else:
        cfg = decode_workload(args)
        leg = OracleDecode(args.workload, cfg)
        unit_bytes = decode_unit_bytes(leg.spec)
        metric = DECODE_METRIC
        what = (f"(batch, KV head) units of {leg.cfg['L']} keys x {leg.g} q-heads, "
                "fp64 dequantize-then-softmax")
        config = decode_config(args.workload, cfg)
    for i in range(args.warmup):
        leg.unit(i)
    t0 = time.perf_counter()
    items = sum(leg.unit(i) for i in range(args.steps))
    dt = time.perf_counter() - t0
    gbs = items * unit_bytes / dt / 1e9
    line = {"impl": "reference", "metric": metric, "value": gbs, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config, "items_per_s": items / dt,
            "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": f"one of {what} per step, one host core (BLAS single-threaded)",
                             "host_cores": os.cpu_count()},
            "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def decode_workload(args):
    """The decode workload's shape, with --B / --L applied."""
    cfg = dict(synth.WORKLOADS[args.workload])
    if getattr(args, "B", None):
        cfg["B"] = args.B
    if getattr(args, "L", None):
        cfg["L"] = args.L
    return cfg


L2_NOTE = "flushed before every step: 256 MB write then a read of it (no dirty lines left)"
L2_B2B_NOTE = "packed K/V larger than twice the L2: steps back to back, no flush"
L2_NOMINAL = 129 << 20  # GB300


def decode_back_to_back(name, cfg, l2=L2_NOMINAL):
    """Whether the decode workload's packed K/V exceed twice the L2 (then the steps run back
    to back without a flush: no step can be served from the L2)."""
    return cfg["B"] * cfg["Hkv"] * cfg["L"] * decode_unit_bytes(DECODE[name]) > 2 * l2


def decode_config(name, cfg, l2=L2_NOMINAL):
    spec = DECODE[name]
    d = spec.get("d", 128)
    return {"workload": f"{name}: B={cfg['B']} Hq={cfg['Hq']} Hkv={cfg['Hkv']} d={d} L={cfg['L']}",
            "B": cfg["B"], "Hq": cfg["Hq"], "Hkv": cfg["Hkv"], "L": cfg["L"], "d": d,
            "k_format": spec["k_fmt"], "v_format": spec["v_fmt"], "rotation": spec["rotation"],
            "q_dtype": cfg["q_dtype"], "l2": L2_B2B_NOTE if decode_back_to_back(name, cfg, l2) else L2_NOTE}


def prefill_config():
    cfg, spec = synth.WORKLOADS["prefill_chunk"], PREFILL["prefill_chunk"]
    return {"workload": (f"prefill_chunk: B={cfg['B']} Hq={cfg['Hq']} Hkv={cfg['Hkv']} d=128 L={cfg['L']} "
                         f"T={cfg['T']} (the last chunk of a {cfg['L']}-token prompt)"),
            "B": cfg["B"], "Hq": cfg["Hq"], "Hkv": cfg["Hkv"], "L": cfg["L"], "T": cfg["T"], "d": 128,
            "k_format": spec["fmt"], "v_format": spec["fmt"], "rotation": spec["rotation"],
            "q_dtype": cfg["q_dtype"], "mask": "causal", "l2": L2_NOTE}


def write_config(args):
    cfg = synth.WORKLOADS["write_chunk"]
    return {"workload": f"write_chunk: {cfg['N']} tokens x {cfg['Hkv']} KV heads x 128, bf16 K and V",
            "rows_per_tensor": cfg["N"] * cfg["Hkv"], "format": args.write_format,
            "rotation": args.write_rotation, "l2": L2_NOTE}


# ----------------------------------------------------------------------------- GPU side

def make_ctx(tq, fmt, spec, seed):
    if fmt == "vgroup2":
        return tq.Ctx("vgroup2")
    return tq.Ctx(fmt, spec["rotation"], seed, spec["qjl_seed"], d=spec.get("d", 128))


def to_device_rows(torch, x32, bits, device):
    if bits is None:
        return torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32)).to(device)
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def generated_units(name, cfg, tensor, workers=None):
    """(b, h, fp32 rows, bf16 bits) of every (batch, KV head) unit in order, drawn by a few
    host threads at a time (numpy's generators release the GIL while they fill arrays)."""
    from concurrent.futures import ThreadPoolExecutor
    units = [(b, h) for b in range(cfg["B"]) for h in range(cfg["Hkv"])]
    workers = workers or max(1, min(16, os.cpu_count() or 1))
    with ThreadPoolExecutor(max_workers=workers) as ex:
        for i in range(0, len(units), workers):
            chunk = units[i:i + workers]
            for (b, h), (x32, bits) in zip(chunk, ex.map(lambda u: unit_rows(name, cfg, tensor, *u), chunk)):
                yield b, h, x32, bits


def build_decode(name, cfg, tq, torch, device):
    spec = DECODE[name]
    B, Hq, Hkv, L = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["L"]
    kctx = make_ctx(tq, spec["k_fmt"], spec, spec["k_seed"])
    vctx = make_ctx(tq, spec["v_fmt"], spec, spec["v_seed"])
    d = spec.get("d", 128)
    kc = tq.alloc_cache(spec["k_fmt"], B * Hkv * L, device, d=d)
    vc = tq.alloc_cache(spec["v_fmt"], B * Hkv * L, device, d=d)
    for tensor, ctx, cache in (("K", kctx, kc), ("V", vctx, vc)):
        for b, h, x32, bits in generated_units(name, cfg, tensor):
            src = to_device_rows(torch, x32, bits, device)
            rows = torch.arange((b * Hkv + h) * L, (b * Hkv + h + 1) * L, dtype=torch.int64, device=device)
            tq.tq_quantize_set_rows(ctx, src, cache, row_ids=rows)
    q32, qbits = decode_queries(name, cfg)
    q = to_device_rows(torch, q32, qbits, device).reshape(B, Hq, d)
    # the step's new token: one K and one V row per (b, KV head), written to slot L-1
    rng = np.random.default_rng([cfg["seed"], 99])
    new = []
    for _ in range(2):
        x = rng.standard_normal((B * Hkv, d), dtype=np.float32)
        new.append(to_device_rows(torch, x, synth.bf16_bits(x) if cfg["kv_dtype"] == "bf16" else None, device))
    slots = torch.tensor([(u + 1) * L - 1 for u in range(B * Hkv)], dtype=torch.int64, device=device)
    ws = tq.alloc_workspace(tq.tq_decode_workspace_size(kctx, vctx, B, Hq, Hkv, L), device)
    out = torch.empty((B, Hq, d), dtype=torch.float32, device=device)
    torch.cuda.synchronize()
    return dict(kctx=kctx, vctx=vctx, kc=kc, vc=vc, q=q, new_k=new[0], new_v=new[1], slots=slots, ws=ws, out=out)


def flusher(torch, device):
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    flush_f32 = flush.view(torch.float32)

    def flush_l2():
        # Write a buffer twice the L2 size, then read it back: the write evicts every line
        # of the inputs, the read leaves the L2 holding clean lines of the flush buffer,
        # so the timed step neither hits cached inputs nor pays for the flush's write-backs.
        flush.zero_()
        flush_f32.sum()
    return flush_l2


def timed_graph_steps(torch, stream, fns, steps, warmup, flush_l2):
    """Time `steps` steps, each one replay of a CUDA graph running the callables `fns` in
    order, with the L2 flushed before every step; returns the per-step times (ms).

    The whole step is one graph, so the kernels of the library keep their programmatic
    launch overlap (each may start its prologue while the previous one finishes).  All
    steps and flushes are queued without a host synchronisation, so the host runs ahead
    of the device and no enqueue gap enters a timed region."""
    for _ in range(warmup):
        flush_l2()
        for fn in fns:
            fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for fn in fns:
            fn()
    for _ in range(warmup):
        flush_l2()
        g.replay()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for e0, e1 in ev:
        flush_l2()
        e0.record(stream)
        g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    return [e0.elapsed_time(e1) for e0, e1 in ev]


def timed_graph_loop(torch, stream, fns, steps, warmup):
    """Time `steps` steps issued back to back: one CUDA graph holding `steps` repetitions of
    the callables `fns`, replayed once between two events; returns the mean step time (ms).

    For inputs larger than twice the L2 (no flush between steps): every step reads the
    whole input again after the other steps' reads evicted it, so no step is served from
    the L2, and the library's kernels keep their programmatic launch overlap from one step
    to the next, as in a decode loop."""
    for _ in range(warmup):
        for fn in fns:
            fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(steps):
            for fn in fns:
                fn()
    g.replay()  # the graph's own first replay, untimed
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def l2_bytes(torch, device):
    return int(getattr(torch.cuda.get_device_properties(device), "L2_cache_size", 0) or (129 << 20))


E2E_MODE = ("value: the public API calls and the copies issued one by one from Python every step "
            "(host validation and enqueue inside the timed region); graph_*: the same calls and copies "
            "captured once in a CUDA graph and replayed every step")


E2E_MODE_DECODE = ("value: one public C-ABI call per step with host buffers (tq_decode_step_host), issued from "
                   "Python every step (host validation and enqueue inside the timed region): with page-locked "
                   "buffers at head dimension 128 the step's kernels read the new K/V rows and q from host "
                   "memory and write the output to host memory in place over the chip-to-chip link; at "
                   "d = 256 one copy in to a device staging area and one copy of the output back; "
                   "graph_*: the same call captured once in a CUDA graph and replayed every step")


def timed_e2e(torch, body, steps, warmup, flush_l2):
    """End-to-end step times (ms, host clock) of `body`: the host-to-device copies of the
    step's inputs from pinned memory, the public API calls and the device-to-host read of
    the result.  Returns (graph, direct): each step one replay of a CUDA graph captured
    from `body` (how a serving loop issues a step), and `body` called directly (host
    enqueue of every copy and call inside the timed region).  Each step starts with the
    L2 flushed and the device idle and ends with a host synchronisation."""
    def run(step):
        out = []
        for i in range(warmup + steps):
            flush_l2()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            step()
            torch.cuda.synchronize()
            if i >= warmup:
                out.append((time.perf_counter() - t0) * 1e3)
        return out

    direct = run(body)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        body()
    return run(g.replay), direct


def common_line(metric, args, world, ms_per_step, value, config, dtype):
    return {"metric": metric, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": dtype, "data": "synthetic", "config": config}


def run_decode(args, rank, world, dist):
    import torch

    import compressed_attention_gb300 as tq

    name = args.workload
    local = int(os.environ.get("LOCAL_RANK", 0))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    cfg, spec = decode_workload(args), DECODE[name]
    B, Hq, Hkv, L = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["L"]
    # the committed ncu summary of the workload holds its named shape: its traffic and
    # instruction counts apply only there (not to a --B / --L point of the sweep)
    base = synth.WORKLOADS[name]
    profiled_shape = (B, L) == (base["B"], base["L"])
    w = build_decode(name, cfg, tq, torch, device)
    stream = torch.cuda.current_stream()
    flush_l2 = flusher(torch, device)

    def step():  # SET_ROWS of K and V, q preparation, split-K decode (merge fused where it applies)
        tq.tq_decode_step(w["kctx"], w["vctx"], w["new_k"], w["new_v"], w["q"], w["kc"], w["vc"], w["out"],
                          w["ws"], B, Hq, Hkv, L, row_ids=w["slots"])

    def partial():  # the split-K kernel alone, writing partials (the stage call)
        tq.tq_decode_partial(w["kctx"], w["vctx"], w["kc"], w["vc"], w["ws"], B, Hq, Hkv, L)

    def partial_merge():  # the split-K kernel as the step launches it, merge fused
        tq.tq_decode_partial_merge(w["kctx"], w["vctx"], w["kc"], w["vc"], w["out"], w["ws"], B, Hq, Hkv, L)

    launches_per_step = tq.tq_decode_step_num_launches(w["kctx"], w["vctx"], w["new_k"].dtype,
                                                       w["new_k"].shape[0], B, Hq, Hkv, L)
    l2 = max(l2_bytes(torch, device), L2_NOMINAL)
    b2b = decode_back_to_back(name, cfg, l2)
    if dist:
        dist.barrier()
    with ClockSampler(local) as clocks:
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        # the step, then the decode kernel alone (the roofline), same workload: as the step
        # launches it (merge fused, over the q the step prepared), and the stage kernel that
        # writes partials only.  Each both back to back (when the packed K/V exceed twice
        # the L2) and with the L2 flushed before every launch.
        loop = {}
        if b2b:
            for key, fn in (("step", step), ("merge", partial_merge), ("stage", partial)):
                loop[key] = timed_graph_loop(torch, stream, (fn,), args.steps, args.warmup)
        step_ms = timed_graph_steps(torch, stream, (step,), args.steps, args.warmup, flush_l2)
        merge_ms = timed_graph_steps(torch, stream, (partial_merge,), args.steps, args.warmup, flush_l2)
        part_ms = timed_graph_steps(torch, stream, (partial,), args.steps, args.warmup, flush_l2)
        if dist:
            dist.barrier()
    clk = clocks.summary()
    flushed = {"step": statistics.mean(step_ms), "merge": statistics.mean(merge_ms),
               "stage": statistics.mean(part_ms)}
    timed = loop if b2b else flushed
    total_ms = max_over_ranks(timed["step"] * args.steps, dist, device)
    merge_avg = max_over_ranks(timed["merge"], dist, device)
    part_avg = max_over_ranks(timed["stage"], dist, device)
    flushed = {k: max_over_ranks(v, dist, device) for k, v in flushed.items()}
    merge_launches = tq.tq_decode_num_launches(w["kctx"], w["vctx"], B, Hq, Hkv, L) - 1

    # end to end through the public API with host buffers, every step: the new K rows, the
    # new V rows and q, back to back in one pinned host buffer, and a pinned output buffer
    # (read and written by the step's kernels in place, or copied through the staging
    # area, as the call decides).
    hstage, _ = tq.pack_step_inputs(w["new_k"], w["new_v"], w["q"])
    h2d = hstage.numel()
    hout = torch.empty(w["out"].shape, dtype=torch.float32, pin_memory=True)
    d2h = hout.numel() * 4
    staging = tq.alloc_workspace(tq.tq_decode_step_host_staging_size(
        w["kctx"], w["new_k"].dtype, w["new_k"].shape[0], w["q"].dtype, B, Hq), device)

    def e2e_body():  # one C-ABI call: input copy, the step, output copy
        tq.tq_decode_step_host(w["kctx"], w["vctx"], hstage, w["new_k"].dtype, w["new_k"].shape[0], w["q"].dtype,
                               hout, w["slots"], w["kc"], w["vc"], staging, w["ws"], B, Hq, Hkv, L)

    e2e_ms, e2e_direct_ms = timed_e2e(torch, e2e_body, args.steps, args.warmup, flush_l2)
    status = tq.tq_ctx_device_status(w["kctx"]) or tq.tq_ctx_device_status(w["vctx"])
    if status:
        raise RuntimeError(f"device status {status} after the benchmark")

    kv_bytes = B * Hkv * L * decode_unit_bytes(spec)
    alg_bytes = kv_bytes + w["q"].numel() * w["q"].element_size() + w["out"].numel() * 4
    ms_per_step = total_ms / args.steps
    value = job_rate(alg_bytes, world, ms_per_step) / 1e9
    peak, peak_kind = measured_peak()
    achieved = kv_bytes / (merge_avg * 1e-3) / 1e9
    achieved_stage = kv_bytes / (part_avg * 1e-3) / 1e9
    e2e_graph_ms = max_over_ranks(statistics.mean(e2e_ms), dist, device)
    e2e_direct_ms = max_over_ranks(statistics.mean(e2e_direct_ms), dist, device)
    if rank != 0:
        return
    cpu = fp32_loop = None
    if world == 1:  # the host-core baselines: N=1 only
        leg = OracleDecode(name, cfg)
        cpu = cpu_sample(leg, decode_unit_bytes(spec),
                         f"whole (batch, KV head) units of {L} keys x {Hq // Hkv} q-heads, "
                         "fp64 dequantize-then-softmax")
        fp32_loop = cpu_fp32_loop(leg)
    line = common_line(DECODE_METRIC, args, world, ms_per_step, value, decode_config(name, cfg, l2), "f32")
    merged = "merge fused" if merge_launches == 1 else "then the combine kernel"
    line.update({
        "timing": (("the steps back to back: one CUDA graph of K tq_decode_step calls (each SET_ROWS of the "
                    "new K/V rows and the q preparation in one launch, then the split-K decode with the merge "
                    "fused), replayed once between two events; the split-K decode alone timed the same way "
                    "for the roofline" if b2b else
                    "each step one CUDA graph replay (tq_decode_step) between two events, the L2 flushed "
                    "before every step; the split-K decode alone timed the same way for the roofline")),
        "l2_flushed_ms": {"step": flushed["step"], "kernel": flushed["merge"], "stage_kernel": flushed["stage"],
                          "note": "the same launches one at a time, the L2 flushed before each"},
        "keys_per_s": job_rate(B * Hkv * L, world, ms_per_step),
        "q_head_scores_per_s": job_rate(B * Hq * L, world, ms_per_step),
        "hbm_frac_of_measured_step": value / peak,
        "algorithmic_bytes_per_step": alg_bytes,
        "operands": "packed K/V decoded in registers to fp16 operands; fp16 hi+lo q and p; fp32 accumulate",
        "roofline": {"bound": "hbm", "kernel": f"{spec['kernel']} (split-K decode, {merged}, as in the step)",
                     "achieved": achieved, "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": achieved / peak,
                     "traffic": profiled_traffic("decode_partial_" + name, spec["source"]) if profiled_shape else None,
                     "algorithmic_bytes_per_launch": kv_bytes, "avg_launch_ms": merge_avg,
                     "launches": merge_launches},
        # (the profiled launch is the split-K kernel alone: where the step follows it with a
        # separate combine, its stage-form time)
        "roofline_issue": issue_roofline("decode_partial_" + name, spec["source"], spec["kernel"],
                                         merge_avg if merge_launches == 1 else part_avg, clk,
                                         torch.cuda.get_device_properties(device).multi_processor_count)
                          if profiled_shape else None,
        "roofline_stage_kernel": {"kernel": f"{spec['kernel']} (stage call: partials only, no merge)",
                                  "achieved": achieved_stage, "frac": achieved_stage / peak,
                                  "avg_launch_ms": part_avg},
        "cpu_baseline": cpu,
        "cpu_fp32_loop": fp32_loop,
        "e2e": {"value": job_rate(alg_bytes, world, e2e_direct_ms) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_direct_ms,
                "mode": E2E_MODE_DECODE, "graph_value": job_rate(alg_bytes, world, e2e_graph_ms) / 1e9,
                "graph_ms_per_step": e2e_graph_ms},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    })
    print(json.dumps(line), flush=True)


def run_prefill(args, rank, world, dist):
    import torch

    import compressed_attention_gb300 as tq

    local = int(os.environ.get("LOCAL_RANK", 0))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    cfg, spec = synth.WORKLOADS["prefill_chunk"], PREFILL["prefill_chunk"]
    B, Hq, Hkv, L, T = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["L"], cfg["T"]
    kctx = tq.Ctx(spec["fmt"], spec["rotation"], spec["k_seed"])
    vctx = tq.Ctx(spec["fmt"], spec["rotation"], spec["v_seed"])
    kc = tq.alloc_cache(spec["fmt"], B * Hkv * L, device)
    vc = tq.alloc_cache(spec["fmt"], B * Hkv * L, device)
    chunk = {}
    for tensor, ctx, cache in (("K", kctx, kc), ("V", vctx, vc)):
        rows = []
        for b in range(B):
            for h in range(Hkv):
                x32, bits = synth.kv_unit(cfg, tensor, b, h)
                src = to_device_rows(torch, x32, bits, device)
                u = b * Hkv + h
                tq.tq_quantize_set_rows(ctx, src, cache,
                                        row_ids=torch.arange(u * L, (u + 1) * L, dtype=torch.int64, device=device))
                rows.append(src[L - T:])
        chunk[tensor] = torch.cat(rows).contiguous()  # the chunk's own rows, rewritten every step
    slots = torch.cat([torch.arange(u * L + L - T, (u + 1) * L, dtype=torch.int64, device=device)
                       for u in range(B * Hkv)])
    q32, qbits = synth.prefill_queries(cfg)
    q = to_device_rows(torch, q32.reshape(-1, 128), qbits.reshape(-1, 128) if qbits is not None else None,
                       device).reshape(B, T, Hq, 128)
    q_start = torch.full((B,), L - T, dtype=torch.int32, device=device)
    ws = tq.alloc_workspace(tq.tq_prefill_workspace_size(kctx, vctx, B, T, Hq, Hkv, L), device)
    out = torch.empty((B, T, Hq, 128), dtype=torch.float32, device=device)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    flush_l2 = flusher(torch, device)

    def write_and_prepare():
        tq.tq_quantize_set_rows(kctx, chunk["K"], kc, row_ids=slots)
        tq.tq_quantize_set_rows(vctx, chunk["V"], vc, row_ids=slots)
        tq.tq_prefill_prepare_q(kctx, vctx, q, ws, B, T, Hq, Hkv, L)

    def partial():
        tq.tq_prefill_partial(kctx, vctx, kc, vc, q_start, ws, B, T, Hq, Hkv, L)

    def combine():
        tq.tq_prefill_combine(kctx, vctx, out, ws, B, T, Hq, Hkv, L)

    if dist:
        dist.barrier()
    with ClockSampler(local) as clocks:
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        step_ms = timed_graph_steps(torch, stream, (write_and_prepare, partial, combine), args.steps,
                                    args.warmup, flush_l2)
        part_ms = timed_graph_steps(torch, stream, (partial,), args.steps, args.warmup, flush_l2)
        if dist:
            dist.barrier()
    clk = clocks.summary()
    total_ms = max_over_ranks(sum(step_ms), dist, device)
    part_avg = max_over_ranks(statistics.mean(part_ms), dist, device)

    # end to end through the public API: q and the chunk's K/V rows in from pinned host
    # memory, SET_ROWS, tq_prefill_attention, the output back
    host = {"q": q, "K": chunk["K"], "V": chunk["V"]}
    pinned = {k: torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t.cpu()) for k, t in host.items()}
    hout = torch.empty(out.shape, dtype=torch.float32, pin_memory=True)
    h2d = sum(t.numel() * t.element_size() for t in pinned.values())
    d2h = hout.numel() * 4
    def e2e_body():
        for k, t in pinned.items():
            host[k].copy_(t, non_blocking=True)
        tq.tq_quantize_set_rows(kctx, chunk["K"], kc, row_ids=slots)
        tq.tq_quantize_set_rows(vctx, chunk["V"], vc, row_ids=slots)
        tq.tq_prefill_attention(kctx, vctx, q, kc, vc, q_start, out, ws, B, T, Hq, Hkv, L)
        hout.copy_(out, non_blocking=True)

    e2e_ms, e2e_direct_ms = timed_e2e(torch, e2e_body, args.steps, args.warmup, flush_l2)
    if tq.tq_ctx_device_status(kctx) or tq.tq_ctx_device_status(vctx):
        raise RuntimeError("device status set after the benchmark")

    flops = prefill_flops(cfg)
    ms_per_step = total_ms / args.steps
    value = job_rate(flops, world, ms_per_step) / 1e12
    peak, peak_kind = measured_tensor_peak()
    achieved = flops / (part_avg * 1e-3) / 1e12
    e2e_step_ms = max_over_ranks(statistics.mean(e2e_ms), dist, device)
    e2e_direct_step_ms = max_over_ranks(statistics.mean(e2e_direct_ms), dist, device)
    if rank != 0:
        return
    cpu = None
    if world == 1:
        leg = OraclePrefill()
        t0, n, work = time.perf_counter(), 0, 0
        while n < 64 and (time.perf_counter() - t0 < 10.0 or n == 0):
            work += leg.unit(n)
            n += 1
        el = time.perf_counter() - t0
        cpu = {"value": work / el / 1e12, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
               "sample": (f"{n} x the last {leg.n} chunk queries x {leg.q.shape[2]} q-heads of one KV head "
                          f"over {L} keys, fp64 dequantize-then-softmax, {el:.1f} s, one host core "
                          "(BLAS single-threaded)"),
               "host_cores": os.cpu_count()}
    line = common_line(PREFILL_METRIC, args, world, ms_per_step, value, prefill_config(), "f16")
    line["unit"] = "TFLOP/s"
    line.update({
        "timing": ("each step one CUDA graph (SET_ROWS of the chunk's K and V rows, q preparation, "
                   "the tensor-core prefill, the combine), steps queued back to back; the prefill "
                   "kernel timed alone the same way for the roofline"),
        "tokens_per_s": job_rate(B * T, world, ms_per_step),
        "flops_per_step": flops,
        "operands": ("fp16 hi+lo q and p against fp16 centroid tiles decoded from the packed cache; "
                     "fp32 accumulate in tensor memory; tensor work executed = 2x the algorithmic FLOPs"),
        "roofline": {"bound": "tensor", "kernel": spec["kernel"], "achieved": achieved, "peak": peak,
                     "peak_kind": peak_kind, "unit": "TFLOP/s", "frac": achieved / peak,
                     "traffic": profiled_traffic("prefill_partial_prefill_chunk", spec["source"]),
                     "algorithmic_flops_per_launch": flops, "avg_launch_ms": part_avg},
        "cpu_baseline": cpu,
        "e2e": {"value": job_rate(flops, world, e2e_direct_step_ms) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_direct_step_ms,
                "mode": E2E_MODE, "graph_value": job_rate(flops, world, e2e_step_ms) / 1e12,
                "graph_ms_per_step": e2e_step_ms},
        "gpu_launches": 5 * args.steps,
        "clocks": clk,
    })
    print(json.dumps(line), flush=True)


def run_write(args, rank, world, dist):
    import torch

    import compressed_attention_gb300 as tq

    local = int(os.environ.get("LOCAL_RANK", 0))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    cfg = synth.WORKLOADS["write_chunk"]
    fmt, rot = args.write_format, args.write_rotation
    kctx, vctx = tq.Ctx(fmt, rot, cfg["seed"]), tq.Ctx(fmt, rot, cfg["seed"] + 100)
    x = {}
    for tensor in ("K", "V"):
        x32, bits = synth.write_rows(cfg, tensor)
        x[tensor] = to_device_rows(torch, x32, bits, device)
    n = x["K"].shape[0]
    caches = {"K": tq.alloc_cache(fmt, n, device), "V": tq.alloc_cache(fmt, n, device)}
    stream = torch.cuda.current_stream()
    flush_l2 = flusher(torch, device)
    fns = (lambda: tq.tq_quantize_set_rows(kctx, x["K"], caches["K"]),
           lambda: tq.tq_quantize_set_rows(vctx, x["V"], caches["V"]))
    if dist:
        dist.barrier()
    with ClockSampler(local) as clocks:
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        step_ms = timed_graph_steps(torch, stream, fns, args.steps, args.warmup, flush_l2)
        launch_ms = timed_graph_steps(torch, stream, fns[:1], args.steps, args.warmup, flush_l2)
        if dist:
            dist.barrier()
    clk = clocks.summary()
    total_ms = max_over_ranks(sum(step_ms), dist, device)
    launch_avg = max_over_ranks(statistics.mean(launch_ms), dist, device)

    # end to end through the public API: the bf16 rows copied in from pinned host memory,
    # quantized, and the packed caches read back, every step.
    hx = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True).copy_(v.cpu()) for k, v in x.items()}
    hc = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in caches.items()}
    h2d = sum(t.numel() * t.element_size() for t in hx.values())
    d2h = sum(t.numel() * t.element_size() for t in hc.values())
    def e2e_body():
        for k in ("K", "V"):
            x[k].copy_(hx[k], non_blocking=True)
        tq.tq_quantize_set_rows(kctx, x["K"], caches["K"])
        tq.tq_quantize_set_rows(vctx, x["V"], caches["V"])
        for k in ("K", "V"):
            hc[k].copy_(caches[k], non_blocking=True)

    e2e_ms, e2e_direct_ms = timed_e2e(torch, e2e_body, args.steps, args.warmup, flush_l2)
    if tq.tq_ctx_device_status(kctx) or tq.tq_ctx_device_status(vctx):
        raise RuntimeError("device status set after the benchmark")

    row_bytes = ROW_BYTES[fmt]
    launch_bytes = n * (256 + row_bytes)
    alg_bytes = 2 * launch_bytes
    ms_per_step = total_ms / args.steps
    value = job_rate(alg_bytes, world, ms_per_step) / 1e9
    peak, peak_kind = measured_peak()
    e2e_step_ms = max_over_ranks(statistics.mean(e2e_ms), dist, device)
    e2e_direct_step_ms = max_over_ranks(statistics.mean(e2e_direct_ms), dist, device)
    if rank != 0:
        return
    cpu = None
    if world == 1:
        leg = OracleWrite(fmt, rot)
        cpu = cpu_sample(leg, 256 + row_bytes, f"blocks of {len(leg.x32)} bf16 rows encoded by the oracle")
    kernel, source = WRITE_KERNEL[rot]
    line = common_line(WRITE_METRIC, args, world, ms_per_step, value, write_config(args), "f32")
    line.update({
        "timing": ("each step one CUDA graph (SET_ROWS of the K rows, then of the V rows), steps queued back "
                   "to back; the first SET_ROWS launch timed alone the same way for the roofline"),
        "rows_per_s": job_rate(2 * n, world, ms_per_step),
        "algorithmic_bytes_per_step": alg_bytes,
        "roofline": {"bound": "hbm", "kernel": kernel, "achieved": launch_bytes / (launch_avg * 1e-3) / 1e9,
                     "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": launch_bytes / (launch_avg * 1e-3) / 1e9 / peak,
                     "traffic": profiled_traffic(f"write_{fmt}_{rot}_write_chunk", source),
                     "algorithmic_bytes_per_launch": launch_bytes, "avg_launch_ms": launch_avg},
        "roofline_issue": issue_roofline(f"write_{fmt}_{rot}_write_chunk", source, kernel, launch_avg, clk,
                                         torch.cuda.get_device_properties(device).multi_processor_count),
        "cpu_baseline": cpu,
        "e2e": {"value": job_rate(alg_bytes, world, e2e_direct_step_ms) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_direct_step_ms,
                "mode": E2E_MODE, "graph_value": job_rate(alg_bytes, world, e2e_step_ms) / 1e9,
                "graph_ms_per_step": e2e_step_ms},
        "gpu_launches": 2 * args.steps,
        "clocks": clk,
    })
    print(json.dumps(line), flush=True)


def relaunch_under_torchrun(n):
    """Run this command again as n ranks under torchrun (one node, 127.0.0.1) and return
    its exit status; rank 0 prints the JSON line."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__), *sys.argv[1:]]
    return subprocess.run(cmd).returncode


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["tq", "reference"], default="tq")
    ap.add_argument("--workload", choices=sorted(DECODE) + ["prefill_chunk", "write_chunk"], default="gqa_lognormal")
    ap.add_argument("--B", type=int, default=None, help="batch of a decode workload (default: the workload's)")
    ap.add_argument("--L", type=int, default=None, help="context of a decode workload (default: the workload's)")
    ap.add_argument("--write-format", choices=["turbo4", "turbo3"], default="turbo4")
    ap.add_argument("--write-rotation", choices=["dense", "wht"], default="dense")
    args = ap.parse_args()
    if args.steps < 1 or args.warmup < 0 or args.gpus < 1:
        ap.error("--steps must be >= 1, --warmup >= 0 and --gpus >= 1")
    if (args.B or args.L) and args.workload not in DECODE:
        ap.error("--B and --L apply to the decode workloads")
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        sys.exit(relaunch_under_torchrun(args.gpus))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world != args.gpus:
        ap.error(f"--gpus {args.gpus} but WORLD_SIZE is {world}")
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    dist = None
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group("nccl")
    try:
        if args.workload == "write_chunk":
            run_write(args, rank, world, dist)
        elif args.workload == "prefill_chunk":
            run_prefill(args, rank, world, dist)
        else:
            run_decode(args, rank, world, dist)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
