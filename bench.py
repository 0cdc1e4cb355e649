"""Benchmark of the ShadowKV decode step on GB300.

Metric: decode tokens/s per layer (b tokens per decode step) on the batch-8,
128K-context Llama-3-8B-style layer, plus the achieved HBM bandwidth of the
dominant kernel against the measured GB300 peak.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config NAME] [--batch B] [--no-cpu-baseline]

One "step" is one decode step through the C ABI (Algorithm 2: landmark
scores, top-k, set-difference value fetch from pinned host memory, key
rebuild with RoPE, attention), for every sequence of the batch, with all
inputs resident in HBM.  Prefill (Algorithm 1) runs once before timing and
is reported separately.  Under torchrun each rank runs its own full batch on
its own GPU (weak scaling, no collective on the data path); rank 0 prints
one JSON line.  `--impl reference` times the CPU oracle instead.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sparse_rank_kv_gb300 import binding, synth  # noqa: E402
from sparse_rank_kv_gb300.synth import CONFIGS  # noqa: E402

METRIC = "ShadowKV decode tokens/s per layer at 128K; achieved HBM GB/s vs GB300 peak"
UNIT = "tokens/s/layer"
DEFAULT_CONFIG = "llama_b8_s128k"
FALLBACK_HBM_GBS = 6800.0


# ----------------------------------------------------------------- helpers
def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def hbm_bytes_per_step(cfg, E, n_loc, alpha=0.0, records=False):
    """Algorithmic HBM bytes of one decode step.

    Row-major contexts follow the pages' step: landmarks, A rows of every
    selected chunk, B, outlier K/V, cached V of the selected chunks,
    local-window K/V.  With K/V records (bf16, d = 128) a cache slot keeps its
    chunk's rebuilt keys, so a step with hit rate `alpha` reads A rows of the
    missed chunks only, reads the keys and values of every selected chunk,
    and writes the missed chunks' rebuilt keys and fetched values."""
    sel = cfg.k * cfg.c                       # selected tokens per (batch, KV head)
    common = cfg.n * cfg.d + cfg.r * cfg.d + 2 * cfg.o * cfg.c * cfg.d + 2 * n_loc * cfg.d
    if records:
        miss = (1.0 - alpha) * sel
        per_pair = common + miss * cfg.r + 2 * sel * cfg.d + 2 * miss * cfg.d
    else:
        per_pair = common + sel * cfg.r + sel * cfg.d
    return E * cfg.b * cfg.h_kv * per_pair


class ClockSampler:
    """Samples SM clock and throttle reasons through NVML (read-only queries)
    in a background thread; falls back to nvidia-smi."""
    REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown",
               0x4: "sw_power_cap", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, index: int, period_s: float = 0.001):
        self.index, self.period = index, period_s
        self.samples, self.reasons, self.max_mhz = [], set(), None
        self._stop = threading.Event()
        self._nvml = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() == 0:
                h = ctypes.c_void_p()
                if nv.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(h)) == 0:
                    self._nvml, self._h = nv, h
                    mx = ctypes.c_uint()
                    if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                        self.max_mhz = mx.value
        except OSError:
            self._nvml = None

    def _poll(self):
        nv, h = self._nvml, getattr(self, "_h", None)
        clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0:
                self.samples.append(clk.value)
            if nv.nvmlDeviceGetCurrentClocksEventReasons(h, ctypes.byref(rs)) == 0:
                for bit, name in self.REASONS.items():
                    if rs.value & bit:
                        self.reasons.add(name)
            time.sleep(self.period)

    def __enter__(self):
        if self._nvml is not None:
            self._t = threading.Thread(target=self._poll, daemon=True)
            self._t.start()
        else:
            q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
                 "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                 "clocks_event_reasons.sw_power_cap")
            self._p = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={q}",
                                        "--format=csv,noheader,nounits", "-lms", "100"],
                                       stdout=subprocess.PIPE, text=True)
        return self

    def __exit__(self, *a):
        if self._nvml is not None:
            self._stop.set()
            self._t.join()
            return
        self._p.terminate()
        out = self._p.communicate()[0]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 6 or not f[0].isdigit():
                continue
            self.samples.append(int(f[0]))
            self.max_mhz = int(f[1])
            for nm, v in zip(names, f[2:]):
                if v.lower() == "active":
                    self.reasons.add(nm)

    def summary(self):
        med = statistics.median(self.samples) if self.samples else None
        return {"sm_mhz": med, "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons),
                "samples": len(self.samples)}


def traffic_from_profile(name: str, src_file: str):
    """Per-launch DRAM bytes of a kernel from its committed ncu summary, if the
    kernel's source has not changed since (sha256 recorded in the summary)."""
    path = os.path.join(ROOT, "profiles", name)
    try:
        text = open(path).read()
    except OSError:
        return None
    rec = {}
    for line in text.splitlines():
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            rec[k.strip()] = v.strip().strip("`")
    src = open(os.path.join(ROOT, "sparse_rank_kv_gb300", "csrc", src_file), "rb").read()
    if rec.get("source_sha256") != hashlib.sha256(src).hexdigest()[:16]:
        return None
    try:
        return float(rec["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def max_over_ranks(x: float, device) -> float:
    """The largest value of x over the ranks of the default process group
    (x itself without one): the job's step time is its slowest rank's."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world: int, b: int, ms_per_step: float) -> float:
    """Whole-job decode throughput: every rank decodes its own batch of b
    sequences, one token each per step, in the job's (slowest) step time."""
    return world * b / (ms_per_step * 1e-3)


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ----------------------------------------------------------- CPU oracle leg
def oracle_decode_timing(cfg, steps: int, warmup: int, seed: int = 0):
    """Times the CPU oracle's decode step on one sequence of cfg (all KV heads)."""
    from oracle import shadowkv_oracle as O
    one = cfg.with_(b=1, steps=warmup + steps, seed=cfg.seed + seed)
    st = synth.make_state(one, device="cpu")
    f = lambda key: st[key].to(torch.float32).numpy()
    state = O.OracleState(c=one.c, theta=one.theta, A=f("A"), B=f("B"), L=f("L"),
                          outlier_ids=st["outlier_ids"].numpy().astype(np.int64),
                          K_out=f("K_out"), V_out=f("V_out"), K_loc=f("K_loc"),
                          V_loc=f("V_loc"), V_cpu=f("v"))
    dec = O.OracleDecoder(state, h_q=one.h_q, k=one.k)
    times = []
    for t in range(warmup + steps):
        q, kn, vn = (st[x][t].to(torch.float32).numpy() for x in ("q", "k_new", "v_new"))
        t0 = time.perf_counter()
        dec.step(q, kn, vn)
        if t >= warmup:
            times.append(time.perf_counter() - t0)
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return sum(times), len(times), cores


# ------------------------------------------------------------------ our arm
def run_ours(args, cfg):
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    K, W = args.steps, args.warmup
    # decode steps appended per pass; every pass starts from the same rewound state
    max_new = W + K
    run_cfg = cfg.with_(steps=max_new)
    E = 2 if cfg.dtype == "bf16" else 4
    dt = synth.torch_dtype(cfg.dtype)

    inp = synth.make_inputs(run_cfg, device=dev)
    p = binding.make_params(run_cfg)
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    ctx = binding.prefill(p, inp["k_pre"], inp["v"], stream)
    torch.cuda.synchronize()
    prefill_ms = (time.perf_counter() - t0) * 1e3
    del inp["k_pre"], inp["v"]
    torch.cuda.empty_cache()
    q, kn, vn = inp["q"], inp["k_new"], inp["v_new"]
    out = torch.empty(cfg.b, cfg.h_q, cfg.d, dtype=dt, device=dev)

    def barrier():
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()

    def decode_pass(timing: bool):
        ctx.rewind(stream)
        ctx.set_option(binding.OPT_TIMING, 1 if timing else 0)
        for t in range(W):
            ctx.decode_step(q[t], kn[t], vn[t], out, stream)
        ctx.reset_timers()
        st0 = ctx.stats()
        barrier()
        torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for t in range(W, W + K):
            ctx.decode_step(q[t], kn[t], vn[t], out, stream)
        ev1.record(stream)
        torch.cuda.synchronize()
        barrier()
        st1 = ctx.stats()
        ms = ev0.elapsed_time(ev1)
        kt = ctx.kernel_times() if timing else None
        ctx.set_option(binding.OPT_TIMING, 0)
        return ms, st0, st1, kt

    # 1) the headline: K decode steps, inputs resident, no per-kernel events
    with ClockSampler(local) as clk:
        ms, st0, st1, _ = decode_pass(False)
    ms = max_over_ranks(ms, dev)
    ms_step = ms / K
    hits = st1.hits - st0.hits
    misses = st1.misses - st0.misses
    alpha = hits / max(1, hits + misses)
    launches = st1.launches - st0.launches

    # 2) the same K steps with CUDA events around every kernel on its stream
    ms_t, _, _, kt = decode_pass(True)

    # 3) end to end through the C ABI from pinned host buffers
    ctx.rewind(stream)
    qh = q.cpu().pin_memory()
    knh, vnh = kn.cpu().pin_memory(), vn.cpu().pin_memory()
    outh = torch.empty(out.shape, dtype=dt).pin_memory()
    qd, knd, vnd = torch.empty_like(q[0]), torch.empty_like(kn[0]), torch.empty_like(vn[0])
    for t in range(W):
        ctx.decode_step(q[t], kn[t], vn[t], out, stream)
    torch.cuda.synchronize()
    barrier()
    t0 = time.perf_counter()
    for t in range(W, W + K):
        qd.copy_(qh[t], non_blocking=True)
        knd.copy_(knh[t], non_blocking=True)
        vnd.copy_(vnh[t], non_blocking=True)
        ctx.decode_step(qd, knd, vnd, out, stream)
        outh.copy_(out, non_blocking=True)
        stream.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, dev)
    barrier()
    h2d = (qd.numel() + knd.numel() + vnd.numel()) * E
    d2h = out.numel() * E

    # host link: bulk pinned -> device copy
    nbytes = 256 << 20
    hbuf = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    dbuf = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    for _ in range(2):
        dbuf.copy_(hbuf, non_blocking=True)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(5):
        dbuf.copy_(hbuf, non_blocking=True)
    e1.record()
    torch.cuda.synchronize()
    bulk_gbs = 5 * nbytes / (e0.elapsed_time(e1) * 1e-3) / 1e9

    ctx.check()
    result = None
    if rank == 0:
        hbm_gbs, peak_src = peaks()
        n_loc_avg = cfg.w + W + (K + 1) / 2.0
        records = cfg.dtype == "bf16" and cfg.d == 128 and cfg.c % 8 == 0 and 128 % cfg.c == 0
        hbm = hbm_bytes_per_step(cfg, E, n_loc_avg, alpha, records)
        link = misses / K * cfg.c * cfg.d * E
        fetch_ms, fetch_n = kt["fetch"]
        fetch_in = "fetch launch"
        if fetch_n == 0:
            # K/V records: the fetch runs as CTAs of the rebuild launch, whose
            # time (bound by the host link) is an upper bound on the fetch's
            fetch_ms, fetch_n = kt["rebuild"]
            fetch_in = "rebuild launch (fetch CTAs inside it)"
        fetch_gbs = link * fetch_n / max(1, K) / (fetch_ms / max(1, fetch_n) * 1e-3) / 1e9 if fetch_ms > 0 else 0.0
        link_gbs = max(bulk_gbs, fetch_gbs)
        t_roof = hbm / (hbm_gbs * 1e9) + link / (link_gbs * 1e9)
        score_ms, score_n = kt["score"]
        # landmarks read + logits P and per-tile softmax partials written
        score_bytes = (E * cfg.b * cfg.h_kv * cfg.n * cfg.d + 4 * cfg.b * cfg.h_q * cfg.n
                       + 8 * 4 * cfg.b * cfg.h_q * ((cfg.n + 127) // 128))
        achieved = score_bytes / (score_ms / score_n * 1e-3) / 1e9
        traffic = traffic_from_profile("score_kernel_b8_s128k.md", "score_tc.cu")
        per_kernel = {k_: {"ms_per_step": v[0] / K, "launches": v[1]} for k_, v in kt.items() if v[1]}
        value = job_tokens_per_s(ws, cfg.b, ms_step)
        result = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": K,
            "warmup": W, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": cfg.dtype, "data": "synthetic",
            "config": {"workload": f"{cfg.name}: ShadowKV decode, b={cfg.b} h_q={cfg.h_q} "
                                   f"h_kv={cfg.h_kv} d={cfg.d} s={cfg.s} c={cfg.c} r={cfg.r} "
                                   f"k={cfg.k} o={cfg.o} w={cfg.w}",
                       "global_batch": ws * cfg.b, "seq_len": cfg.s,
                       "parallelism": f"batch replicas x{ws}" if ws > 1 else "single GPU",
                       "l2": "inputs larger than L2 (landmarks %.0f MB, A %.0f MB per step)" % (
                           E * cfg.b * cfg.h_kv * cfg.n * cfg.d / 1e6, E * cfg.b * cfg.s * cfg.r / 1e6)},
            "roofline": {"bound": "hbm", "kernel": "score", "achieved": achieved,
                         "peak": hbm_gbs, "unit": "GB/s", "frac": achieved / hbm_gbs,
                         "peak_source": peak_src, "traffic": traffic,
                         "algorithmic_bytes_per_launch": score_bytes},
            "step_roofline": {"hbm_bytes": hbm, "link_bytes": link, "hbm_gbs": hbm_gbs,
                              "link_gbs": link_gbs, "bulk_h2d_gbs": bulk_gbs,
                              "fetch_gbs": fetch_gbs, "fetch_timed_in": fetch_in, "t_roof_us": t_roof * 1e6,
                              "t_step_us": ms_step * 1e3, "frac": t_roof / (ms_step * 1e-3)},
            "per_kernel_ms": per_kernel, "timed_with_kernel_events_ms_per_step": ms_t / K,
            "alpha_hit_rate": alpha,
            "equivalent_bandwidth_TBps": 2 * cfg.s * cfg.d * E * cfg.b * cfg.h_kv / (ms_step * 1e-3) / 1e12,
            "prefill_ms": prefill_ms,
            "e2e": {"value": job_tokens_per_s(ws, cfg.b, e2e_s * 1e3 / K), "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": launches,
            "clocks": clk.summary(),
        }
    ctx.close()
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return result


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=32)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default=DEFAULT_CONFIG, choices=sorted(CONFIGS))
    ap.add_argument("--batch", type=int, default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    cfg = CONFIGS[args.config]
    if args.batch:
        cfg = cfg.with_(b=args.batch)
    ws, rank, _ = dist_env()

    if args.impl == "reference":
        if rank != 0:
            return
        tot, n, cores = oracle_decode_timing(cfg, args.steps, args.warmup)
        val = n / tot
        sample = f"1 of {cfg.b} sequences (all {cfg.h_kv} KV heads), {n} decode steps"
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / n,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": f"{cfg.name} (CPU oracle)"},
            "cpu_baseline": {"value": val, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }))
        return

    res = run_ours(args, cfg)
    if res is None:
        return
    if ws == 1 and not args.no_cpu_baseline:
        tot, n, cores = oracle_decode_timing(cfg, 3, 1)
        res["cpu_baseline"] = {"value": n / tot, "unit": UNIT, "cores": cores, "kind": "oracle",
                               "sample": f"1 of {cfg.b} sequences (all {cfg.h_kv} KV heads), "
                                         f"{n} decode steps of the same shape"}
    print(json.dumps(res))


if __name__ == "__main__":
    main()
