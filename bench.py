"""Benchmark of the ShadowKV decode step on GB300.

Metric: decode tokens/s per layer (b tokens per decode step) on the batch-8,
128K-context Llama-3-8B-style layer, plus the achieved HBM bandwidth of the
dominant kernel against the measured GB300 peak.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config NAME] [--batch B] [--sweep B1,B2,...] [--chunk C]
                    [--budget PCT] [--q-sigma S] [--layers L] [--no-cpu-baseline]

One "step" is one decode step through the C ABI (Algorithm 2: landmark
scores, top-k, set-difference value fetch from pinned host memory, key
rebuild with RoPE, attention), for every sequence of the batch, with all
inputs resident in HBM.  Prefill (Algorithm 1) runs once before timing and
is reported separately (wall time, and its kernels' CUDA-event times).
Under torchrun each rank runs its own full batch on its own GPU (weak
scaling, no collective on the data path); rank 0 prints one JSON line.

  --sweep 8,16,24,48   one JSON line per batch size (the 60K batch sweep)
  --chunk/--budget     chunk size c and sparse budget k*c/s in percent
  --q-sigma S          query drift per step (larger: fewer cache hits)
  --layers L           L layers, each its own context and cache, decoded back
                       to back on one stream; reported per layer
With the 256K workload (prefill plus decode) the line also carries the SVD's
reconstruction error over the Eckart-Young optimum and the subspace
similarity <H1, H2> / r of the two sequences' bases.
`--impl reference` times the CPU oracle instead.
"""
from __future__ import annotations

import argparse
import ctypes
import gc
import hashlib
import json
import os
import statistics
import subprocess
import sys
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
_WARM = False
PREFILL_KERNELS = ("chunkstats", "outliers", "gather", "svd_gram", "svd_iter", "orth", "misc", "svd_a")


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
    """HBM bytes of one decode step.

    records=False: the algorithmic bytes of the pages' step -- landmarks, A
    rows of every selected chunk, B, outlier K/V, cached V of the selected
    chunks, local-window K/V.  records=True: the traffic of the K/V-record
    layout, where a cache slot keeps its chunk's rebuilt keys, so a step with
    hit rate `alpha` reads A rows of the missed chunks only, reads the keys
    and values of every selected chunk, and writes the missed chunks'
    rebuilt keys and fetched values."""
    sel = cfg.k * cfg.c                       # selected tokens per (batch, KV head)
    common = cfg.n * cfg.d + cfg.r * cfg.d + 2 * cfg.o * cfg.c * cfg.d + 2 * n_loc * cfg.d
    if records:
        miss = (1.0 - alpha) * sel
        per_pair = common + miss * cfg.r + 2 * sel * cfg.d + 2 * miss * cfg.d
    else:
        per_pair = common + sel * cfg.r + sel * cfg.d
    return E * cfg.b * cfg.h_kv * per_pair


def score_bytes(cfg, E):
    """(algorithmic, written) bytes of one landmark-score launch: the landmarks
    read, and the logits plus per-tile softmax partials the kernel writes for
    the selection (implementation overhead, not in the pages' byte count)."""
    land = E * cfg.b * cfg.h_kv * cfg.n * cfg.d
    extra = 4 * cfg.b * cfg.h_q * cfg.n + 8 * 4 * cfg.b * cfg.h_q * ((cfg.n + 127) // 128)
    return land, extra


def apply_overrides(cfg, chunk=None, budget=None, q_sigma=None, batch=None):
    """The workload with its chunk size, sparse budget (percent of s),
    query drift or batch replaced; k = round(budget * s / c) chunks."""
    pct = 100.0 * cfg.k * cfg.c / cfg.s
    if chunk:
        cfg = cfg.with_(c=chunk)
    if chunk or budget:
        pct = budget if budget else pct
        cfg = cfg.with_(k=max(1, int(round(pct / 100.0 * cfg.s / cfg.c))))
    if q_sigma is not None:
        cfg = cfg.with_(q_sigma=q_sigma)
    if batch:
        cfg = cfg.with_(b=batch)
    return cfg


_SAMPLER = r"""
import ctypes, json, signal, sys, time
idx, period = int(sys.argv[1]), float(sys.argv[2])
REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown",
           0x4: "sw_power_cap", 0x80: "hw_power_brake_slowdown"}
samples, reasons, mx = [], set(), None
stop = []
signal.signal(signal.SIGTERM, lambda *a: stop.append(1))
try:
    nv = ctypes.CDLL("libnvidia-ml.so.1")
    ok = nv.nvmlInit_v2() == 0
except OSError:
    ok = False
if ok:
    h = ctypes.c_void_p()
    ok = nv.nvmlDeviceGetHandleByIndex_v2(idx, ctypes.byref(h)) == 0
if ok:
    m = ctypes.c_uint()
    if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(m)) == 0:
        mx = m.value
    clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
    print("ready", flush=True)
    while not stop:
        if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0:
            samples.append(clk.value)
        if nv.nvmlDeviceGetCurrentClocksEventReasons(h, ctypes.byref(rs)) == 0:
            for bit, name in REASONS.items():
                if rs.value & bit:
                    reasons.add(name)
        time.sleep(period)
else:
    print("ready", flush=True)
    while not stop:
        time.sleep(period)
print(json.dumps({"samples": samples, "reasons": sorted(reasons), "max": mx}), flush=True)
"""


class ClockSampler:
    """Samples the SM clock and throttle reasons through NVML (read-only
    queries) in a separate process, so that the sampling never competes with
    the launching thread for the interpreter lock."""

    def __init__(self, index: int, period_s: float = 0.0005):
        self.index, self.period = index, period_s
        self.samples, self.reasons, self.max_mhz = [], set(), None

    def __enter__(self):
        self._p = subprocess.Popen([sys.executable, "-c", _SAMPLER, str(self.index), str(self.period)],
                                   stdout=subprocess.PIPE, text=True)
        self._p.stdout.readline()          # NVML is up before the timed region starts
        return self

    def __exit__(self, *a):
        self._p.terminate()
        out = self._p.communicate(timeout=30)[0].strip().splitlines()
        try:
            rec = json.loads(out[-1])
        except (IndexError, ValueError):
            return
        self.samples, self.reasons, self.max_mhz = rec["samples"], set(rec["reasons"]), rec["max"]

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


def svd_report(inp, ctx, cfg, dev):
    """Quality of the prefill's rank-r factors, measured with torch in float64
    on the device (a report, not part of the path): for sequence 0,
    |M - A B|^2 and |M - M X^T X|^2 over the Eckart-Young optimum
    sum_{i>r} sigma_i^2 (all from the Gram matrix of M), and the subspace
    similarity <H1, H2> / r = |X_0 X_1^T|_F^2 / r of sequences 0 and 1."""
    b, h, s, d, r = cfg.b, cfg.h_kv, cfg.s, cfg.d, cfg.r
    D = h * d
    X = ctx.export("SVD_BASIS").view(b, r, D).to(dev, torch.float64)
    A = ctx.export("A").view(b, s, r)[0].to(dev, torch.float64)
    B = ctx.export("BT").view(b, h, d, r)[0].to(dev, torch.float64).permute(2, 0, 1).reshape(r, D)
    M = inp["k_pre"][0].to(torch.float64).permute(1, 0, 2).reshape(s, D)
    G = M.T @ M
    tot = float(torch.trace(G))
    lam = torch.linalg.eigvalsh(G)
    opt = float(lam[:-r].sum())
    X0 = X[0]
    Q = X0 @ G @ X0.T
    eb = tot - 2.0 * float(torch.trace(Q)) + float(((X0 @ X0.T) * Q.T).sum())
    es = tot - 2.0 * float(((A.T @ M) * B).sum()) + float(((A.T @ A) * (B @ B.T)).sum())
    rep = {"sequence": 0, "err2_over_opt2_stored": es / opt, "err2_over_opt2_basis": eb / opt,
           "rel_err_stored": (es / tot) ** 0.5, "rel_err_optimal": (opt / tot) ** 0.5}
    m = r - cfg.rank_true
    if m > 0:
        # the same with the r - R directions past the keys' true rank R drawn
        # at random from the noise subspace (expected value)
        noise = lam[:D - cfg.rank_true]
        rep["err2_over_opt2_random_noise_directions"] = float(noise.sum() - m * noise.mean()) / opt
    if b > 1:
        rep["subspace_similarity_seq01"] = float((X[0] @ X[1].T).pow(2).sum()) / r
        rep["subspace_similarity_random_expectation"] = r / D
    del M, G
    return rep


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
def link_bulk_gbs(dev):
    """Best pinned-host -> device copy rate (GB/s) over three copy sizes."""
    best = {}
    for mb in (4, 32, 256):
        nbytes = mb << 20
        hbuf = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
        dbuf = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        for _ in range(2):
            dbuf.copy_(hbuf, non_blocking=True)
        torch.cuda.synchronize()
        reps = max(3, 1024 // mb)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            dbuf.copy_(hbuf, non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        best[f"{mb}MB"] = reps * nbytes / (e0.elapsed_time(e1) * 1e-3) / 1e9
        del hbuf, dbuf
    return best


def run_ours(args, cfg):
    ws, rank, local = dist_env()
    dev = torch.device("cuda", local)
    K, W = args.steps, args.warmup
    L = max(1, args.layers)
    # decode steps appended per pass; every pass starts from the same rewound state
    max_new = W + K
    run_cfg = cfg.with_(steps=max_new)
    E = 2 if cfg.dtype == "bf16" else 4
    dt = synth.torch_dtype(cfg.dtype)
    stream = torch.cuda.current_stream()

    # the first launch of each kernel in a process loads its module: a small
    # prefill of the same kind (same d, G, r, c, dtype) keeps that out of the
    # timed prefill
    global _WARM
    if not _WARM:
        o_w = min(cfg.o, 4096 // cfg.c // 4)
        warm = run_cfg.with_(b=1, s=cfg.w + 4096, o=o_w, k=min(cfg.k, 4096 // cfg.c - o_w))
        wi = synth.make_inputs(warm, device=dev)
        binding.prefill(binding.make_params(warm), wi["k_pre"], wi["v"], stream).close()
        del wi
        _WARM = True

    # ---- prefill: one context (its own cache) per layer
    ctxs, prefill_ms, prefill_kernels, svd = [], [], None, None
    for layer in range(L):
        inp = synth.make_inputs(run_cfg.with_(seed=run_cfg.seed + 1000 * layer), device=dev)
        p = binding.make_params(run_cfg)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        ctx = binding.prefill(p, inp["k_pre"], inp["v"], stream)
        torch.cuda.synchronize()
        prefill_ms.append((time.perf_counter() - t0) * 1e3)
        if args.rebuild_in_attention:
            ctx.set_option(binding.OPT_REBUILD_IN_ATTENTION, 1)
        if layer == 0:
            kt = ctx.kernel_times()
            prefill_kernels = {k_: {"ms": v[0], "launches": v[1]} for k_, v in kt.items()
                               if v[1] and k_ in PREFILL_KERNELS}
            if args.svd_report and rank == 0:
                # kept for the report, which runs after the timed passes: its
                # fp64 products on the device are followed by stalls of some
                # hundreds of microseconds in the next kernels
                svd_keys = inp["k_pre"]
            q, kn, vn = inp["q"], inp["k_new"], inp["v_new"]
        ctx.reset_timers()
        ctxs.append(ctx)
        del inp
        torch.cuda.empty_cache()
    layout = ctxs[0].layout()
    out = torch.empty(cfg.b, cfg.h_q, cfg.d, dtype=dt, device=dev)

    def barrier():
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()

    # every step's C-ABI call with its arguments marshalled in advance, so the
    # timed loops allocate no Python objects (and no collection can run)
    calls = [[ctx.prepared_step(q[t], kn[t], vn[t], out, stream) for ctx in ctxs] for t in range(W + K)]
    host_gap = [0.0]

    def steps(t0, t1, watch=False):
        last = time.perf_counter()
        for t in range(t0, t1):
            for call in calls[t]:
                call()
            if watch:
                now = time.perf_counter()
                if now - last > host_gap[0]:
                    host_gap[0] = now - last
                last = now

    def decode_pass(timing: bool, cache: bool = True):
        for ctx in ctxs:
            ctx.rewind(stream)
            ctx.set_option(binding.OPT_TIMING, 1 if timing else 0)
            ctx.set_option(binding.OPT_CACHE, 1 if cache else 0)
        steps(0, W)
        for ctx in ctxs:
            ctx.reset_timers()
        st0 = [ctx.stats() for ctx in ctxs]
        barrier()
        torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        gc.collect()
        gc.disable()
        ev0.record(stream)
        steps(W, W + K, watch=not timing)
        ev1.record(stream)
        torch.cuda.synchronize()
        gc.enable()
        barrier()
        st1 = [ctx.stats() for ctx in ctxs]
        ms = ev0.elapsed_time(ev1)
        kt = ctxs[0].kernel_times() if timing else None
        for ctx in ctxs:
            ctx.set_option(binding.OPT_TIMING, 0)
            ctx.set_option(binding.OPT_CACHE, 1)
        hits = sum(b_.hits - a_.hits for a_, b_ in zip(st0, st1))
        misses = sum(b_.misses - a_.misses for a_, b_ in zip(st0, st1))
        launches = sum(b_.launches - a_.launches for a_, b_ in zip(st0, st1))
        return ms, hits, misses, launches, kt

    # passes in this order: (a) the cache forced off, so that every selected
    # chunk crosses the host link (it times the fetch's own access pattern at
    # full size; the first pass after a prefill also meets the first GPU
    # accesses to host pages, see the design notes); (b) the same steps with
    # CUDA events around every kernel; (c) the headline: K decode steps (of
    # every layer) after W warm-up steps, inputs resident, no per-kernel
    # events.  Each pass starts from the rewound state.
    _, _, miss_off, _, kt_off = decode_pass(True, cache=False)
    ms_t, _, _, _, kt = decode_pass(True)
    with ClockSampler(local) as clk:
        ms, hits, misses, launches, _ = decode_pass(False)
    ms = max_over_ranks(ms, dev)
    ms_step = ms / K / L                      # per layer
    alpha = hits / max(1, hits + misses)

    # 4) end to end through the C ABI with host buffers: per step and layer,
    #    shadowkv_decode_step_host with the token's q, k_new and v_new in
    #    pinned host memory (q copied to the device inside the call, k_new and
    #    v_new read over the host link) and the output written into pinned
    #    host memory, then a wait for the result
    for ctx in ctxs:
        ctx.rewind(stream)
    nq, nk = q[0].numel(), kn[0].numel()
    per = nq + 2 * nk
    host = torch.empty(W + K, per, dtype=dt).pin_memory()
    host[:, :nq].copy_(q.reshape(W + K, nq))
    host[:, nq:nq + nk].copy_(kn.reshape(W + K, nk))
    host[:, nq + nk:].copy_(vn.reshape(W + K, nk))
    outh = torch.empty(out.shape, dtype=dt).pin_memory()
    hq = [host[t, :nq].view(q[0].shape) for t in range(W + K)]
    hk = [host[t, nq:nq + nk].view(kn[0].shape) for t in range(W + K)]
    hv = [host[t, nq + nk:].view(vn[0].shape) for t in range(W + K)]
    e2e_calls = [[ctx.prepared_step(hq[t], hk[t], hv[t], outh, stream, host=True) for ctx in ctxs]
                 for t in range(W + K)]
    for t in range(W):
        for call in e2e_calls[t]:
            call()
    torch.cuda.synchronize()
    barrier()
    gc.collect()
    gc.disable()
    t0 = time.perf_counter()
    for t in range(W, W + K):
        for call in e2e_calls[t]:
            call()
        stream.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, dev)
    gc.enable()
    barrier()
    h2d = L * per * E
    d2h = L * out.numel() * E

    bulk = link_bulk_gbs(dev)
    for ctx in ctxs:
        ctx.check()
    if args.svd_report and rank == 0:
        svd = svd_report({"k_pre": svd_keys}, ctxs[0], cfg, dev)
        del svd_keys
    result = None
    if rank == 0:
        hbm_gbs, peak_src = peaks()
        n_loc_avg = cfg.w + W + (K + 1) / 2.0
        hbm = hbm_bytes_per_step(cfg, E, n_loc_avg)
        hbm_rec = hbm_bytes_per_step(cfg, E, n_loc_avg, alpha, records=True) if layout["kv_records"] else None
        link = misses / K / L * cfg.c * cfg.d * E
        if layout["fetch_in_attention"]:
            fetch_kid, fetch_in = "attention", "attention launch (fetch warps inside it)"
        elif layout["fetch_in_rebuild"]:
            fetch_kid, fetch_in = "rebuild", "rebuild launch (fetch CTAs inside it)"
        else:
            fetch_kid, fetch_in = "fetch", "fetch launch"

        def rate(kts, nmiss):
            ms_, n_ = kts[fetch_kid]
            byts = nmiss / K / L * cfg.c * cfg.d * E
            return byts / (ms_ / max(1, n_) * 1e-3) / 1e9 if ms_ > 0 else 0.0

        # with the fetch inside the attention's launch, only the cache-off pass
        # (every selected chunk fetched, the launch's time set by the link)
        # measures the host link through it
        fetch_gbs = None if layout["fetch_in_attention"] else rate(kt, misses)
        fetch_off_gbs = rate(kt_off, miss_off)
        link_gbs = max(max(bulk.values()), fetch_off_gbs, fetch_gbs or 0.0)
        t_roof = hbm / (hbm_gbs * 1e9) + link / (link_gbs * 1e9)
        score_ms, score_n = kt["score"]
        land, extra = score_bytes(cfg, E)
        score_s = score_ms / score_n * 1e-3
        achieved = land / score_s / 1e9
        traffic = traffic_from_profile("score_kernel_b8_s128k.md", "score_tc.cu") \
            if (cfg.b, cfg.s, cfg.c) == (8, 131072, 8) else None
        per_kernel = {k_: {"ms_per_step": v[0] / K, "launches": v[1]} for k_, v in kt.items() if v[1]}
        value = job_tokens_per_s(ws, cfg.b, ms_step)
        pct = 100.0 * cfg.k * cfg.c / cfg.s
        step_roof = {"hbm_bytes": hbm, "link_bytes": link, "hbm_gbs": hbm_gbs, "link_gbs": link_gbs,
                     "bulk_h2d_gbs": bulk, "fetch_gbs": fetch_gbs, "fetch_gbs_cache_off": fetch_off_gbs,
                     "fetch_timed_in": fetch_in, "t_roof_us": t_roof * 1e6, "t_step_us": ms_step * 1e3,
                     "frac": t_roof / (ms_step * 1e-3),
                     "bytes": "pages' step (L, A rows of every selected chunk, B, outliers, cached V, local)"}
        if hbm_rec is not None:
            t_rec = hbm_rec / (hbm_gbs * 1e9) + link / (link_gbs * 1e9)
            step_roof.update({"hbm_bytes_records": hbm_rec, "frac_records": t_rec / (ms_step * 1e-3)})
        result = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": K,
            "warmup": W, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": cfg.dtype, "data": "synthetic",
            "config": {"workload": f"{cfg.name}: ShadowKV decode, b={cfg.b} h_q={cfg.h_q} "
                                   f"h_kv={cfg.h_kv} d={cfg.d} s={cfg.s} c={cfg.c} r={cfg.r} "
                                   f"k={cfg.k} ({pct:.2f}% budget) o={cfg.o} w={cfg.w} "
                                   f"q_sigma={cfg.q_sigma}" + (f", {L} layers" if L > 1 else ""),
                       "global_batch": ws * cfg.b, "seq_len": cfg.s,
                       "parallelism": f"batch replicas x{ws}" if ws > 1 else "single GPU",
                       "l2": "inputs larger than L2 (landmarks %.0f MB, A %.0f MB per layer)" % (
                           E * cfg.b * cfg.h_kv * cfg.n * cfg.d / 1e6, E * cfg.b * cfg.s * cfg.r / 1e6)},
            "roofline": {"bound": "hbm", "kernel": "score", "achieved": achieved,
                         "peak": hbm_gbs, "unit": "GB/s", "frac": achieved / hbm_gbs,
                         "peak_source": peak_src, "traffic": traffic,
                         "algorithmic_bytes_per_launch": land,
                         "extra_written_bytes_per_launch": extra,
                         "frac_with_written": (land + extra) / score_s / 1e9 / hbm_gbs},
            "step_roofline": step_roof,
            "per_kernel_ms": per_kernel, "timed_with_kernel_events_ms_per_step": ms_t / K / L,
            "alpha_hit_rate": alpha, "layout": layout,
            "equivalent_bandwidth_TBps": 2 * cfg.s * cfg.d * E * cfg.b * cfg.h_kv / (ms_step * 1e-3) / 1e12,
            "prefill_ms": prefill_ms[0], "prefill_kernels": prefill_kernels,
            "prefill_kernels_ms": sum(v["ms"] for v in prefill_kernels.values()),
            "e2e": {"value": job_tokens_per_s(ws, cfg.b, e2e_s * 1e3 / K / L), "unit": UNIT,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "path": "shadowkv_decode_step_host per layer on each step's q, k_new, v_new in pinned "
                            "host memory (a row of one pinned array per step), then a wait for the output "
                            "in pinned host memory"},
            "gpu_launches": launches,
            "host_max_step_gap_us": host_gap[0] * 1e6,
            "clocks": clk.summary(),
        }
        if svd is not None:
            result["svd"] = svd
        if L > 1:
            result["layers"] = L
            result["prefill_ms_per_layer"] = prefill_ms
    for ctx in ctxs:
        ctx.close()
    return result


def run_prefill(args, cfg):
    """Algorithm 1 alone: a warm-up prefill of the same kind, then the
    workload's prefill, timed on the host around the C-ABI call (which
    synchronizes), with its kernels' CUDA-event times."""
    _, _, local = dist_env()
    dev = torch.device("cuda", local)
    run_cfg = cfg.with_(steps=1)
    stream = torch.cuda.current_stream()
    o_w = min(cfg.o, 4096 // cfg.c // 4)
    warm = run_cfg.with_(b=1, s=cfg.w + 4096, o=o_w, k=min(cfg.k, 4096 // cfg.c - o_w))
    wi = synth.make_inputs(warm, device=dev)
    binding.prefill(binding.make_params(warm), wi["k_pre"], wi["v"], stream).close()
    del wi
    inp = synth.make_inputs(run_cfg, device=dev)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    ctx = binding.prefill(binding.make_params(run_cfg), inp["k_pre"], inp["v"], stream)
    wall = (time.perf_counter() - t0) * 1e3
    kt = ctx.kernel_times()
    kern = {k_: {"ms": v[0], "launches": v[1]} for k_, v in kt.items() if v[1] and k_ in PREFILL_KERNELS}
    E = 2 if cfg.dtype == "bf16" else 4
    D = cfg.h_kv * cfg.d
    res = {"metric": "ShadowKV prefill (Algorithm 1) wall time", "value": wall, "unit": "ms",
           "higher_is_better": False, "dtype": cfg.dtype, "data": "synthetic",
           "config": {"workload": f"{cfg.name}: ShadowKV prefill, b={cfg.b} h_kv={cfg.h_kv} d={cfg.d} "
                                  f"s={cfg.s} c={cfg.c} r={cfg.r} o={cfg.o} w={cfg.w}"},
           "prefill_kernels": kern, "prefill_kernels_ms": sum(v["ms"] for v in kern.values()),
           "key_bytes": E * cfg.b * cfg.s * D, "value_bytes_offloaded": E * cfg.b * cfg.s * D,
           "gram_flops": cfg.b * cfg.s * D * (D + 128), "factor_flops": 4 * cfg.b * cfg.s * D * cfg.r,
           "layout": ctx.layout()}
    if args.svd_report:
        res["svd"] = svd_report(inp, ctx, cfg, dev)
    ctx.check()
    ctx.close()
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=32)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default=DEFAULT_CONFIG, choices=sorted(CONFIGS))
    ap.add_argument("--batch", type=int, default=None)
    ap.add_argument("--sweep", default=None, help="comma-separated batch sizes, one line each")
    ap.add_argument("--chunk", type=int, default=None)
    ap.add_argument("--budget", type=float, default=None, help="sparse budget k*c/s in percent")
    ap.add_argument("--q-sigma", type=float, default=None)
    ap.add_argument("--layers", type=int, default=1)
    ap.add_argument("--rebuild-in-attention", action="store_true",
                    help="rebuild the missed keys inside the attention's launch (three launches per step)")
    ap.add_argument("--svd-report", action="store_true",
                    help="SVD error and subspace similarity (on by default for the 256K workload)")
    ap.add_argument("--prefill-only", action="store_true",
                    help="time Algorithm 1 alone (after a warm-up prefill) and print its line")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.config == "llama_b2_s256k":
        args.svd_report = True
    cfg = apply_overrides(CONFIGS[args.config], args.chunk, args.budget, args.q_sigma, args.batch)
    ws, rank, local = dist_env()

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

    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    if args.prefill_only:
        res = run_prefill(args, cfg)
        if rank == 0:
            print(json.dumps(res), flush=True)
        return
    batches = [int(x) for x in args.sweep.split(",")] if args.sweep else [cfg.b]
    cpu = None
    if ws == 1 and not args.no_cpu_baseline:
        tot, n, cores = oracle_decode_timing(cfg, 3, 1)
        cpu = {"value": n / tot, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"1 sequence (all {cfg.h_kv} KV heads), {n} decode steps of the same shape"}
    for b in batches:
        res = run_ours(args, cfg.with_(b=b))
        if res is None:
            continue
        if cpu is not None:
            res["cpu_baseline"] = cpu
        print(json.dumps(res), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
