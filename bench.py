"""Benchmark of the routed MoE FFN layer on GB300.

Headline: single-token decode through the 40-layer 35B-A3B-shaped stack
(hidden 2048, 256 experts/layer, top-8, expert FFN 512, shared FFN 512,
int4/32-block/fp16-scale experts), as tokens/s, with the achieved HBM
bandwidth of the decode kernel against the measured peak.  Also measured
(under "extra"): the 1+3-token MTP verify batch on the same stack, the
48-layer 125B-A6B-shaped stack with permuted slot tables, and the
8192-token prefill chunk through one 125B-shaped layer (tokens/s and
tensor-core utilisation of its grouped GEMMs).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With torchrun (N > 1) every rank runs its own replica of the workload on its
own GPU (decode tokens are independent: weak scaling, no collective on the
data path); rank 0 prints one JSON line.  --impl reference times the CPU
oracle (test infrastructure) on this host's cores on a bounded sample.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import statistics
import subprocess
import threading
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workload as W  # noqa: E402

HEADLINE = "decode35b"
METRIC = "MoE decode tok/s (40-layer 35B-A3B-shaped stack, 1 token)"
UNIT = "tokens/s"


# --------------------------------------------------------------------------- helpers

def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", 0)), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def decode_bytes_per_layer(cfg, n_units_routed: int) -> int:
    """Algorithmic bytes of one layer: packed codes + scales of the routed
    experts that run plus the shared expert (each byte read once)."""
    b = n_units_routed * cfg.expert_bytes()
    if cfg.shared_ffn:
        b += cfg.expert_bytes(cfg.shared_ffn)
    return b


def router_bytes(cfg) -> int:
    return cfg.n_experts * cfg.hidden * 4


def prefill_flops(cfg, T) -> float:
    H, F, Fs, k, E = cfg.hidden, cfg.ffn, cfg.shared_ffn, cfg.top_k, cfg.n_experts
    return 2.0 * T * (k * 3 * H * F + 3 * H * Fs + E * H)


class ClockSampler:
    """nvidia-smi sampling (every 20 ms) of SM clocks and throttle reasons.

    Started before the warm-up so that it is running when the timed region
    begins; each sample is stamped with the host time it arrived.
    summary() keeps the samples taken between mark_start() and mark_stop()
    (the timed region).  A short timed region (a few ms) may hold no sample,
    so the caller can run the same step for a while after it, untimed, and
    mark that stretch with mark_window(); report() then adds the samples of
    that load window and says so."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 20

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.rows = []
        self.t0 = self.t1 = None
        self.w0 = self.w1 = None
        self.thread = None

    def _reader(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), line))

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", str(self.PERIOD_MS)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True, bufsize=1)
            self.thread = threading.Thread(target=self._reader, daemon=True)
            self.thread.start()
            t_end = time.time() + 5.0
            while not self.rows and time.time() < t_end:  # running before timing starts
                time.sleep(0.01)
        except Exception:
            self.proc = None
        return self

    def mark_start(self):
        self.t0 = time.time()

    def mark_stop(self):
        self.t1 = time.time()

    def mark_window(self, t0: float, t1: float):
        self.w0, self.w1 = t0, t1

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            if self.thread is not None:
                self.thread.join(timeout=5)

    def summary(self, windows=None):
        """Samples whose arrival falls in one of the (t0, t1) windows
        (default: the timed region)."""
        if windows is None:
            windows = [(self.t0, self.t1)] if self.t0 is not None and self.t1 is not None else None
        rows = []
        for t, line in self.rows:
            if windows is not None and not any(a <= t <= b + 0.06 for a, b in windows):
                continue
            r = next(csv.reader(io.StringIO(line)), [])
            if len(r) >= 9:
                rows.append(r)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
            except ValueError:
                continue
            for i, nm in enumerate(names):
                if r[5 + i].strip().lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}

    def report(self):
        """The timed region's summary; when it holds fewer than 3 samples,
        the median and reasons are taken over the timed region and the load
        window after it (same step, untimed), and `source` says so."""
        s = self.summary()
        out = dict(s, samples_timed=s["samples"], source="timed region")
        if s["samples"] < 3 and self.w0 is not None and self.t0 is not None:
            out = dict(self.summary([(self.t0, self.t1), (self.w0, self.w1)]),
                       samples_timed=s["samples"],
                       source="timed region + %.1f s load window of the same step after it"
                              % (self.w1 - self.w0))
        return out


def source_hash(*rel):
    h = hashlib.sha256()
    for r in rel:
        with open(os.path.join(ROOT, r), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_key: str, src_hash: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel source."""
    try:
        with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
            d = json.load(f)
        e = d.get(kernel_key)
        if e and e.get("source_hash") == src_hash:
            return e.get("dram_bytes_per_launch")
    except Exception:
        pass
    return None


# --------------------------------------------------------------------------- GPU arm

class Dist:
    """One process per GPU (replicas: no collective on the data path); the
    process group only carries the barrier and the max over ranks of the
    step time.  backend "gloo" runs it on CPU tensors (tests)."""

    def __init__(self, n_gpus: int, backend: str = "nccl"):
        import torch

        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.n = max(n_gpus, self.world)
        self.pg = None
        self.device = "cuda" if backend == "nccl" else "cpu"
        if self.device == "cuda":
            torch.cuda.set_device(self.local)
        if self.world > 1:
            import torch.distributed as dist

            if self.device == "cuda":
                dist.init_process_group("nccl", device_id=torch.device("cuda", self.local))
            else:
                dist.init_process_group(backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, v: float) -> float:
        if not self.pg:
            return v
        import torch

        t = torch.tensor([v], dtype=torch.float64, device=self.device)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


def job_tokens_per_s(n_ranks: int, tokens_per_rank_step: int, ms_per_step_max: float) -> float:
    """Whole-job throughput: every rank processes its own tokens each step
    (weak scaling); the job's step time is the slowest rank's."""
    return n_ranks * tokens_per_rank_step / (ms_per_step_max / 1e3)


def build_stack(cfg, max_tokens, n_slots=None, profile=False):
    """Library layers of a workload (device-generated weights).  n_slots <
    n_experts keeps only that many experts per layer in HBM (the rest in
    the library's host tier); profile places the Zipf-favoured experts first
    (usage profile = exp of the router's log-Zipf bias)."""
    import quantized_expert_ffn_softmax_gb300 as moe
    import torch

    config = dict(hidden=cfg.hidden, n_experts=cfg.n_experts, top_k=cfg.top_k, ffn=cfg.ffn,
                  shared_ffn=cfg.shared_ffn, max_tokens=max_tokens,
                  routing_flags=cfg.routing_flags, n_slots=n_slots or cfg.n_experts)
    layers = []
    for l in range(cfg.n_layers):
        D = W.device_layer(cfg, l)
        w = {n: D[n] for n in ("router_w", "slot_of_expert", "gate_q", "gate_s", "up_q", "up_s",
                               "down_q", "down_s")}
        w["router_bias"] = D["router_b"]
        if cfg.shared_ffn:
            for n in ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s"):
                w["sh_" + n] = D["sh_" + n]
        if "sh_gate_w" in D:
            w["sh_gate_w"] = D["sh_gate_w"]
        if profile:
            _, b = W.router(cfg, l)
            w["expert_profile"] = torch.from_numpy(np.exp(b.astype(np.float64)).astype(np.float32)).cuda()
        torch.cuda.synchronize()
        layers.append(moe.MoELayer(config, w, True))
        del D, w
    return layers


def time_steps(fn, steps, warmup, dist, ring_len, clk=None):
    import torch

    for i in range(warmup):
        fn(i % ring_len)
    torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if clk is not None:
        clk.mark_start()
    s.record()
    for i in range(steps):
        fn((warmup + i) % ring_len)
    e.record()
    torch.cuda.synchronize()
    if clk is not None:
        clk.mark_stop()
        if clk.t1 - clk.t0 < 1.0:
            # too short for the sampler: run the same step, untimed, for about
            # a second so that clocks under this load are sampled too
            w0 = time.time()
            i = 0
            while time.time() - w0 < 1.0:
                for _ in range(8):
                    fn((warmup + steps + i) % ring_len)
                    i += 1
                torch.cuda.synchronize()
            clk.mark_window(w0, time.time())
    dist.barrier()
    torch.cuda.synchronize()
    return dist.max(s.elapsed_time(e) / steps)


def kernel_profile(fn, steps, ring_len):
    import quantized_expert_ffn_softmax_gb300 as moe
    import torch

    torch.cuda.synchronize()
    moe.moe_profile_read()
    moe.moe_profile_enable(True)
    for i in range(steps):
        fn(i % ring_len)
    torch.cuda.synchronize()
    moe.moe_profile_enable(False)
    return moe.moe_profile_read()


def bench_decode(name, steps, warmup, dist, with_e2e=False, n_slots=None, profile=False):
    import quantized_expert_ffn_softmax_gb300 as moe
    import torch

    cfg = W.CONFIGS[name]
    T = cfg.n_tokens
    layers = build_stack(cfg, max_tokens=8, n_slots=n_slots, profile=profile)
    hs = [l.handle for l in layers]
    ring = [torch.from_numpy(W.activations(cfg, i).view(np.int16)).cuda() for i in range(64)]
    y = torch.empty_like(ring[0])
    # unique routed experts per layer for this input ring (from one traced pass)
    L, k, H = cfg.n_layers, cfg.top_k, cfg.hidden
    ids = torch.empty((L, T, k), dtype=torch.int32, device="cuda")
    hbuf = torch.empty((L, T, H), dtype=torch.int16, device="cuda")
    ubuf = torch.empty_like(hbuf)
    uniq = []
    for i in range(8):
        moe.moe_stack_forward_traced(hs, L, ring[i], T, y, hbuf, ubuf, None, ids)
        a = ids.cpu().numpy()
        uniq.append(sum(len(set(a[l].ravel().tolist())) for l in range(L)))
    assert moe.moe_status_sync(hs[0]) == moe.MOE_OK
    mean_unique_routed = float(np.mean(uniq))  # summed over layers
    bytes_per_step = mean_unique_routed * cfg.expert_bytes() + L * (
        cfg.expert_bytes(cfg.shared_ffn) if cfg.shared_ffn else 0)

    def step(i):
        moe.moe_stack_forward(hs, L, ring[i], T, y)

    for h in hs:
        moe.moe_cache_stats(h, reset=True)
    with ClockSampler(dist.local) as clk:
        ms = time_steps(step, steps, warmup, dist, len(ring), clk)
    cache = [moe.moe_cache_stats(h) for h in hs]
    prof = kernel_profile(step, min(steps, 50), len(ring))
    assert moe.moe_status_sync(hs[0]) == moe.MOE_OK
    kcount, kms = prof.get("moe_decode_kernel", (0, 0.0))
    k_avg = kms / max(kcount, 1)
    launches_per_step = kcount / max(1, min(steps, 50))
    out = {
        "ms_per_step": ms,
        "tok_s": job_tokens_per_s(dist.n, T, ms),
        "bytes_per_step": bytes_per_step,
        "gbs_step": bytes_per_step / (ms / 1e3) / 1e9,
        "kernel_ms": k_avg,
        "gbs_kernel": bytes_per_step / (k_avg / 1e3) / 1e9 if k_avg else None,
        "bytes_incl_router": bytes_per_step + L * router_bytes(cfg),
        "unique_routed_per_layer": mean_unique_routed / L,
        "launches_per_step": launches_per_step,
        "clocks": clk.report(),
    }
    if n_slots and n_slots < cfg.n_experts:
        hits, misses = sum(c[0] for c in cache), sum(c[1] for c in cache)
        out["cache"] = {"n_slots": n_slots, "n_experts": cfg.n_experts, "profile": bool(profile),
                        "hits": hits, "misses": misses,
                        "hit_rate": hits / max(1, hits + misses),
                        "note": "hits/misses over warm-up, timed steps and clock window"}
    if with_e2e:
        xs = [torch.from_numpy(W.activations(cfg, i).view(np.int16)).pin_memory() for i in range(8)]
        yh = torch.empty_like(xs[0]).pin_memory()
        harr = moe.layer_array(hs)  # built once, as a caller running the stack repeatedly would
        strm = torch.cuda.current_stream().cuda_stream
        for i in range(3):
            moe.moe_stack_forward(harr, L, xs[i], T, yh, strm)
        torch.cuda.synchronize()
        dist.barrier()
        t0 = time.perf_counter()
        for i in range(steps):
            # x read from pinned host memory by the kernel, y written back to
            # it, the stream synchronised: the whole step, host to host
            moe.moe_stack_forward(harr, L, xs[i % 8], T, yh, strm)
        dt = dist.max((time.perf_counter() - t0) / steps)
        out["e2e"] = {"value": dist.n * T / dt, "unit": UNIT,
                      "h2d_bytes_per_step": int(xs[0].numel() * 2),
                      "d2h_bytes_per_step": int(yh.numel() * 2)}
    for l in layers:
        l.close()
    del layers
    torch.cuda.empty_cache()
    return out


def bench_prefill(name, steps, warmup, dist, n_layers=1):
    """The prefill chunk through one layer (moe_forward), or through an
    n_layers stack of that shape (moe_stack_forward)."""
    import quantized_expert_ffn_softmax_gb300 as moe
    import torch

    cfg = W.CONFIGS[name].replace(n_layers=n_layers)
    T = cfg.n_tokens
    stack = build_stack(cfg, max_tokens=T)
    layer = stack[0]
    hs = [l.handle for l in stack]
    xs = [torch.from_numpy(W.activations(cfg, i).view(np.int16)).cuda() for i in range(2)]
    y = torch.empty_like(xs[0])

    def step(i):
        if n_layers == 1:
            moe.moe_forward(layer.handle, xs[i], T, y)
        else:
            moe.moe_stack_forward(hs, n_layers, xs[i], T, y)

    with ClockSampler(dist.local) as clk:
        ms = time_steps(step, steps, warmup, dist, 2, clk)
    prof = kernel_profile(step, min(steps, 20), 2)
    assert moe.moe_status_sync(layer.handle) == moe.MOE_OK
    # algorithmic FLOPs per GEMM kernel
    H, F, Fs, k, E = cfg.hidden, cfg.ffn, cfg.shared_ffn, cfg.top_k, cfg.n_experts
    fl = {"moe_gemm_gateup_swiglu": 2.0 * T * (k * 2 * H * F + 2 * H * Fs),
          "moe_gemm_down_scatter": 2.0 * T * (k * H * F + H * Fs),
          "moe_gemm_router": 2.0 * T * E * H}  # per launch (one layer)
    kern = {}
    total_k_ms = 0.0
    for nm, (c, tms) in prof.items():
        avg = tms / max(c, 1)
        total_k_ms += tms
        ent = {"launches": c, "avg_ms": avg}
        if nm in fl:
            ent["tflops"] = fl[nm] / (avg / 1e3) / 1e12
        kern[nm] = ent
    for nm in kern:
        kern[nm]["share"] = prof[nm][1] / total_k_ms if total_k_ms else None
    gemm_ms = sum(kern[n]["avg_ms"] for n in ("moe_gemm_gateup_swiglu", "moe_gemm_down_scatter")
                  if n in kern)
    gemm_fl = fl["moe_gemm_gateup_swiglu"] + fl["moe_gemm_down_scatter"]
    out = {"ms_per_step": ms, "tok_s": dist.n * T / (ms / 1e3), "layers": n_layers,
           "tflops_step": n_layers * prefill_flops(cfg, T) / (ms / 1e3) / 1e12,
           "grouped_gemm_tflops": gemm_fl / (gemm_ms / 1e3) / 1e12 if gemm_ms else None,
           "kernels": kern,
           "launches_per_step": sum(v["launches"] for v in kern.values()) / max(1, min(steps, 20)),
           "clocks": clk.report()}
    for l in stack:
        l.close()
    del stack, layer
    torch.cuda.empty_cache()
    return out


# --------------------------------------------------------------------------- CPU oracle arm

def host_cpu():
    """(nproc, CPU model) of this host."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    import platform

    return os.cpu_count() or 1, model or platform.machine()


def _thread_map(fn, items, workers):
    """fn over items on `workers` host threads (the oracle's C calls release
    the GIL); results in item order."""
    import concurrent.futures as cf

    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        return list(ex.map(fn, items))


def oracle_decode_sample(cfg, n_layers: int, threads: int):
    """Times the oracle as it stands (fp64 C) on `threads` independent tokens
    at once, one per host thread, each through the first `n_layers` layers
    of the stack (its experts drawn before the timed region).  Returns
    (tokens/s for the full stack, description)."""
    import oracle

    routers = [W.router(cfg, l) for l in range(n_layers)]
    shared = [W.shared_expert(cfg, l) for l in range(n_layers)]

    def token_pass(x, plan=None):
        h = x.copy()
        drawn = []
        for l in range(n_layers):
            u = oracle.rmsnorm(h)
            z = oracle.router_logits(*routers[l], u)
            ids, w, _ = oracle.topk_softmax(z, cfg.top_k)
            exs = plan[l] if plan is not None else [W.expert(cfg, l, int(e)) for e in ids[0]]
            drawn.append(exs)
            y = oracle.combine_token(exs, w[0], shared[l], u[0])
            h = oracle.residual(h, y[None, :])
        return drawn

    xs = [W.activations(cfg, 100 + i) for i in range(threads)]
    # route once to know which experts to draw (untimed), then time the pass
    plans = _thread_map(token_pass, xs, threads)
    t0 = time.perf_counter()
    _thread_map(lambda i: token_pass(xs[i], plans[i]), range(threads), threads)
    dt = time.perf_counter() - t0
    tok_s = threads / (dt * cfg.n_layers / n_layers)
    desc = ("oracle (fp64 C, as it stands) on %d independent tokens at once, one per host "
            "thread, each through %d of the %d layers (router, top-%d, %d experts + shared, "
            "residual); expert weights drawn before timing; wall time scaled x%d to the stack"
            % (threads, n_layers, cfg.n_layers, cfg.top_k, cfg.top_k, cfg.n_layers // n_layers))
    return tok_s, desc


def headline_config(n_gpus):
    """The headline workload's config object, shared by both arms."""
    return {"workload": HEADLINE, "layers": 40, "hidden": 2048, "experts": 256, "top_k": 8,
            "ffn": 512, "shared_ffn": 512, "tokens_per_step": 1,
            "weights": "int4, 32-block, fp16 scale", "input_ring": 64,
            "l2": "expert bytes per step 637 MB > 129 MB L2; 64-input ring",
            "parallelism": "replica per GPU" if n_gpus > 1 else "single GPU"}


def run_reference(args):
    """The oracle as it stands (fp64 C), on this host's cores, timed on a
    bounded sample of the headline workload.  One step: `threads` different
    tokens at once, one per host thread, each through layer 0 (router,
    top-k, its k experts and the shared expert; the weights drawn once
    before any timing).  The tokens/s value scales that wall time to the
    40-layer stack; ms_per_step is the time of the work actually timed.
    When K + W such steps would take more than about 150 s, a step is one
    expert FFN per thread instead, scaled by the layer / expert time ratio
    measured once beforehand (untimed)."""
    cfg = W.CONFIGS[HEADLINE]
    import oracle

    oracle.build()
    nproc, model = host_cpu()
    threads = max(1, min(16, nproc))
    wr, b = W.router(cfg, 0)
    sh = W.shared_expert(cfg, 0)
    us = [oracle.rmsnorm(W.activations(cfg, 100 + i)) for i in range(threads)]

    def draw(u):
        ids, _, _ = oracle.topk_softmax(oracle.router_logits(wr, b, u), cfg.top_k)
        return [W.expert(cfg, 0, int(e)) for e in ids[0]]

    experts = _thread_map(draw, us, threads)

    def layer_pass(i):
        zz = oracle.router_logits(wr, b, us[i])
        ii, ww, _ = oracle.topk_softmax(zz, cfg.top_k)
        oracle.combine_token(experts[i], ww[0], sh, us[i][0])

    def expert_pass(i):
        oracle.combine_token(experts[i][:1], np.ones(1), None, us[i][0])

    def timed(fn):
        t0 = time.perf_counter()
        _thread_map(fn, range(threads), threads)
        return time.perf_counter() - t0

    t_layer = min(timed(layer_pass) for _ in range(2))
    n = args.steps + args.warmup
    if n * t_layer <= 150.0:
        fn, scale = layer_pass, float(cfg.n_layers)
        desc = ("oracle (fp64 C, as it stands) on %d host threads: per step %d different tokens "
                "at once, one per thread, through layer 0 (router, top-%d, %d experts + shared); "
                "scaled x%d to the stack" % (threads, threads, cfg.top_k, cfg.top_k, cfg.n_layers))
    else:
        t_exp = min(timed(expert_pass) for _ in range(3))
        fn, scale = expert_pass, cfg.n_layers * t_layer / t_exp
        desc = ("oracle (fp64 C, as it stands) on %d host threads: per step one expert FFN of "
                "layer 0 for each of %d tokens at once, scaled x%.1f (40 layers x the measured "
                "layer/expert time ratio %.2f)" % (threads, threads, scale, t_layer / t_exp))
    for _ in range(args.warmup):
        timed(fn)
    per = [timed(fn) for _ in range(args.steps)]
    step_s = float(np.mean(per))
    v = threads / (step_s * scale)
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3,
            "step_scale_to_stack": scale, "tokens_per_step": threads,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": headline_config(args.gpus),
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": threads, "nproc": nproc,
                             "cpu": model, "kind": "oracle", "sample": desc},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extra", action="store_true", help="headline workload only")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", default=None,
                    help="time one workload only (profiling cases): decode35b, mtp35b, "
                         "decode125b, decode35b_variants or prefill125b")
    ap.add_argument("--layers", type=int, default=None,
                    help="with --only on a decode workload: use the first N layers")
    ap.add_argument("--slots", type=int, default=None,
                    help="with --only on a decode workload: experts per layer kept in HBM")
    ap.add_argument("--profile", action="store_true",
                    help="with --slots: place experts by the usage profile")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            run_reference(args)
        return

    dist = Dist(args.gpus)
    import quantized_expert_ffn_softmax_gb300 as moe

    moe.lib()
    if args.only:
        if args.layers:
            W.CONFIGS[args.only] = W.CONFIGS[args.only].replace(n_layers=args.layers)
        if args.only.startswith("prefill"):
            r = bench_prefill(args.only, args.steps, args.warmup, dist, n_layers=args.layers or 1)
        else:
            r = bench_decode(args.only, args.steps, args.warmup, dist, n_slots=args.slots,
                             profile=args.profile)
        if dist.rank == 0:
            print(json.dumps({"only": args.only, "layers": args.layers, "result": r}), flush=True)
        dist.close()
        return
    hbm, bf16, bf16_sus, peak_kind = peaks()
    head = bench_decode(HEADLINE, args.steps, args.warmup, dist, with_e2e=True)
    extra = {}
    if not args.no_extra:
        for nm in ("mtp35b", "decode125b", "decode35b_variants"):
            r = bench_decode(nm, max(20, args.steps // 2), args.warmup, dist)
            r["frac_of_peak_kernel"] = r["gbs_kernel"] / hbm if r["gbs_kernel"] else None
            extra[nm] = r
        # partial residency: half and a quarter of the experts in HBM (placed
        # by the usage profile), and a quarter placed without one
        for tag, ns, pr in (("decode35b_half_resident", 128, True),
                            ("decode35b_quarter_resident", 64, True),
                            ("decode35b_quarter_resident_noprofile", 64, False)):
            r = bench_decode(HEADLINE, max(20, args.steps // 2), args.warmup, dist, n_slots=ns,
                             profile=pr)
            r["frac_of_peak_kernel"] = r["gbs_kernel"] / hbm if r["gbs_kernel"] else None
            extra[tag] = r
        # routing variants: per-layer time beside the default headline stack
        v = extra["decode35b_variants"]
        v["us_per_layer"] = v["ms_per_step"] * 1e3 / W.CONFIGS["decode35b_variants"].n_layers
        v["default_us_per_layer"] = head["ms_per_step"] * 1e3 / W.CONFIGS[HEADLINE].n_layers
        pf = bench_prefill("prefill125b", max(10, args.steps // 10), args.warmup, dist)
        g = pf["kernels"].get("moe_gemm_gateup_swiglu", {})
        pf["roofline_gateup"] = {"bound": "tensor", "achieved": g.get("tflops"), "peak": bf16,
                                 "unit": "TFLOP/s", "frac": (g.get("tflops") or 0) / bf16,
                                 "note": "fp16 operands; fp16 dense peak = bf16 peak"}
        pf["grouped_gemm_frac"] = (pf["grouped_gemm_tflops"] or 0) / bf16
        extra["prefill125b"] = pf
        # the same chunk through the 48-layer stack of that shape
        ps = bench_prefill("prefill125b", max(3, args.steps // 100), args.warmup, dist, n_layers=48)
        ps["grouped_gemm_frac"] = (ps["grouped_gemm_tflops"] or 0) / bf16
        extra["prefill125b_stack48"] = ps

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cfg = W.CONFIGS[HEADLINE]
        nproc, model = host_cpu()
        threads = max(1, min(16, nproc))
        v, desc = oracle_decode_sample(cfg, 4, threads)
        cpu = {"value": v, "unit": UNIT, "cores": threads, "nproc": nproc, "cpu": model,
               "kind": "oracle", "sample": desc}

    src = source_hash("quantized_expert_ffn_softmax_gb300/csrc/decode.cu",
                      "quantized_expert_ffn_softmax_gb300/csrc/device_common.cuh")
    launches = head["launches_per_step"] * args.steps
    if not args.no_extra:
        launches += 0  # extras are timed separately and not part of the headline region
    line = {
        "metric": METRIC, "value": head["tok_s"], "unit": UNIT, "n_gpus": dist.n,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic",
        "config": headline_config(dist.n),
        "roofline": {"bound": "hbm", "achieved": head["gbs_kernel"], "peak": hbm, "unit": "GB/s",
                     "frac": (head["gbs_kernel"] or 0) / hbm,
                     "traffic": ncu_traffic("moe_decode_kernel:" + HEADLINE, src),
                     "peak_kind": peak_kind, "kernel": "moe_decode_kernel",
                     "bytes_per_launch": head["bytes_per_step"],
                     "kernel_ms": head["kernel_ms"]},
        "cpu_baseline": cpu,
        "e2e": head["e2e"],
        "gpu_launches": int(round(launches)),
        "clocks": head["clocks"],
        "extra": extra,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    dist.close()


if __name__ == "__main__":
    main()
