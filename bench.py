#!/usr/bin/env python3
"""Benchmark of the MoE-layer forward on B300: one JSON line on stdout.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]
                    [--n-group G --topk-group M] [--z-beta B] [--aux-post-drop] [--gather]

A step is one whole layer forward (route, dispatch, expert up/down GEMMs,
combine, aux loss) over one batch of seeded synthetic tokens already resident
in HBM.  Default workload: the largest single-GPU configuration, bf16,
T=32768 tokens, d=4096, 128 experts, top-8, SwiGLU d_ff=1536, dropless
(``--workload`` selects the others, e.g. e8_swiglu: T=4096, 8 experts, top-2,
SwiGLU d_ff=14336, capacity factor 1.25).

Timing: W untimed warm-up steps; then K steps, each preceded (outside the
timed events) by a 512 MB write that flushes the 126 MB L2; CUDA events on
the launching stream around every step and around every call inside it;
barrier + synchronize on both sides; max over ranks.  SM clocks and
clock-event reasons are sampled through NVML during the timed steps.

``e2e``: the same metric through the public API with host buffers: each step
copies x from pinned host memory, runs the layer and reads y and the loss
back, all inside the timed region, pipelined over three streams and two
buffer sets (copy-in of step i+1 and copy-out of step i-1 overlap step i).

``roofline``: the dominant kernel (the expert up-projection GEMM) -- its
algorithmic FLOPs (2 * kept slots * d * N1) over its CUDA-event duration,
against the measured dense bf16 peak.

``roofline_hbm``: the three bandwidth-bound calls (route, dispatch, combine
with the aux loss) -- each one's algorithmic bytes (below) over its CUDA-event
duration, against the measured HBM copy bandwidth and against 8 TB/s:
  route     T*d*b (x) + E*d*4 (router weight) + T*k*8 (indices, gates)
  dispatch  T*k*8 (indices, gates read) + T*k*4 (slot rows) + A*8 (row maps)
            + T_u*d*b (x rows of tokens with a kept slot) + A*d*b (x_perm)
  combine   A*d*b (y_perm) + T*d*b (y) + T*k*4 (slot rows)
with A the kept slots, T_u the tokens with at least one kept slot and b the
bytes of one element.

``cpu_baseline`` (rank 0, N=1): the CPU oracle timed on a bounded sample of
the same workload (its first S tokens, capacity recomputed for S tokens).

``--impl reference``: the CPU oracle alone on the host cores (the method has
no other runnable implementation); rank 0 only.

``--train``: a step is the forward (keeping the pre-activation) and the
backward (input, router and expert weight gradients of <dy, y> + aux loss
(+ z-loss)) for a seeded upstream gradient dy; the JSON line reports
the fwd+bwd rate, per-phase times and the roofline of the largest backward
GEMM (the w1 weight gradient).

Variants (same step, same JSON line; ``config.variant`` names them):
group-limited routing (``--n-group``/``--topk-group``), the router z-loss
(``--z-beta``), the post-drop f_i aux loss (``--aux-post-drop``) and the
up-projection that gathers x rows itself instead of a permuted copy
(``--gather``).

With torchrun (N>1) every rank runs its own independent batch (seed + rank):
the layer forward needs no exchange between GPUs, so scaling is weak (a
global aux loss over all ranks' tokens would add one all-reduce of 2E + 1
numbers: top_routing_expert_02_b300.dist).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from top_routing_expert_02_b300 import synth  # noqa: E402

METRIC = "MoE-layer fwd tokens/s and grouped-GEMM TFLOP/s (% BF16 peak) on 1 B300"
L2_FLUSH_BYTES = 512 << 20
def KERNELS_PER_STEP_TOTAL(cfg, args=None) -> int:
    """Library kernels launched by one layer forward of this workload (the
    device-timed region launches exactly these, K times)."""
    tc_router = cfg.dtype == "bf16" and cfg.E <= 128
    # weight split + logits (E <= 64: with softmax/top-k and the prob sums, written by its last CTA;
    # E > 64: + finishing kernel + prob sums) | CUDA-core router + sums
    route = (2 if cfg.E <= 64 else 4) if tc_router else 2
    gather = bool(args and args.gather)
    n = cfg.T * cfg.k
    # chunk histograms (+ a per-expert scan of them above 65536 assignments) + ranks; T*k = 0: the rank
    # kernel alone
    ranks = 1 if n == 0 else (3 if n > 65536 else 2)
    dispatch = ranks + (0 if gather else 1)      # (+ row copy)
    z = 1 if (args and args.z_beta is not None) else 0
    bwd = BWD_KERNELS if (args and args.train) else 0
    world = int(os.environ.get("WORLD_SIZE", "1"))
    aux = 1 if (world > 1 and not (args and args.train)) else 0   # replicas: the global aux loss is its own launch
    return route + dispatch + 1 + 1 + 1 + aux + z + bwd   # up, down, combine (+ aux) (+ z-loss) (+ backward)


def plan_kwargs(args) -> dict:
    kw = dict(gather=args.gather, n_group=args.n_group, topk_group=args.topk_group, z_beta=args.z_beta,
              aux_post_drop=args.aux_post_drop, train=args.train)
    if args.train:
        kw["grad_dtype"] = torch.bfloat16 if args.grad_dtype == "bf16" else torch.float32
    return kw


BWD_KERNELS = 1 + 2 + 2 + 1 + 6   # combine bwd, 2 data-gradient GEMMs (act bwd fused), 2 weight-gradient GEMMs,
                                  # router bwd, router grads (prep, dl.W GEMM, dx gather, dW GEMM, dW sum, db)


def variant_dict(args) -> dict:
    return {"train": args.train, "weight_grad_dtype": args.grad_dtype if args.train else None,
            "n_group": args.n_group, "topk_group": args.topk_group, "z_beta": args.z_beta,
            "aux_f": "kept slots (post-drop)" if args.aux_post_drop else "every choice (pre-drop)",
            "up_projection": "gathers x rows (no x_perm)" if args.gather else "reads x_perm"}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), float(j["bf16_tflops"]), float(j["bf16_tflops_sustained"]), "measured"
    return 6400.0, 1800.0, 1400.0, "fallback"


# ------------------------------------------------------------------ clocks --
class ClockSampler:
    """NVML samples of SM clock and clock-event reasons (read only)."""
    BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
            0x80: "hw_power_brake_slowdown", 0x2: "applications_clocks_setting", 0x1: "gpu_idle"}

    def __init__(self, device_index: int, period_s: float = 0.01):
        self.samples, self.reasons, self.max_mhz, self.ok, self.err = [], set(), None, False, None
        self._stop = threading.Event()
        self._period = period_s
        self._t = None
        self._smi = None
        try:
            import pynvml
            pynvml.nvmlInit()
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            try:
                self._h = pynvml.nvmlDeviceGetHandleByUUID(uuid.encode())
            except Exception:
                self._h = pynvml.nvmlDeviceGetHandleByUUID(uuid)
            self._nv = pynvml
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self._h, pynvml.NVML_CLOCK_SM)
            self.ok = True
        except Exception as e:   # fall back to nvidia-smi sampling
            self.err = f"nvml: {type(e).__name__}: {e}"
            self._uuid = None
            try:
                self._uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            except Exception:
                pass

    def _run(self):
        nv = self._nv
        while not self._stop.is_set():
            try:
                self.samples.append(nv.nvmlDeviceGetClockInfo(self._h, nv.NVML_CLOCK_SM))
                fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                    nv.nvmlDeviceGetCurrentClocksThrottleReasons
                bits = fn(self._h)
                for b, name in self.BITS.items():
                    if bits & b:
                        self.reasons.add(name)
            except Exception:
                pass
            time.sleep(self._period)

    def _run_smi(self):
        """Fallback: one nvidia-smi process streaming a sample every 20 ms (its own child, ended by PID)."""
        import subprocess
        q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        sel = ["-i", "GPU-" + self._uuid if self._uuid and not self._uuid.startswith("GPU-") else self._uuid] \
            if self._uuid else []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        try:
            proc = subprocess.Popen(["nvidia-smi", *sel, f"--query-gpu={q}", "--format=csv,noheader,nounits",
                                     "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception as e:
            self.err = f"{self.err}; nvidia-smi: {type(e).__name__}: {e}"
            return
        try:
            while not self._stop.is_set():
                line = proc.stdout.readline()
                if not line:
                    break
                try:
                    f = [v.strip() for v in line.split(",")]
                    self.samples.append(float(f[0]))
                    self.max_mhz = float(f[1])
                    for name, v in zip(names, f[2:]):
                        if v.lower().startswith("active"):
                            self.reasons.add(name)
                    self.ok = True
                except (ValueError, IndexError):
                    continue
        finally:
            proc.terminate()
            try:
                proc.wait(timeout=5)
            except Exception:
                proc.kill()

    def __enter__(self):
        target = self._run if self.ok else self._run_smi
        self._t = threading.Thread(target=target, daemon=True)
        self._t.start()
        return self

    def __exit__(self, *a):
        self._stop.set()
        if self._t is not None:
            self._t.join()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0, "error": self.err}
        reasons = sorted(self.reasons - {"gpu_idle"})
        d = {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz, "reasons": reasons,
             "samples": len(self.samples), "source": "nvml" if self.err is None else "nvidia-smi"}
        if self.err:
            d["nvml_error"] = self.err[:200]
        return d


# ------------------------------------------------------------- CPU oracle --
def oracle_variant(args) -> dict:
    """The routing variant's switches in the oracle's terms."""
    return dict(n_group=args.n_group, topk_group=args.topk_group, z_beta=args.z_beta or 0.0,
                aux_post_drop=args.aux_post_drop)


def oracle_sample(cfg: synth.MoEConfig, ri, w1, w2, budget_s: float = 15.0, variant=None):
    """Time the CPU oracle on the first S tokens (S grown until ~budget_s)."""
    import oracle
    w1h, w2h = w1.cpu(), w2.cpu()
    variant = variant or {}

    def run(S):
        sub = ri.x[:S].contiguous()
        cap = oracle.capacity(S, cfg.E, cfg.cf)
        t0 = time.perf_counter()
        oracle.forward(sub, ri.W, ri.b, w1h, w2h, k=cfg.k, cap=cap, act=cfg.act, renorm=cfg.renorm,
                       alpha=cfg.alpha, **variant)
        return time.perf_counter() - t0

    S = min(cfg.T, 8)
    t = run(S)
    for _ in range(3):   # grow the sample towards the budget (the cost is not linear in S)
        if t >= budget_s / 2 or S >= cfg.T:
            break
        S = int(min(cfg.T, max(S + 1, S * (budget_s / max(t, 1e-3)))))
        t = run(S)
    return {"value": S / t, "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"first {S} of {cfg.T} tokens of the workload, whole layer (routing, capacity for {S} "
                      f"tokens, expert FFN, combine, aux loss) in fp64, {t:.1f} s"}, S, t


def reference_arm(args, cfg):
    """--impl reference: the oracle on the host cores, rank 0 only."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    ri = synth.make_routing_inputs(cfg)
    w1, w2 = synth.make_expert_weights(cfg, device="cuda" if torch.cuda.is_available() else "cpu")
    var = oracle_variant(args)
    budget = max(0.2, 120.0 / max(1, args.steps + args.warmup))
    import oracle
    from oracle import backward as ob
    w1h, w2h = w1.cpu(), w2.cpu()
    dy = torch.randn(cfg.T, cfg.d, generator=torch.Generator().manual_seed(777)).to(
        torch.bfloat16 if cfg.dtype == "bf16" else torch.float32)
    if args.train:
        cb = oracle_sample_train(cfg, ri, w1, w2, dy, var, budget_s=budget)
        S = int(cb["sample"].split()[1])
    else:
        cb, S, _ = oracle_sample(cfg, ri, w1, w2, budget_s=budget, variant=var)
    # warm-up and timed steps: each step is the bounded sample
    sub, dys = ri.x[:S].contiguous(), dy[:S].contiguous()
    cap = oracle.capacity(S, cfg.E, cfg.cf)
    bvar = {k: var[k] for k in ("n_group", "topk_group", "z_beta", "aux_post_drop")}
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle.forward(sub, ri.W, ri.b, w1h, w2h, k=cfg.k, cap=cap, act=cfg.act, renorm=cfg.renorm,
                       alpha=cfg.alpha, **var)
        if args.train:
            ob.backward(sub, ri.W, ri.b, w1h, w2h, dys, k=cfg.k, cap=cap, act=cfg.act, renorm=cfg.renorm,
                        alpha=cfg.alpha, **bvar)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    ms = 1000.0 * statistics.mean(times)
    value = S / (ms / 1000.0)
    cb["value"] = value
    metric = "MoE-layer fwd+bwd tokens/s on 1 B300" if args.train else METRIC
    line = {"impl": "reference", "metric": metric, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_dict(cfg, args), "cpu_baseline": cb,
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def enqueue_spin_cycles(host_s: float, tail_s: float) -> int:
    """GPU clock cycles of a device-side wait (torch.cuda._sleep) placed before
    each device-timed step when the host is the slower side: host_s is the
    host time to enqueue one step, tail_s how long the device still ran after
    that.  A short tail means the device kept waiting for launches; then the
    wait lasts twice the host time (capped at 20 ms), so the host has queued
    every launch of the step before the device starts it, and the per-call
    event times hold device work and device-side launch gaps, not host launch
    overhead.  When the device is the slower side the host runs ahead by
    itself and no wait is added (a wait would also let a power-capped GPU
    rest between steps)."""
    if tail_s > 0.25 * host_s:
        return 0
    return int(min(0.02, 2.0 * host_s) * 2.1e9)


def config_dict(cfg, args=None):
    return {"workload": cfg.name, "description": cfg.describe(), "T": cfg.T, "d": cfg.d, "E": cfg.E, "k": cfg.k,
            "F": cfg.F, "act": cfg.act, "cf": cfg.cf, "renorm": cfg.renorm, "alpha": cfg.alpha,
            **({"variant": variant_dict(args)} if args is not None else {}),
            "l2": "device-timed steps: L2 flushed before every step (512 MB write); e2e steps: x arrives by a "
                  "host-to-device copy every step, weights (GBs) exceed L2",
            "timing": "device-timed steps back to back; where the host enqueues a step more slowly than the "
                      "device runs it, each step starts after a GPU-side wait covering the shortfall, so per-call "
                      "times hold no host launch overhead; graph_ms_per_step is the same step as one CUDA-graph "
                      "launch; e2e is the pipelined public-API path"}


def hbm_bytes(cfg, A: int, T_used: int, esz: int, gather: bool = False) -> dict:
    """Algorithmic HBM bytes of one call of each bandwidth-bound step (the
    minimum any implementation must move: every input read once, every output
    written once)."""
    T, d, E, k = cfg.T, cfg.d, cfg.E, cfg.k
    route = T * d * esz + E * d * 4 + T * k * 8
    dispatch = T * k * 8 + T * k * 4 + A * 8 + (0 if gather else T_used * d * esz + A * d * esz)
    combine = A * d * esz + T * d * esz + T * k * 4
    return {"route": route, "dispatch": dispatch, "combine_aux": combine}


def hbm_rooflines(cfg, A, T_used, esz, part, hbm_gbs, peak_src, gather=False) -> dict:
    out = {}
    for name, nbytes in hbm_bytes(cfg, A, T_used, esz, gather).items():
        ms = statistics.mean(part[name])
        gbs = nbytes / (ms * 1e-3) / 1e9
        out[name] = {"bound": "hbm", "bytes": nbytes, "us": 1000.0 * ms, "achieved": gbs, "peak": hbm_gbs,
                     "unit": "GB/s", "frac": gbs / hbm_gbs, "frac_of_8TBs": gbs / 8000.0,
                     "peak_source": f"{peak_src} HBM copy"}
    return out


def traffic_from_profile(kernel_src: str, workload: str):
    """DRAM bytes per launch of the up-projection GEMM from the committed ncu
    summary: one `workload = ...` block per captured workload; a block counts
    only for its own workload and only while the kernel source is unchanged
    since the capture."""
    p = os.path.join(ROOT, "profiles", "expert_up_gemm_traffic.txt")
    if not os.path.exists(p):
        return None
    with open(kernel_src, "rb") as f:
        sha = hashlib.sha256(f.read()).hexdigest()[:16]
    blocks, cur = [], None
    for line in open(p):
        if "=" not in line or line.startswith("#"):
            continue
        k, v = (x.strip() for x in line.split("=", 1))
        if k == "workload":
            cur = {}
            blocks.append(cur)
        if cur is not None:
            cur[k] = v
    for vals in blocks:
        if vals.get("workload") == workload and vals.get("kernel_source_sha256_16") == sha:
            try:
                return float(vals["dram_bytes_per_launch"])
            except (KeyError, ValueError):
                return None
    return None


# -------------------------------------------------------------------- ours --
def our_arm(args, cfg):
    import top_routing_expert_02_b300 as moe
    from top_routing_expert_02_b300 import dist as mdist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    moe.lib()

    rcfg = cfg.replace(seed=cfg.seed + rank)
    ri = synth.make_routing_inputs(rcfg)
    w1, w2 = synth.make_expert_weights(cfg, device=dev)
    x = ri.x.to(dev)
    W = ri.W.to(dev)
    b = None if ri.b is None else ri.b.to(dev)
    tdt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    cap = moe.capacity(cfg.T, cfg.E, cfg.cf)
    pk = plan_kwargs(args)
    plan = moe.MoEPlan(cfg.T, cfg.d, cfg.E, cfg.k, cfg.F, cfg.act, tdt, cap, dev, cfg.alpha, cfg.renorm, **pk)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    D = plan.disp

    def step(evs=None):
        def mark(i):
            if evs is not None:
                evs[i].record(stream)
        mark(0)
        moe.route(x, W, b, plan.k, plan.renorm, topk_idx=plan.topk_idx, topk_gate=plan.topk_gate,
                  prob_sum=plan.prob_sum, ws=plan.ws_route, n_group=plan.n_group, topk_group=plan.topk_group,
                  lse=plan.lse)
        mark(1)
        moe.dispatch(plan.topk_idx, plan.topk_gate, x, plan.E, plan.cap, out=D, ws=plan.ws_dispatch)
        mark(2)
        if plan.gather:
            moe.expert_up_gathered(x, D.row_token, D.offsets, D.kept, w1, plan.F, plan.act, plan.rows_max,
                                   h=plan.h)
        else:
            moe.expert_up(D.x_perm, D.offsets, D.kept, w1, plan.F, plan.act, plan.rows_max, h=plan.h)
        mark(3)
        moe.expert_down(plan.h, D.offsets, D.kept, w2, D.row_gate, plan.rows_max, y_perm=plan.y_perm)
        mark(4)
        f_counts = D.kept if plan.aux_post_drop else D.counts
        if world > 1:
            # token-sharded replicas: the aux loss spans all shards (one all-reduce of 2E sums)
            moe.combine(plan.y_perm, D.slot_row, y=plan.y)
            c, p, t = mdist.global_aux_inputs(f_counts, plan.prob_sum, plan.T, T_total=world * plan.T)
            moe.aux_loss(c, p, t, plan.alpha, loss=plan.loss)
        else:
            moe.combine_aux(plan.y_perm, D.slot_row, f_counts, plan.prob_sum, plan.alpha, y=plan.y, loss=plan.loss)
        if plan.z_beta is not None:
            moe.z_loss(plan.lse, plan.z_beta, loss=plan.z_loss)
        mark(5)

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)

    spin = 0
    for _ in range(args.warmup):
        flush.zero_()
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        step()
        host_s = time.perf_counter() - t0
        torch.cuda.synchronize(dev)
        spin = max(spin, enqueue_spin_cycles(host_s, time.perf_counter() - t0 - host_s))
    moe.check()
    A = int(D.offsets[plan.E].item())
    n_drop = int(D.n_dropped.item())
    counts = D.counts.cpu()
    T_used = int((D.slot_row >= 0).any(dim=1).sum().item()) if cfg.T > 0 else 0

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
    sampler = ClockSampler(local)
    barrier()
    with sampler:
        for i in range(args.steps):
            flush.zero_()
            torch.cuda._sleep(spin)   # the host enqueues the whole step before the device starts it
            step(evs[i])
        barrier()
    moe.check()
    part = {n: [] for n in ("route", "dispatch", "expert_up", "expert_down", "combine_aux", "step")}
    for e in evs:
        part["route"].append(e[0].elapsed_time(e[1]))
        part["dispatch"].append(e[1].elapsed_time(e[2]))
        part["expert_up"].append(e[2].elapsed_time(e[3]))
        part["expert_down"].append(e[3].elapsed_time(e[4]))
        part["combine_aux"].append(e[4].elapsed_time(e[5]))
        part["step"].append(e[0].elapsed_time(e[5]))
    ms_step = sum(part["step"]) / args.steps
    if world > 1:
        ms_step = mdist.max_over_ranks(ms_step, device=dev)

    # the same step as one CUDA-graph replay (removes launch gaps between the calls)
    gx = x.clone()
    gplan = moe.MoEPlan(cfg.T, cfg.d, cfg.E, cfg.k, cfg.F, cfg.act, tdt, cap, dev, cfg.alpha, cfg.renorm, **pk)
    graph = gplan.capture(gx, W, b, w1, w2)
    for _ in range(args.warmup):
        flush.zero_()
        graph.replay()
    gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier()
    for i in range(args.steps):
        flush.zero_()
        gev[i][0].record(stream)
        graph.replay()
        gev[i][1].record(stream)
    barrier()
    moe.check()
    ms_graph = sum(a.elapsed_time(c) for a, c in gev) / args.steps
    if world > 1:
        ms_graph = mdist.max_over_ranks(ms_graph, device=dev)
    del graph, gplan
    value = world * cfg.T / (ms_step / 1000.0)

    # end to end through the public API: pinned host x in, y + loss out, as a
    # three-stream pipeline (copy in / layer / copy out) over two buffer sets, so
    # step i+1's input copy and step i-1's output copy overlap step i's layer
    plans = [plan, moe.MoEPlan(cfg.T, cfg.d, cfg.E, cfg.k, cfg.F, cfg.act, tdt, cap, dev, cfg.alpha, cfg.renorm,
                               **pk)]
    x_host = ri.x.pin_memory()
    y_host = [torch.empty((cfg.T, cfg.d), dtype=tdt).pin_memory() for _ in range(2)]
    loss_host = [torch.empty(1, dtype=torch.float32).pin_memory() for _ in range(2)]
    x_dev = [x.clone() for _ in range(2)]
    graphs = [plans[i].capture(x_dev[i], W, b, w1, w2) for i in range(2)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    comp_done = [None, None]
    out_done = [None, None]

    def e2e_step(i):
        sb = i % 2
        with torch.cuda.stream(s_in):
            if comp_done[sb] is not None:
                s_in.wait_event(comp_done[sb])          # layer i-2 no longer reads x_dev[sb]
            x_dev[sb].copy_(x_host, non_blocking=True)
            in_done = torch.cuda.Event()
            in_done.record(s_in)
        stream.wait_event(in_done)
        if out_done[sb] is not None:
            stream.wait_event(out_done[sb])             # y of step i-2 has reached the host
        graphs[sb].replay()                             # the whole layer: one graph launch
        comp_done[sb] = torch.cuda.Event()
        comp_done[sb].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[sb])
            y_host[sb].copy_(plans[sb].y, non_blocking=True)
            loss_host[sb].copy_(plans[sb].loss, non_blocking=True)
            out_done[sb] = torch.cuda.Event()
            out_done[sb].record(s_out)

    for i in range(args.warmup):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    e_start.record(s_in)
    for i in range(args.warmup, args.warmup + args.steps):
        e2e_step(i)
    for ev in out_done:
        s_out.wait_event(ev)
    e_end.record(s_out)
    torch.cuda.synchronize(dev)
    barrier()
    moe.check()
    ms_e2e = e_start.elapsed_time(e_end) / args.steps
    if world > 1:
        ms_e2e = mdist.max_over_ranks(ms_e2e, device=dev)
    esz = 2 if tdt == torch.bfloat16 else 4

    hbm, bf16_peak, bf16_sust, peak_src = peaks()
    N1 = cfg.N1
    up_flops = 2.0 * A * cfg.d * N1
    down_flops = 2.0 * A * cfg.F * cfg.d
    up_ms = statistics.mean(part["expert_up"])
    down_ms = statistics.mean(part["expert_down"])
    achieved = up_flops / (up_ms * 1e-3) / 1e12
    gemm_tflops = (up_flops + down_flops) / ((up_ms + down_ms) * 1e-3) / 1e12
    traffic = traffic_from_profile(os.path.join(ROOT, "top_routing_expert_02_b300", "csrc", "ffn_tc.cuh"), cfg.name)
    if args.gather:
        traffic = None   # captured on the x_perm kernel

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": cfg.dtype, "data": "synthetic (seeded; weights random-init)",
        "config": config_dict(cfg, args),
        "clocks": sampler.summary(),
        "e2e": {"value": world * cfg.T / (ms_e2e / 1000.0), "unit": "tokens/s", "ms_per_step": ms_e2e,
                "h2d_bytes_per_step": cfg.T * cfg.d * esz, "d2h_bytes_per_step": cfg.T * cfg.d * esz + 4},
        "gpu_launches": KERNELS_PER_STEP_TOTAL(cfg, args) * args.steps,
        "roofline": {"kernel": "expert_up (tcgen05 grouped GEMM + activation)", "bound": "tensor",
                     "achieved": achieved, "peak": bf16_peak, "unit": "TFLOP/s", "frac": achieved / bf16_peak,
                     "peak_source": f"{peak_src} bf16 dense burst", "traffic": traffic,
                     "frac_of_sustained": achieved / bf16_sust,
                     "algorithmic_flops_per_launch": up_flops},
        "gemm_tflops": gemm_tflops, "gemm_frac_of_peak": gemm_tflops / bf16_peak,
        "graph_ms_per_step": ms_graph, "graph_tokens_per_s": world * cfg.T / (ms_graph / 1000.0),
        "kernel_ms": {k: statistics.mean(v) for k, v in part.items()},
        "routing": {"kept_slots": A, "dropped_slots": n_drop, "tokens_with_a_kept_slot": T_used,
                    "max_over_mean_load": float(counts.max()) / (cfg.T * cfg.k / cfg.E)},
        "roofline_hbm": hbm_rooflines(cfg, A, T_used, esz, part, hbm, peak_src, gather=args.gather),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cb, _, _ = oracle_sample(cfg, ri, w1, w2, variant=oracle_variant(args))
        line["cpu_baseline"] = cb
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def train_arm(args, cfg):
    """--train: forward + backward per step (rank 0 prints; ranks run independent batches)."""
    import top_routing_expert_02_b300 as moe
    from top_routing_expert_02_b300 import dist as mdist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    moe.lib()
    if cfg.dtype != "bf16" or args.gather:
        raise SystemExit("--train runs bf16 layers with a materialised x_perm")
    rcfg = cfg.replace(seed=cfg.seed + rank)
    ri = synth.make_routing_inputs(rcfg)
    w1, w2 = synth.make_expert_weights(cfg, device=dev)
    x, W = ri.x.to(dev), ri.W.to(dev)
    b = None if ri.b is None else ri.b.to(dev)
    g = torch.Generator().manual_seed(777 + rank)
    dy_host = torch.randn(cfg.T, cfg.d, generator=g).to(torch.bfloat16)
    dy = dy_host.to(dev)
    cap = moe.capacity(cfg.T, cfg.E, cfg.cf)
    plan = moe.MoEPlan(cfg.T, cfg.d, cfg.E, cfg.k, cfg.F, cfg.act, torch.bfloat16, cap, dev, cfg.alpha, cfg.renorm,
                       **plan_kwargs(args))
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    phases = ["forward", "combine_bwd", "data_grad_gemms", "wgrad_dw2", "wgrad_dw1", "router_and_dx"]

    def step(evs=None):
        def mark(name):
            if evs is not None:
                evs[name].record(stream)
        mark("start")
        plan.run(x, W, b, w1, w2)
        mark("forward")
        plan.backward(x, W, w1, w2, dy, mark=mark)

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)

    spin = 0
    for _ in range(args.warmup):
        flush.zero_()
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        step()
        host_s = time.perf_counter() - t0
        torch.cuda.synchronize(dev)
        spin = max(spin, enqueue_spin_cycles(host_s, time.perf_counter() - t0 - host_s))
    moe.check()
    A = int(plan.disp.offsets[plan.E].item())
    evs = [{n: torch.cuda.Event(enable_timing=True) for n in ["start"] + phases} for _ in range(args.steps)]
    sampler = ClockSampler(local)
    barrier()
    with sampler:
        for i in range(args.steps):
            flush.zero_()
            torch.cuda._sleep(spin)   # the host enqueues the whole step before the device starts it
            step(evs[i])
        barrier()
    moe.check()
    part = {n: [] for n in phases + ["step"]}
    for e in evs:
        prev = "start"
        for n in phases:
            part[n].append(e[prev].elapsed_time(e[n]))
            prev = n
        part["step"].append(e["start"].elapsed_time(e[phases[-1]]))
    ms_step = statistics.mean(part["step"])
    if world > 1:
        ms_step = mdist.max_over_ranks(ms_step, device=dev)

    # the same step as one CUDA-graph replay
    graph = plan.capture(x, W, b, w1, w2, dy=dy)
    for _ in range(args.warmup):
        flush.zero_()
        graph.replay()
    gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier()
    for i in range(args.steps):
        flush.zero_()
        gev[i][0].record(stream)
        graph.replay()
        gev[i][1].record(stream)
    barrier()
    moe.check()
    ms_graph = sum(a.elapsed_time(c) for a, c in gev) / args.steps
    if world > 1:
        ms_graph = mdist.max_over_ranks(ms_graph, device=dev)
    del graph

    # end to end: x and dy from pinned host memory, dx and the loss back; the
    # weight gradients stay on the device where an optimiser would use them.  A
    # three-stream pipeline (copy in / layer / copy out) over two plans, so step
    # i+1's input copies and step i-1's output copies overlap step i's layer.
    plans = [plan, moe.MoEPlan(cfg.T, cfg.d, cfg.E, cfg.k, cfg.F, cfg.act, torch.bfloat16, cap, dev, cfg.alpha,
                               cfg.renorm, **plan_kwargs(args))]
    x_dev, dy_dev = [x, x.clone()], [dy, dy.clone()]
    graphs = [plans[i].capture(x_dev[i], W, b, w1, w2, dy=dy_dev[i]) for i in range(2)]
    x_host, dyh = ri.x.pin_memory(), dy_host.pin_memory()
    dx_host = [torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    loss_host = [torch.empty(1, dtype=torch.float32).pin_memory() for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    comp_done = [None, None]
    out_done = [None, None]

    def e2e_step(i):
        sb = i % 2
        with torch.cuda.stream(s_in):
            if comp_done[sb] is not None:
                s_in.wait_event(comp_done[sb])          # step i-2 no longer reads x_dev[sb], dy_dev[sb]
            x_dev[sb].copy_(x_host, non_blocking=True)
            dy_dev[sb].copy_(dyh, non_blocking=True)
            in_done = torch.cuda.Event()
            in_done.record(s_in)
        stream.wait_event(in_done)
        if out_done[sb] is not None:
            stream.wait_event(out_done[sb])             # dx of step i-2 has reached the host
        graphs[sb].replay()                             # forward + backward: one graph launch
        comp_done[sb] = torch.cuda.Event()
        comp_done[sb].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[sb])
            dx_host[sb].copy_(plans[sb]._bwd["dx"][:cfg.T], non_blocking=True)
            loss_host[sb].copy_(plans[sb].loss, non_blocking=True)
            out_done[sb] = torch.cuda.Event()
            out_done[sb].record(s_out)

    for i in range(args.warmup):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    barrier()
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(s_in)
    for i in range(args.warmup, args.warmup + args.steps):
        e2e_step(i)
    for ev in out_done:
        s_out.wait_event(ev)
    s1.record(s_out)
    torch.cuda.synchronize(dev)
    barrier()
    moe.check()
    ms_e2e = s0.elapsed_time(s1) / args.steps
    if world > 1:
        ms_e2e = mdist.max_over_ranks(ms_e2e, device=dev)
    del graphs

    hbm, bf16_peak, bf16_sust, peak_src = peaks()
    dw1_flops = 2.0 * A * cfg.N1 * cfg.d
    dw1_ms = statistics.mean(part["wgrad_dw1"])
    achieved = dw1_flops / (dw1_ms * 1e-3) / 1e12
    gemm_flops = 2.0 * A * cfg.d * cfg.N1 * 3 + 2.0 * A * cfg.F * cfg.d * 3   # forward 2 + backward 4 GEMMs
    line = {
        "metric": "MoE-layer fwd+bwd tokens/s on 1 B300", "value": world * cfg.T / (ms_step / 1000.0),
        "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": cfg.dtype,
        "data": "synthetic (seeded; weights random-init; seeded upstream gradient)",
        "config": config_dict(cfg, args), "clocks": sampler.summary(),
        "e2e": {"value": world * cfg.T / (ms_e2e / 1000.0), "unit": "tokens/s", "ms_per_step": ms_e2e,
                "h2d_bytes_per_step": 2 * cfg.T * cfg.d * 2, "d2h_bytes_per_step": cfg.T * cfg.d * 2 + 4},
        "gpu_launches": KERNELS_PER_STEP_TOTAL(cfg, args) * args.steps,
        "roofline": {"kernel": "expert_wgrad dw1 (tcgen05 grouped GEMM, per-expert K, fp32 out)", "bound": "tensor",
                     "achieved": achieved, "peak": bf16_peak, "unit": "TFLOP/s", "frac": achieved / bf16_peak,
                     "peak_source": f"{peak_src} bf16 dense burst", "traffic": None,
                     "frac_of_sustained": achieved / bf16_sust, "algorithmic_flops_per_launch": dw1_flops},
        "gemm_tflops_step": gemm_flops / (ms_step * 1e-3) / 1e12,
        "graph_ms_per_step": ms_graph, "graph_tokens_per_s": world * cfg.T / (ms_graph / 1000.0),
        "kernel_ms": {k: statistics.mean(v) for k, v in part.items()},
        "routing": {"kept_slots": A},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = oracle_sample_train(cfg, ri, w1, w2, dy_host, oracle_variant(args))
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def oracle_sample_train(cfg, ri, w1, w2, dy, variant, budget_s: float = 15.0):
    """The CPU oracles (forward + backward) on the first S tokens."""
    import oracle
    from oracle import backward as ob
    w1h, w2h = w1.cpu(), w2.cpu()
    bvar = dict(n_group=variant["n_group"], topk_group=variant["topk_group"], z_beta=variant["z_beta"],
                aux_post_drop=variant["aux_post_drop"])

    def run(S):
        sub, dys = ri.x[:S].contiguous(), dy[:S].contiguous()
        cap = oracle.capacity(S, cfg.E, cfg.cf)
        t0 = time.perf_counter()
        oracle.forward(sub, ri.W, ri.b, w1h, w2h, k=cfg.k, cap=cap, act=cfg.act, renorm=cfg.renorm,
                       alpha=cfg.alpha, **variant)
        ob.backward(sub, ri.W, ri.b, w1h, w2h, dys, k=cfg.k, cap=cap, act=cfg.act, renorm=cfg.renorm,
                    alpha=cfg.alpha, **bvar)
        return time.perf_counter() - t0

    S = min(cfg.T, 8)
    t = run(S)
    if t < budget_s / 4 and S < cfg.T:
        S = int(min(cfg.T, max(S + 1, S * (budget_s / max(t, 1e-3)))))
        t = run(S)
    return {"value": S / t, "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"first {S} of {cfg.T} tokens, forward + backward in fp64 (capacity for {S} tokens), "
                      f"{t:.1f} s"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="e128_top8_T32768", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--n-group", type=int, default=1, help="group-limited routing: contiguous expert groups")
    ap.add_argument("--topk-group", type=int, default=1, help="groups kept per token")
    ap.add_argument("--z-beta", type=float, default=None, help="router z-loss coefficient (off when absent)")
    ap.add_argument("--aux-post-drop", action="store_true", help="aux loss f_i from kept slots")
    ap.add_argument("--gather", action="store_true", help="up-projection gathers x rows (bf16 only)")
    ap.add_argument("--train", action="store_true", help="time forward + backward")
    ap.add_argument("--grad-dtype", default="f32", choices=["f32", "bf16"], help="expert weight gradients (--train)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)      # at least three untimed warm-up steps
    args.steps = max(args.steps, 1)
    cfg = synth.workload(args.workload)
    if args.impl == "reference":
        reference_arm(args, cfg)
    elif args.train:
        train_arm(args, cfg)
    else:
        our_arm(args, cfg)


if __name__ == "__main__":
    main()
