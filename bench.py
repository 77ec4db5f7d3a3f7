"""Benchmark of the routed MoE expert-layer forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config NAME] [--no-cpu-baseline]

One step = one full pass of the layer (route -> sort -> gather -> FC1+SwiGLU ->
FC2 -> finalize) over one batch of seeded synthetic input, launched through the
prepared-launch C ABI.  The default workload is "prefill_many_fine"
(T=8192 tokens, hidden 7168, intermediate 2048, 256 experts, top-8, routing
from fp32 logits with a Zipf(1.2) per-expert bias: the largest configuration,
5.77 TFLOP per step).  Under torchrun every rank runs its own replica of the workload
(tokens are independent; there is no data-path collective), so the scaling is
weak and `value` is the tokens of all ranks divided by the slowest rank's time.

Rank 0 prints one JSON line.  `--impl reference` times the CPU oracle (the only
other place this script runs it) on a bounded token sample of the same
workload per step.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused-MoE tokens/s and TFLOP/s (or GB/s) at 1 GB300; % of BF16/HBM roofline"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except Exception:
        return dict(PEAKS_FALLBACK), "fallback"


# ------------------------------------------------------------------ clocks --

class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: str):
        self.rows = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-i", index,
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.rows.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self, t0: float, t1: float):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        inside = [r for ts, r in self.rows if t0 <= ts <= t1]
        note = None
        if not inside:
            # timed region shorter than one sampling period: nearest samples
            inside = [r for ts, r in self.rows if t0 - 0.5 <= ts <= t1 + 0.5] or [r for _, r in self.rows]
            note = "timed region shorter than the 200 ms sampling period; nearest samples used"

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in inside if num(r[1]) is not None]
        smax = [num(r[2]) for r in inside if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i in range(4) if r[5 + i].lower().startswith("active")})
        out = {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
               "reasons": reasons, "samples": len(inside)}
        if note:
            out["note"] = note
        return out


# ------------------------------------------------------------ distributed --

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, value: float) -> float:
    if world == 1:
        return value
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if torch.cuda.is_available() else torch.device("cpu")
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# -------------------------------------------------------------- workload --

def layer_flops(M: int, H: int, I: int) -> float:
    return 2.0 * M * (H * 2 * I + I * H)


def layer_bytes(wl, ids: np.ndarray, wbytes_per_elem: float = 2.0) -> float:
    """Algorithmic bytes: weights of non-empty local experts, x read, out
    written, routing inputs read."""
    L = wl.num_local
    local = ids[(ids >= wl.local_offset) & (ids < wl.local_offset + L)] - wl.local_offset
    active = len(np.unique(local))
    wbytes = active * (2 * wl.I * wl.H + wl.H * wl.I) * wbytes_per_elem
    route = wl.T * wl.E * 4.0 if wl.mode == "logits" else wl.T * wl.top_k * 8.0
    return wbytes + wl.T * wl.H * 2.0 * 2 + route, active


def oracle_sample_rate(wl, ids, w, n_tok: int, seed: int, threads: int, host_w=None):
    """Time the CPU oracle on n_tok sampled tokens (route + layer for them).
    Returns (tokens/s, seconds, tokens)."""
    import oracle
    from mixture_experts_expert_router_gb300 import workloads as W
    rng = np.random.default_rng(seed)
    tokens = np.sort(rng.choice(wl.T, size=min(n_tok, wl.T), replace=False)).astype(np.int32)
    x = W.bf16_bits(wl.x)
    w1, w2 = host_w[:2]
    t0 = time.perf_counter()
    if wl.mode == "logits":
        lg = wl.logits.cpu().numpy()[tokens]
        ids_s, w_s = oracle.route(lg, wl.top_k, nthreads=threads)
        ids_full = np.zeros((wl.T, wl.top_k), np.int32)
        w_full = np.zeros((wl.T, wl.top_k), np.float32)
        ids_full[tokens], w_full[tokens] = ids_s, w_s
    else:
        ids_full, w_full = ids, w
    if len(host_w) > 2:  # E4M3 family: (w1q, w2q, s1, s2, a1, a2)
        oracle.moe_tokens_fp8(x, ids_full, w_full, *host_w, wl.E, tokens=tokens, local_offset=wl.local_offset,
                              num_local=wl.num_local, nthreads=threads)
    else:
        oracle.moe_tokens(x, ids_full, w_full, w1, w2, wl.E, tokens=tokens, local_offset=wl.local_offset,
                          num_local=wl.num_local, nthreads=threads)
    dt = time.perf_counter() - t0
    return len(tokens) / dt, dt, len(tokens)


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def calibrated_tokens(wl, ids, w, threads, host_w, budget_s: float):
    rate, _, _ = oracle_sample_rate(wl, ids, w, min(max(8, 2 * threads), wl.T), 12345, threads, host_w)
    return int(max(1, min(wl.T, rate * budget_s)))


# ------------------------------------------------------------------- main --

def run_reference(args, world, rank):
    if rank != 0:
        return 0
    import oracle
    from mixture_experts_expert_router_gb300 import workloads as W
    oracle.build()
    # the same seeded weight banks as the other arm (drawn where that arm draws
    # them, then read back for the oracle); only the random draw uses the GPU
    wdev = torch.device("cuda", 0) if torch.cuda.is_available() else "cpu"
    wl = make_workload(args, 0, wdev)
    threads = host_cores()
    ids = wl.topk_ids.numpy() if wl.topk_ids is not None else None
    w = wl.topk_w.numpy() if wl.topk_w is not None else None
    host_w = (W.bf16_bits(wl.w1), W.bf16_bits(wl.w2))
    steps, warm = args.steps, args.warmup
    per_step = max(0.5, args.reference_budget / max(1, steps + warm))
    n_tok = calibrated_tokens(wl, ids, w, threads, host_w, per_step)
    for i in range(warm):
        oracle_sample_rate(wl, ids, w, n_tok, 100 + i, threads, host_w)
    total_tok, total_t = 0, 0.0
    for i in range(steps):
        _, dt, n = oracle_sample_rate(wl, ids, w, n_tok, 1000 + i, threads, host_w)
        total_tok += n
        total_t += dt
    value = total_tok / total_t
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": steps, "warmup": warm, "ms_per_step": 1000.0 * total_t / steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded)",
        "config": config_dict(wl, world, weight_banks(wl)),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": f"{n_tok} random tokens of the {wl.T}-token batch per step "
                                   f"(routing + FC1/SwiGLU + FC2 + combine for those tokens)"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def make_workload(args, rank, weights_device):
    from mixture_experts_expert_router_gb300 import workloads as W
    if args.shape:
        T, H, I, E, k = (int(v) for v in args.shape.split(","))
        wl = W.make_moe(T=T, H=H, I=I, E=E, top_k=k, mode="logits", seed=args.seed + rank, device="cpu",
                        weights_device=weights_device, bias=f"zipf{args.zipf}" if args.zipf else None)
        wl.name = f"custom_T{T}_H{H}_I{I}_E{E}_k{k}" + (f"_zipf{args.zipf}" if args.zipf else "")
        return wl
    return W.make_moe(args.config, seed=args.seed + rank, device="cpu", weights_device=weights_device)


def timed_steps(fn, steps, stream):
    """Device time (ms) of `steps` back-to-back calls of fn, by CUDA events
    on `stream`."""
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1)


def recorded_traffic(workload: str, kernel: str):
    """DRAM bytes per stage launch (read + write, summed over the stage's
    kernels) recorded from an ncu capture in profiles/traffic.json, or None
    when none exists or a kernel source file changed since the capture (their
    sha256 prefixes are stored beside it)."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)
        for entry in rec.get("captures", []):
            if entry.get("workload") != workload or entry.get("kernel") != kernel:
                continue
            for src, want in zip(entry["sources"], entry["sources_sha16"]):
                sha = hashlib.sha256(open(os.path.join(ROOT, src), "rb").read()).hexdigest()[:16]
                if sha != want:
                    return None
            return int(entry["bytes"])
    except (OSError, ValueError, KeyError):
        pass
    return None


# A timed region shorter than this runs at burst clocks; longer ones settle
# under the power cap (the two measured bf16 peaks).
SUSTAINED_AFTER_S = 1.0


def roofline_entry(decode_path, fc1_s, F_fc1, B_fc1, peaks, peak_src, region_s, traffic, B_layer=None):
    """Dominant kernel (FC1 + SwiGLU): tensor-bound on the grouped path,
    HBM-bound (weight streaming) on the decode path.  With B_layer the decode
    chain runs as one kernel (FC1, FC2 and the combine), timed whole against
    the layer's algorithmic bytes.  The bf16 peak is the burst one when the
    kernel's timed region (region_s) is shorter than SUSTAINED_AFTER_S, else
    the sustained one; the fraction against the other is reported beside it."""
    if fc1_s <= 0:
        return None
    peak_b = float(peaks["hbm_gbs"])
    if B_layer is not None:
        gbs = B_layer / fc1_s / 1e9
        return {"kernel": "decode chain in one launch (FC1 + SwiGLU, FC2, combine)", "bound": "hbm",
                "achieved": gbs, "peak": peak_b, "unit": "GB/s", "frac": gbs / peak_b, "traffic": traffic,
                "peak_kind": f"{peak_src} HBM copy bandwidth", "bytes_per_launch": B_layer}
    if decode_path:
        gbs = B_fc1 / fc1_s / 1e9
        return {"kernel": "fc1_swiglu (decode form)", "bound": "hbm", "achieved": gbs, "peak": peak_b,
                "unit": "GB/s", "frac": gbs / peak_b, "traffic": traffic,
                "peak_kind": f"{peak_src} HBM copy bandwidth", "bytes_per_launch": B_fc1}
    burst = float(peaks["bf16_tflops"])
    sustained = float(peaks.get("bf16_tflops_sustained", burst))
    long_region = region_s >= SUSTAINED_AFTER_S
    peak_t = sustained if long_region else burst
    tf = F_fc1 / fc1_s / 1e12
    return {"kernel": "fc1_swiglu", "bound": "tensor", "achieved": tf, "peak": peak_t, "unit": "TFLOP/s",
            "frac": tf / peak_t, "traffic": traffic,
            "peak_kind": (f"{peak_src} {'sustained' if long_region else 'burst'} bf16 (the kernel's timed "
                          f"region lasted {region_s:.2f} s)"),
            "frac_vs_burst": tf / burst, "frac_vs_sustained": tf / sustained, "flops_per_launch": F_fc1}


L2_NOMINAL = 128 << 20  # GB300's L2, rounded
MAX_BANKS = 32


def weight_banks(wl) -> int:
    """Copies of the expert banks the steps rotate over (one per layer of a
    model), so that the active weights of all copies exceed three times the
    L2: every step streams its own weights from HBM.  1 when one step's
    active weights already do (every routed expert distinct)."""
    experts = min(wl.num_local, wl.T * wl.top_k)
    active = experts * 3.0 * wl.H * wl.I * 2
    return 1 if active >= 3 * L2_NOMINAL else min(MAX_BANKS, int(np.ceil(3 * L2_NOMINAL / active)))


def config_dict(wl, world, banks=1):
    experts = min(wl.num_local, wl.T * wl.top_k)
    rotated = banks * experts * 3.0 * wl.H * wl.I * 2
    return {"workload": wl.name, "T": wl.T, "H": wl.H, "I": wl.I, "E": wl.E, "top_k": wl.top_k,
            "routing": wl.mode, "global_batch": wl.T * world,
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "l2": ("inputs larger than L2: the expert weights stream from HBM every step" if banks == 1 else
                   f"inputs larger than L2: consecutive steps rotate over {banks} copies of the expert "
                   f"banks (one per layer), whose active weights together exceed three times the L2, "
                   f"so every step streams its weights from HBM" if rotated >= 3 * L2_NOMINAL else
                   f"small workload: the steps rotate over {banks} copies of the expert banks, which "
                   f"still fit in L2")}


def run_ours(args, world, rank, local):
    import mixture_experts_expert_router_gb300 as moe
    from mixture_experts_expert_router_gb300 import workloads as W
    moe.library()
    dev = torch.device("cuda", local)
    wl = make_workload(args, rank, dev)
    x = wl.x.to(dev)
    logits = wl.logits.to(dev) if wl.logits is not None else None
    tids = wl.topk_ids.to(dev) if wl.topk_ids is not None else None
    tw = wl.topk_w.to(dev) if wl.topk_w is not None else None
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    opts = dict(decode_chain=True if args.decode_chain else (False if args.decode_separate else None),
                one_cta_gemm=args.one_cta_gemm, fused_gather=args.fused_gather,
                decode_one_launch=args.decode_one_launch, no_tail_tiles=args.no_tail_tiles,
                small_group_kernel={"auto": None, "on": True, "off": False}[args.small_group_kernel])
    # one plan per copy of the expert banks; the steps rotate over them
    banks = weight_banks(wl)
    fw = None
    if args.e4m3:  # the fp8 per-tensor family: E4M3 codes with per-expert scales
        fw = W.make_fp8_weights(wl.num_local, wl.H, wl.I, seed=args.seed + rank, device=dev)
        opts["e4m3"] = dict(w1_scale=fw.s1, w2_scale=fw.s2, x_scale=fw.a1, h_scale=fw.a2)
        base1, base2 = fw.w1q, fw.w2q
        wl.w1, wl.w2 = None, None  # the bf16 banks are not used
        torch.cuda.empty_cache()
    else:
        base1, base2 = wl.w1, wl.w2
    w1s = [base1] + [base1.clone() for _ in range(banks - 1)]
    w2s = [base2] + [base2.clone() for _ in range(banks - 1)]
    plans, plans_t = [], []
    for b in range(banks):
        p_b = moe.MoEPlan(x, w1s[b], w2s[b], wl.E, wl.top_k, logits=logits, topk_ids=tids, topk_w=tw,
                          local_offset=wl.local_offset, status=status,
                          out=plans[0].out if plans else None, **opts)
        # a second plan on the same buffers records CUDA events around every stage
        plans_t.append(moe.MoEPlan(x, w1s[b], w2s[b], wl.E, wl.top_k, logits=logits, topk_ids=tids,
                                   topk_w=tw, local_offset=wl.local_offset, status=status, out=p_b.out,
                                   workspace=p_b.workspace, stage_timing=True, **opts))
        plans.append(p_b)
    plan, plan_t = plans[0], plans_t[0]
    kernels = plan.kernels_per_launch()
    stream = torch.cuda.current_stream(dev)

    # routed rows of this batch (for FLOP and byte counts)
    plan.launch()
    torch.cuda.synchronize()
    R = wl.T * wl.top_k
    if wl.mode == "logits":  # the routed ids the plan left in its workspace
        off = plan.buffers()["topk_ids"] - plan.workspace.data_ptr()
        ids_np = plan.workspace[off:off + R * 4].view(torch.int32).cpu().numpy()
    else:
        ids_np = wl.topk_ids.numpy().ravel()
    L = wl.num_local
    M = int(np.sum((ids_np >= wl.local_offset) & (ids_np < wl.local_offset + L)))
    F = layer_flops(M, wl.H, wl.I)
    F_fc1 = 2.0 * M * wl.H * 2 * wl.I
    B, active = layer_bytes(wl, ids_np, 1.0 if fw is not None else 2.0)

    # one step = one replay of the prepared launch captured in a CUDA graph
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        for _ in range(3):
            for p_b in plans:
                p_b.launch()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    graphs = []
    if not args.no_graph:
        for p_b in plans:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                p_b.launch()
            graphs.append(g)
    calls = [g.replay for g in graphs] if graphs else [p_b.launch for p_b in plans]
    graph = graphs[0] if graphs else None

    def rotating(fns):
        k = [0]

        def call():
            fns[k[0] % len(fns)]()
            k[0] += 1
        return call
    step = rotating(calls)

    dev_index = str(local)
    try:
        uuid = torch.cuda.get_device_properties(dev).uuid
        dev_index = "GPU-" + str(uuid) if uuid is not None else dev_index
    except Exception:
        pass
    clocks = ClockSampler(dev_index)
    time.sleep(0.3)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    ms_local = timed_steps(step, args.steps, stream)
    t_wall1 = time.time()
    barrier(world)

    # stage pass: the same steps with CUDA events between the stages (no PDL
    # overlap between them); gives each kernel's mean duration
    for _ in range(3):
        for p_b in plans_t:
            p_b.launch()
    torch.cuda.synchronize()
    for p_b in plans_t:
        p_b.stage_reset()
    n_stage_steps = min(args.steps, 200)
    stage_pass_total_ms = timed_steps(rotating([p_b.launch for p_b in plans_t]), n_stage_steps, stream)
    stage_pass_ms = stage_pass_total_ms / n_stage_steps
    stage_ms, n_timed = {}, 0
    for p_b in plans_t:
        ms_b, n_b = p_b.stage_times()
        n_timed += n_b
        for key, v in ms_b.items():
            stage_ms[key] = stage_ms.get(key, 0.0) + v
    time.sleep(0.25)

    # end to end: pinned host inputs in, result out, every step
    x_h = wl.x.pin_memory()
    lg_h = wl.logits.pin_memory() if logits is not None else None
    ids_h = wl.topk_ids.pin_memory() if tids is not None else None
    w_h = wl.topk_w.pin_memory() if tw is not None else None
    out_h = torch.empty(plan.out.shape, dtype=plan.out.dtype).pin_memory()
    h2d = x_h.numel() * 2 + (lg_h.numel() * 4 if lg_h is not None else 0) + \
        (ids_h.numel() * 4 + w_h.numel() * 4 if ids_h is not None else 0)
    d2h = out_h.numel() * 2

    decode_path = plan.buffers()["path"] == moe.PATH_DECODE

    def e2e_serial():
        # decode steps (tens of microseconds, a few KB copied): one stream
        x.copy_(x_h, non_blocking=True)
        if lg_h is not None:
            logits.copy_(lg_h, non_blocking=True)
        if ids_h is not None:
            tids.copy_(ids_h, non_blocking=True)
            tw.copy_(w_h, non_blocking=True)
        e2e_launch()
        out_h.copy_(plan.out, non_blocking=True)
    e2e_launch = rotating([p_b.launch for p_b in plans])

    # Grouped path: two sets of device buffers, each with its plans, so that
    # the copies of one step (inputs in on one stream, the result out on
    # another) overlap the kernels of its neighbours, as a serving loop would
    # pipeline them.
    def like(t):
        return None if t is None else torch.empty_like(t)
    x2, logits2, tids2, tw2 = like(x), like(logits), like(tids), like(tw)
    plans2 = []
    for b in range(0 if decode_path else banks):
        plans2.append(moe.MoEPlan(x2, w1s[b], w2s[b], wl.E, wl.top_k, logits=logits2, topk_ids=tids2, topk_w=tw2,
                                  local_offset=wl.local_offset, status=status,
                                  out=plans2[0].out if plans2 else None, **opts))
    sets = [(x, logits, tids, tw, plans, out_h), (x2, logits2, tids2, tw2, plans2,
                                                  out_h if decode_path else
                                                  torch.empty(plan.out.shape, dtype=plan.out.dtype).pin_memory())]
    copy_in, copy_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_free = [torch.cuda.Event() for _ in range(2)]
    e2e_n = [0]

    def e2e_step():
        n = e2e_n[0]
        e2e_n[0] += 1
        b = n % 2
        xb, lgb, idb, twb, pls, outb_h = sets[b]
        if n >= 2:
            copy_in.wait_event(ev_free[b])  # step n - 2 has read these inputs and written its result out
        with torch.cuda.stream(copy_in):
            xb.copy_(x_h, non_blocking=True)
            if lg_h is not None:
                lgb.copy_(lg_h, non_blocking=True)
            if ids_h is not None:
                idb.copy_(ids_h, non_blocking=True)
                twb.copy_(w_h, non_blocking=True)
            ev_in[b].record(copy_in)
        stream.wait_event(ev_in[b])
        pls[(n // 2) % len(pls)].launch(stream)
        ev_done[b].record(stream)
        copy_out.wait_event(ev_done[b])
        with torch.cuda.stream(copy_out):
            outb_h.copy_(pls[0].out, non_blocking=True)
            ev_free[b].record(copy_out)

    run = e2e_serial if decode_path else e2e_step
    for _ in range(max(2, args.warmup)):
        run()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    if decode_path:
        ms_e2e_local = timed_steps(e2e_serial, args.steps, stream)
    else:
        e_a, e_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e_a.record(copy_in)
        for _ in range(args.steps):
            e2e_step()
        copy_out.wait_stream(stream)
        e_b.record(copy_out)
        torch.cuda.synchronize()
        ms_e2e_local = e_a.elapsed_time(e_b)
    barrier(world)
    clocks.stop()
    st = int(status.item())

    ms = max_over_ranks(world, ms_local)
    ms_e2e = max_over_ranks(world, ms_e2e_local)
    tokens_all = wl.T * world * args.steps
    value = tokens_all / (ms / 1000.0)
    e2e_value = tokens_all / (ms_e2e / 1000.0)
    step_s = ms / 1000.0 / args.steps

    peaks, peak_src = load_peaks()
    fc1_s = stage_ms.get("fc1_swiglu", 0.0) / 1000.0 / max(1, n_timed)
    peak_b = float(peaks.get("hbm_gbs", PEAKS_FALLBACK["hbm_gbs"]))
    # E4M3 MMAs: the nominal fp8 / bf16 ratio (4.5 / 2.25 PFLOP/s) times the measured bf16 peaks
    tmul = 2.0 if fw is not None else 1.0
    if fw is not None:
        peaks = dict(peaks, bf16_tflops=tmul * float(peaks["bf16_tflops"]),
                     bf16_tflops_sustained=tmul * float(peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])))
    roofline_t = max(F / (float(peaks["bf16_tflops"]) * 1e12), B / (peak_b * 1e9))
    # FC1's algorithmic bytes: W1 of the active experts, its gathered input rows, h written
    esz = 1.0 if fw is not None else 2.0
    B_fc1 = active * 2.0 * wl.I * wl.H * esz + M * wl.H * esz + M * wl.I * esz
    decode_path = plan.buffers()["path"] == moe.PATH_DECODE
    # the captures are of the default bf16 plan's kernels; other kernel choices have none recorded
    default_kernels = not (args.e4m3 or args.one_cta_gemm or args.no_tail_tiles or args.fused_gather
                           or args.small_group_kernel != "auto")
    traffic = recorded_traffic(wl.name, "fc1_swiglu") if (default_kernels and not decode_path) else None
    # the decode chain in one launch: one kernel (plus the router with logits)
    one_kernel = decode_path and kernels == (1 if logits is None else 2)

    if rank != 0:
        return 0
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3" if fw is not None else "bf16",
        "data": "synthetic (seeded)",
        "config": dict(config_dict(wl, world, banks), **({"weights": "e4m3 per-tensor (fp8 family); tensor peak "
                                                         "= 2 x the measured bf16 peak"} if fw is not None else {})),
        "tflops": F * world / step_s / 1e12,
        "hbm_gbs": B * world / step_s / 1e9,
        "roofline_step": {"time_ms": roofline_t * 1000.0, "frac": roofline_t / step_s,
                          "flops": F, "bytes": B, "active_experts": active,
                          "peaks": f"{peak_src}: {peaks['bf16_tflops']} TFLOP/s bf16, {peaks['hbm_gbs']} GB/s"},
        "roofline": roofline_entry(decode_path, fc1_s, F_fc1, B_fc1, peaks, peak_src, stage_pass_total_ms / 1000.0,
                                   traffic, B if one_kernel else None),
        "stage_ms": {k: v / max(1, n_timed) for k, v in stage_ms.items()},
        "stage_pass_ms_per_step": stage_pass_ms,
        "timing": ("CUDA-graph replay of the prepared launch" if graph is not None else "prepared launch")
                  + "; dominant-kernel time from a second pass with CUDA events around each stage",
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "timing": "every step copies its inputs in from pinned host memory and its output back; " +
                          ("one stream" if decode_path else
                           "two sets of device buffers let one step's copies overlap its neighbours' kernels")},
        "gpu_launches": kernels * args.steps,
        "kernels_per_step": kernels,
        "clocks": clocks.summary(t_wall0, t_wall1),
        "device_status": st,
    }
    if world == 1 and not args.no_cpu_baseline:
        threads = host_cores()
        host_w = ((fw.w1q.cpu().numpy(), fw.w2q.cpu().numpy(), fw.s1.cpu().numpy(), fw.s2.cpu().numpy(), fw.a1, fw.a2)
                  if fw is not None else (W.bf16_bits(wl.w1), W.bf16_bits(wl.w2)))
        ids2 = wl.topk_ids.numpy() if wl.topk_ids is not None else None
        w2 = wl.topk_w.numpy() if wl.topk_w is not None else None
        n_tok = calibrated_tokens(wl, ids2, w2, threads, host_w, args.cpu_budget)
        rate, dt, n = oracle_sample_rate(wl, ids2, w2, n_tok, 7, threads, host_w)
        line["cpu_baseline"] = {"value": rate, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                                "sample": f"{n} random tokens of the {wl.T}-token batch "
                                          f"({dt:.1f} s wall on {threads} threads)"}
    print(json.dumps(line), flush=True)
    return 0


def run_grouped_gemm(args, world, rank, local):
    """One step = one ragged grouped GEMM forward (Y[g] = X[g] W[g]^T, bf16),
    sum_m=16384 rows over 64 Dirichlet(0.3)-sized groups, K=4096, N=1536."""
    import mixture_experts_expert_router_gb300 as moe
    from mixture_experts_expert_router_gb300 import workloads as W
    moe.library()
    dev = torch.device("cuda", local)
    d = W.make_grouped_gemm(seed=args.seed + rank, device="cpu", weights_device=dev)
    X, Wt, offs = d["X"].to(dev), d["W"], d["offs"].to(dev)
    Y = torch.empty((d["sum_m"], d["N"]), dtype=torch.bfloat16, device=dev)
    sizes = d["sizes"]
    active = int((sizes > 0).sum())
    F = 2.0 * d["sum_m"] * d["K"] * d["N"]
    B = active * d["N"] * d["K"] * 2.0 + d["sum_m"] * d["K"] * 2.0 + d["sum_m"] * d["N"] * 2.0
    stream = torch.cuda.current_stream(dev)
    counters = torch.empty(moe.GROUPED_GEMM_COUNTERS, dtype=torch.int32, device=dev)
    gopts = dict(no_tail_tiles=args.no_tail_tiles, counters=counters,
                 small_group_kernel={"auto": None, "on": True, "off": False}[args.small_group_kernel])
    # the CTA-pair kernel, and the small-group kernel beside it where the call runs it (on request)
    with_small = bool(gopts["small_group_kernel"]) and not args.no_tail_tiles and d["N"] % 256 == 0
    kernels_per_call = 2 if with_small else 1
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        for _ in range(3):
            moe.grouped_gemm_fwd(X, Wt, offs, Y, **gopts)
    stream.wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        moe.grouped_gemm_fwd(X, Wt, offs, Y, **gopts)
    clocks = ClockSampler(str(local))
    time.sleep(0.3)
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    e0.record(stream)
    for _ in range(args.steps):
        graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    barrier(world)
    ms = max_over_ranks(world, e0.elapsed_time(e1))
    # end to end: X in from pinned host memory, Y back, every step; two sets of
    # device buffers let one call's copies (X in on one stream, Y out on
    # another) overlap its neighbours' kernels
    X_h = d["X"].pin_memory()
    bufs = [(X, Y, torch.empty(Y.shape, dtype=Y.dtype).pin_memory()),
            (torch.empty_like(X), torch.empty_like(Y), torch.empty(Y.shape, dtype=Y.dtype).pin_memory())]
    cnts = [counters, torch.empty_like(counters)]
    copy_in, copy_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_free = [torch.cuda.Event() for _ in range(2)]

    def e2e_call(n):
        b = n % 2
        Xb, Yb, Yb_h = bufs[b]
        if n >= 2:
            copy_in.wait_event(ev_free[b])
        with torch.cuda.stream(copy_in):
            Xb.copy_(X_h, non_blocking=True)
            ev_in[b].record(copy_in)
        stream.wait_event(ev_in[b])
        moe.grouped_gemm_fwd(Xb, Wt, offs, Yb, **dict(gopts, counters=cnts[b]))
        ev_done[b].record(stream)
        copy_out.wait_event(ev_done[b])
        with torch.cuda.stream(copy_out):
            Yb_h.copy_(Yb, non_blocking=True)
            ev_free[b].record(copy_out)

    n_call = 0
    for _ in range(max(2, args.warmup)):
        e2e_call(n_call)
        n_call += 1
    torch.cuda.synchronize()
    e0.record(copy_in)
    for _ in range(args.steps):
        e2e_call(n_call)
        n_call += 1
    copy_out.wait_stream(stream)
    e1.record(copy_out)
    torch.cuda.synchronize()
    Y_h = bufs[0][2]
    clocks.stop()
    ms_e2e = max_over_ranks(world, e0.elapsed_time(e1))
    if rank != 0:
        return 0
    peaks, src = load_peaks()
    step = ms / 1000.0 / args.steps
    gbs = B / step / 1e9
    rows_all = d["sum_m"] * world * args.steps
    line = {
        "metric": METRIC, "value": rows_all / (ms / 1000.0), "unit": "rows/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded)",
        "config": {"workload": "grouped_gemm", "sum_m": d["sum_m"], "E": d["E"], "K": d["K"], "N": d["N"],
                   "empty_groups": int((sizes == 0).sum()), "l2": "inputs larger than L2 (W is 805 MB)",
                   "parallelism": "single GPU" if world == 1 else f"replicas x{world}"},
        "tflops": F / step / 1e12,
        "roofline": {"kernel": "grouped_gemm_fwd", "bound": "hbm", "achieved": gbs,
                     "peak": float(peaks["hbm_gbs"]), "unit": "GB/s", "frac": gbs / float(peaks["hbm_gbs"]),
                     "traffic": None, "bytes_per_launch": B, "flops_per_launch": F,
                     "peak_kind": f"{src} HBM copy bandwidth"},
        "roofline_step": {"time_ms": max(F / (float(peaks["bf16_tflops"]) * 1e12),
                                         B / (float(peaks["hbm_gbs"]) * 1e9)) * 1000.0},
        "e2e": {"value": rows_all / (ms_e2e / 1000.0), "unit": "rows/s",
                "h2d_bytes_per_step": X_h.numel() * 2, "d2h_bytes_per_step": Y_h.numel() * 2},
        "gpu_launches": args.steps * kernels_per_call, "clocks": clocks.summary(t0, t1),
    }
    line["roofline_step"]["frac"] = line["roofline_step"]["time_ms"] / (ms / args.steps)
    print(json.dumps(line), flush=True)
    return 0


def run_grouped_gemm_bwd(args, world, rank, local):
    """One step = the backward of the ragged grouped GEMM on the grouped-GEMM
    workload (sum_m=16384 rows over 64 Dirichlet(0.3)-sized groups, K=4096,
    N=1536): dX = G W[g] (dgrad, bf16) and dW[g] = G^T X (wgrad, fp32), each
    timed alone as back-to-back CUDA-graph replays, inputs resident in HBM."""
    import mixture_experts_expert_router_gb300 as moe
    from mixture_experts_expert_router_gb300 import workloads as W
    moe.library()
    dev = torch.device("cuda", local)
    d = W.make_grouped_gemm(seed=args.seed + rank, device="cpu", weights_device=dev, with_grad=True)
    X, G, Wt, offs = d["X"].to(dev), d["G"].to(dev), d["W"], d["offs"].to(dev)
    sum_m, E, K, N = d["sum_m"], d["E"], d["K"], d["N"]
    dX = torch.empty((sum_m, K), dtype=torch.bfloat16, device=dev)
    dW = torch.empty((E, N, K), dtype=torch.float32, device=dev)
    active = int((d["sizes"] > 0).sum())
    F = 2.0 * sum_m * K * N
    B_dgrad = active * N * K * 2.0 + sum_m * N * 2.0 + sum_m * K * 2.0       # W (non-empty), G, dX
    B_wgrad = sum_m * N * 2.0 + sum_m * K * 2.0 + E * N * K * 4.0            # G, X, every dW[e] (fp32)
    stream = torch.cuda.current_stream(dev)
    calls = {"dgrad": lambda: moe.grouped_gemm_dgrad(G, Wt, offs, dX),
             "wgrad": lambda: moe.grouped_gemm_wgrad(G, X, offs, out_dtype=torch.float32, dW=dW)}
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        for _ in range(3):
            for fn in calls.values():
                fn()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    graphs = {}
    for name, fn in calls.items():
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        graphs[name] = g
    clocks = ClockSampler(str(local))
    time.sleep(0.3)
    for _ in range(args.warmup):
        for g in graphs.values():
            g.replay()
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.time()
    ms = {}
    for name, g in graphs.items():
        ms[name] = max_over_ranks(world, timed_steps(g.replay, args.steps, stream)) / args.steps
    t1 = time.time()
    # end to end: G and X in from pinned host memory, dX and dW back, every step
    G_h, X_h = d["G"].pin_memory(), d["X"].pin_memory()
    dX_h = torch.empty(dX.shape, dtype=dX.dtype).pin_memory()
    dW_h = torch.empty(dW.shape, dtype=dW.dtype).pin_memory()

    def e2e():
        G.copy_(G_h, non_blocking=True)
        X.copy_(X_h, non_blocking=True)
        calls["dgrad"]()
        calls["wgrad"]()
        dX_h.copy_(dX, non_blocking=True)
        dW_h.copy_(dW, non_blocking=True)
    for _ in range(args.warmup):
        e2e()
    torch.cuda.synchronize()
    n_e2e = min(args.steps, 50)
    ms_e2e = max_over_ranks(world, timed_steps(e2e, n_e2e, stream)) / n_e2e
    clocks.stop()
    if rank != 0:
        return 0
    peaks, src = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    step_ms = ms["dgrad"] + ms["wgrad"]
    rows_all = sum_m * world

    def roof(name, B):
        gbs = B / (ms[name] / 1000.0) / 1e9
        return {"kernel": f"grouped_gemm_{name}", "bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                "frac": gbs / hbm, "traffic": None, "bytes_per_launch": B, "flops_per_launch": F,
                "tflops": F / (ms[name] / 1000.0) / 1e12, "ms": ms[name], "peak_kind": f"{src} HBM copy bandwidth"}
    r_d, r_w = roof("dgrad", B_dgrad), roof("wgrad", B_wgrad)
    line = {
        "metric": METRIC, "value": rows_all / (step_ms / 1000.0), "unit": "rows/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded)",
        "config": {"workload": "grouped_gemm_bwd", "sum_m": sum_m, "E": E, "K": K, "N": N,
                   "empty_groups": int((d["sizes"] == 0).sum()), "dW": "fp32",
                   "l2": "inputs larger than L2 (W is 805 MB, dW 1.6 GB)",
                   "parallelism": "single GPU" if world == 1 else f"replicas x{world}"},
        "roofline": r_w if r_w["ms"] >= r_d["ms"] else r_d,
        "kernels": {"dgrad": r_d, "wgrad": r_w},
        "timing": "each kernel as back-to-back CUDA-graph replays; step = dgrad + wgrad",
        "e2e": {"value": rows_all / (ms_e2e / 1000.0), "unit": "rows/s",
                "h2d_bytes_per_step": (G_h.numel() + X_h.numel()) * 2,
                "d2h_bytes_per_step": dX_h.numel() * 2 + dW_h.numel() * 4},
        "gpu_launches": 2 * args.steps, "clocks": clocks.summary(t0, t1),
    }
    print(json.dumps(line), flush=True)
    return 0


BGMV_WORKLOAD = dict(T=2048, H=3072, R=32, E=64, num_loras=4, top_k=2)


def run_bgmv(args, world, rank, local):
    """One step = one BGMV LoRA-MoE shrink + expand (moe_bgmv) over T=2048
    tokens, hidden 3072 (feat_out = hidden), rank 32, 64 experts, 4 LoRAs,
    contiguous top-2 pairs; inputs resident in HBM, steps rotating over
    copies of the LoRA banks whose used weights together exceed L2."""
    import mixture_experts_expert_router_gb300 as moe
    from mixture_experts_expert_router_gb300 import workloads as W
    moe.library()
    dev = torch.device("cuda", local)
    c = BGMV_WORKLOAD
    wl = W.make_bgmv(T=c["T"], H=c["H"], R=c["R"], E=c["E"], num_loras=c["num_loras"], top_k=c["top_k"],
                     seed=args.seed + rank, device="cpu", weights_device=dev)
    x, tok, eid, lora, w = (t.to(dev) for t in (wl.x, wl.tok, wl.eid, wl.lora, wl.w))
    T, H, R, P = wl.T, wl.H, wl.R, wl.tok.numel()
    used = len(set(zip(wl.lora.numpy()[wl.tok.numpy()].tolist(), wl.eid.numpy().tolist())))
    w_bytes = used * (R * H + H * R) * 2.0            # A and B of every (LoRA, expert) pair used
    B = w_bytes + T * H * 2.0 + T * H * 4.0 + P * (4 + 4 + 4) + T * 4 + 2 * P * R * 2.0
    banks = 1 if 3 * w_bytes >= 3 * L2_NOMINAL else min(MAX_BANKS, int(np.ceil(3 * L2_NOMINAL / w_bytes)))
    A = [wl.lora_a[0]] + [wl.lora_a[0].clone() for _ in range(banks - 1)]
    Bw = [wl.lora_b[0]] + [wl.lora_b[0].clone() for _ in range(banks - 1)]
    y = torch.empty((T, H), dtype=torch.float32, device=dev)
    sh = torch.empty((1, P, R), dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    calls = [(lambda i=i: moe.bgmv(x, [A[i]], [Bw[i]], tok, eid, lora, w, contiguous_top_k=wl.top_k,
                                   shrink_out=sh, y_accum=y, status=status)) for i in range(banks)]
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        for fn in calls:
            fn()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    graphs = []
    for fn in calls:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        graphs.append(g)
    k = [0]

    def step():
        graphs[k[0] % banks].replay()
        k[0] += 1
    clocks = ClockSampler(str(local))
    time.sleep(0.3)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.time()
    ms = max_over_ranks(world, timed_steps(step, args.steps, stream))
    t1 = time.time()
    x_h = wl.x.pin_memory()
    y_h = torch.empty(y.shape, dtype=y.dtype).pin_memory()

    def e2e():
        x.copy_(x_h, non_blocking=True)
        step()
        y_h.copy_(y, non_blocking=True)
    for _ in range(args.warmup):
        e2e()
    torch.cuda.synchronize()
    ms_e2e = max_over_ranks(world, timed_steps(e2e, args.steps, stream))
    clocks.stop()
    if rank != 0:
        return 0
    peaks, src = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    step_s = ms / 1000.0 / args.steps
    gbs = B / step_s / 1e9
    line = {
        "metric": METRIC, "value": T * world / step_s, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded)",
        "config": {"workload": "bgmv", **c, "feat_out": H, "slices": 1, "pairs": "contiguous top-k",
                   "lora_pairs_used": used,
                   "l2": f"steps rotate over {banks} copies of the LoRA banks" if banks > 1 else "weights exceed L2",
                   "parallelism": "single GPU" if world == 1 else f"replicas x{world}"},
        "roofline": {"kernel": "moe_bgmv (shrink + expand)", "bound": "hbm", "achieved": gbs, "peak": hbm,
                     "unit": "GB/s", "frac": gbs / hbm, "traffic": None, "bytes_per_launch": B,
                     "peak_kind": f"{src} HBM copy bandwidth"},
        "e2e": {"value": T * world / (ms_e2e / 1000.0 / args.steps), "unit": "tokens/s",
                "h2d_bytes_per_step": x_h.numel() * 2, "d2h_bytes_per_step": y_h.numel() * 4},
        "gpu_launches": 2 * args.steps, "clocks": clocks.summary(t0, t1), "device_status": int(status.item()),
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="prefill_many_fine")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--shape", default=None,
                    help="T,H,I,E,top_k of a custom logits-routed workload (profiling runs)")
    ap.add_argument("--zipf", type=float, default=None,
                    help="with --shape: per-expert logit bias ln p_e, p_e ~ rank^-s (imbalanced groups)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e4m3", action="store_true", help="the fp8 per-tensor weight family (E4M3 weights)")
    ap.add_argument("--no-tail-tiles", action="store_true",
                    help="CTA-pair GEMMs: remainders as main tiles instead of swap-AB tail tiles")
    ap.add_argument("--no-graph", action="store_true", help="launch the plan directly instead of a CUDA graph")
    ap.add_argument("--decode-chain", action="store_true", help="decode path: always the two-kernel chain")
    ap.add_argument("--decode-one-launch", action="store_true",
                    help="decode path: the two-kernel chain as one kernel")
    ap.add_argument("--decode-separate", action="store_true",
                    help="decode path: always the five separate kernels (comparison)")
    ap.add_argument("--one-cta-gemm", action="store_true", help="grouped path: one-CTA GEMMs (comparison)")
    ap.add_argument("--small-group-kernel", default="auto", choices=["auto", "on", "off"],
                    help="grouped path: groups of at most 64 rows in their own kernel beside the CTA-pair GEMMs")
    ap.add_argument("--fused-gather", action="store_true",
                    help="grouped path: FC1 copies its token rows from x (no gather kernel)")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--reference-budget", type=float, default=120.0,
                    help="seconds of oracle work for the whole --impl reference run")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world, rank, local = dist_setup()
    try:
        if args.impl == "reference":
            return run_reference(args, world, rank)
        if args.config == "grouped_gemm":
            return run_grouped_gemm(args, world, rank, local)
        if args.config == "grouped_gemm_bwd":
            return run_grouped_gemm_bwd(args, world, rank, local)
        if args.config == "bgmv":
            return run_bgmv(args, world, rank, local)
        return run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
