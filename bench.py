"""Benchmark of the sparse-MoE layer forward pass on one B300 (or N replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload mixtral]
                    [--configs all|none|name,name...] [--only-route]
    python bench.py --impl reference ...     # the CPU oracle, timed on host cores

One step = one moe_layer_fwd (router -> capacity/dispatch -> grouped expert
GEMMs -> combine -> statistics; plus the loss-free bias update where the
workload has one) over one batch of T synthetic tokens. Prints one JSON line.

The headline workload (default: the Mixtral-shaped layer, the largest by
FLOPs and tokens) is timed for exactly K steps; every other workload named by
--configs (default: all of them) is then measured the same way, with its own
step count, and reported under the line's "configs" key.

value      tokens/s over all ranks, inputs already resident in HBM
e2e        the same call with the step's inputs (x, and the router noise where
           the workload passes it in) copied from pinned host memory and the
           result (y, aux) copied back inside the timed region; two buffer sets
           let the copies of neighbouring steps overlap the compute; at least
           200 steps and one second of wall time
roofline   the grouped expert GEMM (the dominant kernel): algorithmic bytes
           (weights of touched experts + activations in/out) per launch over its
           CUDA-event duration, against the measured HBM copy bandwidth; or, when
           its FLOPs at the measured bf16 rate take longer than its bytes at the
           HBM rate (the Mixtral- and DeepSeek-shaped layers), its TFLOP/s
           against that bf16 rate
hbm_stages the router, dispatch, combine and statistics entry points alone:
           their algorithmic bytes over their time, against the HBM peak
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
METRIC = "MoE-layer fwd tokens/s on 1 B300; grouped-GEMM TFLOP/s & HBM GB/s vs peak"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="mixtral")
    ap.add_argument("--configs", default="all",
                    help="other workloads measured after the headline: all, none, or a "
                         "comma-separated list")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only-route", action="store_true",
                    help="time moe_route alone on the headline workload (no expert weights)")
    ap.add_argument("--override", default="",
                    help="comma-separated field=value changes to the headline workload "
                         "(e.g. d_ff=64 keeps the router, dispatch and combine shapes of a "
                         "layer with small expert weights, for profiling)")
    a = ap.parse_args()
    a.warmup = max(a.warmup, 3)
    a.steps = max(a.steps, 1)
    return a


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value: float, pg, device) -> float:
    """The largest value over all ranks: a job's time is its slowest rank's."""
    if pg is None:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def tokens_per_s(world: int, T: int, steps: int, ms_total: float) -> float:
    """Whole-job throughput: every rank processes T tokens per step."""
    return world * T * steps / (ms_total / 1e3)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


def ffn_kernels(wl, R_max):
    """(launches, kernel names) of one expert-FFN call, chosen as the library
    chooses them from the layer's shape (R_max = the expert-sorted rows' bound,
    moe_capacity): bf16 experts of at least 1024 rows on average run on CTA
    pairs; 256 or more (T > 128) as two launches per projection; the rest as
    one single-CTA launch per projection."""
    c = wl.cfg
    T, E, k = c.T, c.n_experts, c.top_k
    if c.dtype != 1:
        return 2, "grouped_gemm_simt_kernel (expert FFN: up + down launches)"
    if R_max >= 1024 * E:
        return 2, "grouped_gemm_pair_kernel (CTA pairs; expert FFN: up + down launches)"
    if T > 128 and T * k >= 256 * E:
        return 4, ("grouped_gemm_tc_kernel + grouped_gemm_pair_kernel (few-row experts on "
                   "single CTAs, then many-row and shared experts on CTA pairs; expert FFN: "
                   "2 launches per projection)")
    return 2, "grouped_gemm_tc_kernel (expert FFN: up + down launches)"


def roofline_record(flops, ffn_bytes, ffn_ms, pk, pk_kind, traffic, launches=2,
                    kernel="grouped_gemm_tc_kernel (expert FFN: up + down launches)"):
    """The JSON roofline object of the expert FFN (`launches` grouped-GEMM
    launches of flops and ffn_bytes in total, ffn_ms per call). The bound is
    the larger of the two floors: the algorithmic bytes at the measured HBM
    rate, or the FLOPs at the measured bf16 rate. An FFN of a millisecond or
    more per call, timed back to back, runs under the power cap, so its bf16
    rate is the sustained one, else the burst one."""
    hbm = pk["hbm_gbs"]
    achieved_gbs = ffn_bytes / (ffn_ms / 1e3) / 1e9
    tflops = flops / (ffn_ms / 1e3) / 1e12
    sustained = ffn_ms >= 1.0
    peak_t = pk["bf16_tflops_sustained"] if sustained else pk["bf16_tflops"]
    if ffn_bytes / (hbm * 1e9) >= flops / (peak_t * 1e12):
        return {"bound": "hbm", "achieved": achieved_gbs, "peak": hbm, "unit": "GB/s",
                "frac": achieved_gbs / hbm, "traffic": traffic, "kernel": kernel,
                "algorithmic_bytes_per_launch": ffn_bytes / launches, "peak_kind": pk_kind,
                "tflops": tflops, "tflops_frac_of_bf16_peak": tflops / pk["bf16_tflops"]}
    return {"bound": "tensor", "achieved": tflops, "peak": peak_t, "unit": "TFLOP/s",
            "frac": tflops / peak_t, "traffic": traffic, "kernel": kernel,
            "algorithmic_flops_per_launch": flops / launches,
            "peak_kind": pk_kind + (" sustained" if sustained else " burst"),
            "hbm_gbs": achieved_gbs, "hbm_frac": achieved_gbs / hbm}


def workload_desc(wl):
    c = wl.cfg
    act = {0: "ReLU", 1: "GELU", 2: "SwiGLU"}[c.act]
    s = (f"{wl.name}: T={c.T} d={c.d_model} E={c.n_experts} k={c.top_k} F={c.d_ff} {act}"
         f" shared={c.n_shared} cf={c.capacity_factor:g}")
    if wl.noisy:
        s += " noisy-KeepTopK" + (" (noise drawn on the device)" if c.noise_draw else "")
    if wl.zipf_s:
        s += f" zipf-offset={wl.zipf_s}"
    if wl.sel_bias:
        s += f" sel-bias+update(rate={wl.bias_rate:g})"
    if c.reroute:
        s += f" reroute={c.reroute} priority={'rank' if c.priority else 'token'}"
    elif c.priority:
        s += " priority=rank"
    if c.pad_to_capacity:
        s += " padded-to-capacity"
    if c.routing == 1:
        s += " expert-choice"
    return s


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            out, _ = self.proc.communicate(timeout=10)
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def source_hash():
    """Hash of the grouped-GEMM kernel code (comments and blank lines left
    out), which names the kernel version an ncu traffic figure was taken on."""
    h = hashlib.sha256()
    for f in ("gemm_tc.cu", "group_table.cuh"):
        text = open(os.path.join(ROOT, "sparse_mixture_experts_69_b300", "csrc", f)).read()
        for line in text.splitlines():
            code = line.split("//", 1)[0].rstrip()
            if code:
                h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def ncu_traffic(workload):
    """dram bytes per grouped-GEMM launch from the committed ncu summary, if it
    was taken on the current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    rec = d.get(workload)
    if not rec or rec.get("source_hash") != source_hash():
        return None
    return rec.get("dram_bytes_per_launch")


# ----------------------------------------------------------------- CPU oracle leg

class OracleInputs:
    """Host-side inputs for the oracle: the small tensors whole, expert weights
    fetched per expert on first use (copied from the device, or generated on
    the host with the same seeded generator) and cached as float32."""

    def __init__(self, wl, inp=None):
        import numpy as np

        from sparse_mixture_experts_69_b300 import synth
        from sparse_mixture_experts_69_b300.workloads import W_STD, make_inputs

        self.wl, self._np, self._synth, self._std = wl, np, synth, W_STD
        c = wl.cfg
        if inp is None:  # host only: generate all but the expert weights
            small = make_inputs(wl.with_(n_experts=c.n_experts), "cpu", experts=False)
            self.inp, self.dev = small, None
        else:
            self.inp, self.dev = inp, inp["x"].device
        self.small = {k: (None if v is None or k in ("W1", "W2", "W1s", "W2s") else v.cpu())
                      for k, v in self.inp.items()}
        if wl.noisy and self.small["noise"] is None:  # the library draws it: the oracle's draws
            import oracle
            eps = oracle.draw_noise(c.T, c.n_experts, c.noise_seed, c.noise_counter)
            self.small["noise"] = torch.from_numpy(eps.astype(np.float32))
        self.cache = {}

    def _get(self, key, tid, e, shape):
        if (key, e) in self.cache:
            return self.cache[(key, e)]
        if self.dev is not None:
            t = self.inp[key][e].float().cpu()
        else:
            import math
            t = self._synth.normal(shape, self.wl.seed, tid, self._std, self.wl.cfg.torch_dtype,
                                   "cpu", offset=e * math.prod(shape)).float()
        a = self._np.ascontiguousarray(t.numpy(), dtype=self._np.float32)
        self.cache[(key, e)] = a
        return a

    def W1(self, e):
        c = self.wl.cfg
        return self._get("W1", 10, e, (c.F1, c.d_model))

    def W2(self, e):
        c = self.wl.cfg
        return self._get("W2", 11, e, (c.d_model, c.d_ff))

    def W1s(self, s):
        c = self.wl.cfg
        return self._get("W1s", 12, s, (c.F1, c.d_model))

    def W2s(self, s):
        c = self.wl.cfg
        return self._get("W2s", 13, s, (c.d_model, c.d_ff))


def oracle_tokens_per_s(oi, n_tok, seed=5):
    """Time the oracle (as it stands) on n_tok sampled tokens of the workload:
    router, then every expert FFN those tokens chose, then combine. Expert
    weights are fetched before the clock starts."""
    import numpy as np

    import oracle
    from sparse_mixture_experts_69_b300 import synth

    wl = oi.wl
    c = wl.cfg
    tok = sorted(set(synth.randint((n_tok,), seed, 400, c.T).tolist()))
    tt = torch.as_tensor(tok)
    g = lambda n: oi.small[n]
    rows = lambda n: None if oi.small[n] is None else oi.small[n][tt]
    rd = oracle.ROUND_BF16 if c.dtype == 1 else oracle.ROUND_F32
    slot = np.zeros((len(tok), c.top_k), np.int32)
    # routing decides which experts are needed: fetch them untimed, then time it all
    r0 = oracle.router(rows("x"), g("Wg"), c.top_k, Wnoise=g("Wnoise"), noise=rows("noise"),
                       offset=g("logit_offset"), bias=g("sel_bias"), renorm=bool(c.renorm_topk))
    for e in sorted(set(r0["ids"].ravel().tolist())):
        oi.W1(e), oi.W2(e)
    for s in range(c.n_shared):
        oi.W1s(s), oi.W2s(s)
    x_rows = rows("x")
    t0 = time.perf_counter()
    r = oracle.router(x_rows, g("Wg"), c.top_k, Wnoise=g("Wnoise"), noise=rows("noise"),
                      offset=g("logit_offset"), bias=g("sel_bias"), renorm=bool(c.renorm_topk))
    O, Os = oracle.ffn_for_tokens(x_rows, list(range(len(tok))), r["ids"], slot, oi.W1, oi.W2,
                                  c.act, rd, c.n_shared, oi.W1s, oi.W2s)
    oracle.combine(r["w"], slot, O, Os, rd)
    dt = time.perf_counter() - t0
    return len(tok), dt


def cpu_baseline(wl, inp, budget_s=12.0):
    import oracle
    oracle.build()
    oi = OracleInputs(wl, inp)
    # grow the sample until it takes about budget_s (the per-token cost falls
    # as the rows fill the OpenMP threads, so one calibration is not enough)
    n2, dt2 = oracle_tokens_per_s(oi, 16)
    for it in range(8):
        if dt2 >= 0.7 * budget_s or n2 >= wl.cfg.T:
            break
        want = int(max(16, min(wl.cfg.T, n2 * budget_s / max(dt2, 1e-6))))
        n2, dt2 = oracle_tokens_per_s(oi, want, seed=6 + it)
    cores = len(os.sched_getaffinity(0))
    return {"value": n2 / dt2, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{n2} sampled tokens of the {wl.name} workload (router + chosen expert "
                      f"FFNs + combine, plain double loops, OpenMP over rows); {dt2:.1f} s"}


def run_reference(a):
    """--impl reference: the CPU oracle, timed on the host cores, same workload.
    The synthetic inputs are made on the GPU when one is present (the
    generator is the same on both devices; generating the Mixtral-shaped
    layer's 2.8 GB of expert weights on the host would take minutes), then
    copied to the host; the oracle itself runs on the host only."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from sparse_mixture_experts_69_b300.workloads import WORKLOADS, make_inputs
    import oracle
    oracle.build()
    wl = WORKLOADS[a.workload]
    inp = make_inputs(wl, "cuda") if torch.cuda.is_available() else None
    oi = OracleInputs(wl, inp)
    # per-step sample sized so warm-up + steps take about two minutes of compute
    n, dt = oracle_tokens_per_s(oi, 4)
    per_tok = dt / max(n, 1)
    n_step = int(max(1, min(256, 120.0 / (a.steps + a.warmup) / max(per_tok, 1e-6))))
    for i in range(a.warmup):
        oracle_tokens_per_s(oi, n_step, seed=10 + i)
    done, total = 0, 0.0
    for i in range(a.steps):
        m, dt = oracle_tokens_per_s(oi, n_step, seed=1000 + i)
        done += m
        total += dt
    value = done / total
    cores = len(os.sched_getaffinity(0))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": a.gpus, "steps": a.steps, "warmup": a.warmup,
            "ms_per_step": 1e3 * total / a.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_desc(wl), "global_batch": wl.cfg.T,
                       "parallelism": "host cores"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores,
                             "kind": "oracle",
                             "sample": f"{n_step} sampled tokens per step of the {wl.name} "
                                       "workload (router + chosen expert FFNs + combine)"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- our arm

ALL_CONFIGS = ["tiny", "switch", "mixtral", "deepseek", "decode"]


def router_selects_in_gemm(c, noisy):
    """The library's rule for selecting in the router GEMM's epilogue (no
    selection launch): bf16, no noise, at most 32 experts and 8 candidates,
    and a router plan of one K part (the library's router_plan for 32-wide
    column tiles: 128-row tiles, or one tile of ceil(T / 148) >= 64 rows per
    SM when 128-row tiles would leave SMs idle and no split applies; then
    the K range splits while 2x the tiles fit 148 SMs and each part keeps 4
    blocks of 64)."""
    if c.dtype != 1 or noisy or c.n_experts > 32 or c.n_cand > 8:
        return False
    T, nkb = c.T, (c.d_model + 63) // 64
    tm = 128
    t128 = (T + 127) // 128
    if t128 < 148 and not (t128 * 2 <= 148 and nkb // 2 >= 4):
        want = (T + 147) // 148
        if 64 <= want < 128:
            tm = want
    tiles = (T + tm - 1) // tm
    return not (tiles * 2 <= 148 and nkb // 2 >= 4)


def launches_per_step(wl):
    """Kernels of this library one step launches. Layer path: [Wg transpose
    (bf16)], router GEMM, fused selection + histogram + statistics (none when
    the router GEMM selects itself), capacity
    scan + slots (one launch up to 256 token blocks), permute, up GEMM, down
    GEMM (each two launches for layers of mixed expert sizes), [combine: skipped where the down GEMM writes y itself, by its
    folded combine (bf16, packed rows, combine_mode = 1) or, for top-1
    without shared experts, by scattering gate * output], [bias update]. Overflow policies:
    one capacity kernel instead of scan + slots; expert choice: select +
    gather instead of capacity + permute, its own combine."""
    c = wl.cfg
    T, k, nc = c.T, c.top_k, c.n_cand
    ec = c.routing == 1
    scatter = c.top_k == 1 and nc == 1 and c.n_shared == 0
    combine_in_gemm = c.dtype == 1 and not c.pad_to_capacity and (
        scatter or c.combine_mode == 1)
    policy = nc > k or c.priority != 0
    route_launches = (1 if c.dtype == 1 else 0) + (1 if router_selects_in_gemm(c, wl.noisy) else 2)
    if ec:
        return route_launches + 2 + 2 + 1
    cap_launches = 1 if policy else (1 if (T + 255) // 256 <= 256 else 2)
    # expert projections: one launch each, or two for layers of mixed expert
    # sizes (ffn_kernels)
    from sparse_mixture_experts_69_b300 import moe
    gemm_launches = ffn_kernels(wl, moe.moe_capacity(c)[1])[0]
    return (route_launches + cap_launches + 1 + gemm_launches + (0 if combine_in_gemm else 1)
            + (1 if wl.bias_rate else 0))


def time_graph(fn, n, stream, dev):
    """Device time of one call of fn: n calls captured in one CUDA graph and
    replayed between CUDA events (a single small call is host-bound)."""
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        with torch.cuda.graph(g, stream=cap, capture_error_mode="relaxed"):
            for _ in range(n):
                fn()
    torch.cuda.synchronize()
    g.replay()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / n


def hbm_record(nbytes, ms, hbm):
    gbs = nbytes / (ms / 1e3) / 1e9
    return {"bytes": nbytes, "ms": ms, "gbs": gbs, "frac": gbs / hbm}


def measure(wl, steps, warmup, dev, pg, world, local, cpu_budget, want_cpu, auto_steps=False):
    """Time one workload: the layer with inputs resident (steps x
    moe_layer_fwd), each entry point alone, and end to end with host buffers.
    Returns the workload's record (the JSON line's fields)."""
    from sparse_mixture_experts_69_b300 import moe
    from sparse_mixture_experts_69_b300.workloads import make_inputs

    c = wl.cfg
    T, E, k, d, nc = c.T, c.n_experts, c.top_k, c.d_model, c.n_cand
    ec = c.routing == moe.MOE_EXPERT_CHOICE
    inp = make_inputs(wl, dev)
    ws = moe.workspace(c, dev)
    y = torch.empty((T, d), dtype=c.torch_dtype, device=dev)
    ids = torch.empty((T, nc), dtype=torch.int32, device=dev)
    w = torch.empty((T, nc), dtype=torch.float32, device=dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    aux_vecs = torch.empty((3, E), dtype=torch.float32, device=dev)
    out3 = torch.empty(3, dtype=torch.float32, device=dev)
    bias = inp["sel_bias"].clone() if inp["sel_bias"] is not None else None
    stream = torch.cuda.current_stream(dev)
    # expert choice: the token-choice outputs (ids, gates, counts, statistics) do not apply
    tc_out = (None,) * 5 if ec else (ids, w, counts, aux_vecs, out3)

    def step(x, noise):
        moe.moe_layer_fwd(c, x, inp["Wg"], inp["Wnoise"], noise, inp["logit_offset"], bias,
                          inp["W1"], inp["W2"], inp["W1s"], inp["W2s"], y, *tc_out, ws, stream)
        if wl.bias_rate:
            moe.moe_bias_update(c, counts, bias, wl.bias_rate, stream)

    def barrier():
        if pg:
            pg.barrier()

    def reset_bias():
        # every timed phase starts from the workload's initial selection bias:
        # the bias update moves the routing a little each step
        if bias is not None:
            bias.copy_(inp["sel_bias"])

    # ------------------------------------------------ device-resident timing
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(warmup):
        step(inp["x"], inp["noise"])
    ev1.record(stream)
    st = moe.moe_read_device_error(c, ws)
    if st != 0:
        raise RuntimeError(f"{wl.name}: device status after warm-up: " + moe.moe_status_string(st))
    if auto_steps:  # about half a second of timed work
        est = ev0.elapsed_time(ev1) / warmup
        steps = int(min(4000, max(20, 500.0 / max(est, 1e-3))))
    reset_bias()
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        ev0.record(stream)
        for _ in range(steps):
            step(inp["x"], inp["noise"])
        ev1.record(stream)
        torch.cuda.synchronize()
    barrier()
    ms = ev0.elapsed_time(ev1)
    ms_max = max_over_ranks(ms, pg, dev)
    st = moe.moe_read_device_error(c, ws)
    if st != 0:
        raise RuntimeError(f"{wl.name}: device status after timing: " + moe.moe_status_string(st))
    value = tokens_per_s(world, T, steps, ms_max)

    # ------------------------------------------------ each entry point alone
    C, R_max = moe.moe_capacity(c)
    logits = torch.empty((T, E), device=dev)
    probs = torch.empty((T, E), device=dev)
    kept = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    slot = torch.empty((T, nc), dtype=torch.int32, device=dev)
    row_token = torch.empty(R_max, dtype=torch.int32, device=dev)
    xp = torch.empty((R_max, d), dtype=c.torch_dtype, device=dev)
    yp = torch.empty((R_max, d), dtype=c.torch_dtype, device=dev)
    ys = torch.empty((c.n_shared, T, d), dtype=c.torch_dtype, device=dev) if c.n_shared else None
    fP = torch.empty((3, E), device=dev)
    row_w = torch.empty(R_max, device=dev)
    tok_row = torch.empty((T, E), dtype=torch.int32, device=dev) if ec else None
    n_seq = 8
    seq_offsets = torch.arange(0, T + 1, max(1, T // n_seq), dtype=torch.int32,
                               device=dev)[:n_seq + 1].clone()
    n_seq = seq_offsets.numel() - 1
    seq_offsets[-1] = T
    seq_out = torch.empty((2, n_seq, E), device=dev)
    seq_aux = torch.empty(n_seq + 1, device=dev)
    n_split = 20
    # the stage calls take torch's current stream, which is the capture stream in time_graph
    route = lambda: moe.moe_route(
        c, inp["x"], inp["Wg"], inp["Wnoise"], inp["noise"], inp["logit_offset"], bias, logits,
        probs, None, None if ec else ids, None if ec else w, 0, ws)
    ffn = lambda: moe.moe_expert_ffn(c, xp, offsets, inp["W1"], inp["W2"], inp["x"], inp["W1s"],
                                     inp["W2s"], yp, ys, ws)
    tg = lambda fn: time_graph(fn, n_split, stream, dev)
    if ec:
        stage_ms = {
            "route": tg(route),
            "dispatch": tg(lambda: moe.moe_expert_choice_dispatch(
                c, inp["x"], probs, offsets, row_token, row_w, tok_row, xp, ws)),
            "expert_ffn": tg(ffn),
            "combine": tg(lambda: moe.moe_expert_choice_combine(
                c, yp, tok_row, probs, ys, y, ws)),
        }
    else:
        stage_ms = {
            "route": tg(route),
            "dispatch": tg(lambda: moe.moe_dispatch(
                c, inp["x"], ids, counts, kept, offsets, slot, xp, row_token, ws)),
            "expert_ffn": tg(ffn),
            "combine": tg(lambda: moe.moe_combine(c, yp, slot, w, ys, y, ws)),
            "aux": tg(lambda: moe.moe_aux_stats(c, probs, ids, w, fP[0], fP[1], fP[2], out3,
                                                ws)),
            f"seq_aux_{n_seq}_sequences": tg(lambda: moe.moe_seq_aux_stats(
                c, probs, ids, seq_offsets, n_seq, seq_out[0], seq_out[1], seq_aux[:n_seq],
                seq_aux[n_seq:], ws)),
        }
    st = moe.moe_read_device_error(c, ws)
    if st != 0:
        raise RuntimeError(f"{wl.name}: device status after the stage timing: "
                           + moe.moe_status_string(st))

    # algorithmic work of the expert FFN (two grouped-GEMM launches): rows the
    # GEMMs run on (padding rows included where the blocks are padded), and the
    # weights of every expert that owns at least one row
    R = int(offsets[E].item())
    touched = E if (ec or c.pad_to_capacity) else int((kept.cpu() > 0).sum())
    es = 2 if c.dtype == 1 else 4
    F, F1, S = c.d_ff, c.F1, c.n_shared
    w_bytes = (touched + S) * (F1 * d + d * F) * es
    act_bytes = (R + S * T) * (d + F + F + d) * es  # up: read x rows, write h; down: read h, write y
    ffn_bytes = w_bytes + act_bytes
    flops = 2 * (R + S * T) * d * (F1 + F)
    ffn_ms = stage_ms["expert_ffn"]
    pk, pk_kind = peaks()
    n_launch, kname = ffn_kernels(wl, R_max)
    roofline = roofline_record(flops, ffn_bytes, ffn_ms, pk, pk_kind, ncu_traffic(wl.name),
                               n_launch, kname)
    # the memory-bound entry points: algorithmic bytes (inputs read once,
    # outputs written once) over their time
    noisy_b = (d * E * es + (T * E * 4 if inp["noise"] is not None else 0)) if wl.noisy else 0
    route_b = (T * d * es + d * E * es + noisy_b + 2 * T * E * 4
               + (0 if ec else T * nc * 8))
    hbm = pk["hbm_gbs"]
    hbm_stages = {"route": hbm_record(route_b, stage_ms["route"], hbm)}
    if not ec:
        hbm_stages["dispatch"] = hbm_record(T * d * es + 2 * T * nc * 4 + R * (d * es + 4),
                                            stage_ms["dispatch"], hbm)
        hbm_stages["combine"] = hbm_record(R * d * es + T * nc * 8 + S * T * d * es + T * d * es,
                                           stage_ms["combine"], hbm)
        hbm_stages["aux"] = hbm_record(T * E * 4 + T * k * 8, stage_ms["aux"], hbm)

    # ------------------------------------------------ end to end (host buffers)
    # Every step uploads its inputs (x, and the router noise where it is passed
    # in) from pinned host memory and downloads its result (y, and the aux
    # scalars) to pinned host memory. Two buffer sets and separate upload /
    # download streams let step i+1's upload and step i-1's download run under
    # step i's compute, as a caller streaming batches through the layer would.
    x_host = inp["x"].cpu().pin_memory()
    noise_host = inp["noise"].cpu().pin_memory() if inp["noise"] is not None else None
    nbuf = 2
    x_dev = [torch.empty_like(inp["x"]) for _ in range(nbuf)]
    noise_dev = [torch.empty_like(inp["noise"]) if noise_host is not None else None
                 for _ in range(nbuf)]
    y_dev = [torch.empty_like(y) for _ in range(nbuf)]
    o3_dev = [torch.empty(3, dtype=torch.float32, device=dev) for _ in range(nbuf)]
    y_host = [torch.empty_like(y, device="cpu").pin_memory() for _ in range(nbuf)]
    o3_host = [torch.empty(3, dtype=torch.float32).pin_memory() for _ in range(nbuf)]
    up_st, comp_st, down_st = (torch.cuda.Stream(dev) for _ in range(3))
    uploaded = [torch.cuda.Event() for _ in range(nbuf)]
    computed = [torch.cuda.Event() for _ in range(nbuf)]
    downloaded = [torch.cuda.Event() for _ in range(nbuf)]
    for e_ in computed + downloaded:
        e_.record(stream)  # every buffer starts free

    def e2e_step(i):
        bi = i % nbuf
        up_st.wait_event(computed[bi])  # step i-2 has finished reading x_dev[bi]
        with torch.cuda.stream(up_st):
            x_dev[bi].copy_(x_host, non_blocking=True)
            if noise_host is not None:
                noise_dev[bi].copy_(noise_host, non_blocking=True)
        uploaded[bi].record(up_st)
        comp_st.wait_event(uploaded[bi])
        comp_st.wait_event(downloaded[bi])  # step i-2's y and aux have been read back
        outs = (None,) * 5 if ec else (ids, w, counts, aux_vecs, o3_dev[bi])
        moe.moe_layer_fwd(c, x_dev[bi], inp["Wg"], inp["Wnoise"], noise_dev[bi],
                          inp["logit_offset"], bias, inp["W1"], inp["W2"], inp["W1s"],
                          inp["W2s"], y_dev[bi], *outs, ws, comp_st)
        if wl.bias_rate:
            moe.moe_bias_update(c, counts, bias, wl.bias_rate, comp_st)
        computed[bi].record(comp_st)
        down_st.wait_event(computed[bi])
        with torch.cuda.stream(down_st):
            y_host[bi].copy_(y_dev[bi], non_blocking=True)
            if not ec:
                o3_host[bi].copy_(o3_dev[bi], non_blocking=True)
        downloaded[bi].record(down_st)

    # an estimate first, then at least 200 steps and one second of wall time
    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(10):
        e2e_step(i)
    torch.cuda.synchronize()
    est = (time.perf_counter() - t0) / 10
    K2 = int(max(200, 1.2 / max(est, 1e-6)))
    reset_bias()
    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(K2):
        e2e_step(i)
    torch.cuda.synchronize()
    e2e_s = time.perf_counter() - t0
    barrier()
    e2e_s = max_over_ranks(e2e_s, pg, dev)
    h2d = x_host.numel() * x_host.element_size() + (
        noise_host.numel() * 4 if noise_host is not None else 0)
    d2h = y_host[0].numel() * y_host[0].element_size() + (0 if ec else 12)
    e2e_value = tokens_per_s(world, T, K2, e2e_s * 1e3)
    st = moe.moe_read_device_error(c, ws)
    if st != 0:
        raise RuntimeError(f"{wl.name}: device status after e2e: " + moe.moe_status_string(st))

    cb = None
    # the oracle's per-token sample has no expert-choice counterpart (an expert's
    # choice depends on the whole batch); that variant reports none
    if want_cpu and world == 1 and not ec:
        cb = cpu_baseline(wl, inp, cpu_budget)
    rec = {
        "workload": workload_desc(wl), "value": value, "unit": "tokens/s",
        "ms_per_step": ms_max / steps, "steps": steps,
        "dtype": "bf16" if c.dtype == 1 else "f32",
        "roofline": roofline, "hbm_stages": hbm_stages, "cpu_baseline": cb,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": K2, "wall_s": e2e_s,
                "copies": "pinned host buffers, double-buffered, upload / download streams "
                          "overlapping the compute stream"},
        "clocks": clk.summary(), "stage_ms": stage_ms, "rows_kept": R,
        "experts_touched": touched, "weights_gb": w_bytes / 1e9,
        "gpu_launches": launches_per_step(wl) * steps,
    }
    return rec


def headline_workload(a):
    """The --workload entry of WORKLOADS with the --override changes."""
    from sparse_mixture_experts_69_b300.workloads import WORKLOADS
    wl = WORKLOADS[a.workload]
    kw = {}
    for item in filter(None, a.override.split(",")):
        key, val = item.split("=", 1)
        kw[key.strip()] = float(val) if "." in val else int(val, 0)
    if kw:
        wl = wl.with_(name=wl.name + "[" + a.override + "]", **kw)
    return wl


def run_only_route(a, dev):
    """Time moe_route alone on the headline workload (router inputs only, no
    expert weights): its HBM rate against the measured peak."""
    from sparse_mixture_experts_69_b300 import moe
    from sparse_mixture_experts_69_b300.workloads import make_inputs
    wl = headline_workload(a)
    c = wl.cfg
    T, E, d, nc = c.T, c.n_experts, c.d_model, c.n_cand
    inp = make_inputs(wl, dev, experts=False)
    ws = moe.workspace(c, dev)
    logits = torch.empty((T, E), device=dev)
    probs = torch.empty((T, E), device=dev)
    ids = torch.empty((T, nc), dtype=torch.int32, device=dev)
    w = torch.empty((T, nc), device=dev)
    stream = torch.cuda.current_stream(dev)
    fn = lambda: moe.moe_route(c, inp["x"], inp["Wg"], inp["Wnoise"], inp["noise"],
                               inp["logit_offset"], inp["sel_bias"], logits, probs, None, ids,
                               w, 0, ws)
    for _ in range(a.warmup):
        fn()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    ev0.record(stream)
    for _ in range(a.steps):
        fn()
    ev1.record(stream)
    torch.cuda.synchronize()
    st = moe.moe_read_device_error(c, ws)
    if st != 0:
        raise RuntimeError("device status: " + moe.moe_status_string(st))
    ms = ev0.elapsed_time(ev1) / a.steps
    es = 2 if c.dtype == 1 else 4
    noisy_b = (d * E * es + (T * E * 4 if inp["noise"] is not None else 0)) if wl.noisy else 0
    nbytes = T * d * es + d * E * es + noisy_b + 2 * T * E * 4 + T * nc * 8
    pk, pk_kind = peaks()
    line = {"mode": "only-route", "workload": workload_desc(wl), "steps": a.steps,
            "route_ms": ms, "graph_route_ms": time_graph(fn, 20, stream, dev),
            "route": hbm_record(nbytes, ms, pk["hbm_gbs"]), "peak_kind": pk_kind,
            "router_gflop": 2.0 * T * d * (2 * E if wl.noisy else E) / 1e9}
    print(json.dumps(line), flush=True)
    return 0


def main():
    a = parse()
    if a.impl == "reference":
        return run_reference(a)
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if a.only_route:
        return run_only_route(a, dev)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    from sparse_mixture_experts_69_b300.workloads import WORKLOADS

    wl = headline_workload(a).with_(seed=rank)
    head = measure(wl, a.steps, a.warmup, dev, pg, world, local, 12.0,
                   not a.no_cpu_baseline and rank == 0)
    torch.cuda.empty_cache()
    # the other workloads, one after another (each one's tensors are freed
    # before the next is made); replicas under torchrun time the headline only
    others = {}
    names = ALL_CONFIGS if a.configs == "all" else (
        [] if a.configs == "none" else [n for n in a.configs.split(",") if n])
    if world == 1:
        for name in names:
            if name == a.workload:
                continue
            others[name] = measure(WORKLOADS[name], 0, max(3, min(a.warmup, 10)), dev, None, 1,
                                   local, 6.0, not a.no_cpu_baseline, auto_steps=True)
            torch.cuda.empty_cache()
    if rank != 0:
        if pg:
            pg.destroy_process_group()
        return 0
    c = wl.cfg
    line = {
        "metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": world,
        "steps": a.steps, "warmup": a.warmup, "ms_per_step": head["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": head["dtype"], "data": "synthetic",
        "config": {"workload": head["workload"], "global_batch": world * c.T,
                   "seq_len": None, "parallelism": "replicas" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2: each step streams "
                         f"{head['weights_gb']:.2f} GB of expert weights through the 126 MB L2"},
        "roofline": head["roofline"],
        "cpu_baseline": head["cpu_baseline"],
        "e2e": head["e2e"],
        "gpu_launches": head["gpu_launches"],
        "clocks": head["clocks"],
        "stage_ms": head["stage_ms"],
        "hbm_stages": head["hbm_stages"],
        "rows_kept": head["rows_kept"], "experts_touched": head["experts_touched"],
        "configs": others,
    }
    print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
